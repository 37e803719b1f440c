"""INT8 compressed checkpoints: the oracle's codec and record layout.

TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU legs of bench.py
use this module; the CUDA library never calls it and shares no code with it.

Source: "KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제" (KDA's AI-infrastructure challenges),
§0x05 5.3 and §0x06 6.6.  Checkpoints that wait in the cache may hold the recurrent state in
INT8 while the small conv window keeps its native precision; the quantisation is symmetric,
with one scale per key channel taken as the max-abs along the value channels; on a hit the
checkpoint is dequantised once into a fresh active (full-precision) slot and the recurrence
continues there, so quantisation error does not accumulate step after step.

Readings where the pages are silent (each listed in the design notes):
  - codes are int8 in [-127, 127] (symmetric, -128 unused); scale_i = max_j |S[i][j]| / 127;
  - every step in fp32 with IEEE rounding: the division x / scale_i, then round to nearest,
    ties to even; a row of zeros has scale 0 and codes 0; dequantisation is code * scale_i;
  - record layout (per head, in head order inside an object like the fp32 record):
        scale  fp32 [d]          (key channel i)
        codes  int8 [d][d]       (row i = key channel, column j = value channel)
        window [3][3d] in dtype  (unchanged)
    zero-padded to a multiple of 256 bytes (19,200 B at d = 128 bf16: 3.53x smaller).
"""
from __future__ import annotations

import numpy as np
import torch

from . import policy

QMAX = 127


def record_bytes(d: int, dtype: str) -> int:
    raw = 4 * d + d * d + 3 * 3 * d * policy.DTYPE_SIZE[dtype]
    return (raw + 255) // 256 * 256


def object_bytes(H: int, d: int, dtype: str) -> int:
    return H * record_bytes(d, dtype)


def object_pages(H: int, d: int, dtype: str, page_bytes: int) -> int:
    return -(-object_bytes(H, d, dtype) // page_bytes)


def quantize(S) -> tuple[np.ndarray, np.ndarray]:
    """Per-row symmetric INT8 of a [d][d] state (values taken as fp32)."""
    S = np.asarray(S, dtype=np.float32)
    amax = np.max(np.abs(S), axis=1).astype(np.float32)
    scale = (amax / np.float32(QMAX)).astype(np.float32)
    safe = np.where(scale > 0, scale, np.float32(1)).astype(np.float32)
    q = np.rint((S / safe[:, None]).astype(np.float32))
    q = np.clip(q, -QMAX, QMAX)
    q = np.where(scale[:, None] > 0, q, 0).astype(np.int8)
    return scale, q


def dequantize(scale, codes) -> np.ndarray:
    scale = np.asarray(scale, dtype=np.float32)
    return (np.asarray(codes, dtype=np.int8).astype(np.float32) * scale[:, None]).astype(np.float32)


def pack_record(S, win, dtype: str) -> bytes:
    d = np.asarray(S).shape[0]
    scale, q = quantize(S)
    body = scale.tobytes() + q.tobytes() + policy._window_bytes(np.asarray(win).reshape(3, 3 * d), dtype)
    return body + bytes(record_bytes(d, dtype) - len(body))


def unpack_record(buf: bytes, d: int, dtype: str):
    """-> (scale fp32 [d], codes int8 [d][d], window [3][3d] as float64)."""
    scale = np.frombuffer(buf[:4 * d], dtype=np.float32).copy()
    codes = np.frombuffer(buf[4 * d:4 * d + d * d], dtype=np.int8).reshape(d, d).copy()
    off = 4 * d + d * d
    wb = buf[off:off + 9 * d * policy.DTYPE_SIZE[dtype]]
    if dtype == "f32":
        win = np.frombuffer(wb, dtype=np.float32).astype(np.float64)
    else:
        win = torch.from_numpy(np.frombuffer(wb, dtype=np.int16).copy()).view(torch.bfloat16).double().numpy()
    return scale, codes, win.reshape(3, 3 * d)


def pack_object(S, win, dtype: str) -> bytes:
    S = np.asarray(S)
    return b"".join(pack_record(S[h], win[h], dtype) for h in range(S.shape[0]))


def unpack_object(buf: bytes, H: int, d: int, dtype: str):
    R = record_bytes(d, dtype)
    out = [unpack_record(buf[h * R:(h + 1) * R], d, dtype) for h in range(H)]
    return (np.stack([o[0] for o in out]), np.stack([o[1] for o in out]), np.stack([o[2] for o in out]))
