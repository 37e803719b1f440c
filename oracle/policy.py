"""Host-side policy of the KDA state path, written plainly: checkpoint positions, the
resume-boundary arithmetic, a lowest-free page allocator simulation and the byte layout of
state records in the paged pool.

TEST INFRASTRUCTURE ONLY (see the package docstring).  The CUDA library implements the same
rules independently in C++; tests compare the two bit for bit.

Sources
-------
* "Cache de préfixe hybride KDA–MLA": checkpoints only at a sparse subset of 512-token
  hash-block ends (§"La solution : découpler les deux granularités"); after each forward the
  state at the last hash-aligned position processed is persisted (§"Le fonctionnement du
  prefill"); the hit is the longest boundary with a stored checkpoint, always a multiple of
  the hash block (§"La recherche en deux étages", worked hit 2800 -> 2560); one page byte
  size for every cache type and heads stored contiguously one after another inside the
  pages (§"La mise en page unifiée"); checkpoints are read-only, new ones go to fresh slots
  and a hit is copied into the private state (§"Les checkpoints sont en lecture seule").
* "KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제" (KDA's AI-infrastructure challenges):
  rollback to the largest stored checkpoint not above the matched length (§0x03, 6000 ->
  4096; §0x09 9.2, 15k -> 10k).

Readings taken where the sources are silent
-------------------------------------------
* Checkpoint positions of one forward over absolute positions [start, end): every p with
  p % (hash_block * stride) == 0 and start < p <= end, plus, when include_last is set, the
  last hash-aligned position floor(end / hash_block) * hash_block if it is > start.
* Allocation is lowest-free-first; the pages of the checkpoints of one call are taken in
  (sequence ascending, position ascending) order, all or nothing.
* A state record of one head is S as fp32 row-major [d_k][d_v] followed by the conv window
  [3][q | k | v] (oldest token first) in the input dtype, zero-padded to a multiple of 256
  bytes.  An object is the H records of one sequence in head order; logical byte offset x of
  an object lives in page list[x // page_bytes] at byte x % page_bytes.
"""
from __future__ import annotations

import numpy as np
import torch

DTYPE_SIZE = {"f32": 4, "bf16": 2}


# ----------------------------------------------------------------------------- positions
def ckpt_positions(start: int, end: int, hash_block: int = 512, stride: int = 1,
                   include_last: bool = False) -> list[int]:
    """Absolute checkpoint positions for one forward over [start, end)."""
    if hash_block <= 0 or stride <= 0 or start < 0 or end < start:
        raise ValueError("bad arguments")
    step = hash_block * stride
    first = (start // step + 1) * step
    out = list(range(first, end + 1, step))
    if include_last:
        last = (end // hash_block) * hash_block
        if last > start and (not out or out[-1] != last):
            out.append(last)
            out.sort()
    return out


def decode_ckpt_due(pos: int, interval: int) -> bool:
    """A decode step that starts from `pos` consumed tokens keeps the state at `pos` as a
    checkpoint when pos is a positive multiple of the interval ("KIMI K3 경량 복제에서 본 KDA의
    AI 인프라 과제", §0x05 5.2: decode checkpoints at a fixed interval)."""
    return pos > 0 and pos % interval == 0


def pingpong_plan(pool: "PoolSim", pos: list[int], interval: int, active: list[list[int]],
                  pages_per_object: int):
    """Destination page lists of a ping-pong step: fresh pages (lowest free first, in request
    order) for the requests that are due, the active pages for the others."""
    due = [r for r, p in enumerate(pos) if decode_ckpt_due(p, interval)]
    if pool.free_count() < len(due) * pages_per_object:
        raise AllocError("no pages")
    dst = [list(a) for a in active]
    for r in due:
        dst[r] = pool.alloc(pages_per_object)
    return dst, due


def hit_boundary(stored: list[int], matched: int) -> int:
    """Resume point: the largest stored checkpoint position not above the matched length
    (0, a fresh start, when none qualifies)."""
    best = 0
    for p in stored:
        if p <= matched and p > best:
            best = p
    return best


# ----------------------------------------------------------------------------- layout
def record_bytes(d: int, dtype: str) -> int:
    raw = d * d * 4 + 3 * 3 * d * DTYPE_SIZE[dtype]
    return (raw + 255) // 256 * 256


def object_bytes(H: int, d: int, dtype: str) -> int:
    return H * record_bytes(d, dtype)


def object_pages(H: int, d: int, dtype: str, page_bytes: int) -> int:
    return (object_bytes(H, d, dtype) + page_bytes - 1) // page_bytes


def _window_bytes(win: np.ndarray, dtype: str) -> bytes:
    t = torch.from_numpy(np.ascontiguousarray(win, dtype=np.float64))
    if dtype == "f32":
        return t.to(torch.float32).numpy().tobytes()
    return t.to(torch.bfloat16).view(torch.int16).numpy().tobytes()


def pack_record(S: np.ndarray, win: np.ndarray, dtype: str) -> bytes:
    """One head record: S (d x d) as fp32 row-major, window (3 x 3d) in dtype, zero pad."""
    d = S.shape[0]
    body = np.ascontiguousarray(S, dtype=np.float64).astype(np.float32).tobytes()
    body += _window_bytes(np.asarray(win).reshape(3, 3 * d), dtype)
    return body + b"\0" * (record_bytes(d, dtype) - len(body))


def unpack_record(buf: bytes, d: int, dtype: str):
    """Inverse of pack_record: returns (S float64 [d, d], window float64 [3, 3d])."""
    nS = d * d * 4
    S = np.frombuffer(buf[:nS], dtype=np.float32).astype(np.float64).reshape(d, d)
    nW = 9 * d * DTYPE_SIZE[dtype]
    wb = buf[nS:nS + nW]
    if dtype == "f32":
        win = np.frombuffer(wb, dtype=np.float32).astype(np.float64)
    else:
        bits = torch.from_numpy(np.frombuffer(wb, dtype=np.int16).copy())
        win = bits.view(torch.bfloat16).double().numpy()
    return S, win.reshape(3, 3 * d)


def pack_object(S_heads: np.ndarray, win_heads: np.ndarray, dtype: str) -> bytes:
    """An object = the H head records of one sequence, one after another in head order."""
    return b"".join(pack_record(S_heads[h], win_heads[h], dtype) for h in range(S_heads.shape[0]))


def unpack_object(buf: bytes, H: int, d: int, dtype: str):
    R = record_bytes(d, dtype)
    Ss, Ws = [], []
    for h in range(H):
        S, W = unpack_record(buf[h * R:(h + 1) * R], d, dtype)
        Ss.append(S)
        Ws.append(W)
    return np.stack(Ss), np.stack(Ws)


def scatter_object(pool: np.ndarray, pages: list[int], page_bytes: int, obj: bytes) -> None:
    """Write object bytes into a pool byte array (uint8 [num_pages * page_bytes])."""
    mv = np.frombuffer(obj, dtype=np.uint8)
    for x0 in range(0, len(obj), page_bytes):
        n = min(page_bytes, len(obj) - x0)
        p = pages[x0 // page_bytes]
        pool[p * page_bytes:p * page_bytes + n] = mv[x0:x0 + n]


def gather_object(pool: np.ndarray, pages: list[int], page_bytes: int, nbytes: int) -> bytes:
    """Read object bytes back from a pool byte array."""
    parts = []
    for x0 in range(0, nbytes, page_bytes):
        n = min(page_bytes, nbytes - x0)
        p = pages[x0 // page_bytes]
        parts.append(pool[p * page_bytes:p * page_bytes + n].tobytes())
    return b"".join(parts)


# ----------------------------------------------------------------------------- allocator
class AllocError(Exception):
    pass


class PoolSim:
    """Lowest-free-first page allocator with reference counts (a page is free at 0)."""

    def __init__(self, num_pages: int):
        self.ref = [0] * num_pages

    def free_count(self) -> int:
        return sum(1 for r in self.ref if r == 0)

    def alloc(self, n: int) -> list[int]:
        free = [i for i, r in enumerate(self.ref) if r == 0]
        if n < 0 or len(free) < n:
            raise AllocError("no pages")
        ids = free[:n]
        for i in ids:
            self.ref[i] = 1
        return ids

    def claim(self, ids: list[int]) -> None:
        if len(set(ids)) != len(ids) or any(i < 0 or i >= len(self.ref) or self.ref[i] != 0
                                            for i in ids):
            raise AllocError("claim of a used or invalid page")
        for i in ids:
            self.ref[i] = 1

    def incref(self, ids: list[int]) -> None:
        if any(i < 0 or i >= len(self.ref) or self.ref[i] == 0 for i in ids):
            raise AllocError("incref of a free or invalid page")
        for i in ids:
            self.ref[i] += 1

    def decref(self, ids: list[int]) -> None:
        need: dict[int, int] = {}
        for i in ids:
            need[i] = need.get(i, 0) + 1
        if any(i < 0 or i >= len(self.ref) or self.ref[i] < c for i, c in need.items()):
            raise AllocError("decref below zero or of an invalid page")
        for i in ids:
            self.ref[i] -= 1


def plan_checkpoints(pool: PoolSim, seqs: list[tuple[int, int]], pages_per_object: int,
                     hash_block: int = 512, stride: int = 1, include_last: bool = False):
    """Checkpoint list of one prefill call: [(seq, position, [pages])] in (seq, pos) order,
    pages taken lowest-free-first, all or nothing.  seqs = [(start, end)] absolute."""
    items = []
    for s, (start, end) in enumerate(seqs):
        for p in ckpt_positions(start, end, hash_block, stride, include_last):
            items.append((s, p))
    if pool.free_count() < len(items) * pages_per_object:
        raise AllocError("no pages")
    return [(s, p, pool.alloc(pages_per_object)) for s, p in items]
