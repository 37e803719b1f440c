"""Python binding of libkda.so, the GB300 (sm_103a) KDA state library.

Argument marshalling only: every step of the state path runs in the library's CUDA kernels.
Functions carry the C names declared in include/kda.h; device arrays are torch CUDA tensors,
host arrays are Python sequences or numpy arrays.  A non-OK status raises KdaError.

The library is loaded from kda_state_chunked_gb300/_build/libkda.so (built by
``python -m kda_state_chunked_gb300.build`` or ``__graft_entry__.build()``); if it is
missing, the first call raises: there is no other implementation behind these names.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import workloads  # noqa: F401  (seeded synthetic inputs; no method arithmetic)

_SO = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libkda.so")
_lock = threading.Lock()
_lib = None

KDA_OK, KDA_EINVAL, KDA_ENOPAGES, KDA_EREF, KDA_ECUDA, KDA_EDEVICE = 0, -1, -2, -3, -4, -5
KDA_F32, KDA_BF16 = 0, 1
KDA_DEV_BAD_PAGE, KDA_DEV_BAD_META, KDA_DEV_TIMEOUT, KDA_DEV_RANGE = 1, 2, 4, 8
DTYPES = {"f32": KDA_F32, "bf16": KDA_BF16}

# Every symbol include/kda.h declares, with (restype, argtypes).
_P = ctypes.c_void_p
_I32, _I64 = ctypes.c_int32, ctypes.c_int64
_SIGS = {
    "kda_record_bytes": (_I64, [_I32, _I32]),
    "kda_object_bytes": (_I64, [_I32, _I32, _I32]),
    "kda_object_pages": (_I32, [_P, _I32, _I32, _I32]),
    "kda_pool_create": (ctypes.c_int, [_I64, _I32, _P]),
    "kda_pool_destroy": (ctypes.c_int, [_P]),
    "kda_pool_page_bytes": (_I64, [_P]),
    "kda_pool_num_pages": (_I32, [_P]),
    "kda_pool_free_count": (_I32, [_P]),
    "kda_page_alloc": (ctypes.c_int, [_P, _I32, _P]),
    "kda_page_claim": (ctypes.c_int, [_P, _I32, _P]),
    "kda_page_incref": (ctypes.c_int, [_P, _I32, _P]),
    "kda_page_decref": (ctypes.c_int, [_P, _I32, _P]),
    "kda_page_refcount": (_I32, [_P, _I32]),
    "kda_ckpt_positions": (_I32, [_I64, _I64, _I32, _I32, _I32, _P, _I32]),
    "kda_ckpt_plan": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P, _I32, _I32, _I32, _I32,
                                     _P, _P, _P, _P]),
    "kda_prefill_workspace_bytes": (_I64, [_I32, _I32, _I32, _I32, _P, _P, _I32, _I32]),
    "kda_prefill_kernel_launches": (_I32, [_I32, _I32, _I32, _I32, _P, _P]),
    "kda_prefill_waves": (_I32, [_I32, _I32, _I32, _I32, _P, _P, _P, _I32]),
    "kda_prefill_varlen": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                          _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _I64, _P, _P]),
    "kda_prefill_varlen_noalloc": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P,
                                                  _P, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P, _P]),
    "kda_decode_step": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P, _P, _P]),
    "kda_decode_step_pp": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P,
                                          _P, _P, _P, _P, _P]),
    "kda_decode_pingpong_plan": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _I32, _P, _P, _P, _P]),
    "kda_verify_plan": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _I32, _P]),
    "kda_verify_step": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _P, _P, _P, _P,
                                       _P, _P, _P, _P]),
    "kda_verify_accept": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _I32, _P, _P, _P, _P]),
    "kda_copy_workspace_bytes": (_I64, [_I32, _I32]),
    "kda_ckpt_write": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _I64, _P, _P]),
    "kda_ckpt_restore": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _I64, _P, _P]),
    "kda_ckpt_release": (ctypes.c_int, [_P, _I32, _I32, _P]),
    "kda_ckpt_offload": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P, _I64, _P, _P, _I64, _P, _P]),
    "kda_ckpt_prefetch": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _I64, _P, _P, _P, _I64, _P, _P]),
    "kda_record_bytes_q8": (_I64, [_I32, _I32]),
    "kda_object_bytes_q8": (_I64, [_I32, _I32, _I32]),
    "kda_object_pages_q8": (_I32, [_P, _I32, _I32, _I32]),
    "kda_ckpt_write_q8": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _I64, _P, _P]),
    "kda_ckpt_restore_q8": (ctypes.c_int, [_P, _I32, _I32, _I32, _I32, _P, _P, _P, _P, _I64, _P, _P]),
    "kda_sync_status": (ctypes.c_int, [_P, _P, _P]),
    "kda_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}


class KdaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = lib().kda_status_string(code).decode() if _lib is not None else str(code)
        super().__init__(f"{where}: {msg} ({code})")


def library_path() -> str:
    return _SO


def lib() -> ctypes.CDLL:
    """Load libkda.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_SO):
                raise RuntimeError(f"libkda.so is not built ({_SO}); run "
                                   "`python -m kda_state_chunked_gb300.build` first")
            L = ctypes.CDLL(_SO)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
    return _lib


def _check(rc: int, where: str) -> int:
    if rc < 0:
        raise KdaError(rc, where)
    return rc


def _i32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32).reshape(-1))


def _i64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.int64).reshape(-1))


def _ptr(a) -> ctypes.c_void_p | None:
    if a is None:
        return None
    if isinstance(a, np.ndarray):
        return a.ctypes.data_as(ctypes.c_void_p)
    return ctypes.c_void_p(a.data_ptr())


def _dev(t):
    """Device pointer of a CUDA tensor (checked contiguous)."""
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("expected a contiguous CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def dtype_of(t) -> int:
    import torch
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


# ------------------------------------------------------------------------------ sizes
def kda_record_bytes(d: int, dtype: int) -> int:
    return _check(lib().kda_record_bytes(d, dtype), "kda_record_bytes")


def kda_object_bytes(H: int, d: int, dtype: int) -> int:
    return _check(lib().kda_object_bytes(H, d, dtype), "kda_object_bytes")


def kda_object_pages(pool: "Pool", H: int, d: int, dtype: int) -> int:
    return _check(lib().kda_object_pages(pool.handle, H, d, dtype), "kda_object_pages")


# ------------------------------------------------------------------------------ pool
class Pool:
    """Owns a kda_pool (host metadata) and, when `device` is given, the device pages
    (a uint8 tensor of num_pages * page_bytes bytes)."""

    def __init__(self, page_bytes: int, num_pages: int, device=None):
        h = ctypes.c_void_p()
        _check(lib().kda_pool_create(page_bytes, num_pages, ctypes.byref(h)), "kda_pool_create")
        self.handle = h
        self.page_bytes = page_bytes
        self.num_pages = num_pages
        self.base = None
        if device is not None:
            import torch
            self.base = torch.zeros(num_pages * page_bytes, dtype=torch.uint8, device=device)

    def close(self):
        if self.handle is not None and _lib is not None:
            _lib.kda_pool_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def free_count(self) -> int:
        return _check(lib().kda_pool_free_count(self.handle), "kda_pool_free_count")

    def object_pages(self, H: int, d: int, dtype: int) -> int:
        return kda_object_pages(self, H, d, dtype)

    def page_view(self, page: int):
        return self.base[page * self.page_bytes:(page + 1) * self.page_bytes]


def kda_page_alloc(pool: Pool, n: int) -> np.ndarray:
    out = np.zeros(max(n, 1), dtype=np.int32)
    _check(lib().kda_page_alloc(pool.handle, n, _ptr(out)), "kda_page_alloc")
    return out[:n]


def kda_page_claim(pool: Pool, ids) -> None:
    a = _i32(ids)
    _check(lib().kda_page_claim(pool.handle, len(a), _ptr(a)), "kda_page_claim")


def kda_page_incref(pool: Pool, ids) -> None:
    a = _i32(ids)
    _check(lib().kda_page_incref(pool.handle, len(a), _ptr(a)), "kda_page_incref")


def kda_page_decref(pool: Pool, ids) -> None:
    a = _i32(ids)
    _check(lib().kda_page_decref(pool.handle, len(a), _ptr(a)), "kda_page_decref")


def kda_page_refcount(pool: Pool, page: int) -> int:
    return _check(lib().kda_page_refcount(pool.handle, page), "kda_page_refcount")


# ------------------------------------------------------------------------------ policy
def kda_ckpt_positions(start: int, end: int, hash_block: int = 512, stride: int = 1,
                       include_last: bool = False) -> list[int]:
    n = _check(lib().kda_ckpt_positions(start, end, hash_block, stride, int(include_last), None, 0),
               "kda_ckpt_positions")
    out = np.zeros(max(n, 1), dtype=np.int64)
    lib().kda_ckpt_positions(start, end, hash_block, stride, int(include_last), _ptr(out), n)
    return [int(x) for x in out[:n]]


def kda_ckpt_plan(pool: Pool, H: int, d: int, dtype: int, cu_seqlens, start_pos,
                  hash_block: int = 512, stride: int = 1, include_last: bool = False):
    """Returns (seq int32[n], pos int64[n], pages int32[n, P]); pages are allocated."""
    cu = _i32(cu_seqlens)
    sp = _i64(start_pos)
    nseq = len(cu) - 1
    P = kda_object_pages(pool, H, d, dtype)
    cap = sum(len(kda_ckpt_positions(int(sp[s]), int(sp[s]) + int(cu[s + 1] - cu[s]), hash_block,
                                     stride, include_last)) for s in range(nseq))
    seq = np.zeros(max(cap, 1), dtype=np.int32)
    pos = np.zeros(max(cap, 1), dtype=np.int64)
    pages = np.zeros(max(cap, 1) * P, dtype=np.int32)
    n = ctypes.c_int32(0)
    _check(lib().kda_ckpt_plan(pool.handle, H, d, dtype, nseq, _ptr(cu), _ptr(sp), hash_block,
                               stride, int(include_last), cap, ctypes.byref(n), _ptr(seq),
                               _ptr(pos), _ptr(pages)), "kda_ckpt_plan")
    n = n.value
    return seq[:n], pos[:n], pages[:n * P].reshape(n, P)


# ------------------------------------------------------------------------------ prefill
def kda_prefill_workspace_bytes(H: int, d: int, dtype: int, cu_seqlens, start_pos, n_ckpt: int,
                                pages_per_object: int) -> int:
    """Workspace bytes of kda_prefill_varlen for this batch (host cu_seqlens / start_pos)."""
    cu = _i32(cu_seqlens)
    sp = _i64(start_pos)
    return _check(lib().kda_prefill_workspace_bytes(H, d, dtype, len(cu) - 1, _ptr(cu), _ptr(sp), n_ckpt,
                                                    pages_per_object), "kda_prefill_workspace_bytes")


def kda_prefill_kernel_launches(H: int, d: int, dtype: int, cu_seqlens, start_pos) -> int:
    """Kernel launches one kda_prefill_varlen call makes for this batch."""
    cu = _i32(cu_seqlens)
    sp = _i64(start_pos)
    return _check(lib().kda_prefill_kernel_launches(H, d, dtype, len(cu) - 1, _ptr(cu), _ptr(sp)),
                  "kda_prefill_kernel_launches")


def kda_prefill_waves(H: int, d: int, dtype: int, cu_seqlens, start_pos) -> np.ndarray:
    """Wave bounds of the bf16 d=128 prefill for this batch: wave w = local chunks
    [b[w], b[w + 1]) of every sequence (empty for other shapes or only empty sequences)."""
    cu = _i32(cu_seqlens)
    sp = _i64(start_pos)
    n = _check(lib().kda_prefill_waves(H, d, dtype, len(cu) - 1, _ptr(cu), _ptr(sp), None, 0), "kda_prefill_waves")
    if n == 0:
        return np.zeros(0, dtype=np.int32)
    out = np.zeros(n + 1, dtype=np.int32)
    _check(lib().kda_prefill_waves(H, d, dtype, len(cu) - 1, _ptr(cu), _ptr(sp), _ptr(out), n + 1), "kda_prefill_waves")
    return out


def prefill_workspace(q, cu_seqlens, start_pos, n_ckpt: int, pages_per_object: int):
    """A device byte tensor sized for kda_prefill_varlen on this batch."""
    import torch
    T_tot, H, d = q.shape
    nb = kda_prefill_workspace_bytes(H, d, dtype_of(q), cu_seqlens, start_pos, n_ckpt, pages_per_object)
    return torch.empty(nb, dtype=torch.uint8, device=q.device)


def kda_prefill_varlen(pool: Pool, cu_seqlens, start_pos, has_init, q, k, v, alpha, beta, conv_w,
                       o, active_pages, ckpt_seq=(), ckpt_pos=(), ckpt_pages=None,
                       workspace=None, status=None, stream=None) -> None:
    """q, k, v, alpha, o: [T_tot, H, d]; beta: [T_tot, H]; conv_w: fp32 [H, 3d, 4] (CUDA).
    active_pages: host [nseq, P]; ckpt_*: as returned by kda_ckpt_plan."""
    T_tot, H, d = q.shape
    cu = _i32(cu_seqlens)
    sp = _i64(start_pos)
    hi = np.ascontiguousarray(np.asarray(has_init, dtype=np.uint8).reshape(-1))
    act = _i32(active_pages)
    cs = _i32(ckpt_seq)
    cp = _i64(ckpt_pos)
    n_ck = len(cs)
    cpg = _i32(ckpt_pages if ckpt_pages is not None else np.zeros(0, np.int32))
    nseq = len(cu) - 1
    rc = lib().kda_prefill_varlen(
        pool.handle, H, d, dtype_of(q), nseq, _ptr(cu), _ptr(sp), _ptr(hi), _dev(q), _dev(k),
        _dev(v), _dev(alpha), _dev(beta), _dev(conv_w), _dev(o), _dev(pool.base), _ptr(act), n_ck,
        _ptr(cs) if n_ck else None, _ptr(cp) if n_ck else None, _ptr(cpg) if n_ck else None,
        _dev(workspace), workspace.numel() * workspace.element_size(), _dev(status),
        _stream(stream))
    _check(rc, "kda_prefill_varlen")


KDA_NOALLOC_SCRATCH_BYTES = 1 << 20


def kda_prefill_varlen_noalloc(pool: Pool, cu_seqlens, start_pos, has_init, q, k, v, alpha, beta,
                               conv_w, o, active_pages, ckpt_seq=(), ckpt_pos=(), ckpt_pages=None,
                               status=None, stream=None) -> None:
    """kda_prefill_varlen without a workspace, for callers that cannot allocate device memory
    at call time: the per-call metadata lives in a fixed 1 MiB array inside the library
    (see include/kda.h for the limit and the rules on concurrent calls)."""
    T_tot, H, d = q.shape
    cu = _i32(cu_seqlens)
    sp = _i64(start_pos)
    hi = np.ascontiguousarray(np.asarray(has_init, dtype=np.uint8).reshape(-1))
    act = _i32(active_pages)
    cs = _i32(ckpt_seq)
    cp = _i64(ckpt_pos)
    n_ck = len(cs)
    cpg = _i32(ckpt_pages if ckpt_pages is not None else np.zeros(0, np.int32))
    rc = lib().kda_prefill_varlen_noalloc(
        pool.handle, H, d, dtype_of(q), len(cu) - 1, _ptr(cu), _ptr(sp), _ptr(hi), _dev(q), _dev(k),
        _dev(v), _dev(alpha), _dev(beta), _dev(conv_w), _dev(o), _dev(pool.base), _ptr(act), n_ck,
        _ptr(cs) if n_ck else None, _ptr(cp) if n_ck else None, _ptr(cpg) if n_ck else None,
        _dev(status), _stream(stream))
    _check(rc, "kda_prefill_varlen_noalloc")


# ------------------------------------------------------------------------------ decode
def kda_decode_step(pool: Pool, q, k, v, alpha, beta, conv_w, o, state_pages, status,
                    stream=None) -> None:
    """q, k, v, alpha, o: [B, H, d]; beta: [B, H]; state_pages: int32 CUDA [B, P]."""
    B, H, d = q.shape
    rc = lib().kda_decode_step(pool.handle, H, d, dtype_of(q), B, _dev(q), _dev(k), _dev(v),
                               _dev(alpha), _dev(beta), _dev(conv_w), _dev(o), _dev(pool.base),
                               _dev(state_pages), _dev(status), _stream(stream))
    _check(rc, "kda_decode_step")


def kda_decode_step_pp(pool: Pool, q, k, v, alpha, beta, conv_w, o, src_pages, dst_pages, status,
                       stream=None) -> None:
    """Ping-pong decode step: read each request's state from src_pages, write it to dst_pages
    (both int32 CUDA [B, P]); requests whose lists are equal update in place."""
    B, H, d = q.shape
    rc = lib().kda_decode_step_pp(pool.handle, H, d, dtype_of(q), B, _dev(q), _dev(k), _dev(v),
                                  _dev(alpha), _dev(beta), _dev(conv_w), _dev(o), _dev(pool.base),
                                  _dev(src_pages), _dev(dst_pages), _dev(status), _stream(stream))
    _check(rc, "kda_decode_step_pp")


def kda_decode_pingpong_plan(pool: Pool, H: int, d: int, dtype: int, pos, interval: int, active_pages):
    """-> (dst_pages [B, P], donated request indices): fresh destination objects for the
    requests at a decode-checkpoint boundary (pos > 0, pos % interval == 0)."""
    act = _i32(active_pages)
    P = kda_object_pages(pool, H, d, dtype)
    B = len(act) // P
    p = _i64(pos)
    dst = np.zeros(max(B * P, 1), dtype=np.int32)
    don = np.zeros(max(B, 1), dtype=np.int32)
    n = ctypes.c_int32(0)
    _check(lib().kda_decode_pingpong_plan(pool.handle, H, d, dtype, B, _ptr(p), interval, _ptr(act), _ptr(dst),
                                          _ptr(don), ctypes.byref(n)), "kda_decode_pingpong_plan")
    return dst[:B * P].reshape(B, P), don[:n.value]


def kda_verify_plan(pool: Pool, H: int, d: int, dtype: int, B: int, K: int) -> np.ndarray:
    """Intermediate objects of a verify step: pages [K, B, P]."""
    P = kda_object_pages(pool, H, d, dtype)
    out = np.zeros(max(K * B * P, 1), dtype=np.int32)
    _check(lib().kda_verify_plan(pool.handle, H, d, dtype, B, K, _ptr(out)), "kda_verify_plan")
    return out[:K * B * P].reshape(K, B, P)


def kda_verify_step(pool: Pool, q, k, v, alpha, beta, conv_w, o, src_pages, inter_pages, status,
                    stream=None) -> None:
    """q, k, v, alpha, o: [K, B, H, d]; beta: [K, B, H]; src_pages int32 CUDA [B, P];
    inter_pages int32 CUDA [K, B, P]."""
    K, B, H, d = q.shape
    rc = lib().kda_verify_step(pool.handle, H, d, dtype_of(q), B, K, _dev(q), _dev(k), _dev(v), _dev(alpha),
                               _dev(beta), _dev(conv_w), _dev(o), _dev(pool.base), _dev(src_pages),
                               _dev(inter_pages), _dev(status), _stream(stream))
    _check(rc, "kda_verify_step")


def kda_verify_accept(pool: Pool, H: int, d: int, dtype: int, accepted, src_pages, inter_pages) -> np.ndarray:
    """Keep the object at each request's accepted length; release the rest.  Returns the new
    active pages [B, P]."""
    acc = _i32(accepted)
    src = _i32(src_pages)
    inter = _i32(inter_pages)
    P = kda_object_pages(pool, H, d, dtype)
    B = len(acc)
    K = len(inter) // (B * P)
    out = np.zeros(max(B * P, 1), dtype=np.int32)
    _check(lib().kda_verify_accept(pool.handle, H, d, dtype, B, K, _ptr(acc), _ptr(src), _ptr(inter), _ptr(out)),
           "kda_verify_accept")
    return out[:B * P].reshape(B, P)


# ------------------------------------------------------------------------------ copies
def kda_copy_workspace_bytes(n: int, pages_per_object: int) -> int:
    return _check(lib().kda_copy_workspace_bytes(n, pages_per_object), "kda_copy_workspace_bytes")


def kda_ckpt_write(pool: Pool, H: int, d: int, dtype: int, src_pages, workspace, status,
                   stream=None) -> np.ndarray:
    src = _i32(src_pages)
    P = kda_object_pages(pool, H, d, dtype)
    n = len(src) // P
    dst = np.zeros(max(len(src), 1), dtype=np.int32)
    rc = lib().kda_ckpt_write(pool.handle, H, d, dtype, n, _ptr(src), _ptr(dst), _dev(pool.base),
                              _dev(workspace), workspace.numel() * workspace.element_size(),
                              _dev(status), _stream(stream))
    _check(rc, "kda_ckpt_write")
    return dst[:len(src)].reshape(n, P)


def kda_ckpt_restore(pool: Pool, H: int, d: int, dtype: int, ckpt_pages, active_pages, workspace,
                     status, stream=None) -> None:
    ck = _i32(ckpt_pages)
    act = _i32(active_pages)
    P = kda_object_pages(pool, H, d, dtype)
    n = len(ck) // P
    if len(act) != len(ck):
        raise ValueError("ckpt_pages and active_pages differ in length")
    rc = lib().kda_ckpt_restore(pool.handle, H, d, dtype, n, _ptr(ck), _ptr(act), _dev(pool.base),
                                _dev(workspace), workspace.numel() * workspace.element_size(),
                                _dev(status), _stream(stream))
    _check(rc, "kda_ckpt_restore")


def kda_ckpt_release(pool: Pool, ckpt_pages, pages_per_object: int) -> None:
    ck = _i32(ckpt_pages)
    _check(lib().kda_ckpt_release(pool.handle, len(ck) // pages_per_object, pages_per_object,
                                  _ptr(ck)), "kda_ckpt_release")


# ------------------------------------------------------------------------------ host offload
def kda_ckpt_offload(pool: Pool, H: int, d: int, dtype: int, pages, host, workspace, status, stream=None) -> None:
    """Copy objects (pages [n, P]) into a pinned host uint8 tensor (object i at i * object_bytes)."""
    pg = _i32(pages)
    P = kda_object_pages(pool, H, d, dtype)
    n = len(pg) // P
    rc = lib().kda_ckpt_offload(pool.handle, H, d, dtype, n, _ptr(pg), ctypes.c_void_p(host.data_ptr()),
                                host.numel() * host.element_size(), _dev(pool.base), _dev(workspace),
                                workspace.numel() * workspace.element_size(), _dev(status), _stream(stream))
    _check(rc, "kda_ckpt_offload")


def kda_ckpt_prefetch(pool: Pool, H: int, d: int, dtype: int, n: int, host, workspace, status,
                      stream=None) -> np.ndarray:
    """Allocate n fresh objects and copy them in from a pinned host uint8 tensor; returns the
    pages [n, P]."""
    P = kda_object_pages(pool, H, d, dtype)
    out = np.zeros(max(n * P, 1), dtype=np.int32)
    rc = lib().kda_ckpt_prefetch(pool.handle, H, d, dtype, n, ctypes.c_void_p(host.data_ptr()),
                                 host.numel() * host.element_size(), _ptr(out), _dev(pool.base), _dev(workspace),
                                 workspace.numel() * workspace.element_size(), _dev(status), _stream(stream))
    _check(rc, "kda_ckpt_prefetch")
    return out[:n * P].reshape(n, P)


# ------------------------------------------------------------------------------ INT8 checkpoints
def kda_record_bytes_q8(d: int, dtype: int) -> int:
    return _check(lib().kda_record_bytes_q8(d, dtype), "kda_record_bytes_q8")


def kda_object_bytes_q8(H: int, d: int, dtype: int) -> int:
    return _check(lib().kda_object_bytes_q8(H, d, dtype), "kda_object_bytes_q8")


def kda_object_pages_q8(pool: Pool, H: int, d: int, dtype: int) -> int:
    return _check(lib().kda_object_pages_q8(pool.handle, H, d, dtype), "kda_object_pages_q8")


def kda_ckpt_write_q8(pool: Pool, H: int, d: int, dtype: int, src_pages, workspace, status,
                      stream=None) -> np.ndarray:
    """Snapshot full objects into new INT8 checkpoints; returns their pages [n, Pq]."""
    src = _i32(src_pages)
    P = kda_object_pages(pool, H, d, dtype)
    Pq = kda_object_pages_q8(pool, H, d, dtype)
    n = len(src) // P
    dst = np.zeros(max(n * Pq, 1), dtype=np.int32)
    rc = lib().kda_ckpt_write_q8(pool.handle, H, d, dtype, n, _ptr(src), _ptr(dst), _dev(pool.base),
                                 _dev(workspace), workspace.numel() * workspace.element_size(),
                                 _dev(status), _stream(stream))
    _check(rc, "kda_ckpt_write_q8")
    return dst[:n * Pq].reshape(n, Pq)


def kda_ckpt_restore_q8(pool: Pool, H: int, d: int, dtype: int, ckpt_pages, active_pages, workspace,
                        status, stream=None) -> None:
    """Dequantise INT8 checkpoints [n, Pq] into private full objects [n, P]."""
    ck = _i32(ckpt_pages)
    act = _i32(active_pages)
    P = kda_object_pages(pool, H, d, dtype)
    Pq = kda_object_pages_q8(pool, H, d, dtype)
    n = len(act) // P
    if len(ck) != n * Pq:
        raise ValueError("ckpt_pages and active_pages hold different object counts")
    rc = lib().kda_ckpt_restore_q8(pool.handle, H, d, dtype, n, _ptr(ck), _ptr(act), _dev(pool.base),
                                   _dev(workspace), workspace.numel() * workspace.element_size(),
                                   _dev(status), _stream(stream))
    _check(rc, "kda_ckpt_restore_q8")


# ------------------------------------------------------------------------------ status
def kda_sync_status(status, stream=None) -> tuple[int, int]:
    """Returns (status code, device bits); does not raise on KDA_EDEVICE."""
    bits = ctypes.c_int32(0)
    rc = lib().kda_sync_status(_dev(status), _stream(stream), ctypes.byref(bits))
    if rc not in (KDA_OK, KDA_EDEVICE):
        raise KdaError(rc, "kda_sync_status")
    return rc, bits.value
