"""KDA oracle: slow, plain fp64 CPU reference of the KDA state path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package.  It shares no code with the CUDA library
(``kda_state_chunked_gb300``) and neither imports the other.

Contents
--------
* ``kda_oracle.c`` (built into ``_build/liboracle.so`` with gcc): the token-by-token
  recurrence with the short causal conv, checkpoint emission, and the explicit segment
  affine map.  See the header of that file for the sources each step follows.
* ``policy.py``: checkpoint positions, hit-boundary arithmetic, a lowest-free page
  allocator simulation and the byte packer for the paged record layout.

Every function here is pinned by ``tests/test_oracle_*.py`` against facts the sources and
the mathematics fix (closed forms, invariants, brute force, the sources' worked examples).
Parity pinned for: conv, recurrence, checkpoint emission, segment maps, positions,
allocation order and the byte layout.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP, no fp contraction, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared",
               "-fPIC", "-std=c11", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_SO)
            P = ctypes.c_void_p
            L.oracle_scan.argtypes = [ctypes.c_int64, ctypes.c_int32, P, P, P, P, P, P, P]
            L.oracle_segment_affine.argtypes = [ctypes.c_int64, ctypes.c_int32, P, P, P, P, P, P]
            L.oracle_kda_run.argtypes = ([ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int32]
                                         + [P] * 16)
            L.oracle_num_threads.argtypes = []
            for f in (L.oracle_scan, L.oracle_segment_affine, L.oracle_kda_run,
                      L.oracle_num_threads):
                f.restype = ctypes.c_int
            _lib = L
    return _lib


def _f64(x):
    """Exact float64 copy of an array-like (torch tensors of any float dtype included)."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor: widen exactly on the CPU
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def scan(qbar, kbar, vbar, alpha, beta, S0=None):
    """Recurrence on post-conv inputs of one (sequence, head).

    qbar, kbar, vbar, alpha: [T, d]; beta: [T]; S0: [d, d] (zeros if None).
    Returns (o [T, d], S_T [d, d]).
    """
    qbar, kbar, vbar, alpha, beta = map(_f64, (qbar, kbar, vbar, alpha, beta))
    T, d = kbar.shape
    S = np.zeros((d, d)) if S0 is None else _f64(S0).copy()
    o = np.zeros((T, d))
    rc = lib().oracle_scan(T, d, _p(qbar), _p(kbar), _p(vbar), _p(alpha), _p(beta), _p(S), _p(o))
    assert rc == 0, rc
    return o, S


def segment_affine(kbar, vbar, alpha, beta):
    """Explicit (M_C, b_C) of a token segment (post-conv inputs), F_C(S) = M_C S + b_C."""
    kbar, vbar, alpha, beta = map(_f64, (kbar, vbar, alpha, beta))
    T, d = kbar.shape
    M = np.zeros((d, d))
    b = np.zeros((d, d))
    rc = lib().oracle_segment_affine(T, d, _p(kbar), _p(vbar), _p(alpha), _p(beta), _p(M), _p(b))
    assert rc == 0, rc
    return M, b


def kda_run(q, k, v, alpha, beta, conv_w, cu_seqlens, S0=None, win0=None, ckpt_counts=None,
            want_xbar=False):
    """Full path on a packed varlen batch.

    q, k, v, alpha: [T_tot, H, d]; beta: [T_tot, H]; conv_w: [H, 3d, 4];
    cu_seqlens: [nseq+1] ints; S0: [nseq, H, d, d] or None; win0: [nseq, H, 3, 3d] or None;
    ckpt_counts: list (per sequence) of ascending token counts p at which (S, window) is
    copied out.  Returns a dict with o, S, win, ck_S, ck_win (lists per sequence) and
    optionally xbar [T_tot, H, 3d].
    """
    q, k, v, alpha, beta, conv_w = map(_f64, (q, k, v, alpha, beta, conv_w))
    T_tot, H, d = q.shape
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    nseq = len(cu) - 1
    S0 = _f64(S0)
    win0 = _f64(win0)
    if ckpt_counts is None:
        ckpt_counts = [[] for _ in range(nseq)]
    ck_off = np.zeros(nseq + 1, dtype=np.int64)
    for s in range(nseq):
        ck_off[s + 1] = ck_off[s] + len(ckpt_counts[s])
    ck_at = np.ascontiguousarray(np.array([p for lst in ckpt_counts for p in lst] or [0],
                                          dtype=np.int64))
    nck = int(ck_off[-1])
    o = np.zeros((T_tot, H, d))
    S = np.zeros((nseq, H, d, d))
    win = np.zeros((nseq, H, 3, 3 * d))
    ck_S = np.zeros((max(nck, 1), H, d, d))
    ck_win = np.zeros((max(nck, 1), H, 3, 3 * d))
    xbar = np.zeros((T_tot, H, 3 * d)) if want_xbar else None
    rc = lib().oracle_kda_run(nseq, _p(cu), H, d, _p(q), _p(k), _p(v), _p(alpha), _p(beta),
                              _p(conv_w), _p(S0), _p(win0), _p(o), _p(S), _p(win), _p(xbar),
                              _p(ck_off), _p(ck_at), _p(ck_S), _p(ck_win))
    assert rc == 0, rc
    out = {"o": o, "S": S, "win": win, "xbar": xbar, "ck_S": [], "ck_win": []}
    for s in range(nseq):
        a, b = int(ck_off[s]), int(ck_off[s + 1])
        out["ck_S"].append(ck_S[a:b])
        out["ck_win"].append(ck_win[a:b])
    return out
