"""kda_prefill_varlen_noalloc, the prefill entry point for callers that cannot allocate
device memory at call time (for example a serving runtime that reserved all of HBM for its
own pool at start-up, or a latency-critical path where cudaMalloc / cudaFree are not
allowed).  It keeps its per-call metadata in a fixed array inside the library instead of a
caller-provided workspace, and runs the single-kernel tensor-core prefill for bf16 d = 128
(the CUDA-core kernel for fp32).

Checked here through the C ABI:
  * its outputs, final states and windows, checkpoint states and windows against the fp64
    oracle on the same inputs (1e-4 for fp32, 2e-2 for bf16 per (sequence, head) block;
    windows, positions and pages exactly), on two calls in a row of different sizes, so
    that metadata left in the shared array by the first call would show;
  * the same results as kda_prefill_varlen on the same inputs, within that tolerance;
  * a first call in a fresh process, made before any other prefill call of that process,
    on a fragmented pool of 19 x 256-byte pages (page translation without a power-of-two
    shift, records across non-adjacent pages), against the oracle;
  * metadata larger than the fixed array is refused.
The file is collected last so that a run stopping at the first failure has already run
every other test; it also passes alone in a fresh process."""
import ctypes
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import kda_state_chunked_gb300 as kda
from kda_state_chunked_gb300 import workloads

from kda_cases import (TOL, Prefill, assert_close, compare_prefill, oracle_positions, oracle_prefill,
                       random_state, read_object, record_margin, write_object)

pytestmark = pytest.mark.gpu
DEV = "cuda"
HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


class NoallocPrefill:
    """One kda_prefill_varlen_noalloc call, with the same fields as kda_cases.Prefill."""

    def __init__(self, pool, toks, cu, start_pos, has_init, active_pages, stride=1, include_last=True):
        q = toks["q"]
        _, H, d = q.shape
        self.H, self.d = H, d
        self.seq, self.pos, self.pages = kda.kda_ckpt_plan(pool, H, d, kda.dtype_of(q), cu, start_pos, 512,
                                                           stride, include_last)
        self.status = torch.zeros(1, dtype=torch.int32, device=q.device)
        self.o = torch.full_like(q, float("nan"))
        kda.kda_prefill_varlen_noalloc(pool, cu, start_pos, has_init, q, toks["k"], toks["v"], toks["alpha"],
                                       toks["beta"], toks["conv_w"], self.o, active_pages, self.seq, self.pos,
                                       self.pages, self.status)
        rc, bits = kda.kda_sync_status(self.status)
        assert rc == kda.KDA_OK, f"device status bits {bits}"


def _inputs(dtype, d, H, lens, starts, init, seed):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cpu = workloads.make_tokens(int(cu[-1]), H, d, dtype, seed, "cpu")
    dev = {k: v.to(DEV) for k, v in cpu.items()}
    g = torch.Generator().manual_seed(seed)
    n = len(lens)
    S0 = np.zeros((n, H, d, d))
    W0 = np.zeros((n, H, 3, 3 * d))
    for s in range(n):
        if init[s]:
            S0[s], W0[s] = random_state(H, d, dtype, g)
    return cu, cpu, dev, S0, W0


def _run(kind, pool, dtype, d, H, cu, dev, starts, init, S0, W0, stride):
    P = pool.object_pages(H, d, kda.DTYPES[dtype])
    n = len(cu) - 1
    act = kda.kda_page_alloc(pool, n * P).reshape(n, P)
    for s in range(n):
        if init[s]:
            write_object(pool, act[s], S0[s], W0[s], dtype)
    cls = NoallocPrefill if kind == "noalloc" else Prefill
    return cls(pool, dev, cu, starts, init, act, stride=stride, include_last=True), act


def _case(pool, dtype, d, H, lens, starts, init, seed, stride=1):
    """Both entry points against the oracle, then against each other."""
    cu, cpu, dev, S0, W0 = _inputs(dtype, d, H, lens, starts, init, seed)
    ck = oracle_positions(cu, starts, stride, True)
    ref = oracle_prefill(cpu, cu, starts, S0=S0, win0=W0, ckpt_abs=ck)
    tol = TOL[dtype]
    na, act_na = _run("noalloc", pool, dtype, d, H, cu, dev, starts, init, S0, W0, stride)
    compare_prefill(pool, na, ref, cu, act_na, dtype, ck, name=f"noalloc prefill vs oracle ({dtype})")
    ws, act_ws = _run("workspace", pool, dtype, d, H, cu, dev, starts, init, S0, W0, stride)
    compare_prefill(pool, ws, ref, cu, act_ws, dtype, ck)
    # the two entry points agree with each other as well
    assert [int(p) for p in na.pos] == [int(p) for p in ws.pos]
    o1, o2 = ws.o.float().cpu().numpy(), na.o.float().cpu().numpy()
    for s in range(len(lens)):
        a, b = int(cu[s]), int(cu[s + 1])
        S1, W1 = read_object(pool, act_ws[s], H, d, dtype)
        S2, W2 = read_object(pool, act_na[s], H, d, dtype)
        for h in range(H):
            if b > a:
                assert_close(o2[a:b, h], o1[a:b, h], tol, f"o seq {s} head {h}")
            assert_close(S2[h], S1[h], tol, f"state seq {s} head {h}")
        assert np.array_equal(W2, W1)
    for i in range(len(na.pos)):
        S1, W1 = read_object(pool, ws.pages[i], H, d, dtype)
        S2, W2 = read_object(pool, na.pages[i], H, d, dtype)
        for h in range(H):
            assert_close(S2[h], S1[h], tol, f"checkpoint {i} head {h}")
        assert np.array_equal(W2, W1)


def test_noalloc_prefill_matches_oracle_twice():
    pool = kda.Pool(65536, 2048, DEV)
    # first call: a larger batch; second call: a smaller one, so that any stale metadata
    # left in the shared array by the first call would show
    _case(pool, "bf16", 128, 4, [1300, 700, 2100], [0, 512, 96], [0, 1, 1], seed=31)
    _case(pool, "bf16", 128, 2, [640], [1024], [1], seed=32)


def test_noalloc_prefill_fp32_matches_oracle():
    pool = kda.Pool(65536, 256, DEV)
    _case(pool, "f32", 64, 2, [1024, 5], [0, 2048], [0, 1], seed=33)


def fresh_process_case():
    """Body of the fresh-process test: the first prefill call of the process is the
    allocation-free one, on a fragmented pool of 19 x 256-byte pages whose objects' pages are
    three ids apart; compared with the oracle.  Prints the worst error."""
    dtype, d, H = "bf16", 128, 3
    lens, starts, init = [700, 1, 1500, 333, 0, 2100], [0, 512, 96, 2048 + 37, 4096, 5], [0, 1, 1, 1, 1, 1]
    cu, cpu, dev, S0, W0 = _inputs(dtype, d, H, lens, starts, init, seed=41)
    pool = kda.Pool(19 * 256, 3000, DEV)
    held = kda.kda_page_alloc(pool, 3000)
    kda.kda_page_decref(pool, held[1::3])          # later allocations get ids 1, 4, 7, ...
    P = pool.object_pages(H, d, kda.DTYPES[dtype])
    act = kda.kda_page_alloc(pool, len(lens) * P).reshape(len(lens), P)
    assert np.all(np.diff(act.reshape(-1)) == 3)
    for s in range(len(lens)):
        if init[s]:
            write_object(pool, act[s], S0[s], W0[s], dtype)
    run = NoallocPrefill(pool, dev, cu, starts, init, act, stride=2, include_last=True)
    ck = oracle_positions(cu, starts, 2, True)
    ref = oracle_prefill(cpu, cu, starts, S0=S0, win0=W0, ckpt_abs=ck)
    worst = compare_prefill(pool, run, ref, cu, act, dtype, ck)
    print(f"WORST {worst:.6e}")


def test_noalloc_first_call_in_fresh_process_on_scattered_pages():
    code = ("import sys; sys.path.insert(0, %r); sys.path.insert(0, %r); "
            "import test_zz_no_alloc as t; t.fresh_process_case()" % (ROOT, HERE))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    worst = float(r.stdout.split("WORST")[-1].split()[0])
    record_margin("noalloc prefill vs oracle, fresh process, 19x256 B pages (bf16)", worst, TOL["bf16"])


def test_noalloc_prefill_refuses_oversized_metadata():
    """(nseq + n_ckpt) page lists beyond the fixed array are refused before any GPU work."""
    H, d, dt = 32, 128, kda.KDA_BF16
    pool = kda.Pool(65536, 64, DEV)
    P = pool.object_pages(H, d, dt)            # 34 pages per object
    nseq = (kda.KDA_NOALLOC_SCRATCH_BYTES // (4 * P)) + 8
    act = np.zeros(nseq * P, dtype=np.int32)   # the size check comes before any page check
    cu = np.zeros(nseq + 1, dtype=np.int32)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L = kda.lib()
    rc = L.kda_prefill_varlen_noalloc(pool.handle, H, d, dt, nseq, kda._ptr(cu),
                                      kda._ptr(np.zeros(nseq, np.int64)), kda._ptr(np.zeros(nseq, np.uint8)),
                                      None, None, None, None, None,
                                      ctypes.c_void_p(torch.zeros(H, 3 * d, 4, device=DEV).data_ptr()),
                                      None, kda._dev(pool.base), kda._ptr(act), 0, None, None, None,
                                      kda._dev(st), kda._stream(None))
    assert rc == kda.KDA_EINVAL
