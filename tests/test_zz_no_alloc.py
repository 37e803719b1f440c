"""kda_prefill_varlen_noalloc, the prefill entry point for callers that cannot allocate
device memory at call time (for example a serving runtime that reserved all of HBM for its
own pool at start-up, or a latency-critical path where cudaMalloc / cudaFree are not
allowed).  It keeps its per-call metadata in a fixed array inside the library instead of a
caller-provided workspace.

Checked here through the C ABI: two calls in a row give the same outputs, final states and
checkpoints as kda_prefill_varlen on the same inputs, within the tolerance the other GPU
tests use, and metadata larger than the fixed array is refused.  The file is collected
last so that a run stopping at the first failure has already run every other test; it
also passes alone in a fresh process, where its first call sets the array up."""
import ctypes

import numpy as np
import pytest
import torch

import kda_state_chunked_gb300 as kda
from kda_state_chunked_gb300 import workloads

from kda_cases import TOL, assert_close, random_state, read_object, write_object

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _case(pool, dtype, d, H, lens, starts, init, seed):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    toks = workloads.make_tokens(int(cu[-1]), H, d, dtype, seed, DEV)
    dt = kda.DTYPES[dtype]
    P = pool.object_pages(H, d, dt)
    n = len(lens)
    g = torch.Generator().manual_seed(seed)
    S0 = [random_state(H, d, dtype, g) for _ in range(n)]
    outs = []
    for which in ("workspace", "noalloc"):
        act = kda.kda_page_alloc(pool, n * P).reshape(n, P)
        for s in range(n):
            if init[s]:
                write_object(pool, act[s], S0[s][0], S0[s][1], dtype)
        seq, pos, pages = kda.kda_ckpt_plan(pool, H, d, dt, cu, starts, 512, 1, True)
        o = torch.full_like(toks["q"], float("nan"))
        st = torch.zeros(1, dtype=torch.int32, device=DEV)
        if which == "workspace":
            ws = kda.prefill_workspace(toks["q"], cu, starts, len(seq), P)
            kda.kda_prefill_varlen(pool, cu, starts, init, toks["q"], toks["k"], toks["v"], toks["alpha"],
                                   toks["beta"], toks["conv_w"], o, act, seq, pos, pages, ws, st)
        else:
            kda.kda_prefill_varlen_noalloc(pool, cu, starts, init, toks["q"], toks["k"], toks["v"],
                                           toks["alpha"], toks["beta"], toks["conv_w"], o, act, seq, pos,
                                           pages, st)
        rc, bits = kda.kda_sync_status(st)
        assert rc == kda.KDA_OK, bits
        states = [read_object(pool, act[s], H, d, dtype) for s in range(n)]
        ckpts = [read_object(pool, pages[i], H, d, dtype) for i in range(len(seq))]
        outs.append((o.float().cpu().numpy(), states, ckpts, list(pos)))
    (o1, st1, ck1, pos1), (o2, st2, ck2, pos2) = outs
    tol = TOL[dtype]
    assert pos1 == pos2 and len(ck1) == len(ck2)
    for s in range(len(lens)):
        a, b = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            if b > a:
                assert_close(o2[a:b, h], o1[a:b, h], tol, f"o seq {s} head {h}")
            assert_close(st2[s][0][h], st1[s][0][h], tol, f"state seq {s} head {h}")
        assert np.array_equal(st2[s][1], st1[s][1])
    for i in range(len(ck1)):
        for h in range(H):
            assert_close(ck2[i][0][h], ck1[i][0][h], tol, f"checkpoint {i} head {h}")
        assert np.array_equal(ck2[i][1], ck1[i][1])


def test_noalloc_prefill_matches_workspace_prefill_twice():
    pool = kda.Pool(65536, 2048, DEV)
    # first call: a larger batch; second call: a smaller one, so that any stale metadata
    # left in the shared array by the first call would show
    _case(pool, "bf16", 128, 4, [1300, 700, 2100], [0, 512, 96], [0, 1, 1], seed=31)
    _case(pool, "bf16", 128, 2, [640], [1024], [1], seed=32)


def test_noalloc_prefill_fp32_matches():
    pool = kda.Pool(65536, 256, DEV)
    _case(pool, "f32", 64, 2, [1024, 5], [0, 2048], [0, 1], seed=33)


def test_noalloc_prefill_refuses_oversized_metadata():
    """(nseq + n_ckpt) page lists beyond the fixed array are refused before any GPU work."""
    H, d, dt = 32, 128, kda.KDA_BF16
    pool = kda.Pool(65536, 64, DEV)
    P = pool.object_pages(H, d, dt)            # 34 pages per object
    nseq = (kda.KDA_NOALLOC_SCRATCH_BYTES // (4 * P)) + 8
    act = np.zeros(nseq * P, dtype=np.int32)   # the size check comes before any page check
    cu = np.zeros(nseq + 1, dtype=np.int32)
    q = torch.zeros(1, H, d, dtype=torch.bfloat16, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L = kda.lib()
    rc = L.kda_prefill_varlen_noalloc(pool.handle, H, d, dt, nseq, kda._ptr(cu),
                                      kda._ptr(np.zeros(nseq, np.int64)), kda._ptr(np.zeros(nseq, np.uint8)),
                                      None, None, None, None, None,
                                      ctypes.c_void_p(torch.zeros(H, 3 * d, 4, device=DEV).data_ptr()),
                                      None, kda._dev(pool.base), kda._ptr(act), 0, None, None, None,
                                      kda._dev(st), kda._stream(None))
    assert rc == kda.KDA_EINVAL
    del q
