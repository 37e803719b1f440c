"""GPU parity of the speculative verify step: K draft tokens per request, the output of each and
the state after each kept in its own object (token by token against the oracle), the source
untouched; accepting a prefix makes its state the active one, and decoding continues from it."""
import numpy as np
import pytest
import torch

import kda_state_chunked_gb300 as kda
from kda_state_chunked_gb300 import workloads
import oracle
from oracle import policy

from kda_cases import TOL, assert_close, random_state, read_object, read_object_bytes, write_object

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("dtype,d,page_bytes", [("bf16", 128, 65536), ("bf16", 128, 260 * 256), ("f32", 64, 4096)])
def test_verify_intermediate_states_and_accept(dtype, d, page_bytes):
    dt = kda.DTYPES[dtype]
    B, H, K = 3, 2, 4
    P = policy.object_pages(H, d, dtype, page_bytes)
    nb = policy.object_bytes(H, d, dtype)
    pool = kda.Pool(page_bytes, (K + 2) * B * P + 8, DEV)
    src = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    g = torch.Generator().manual_seed(50 + d)
    S0 = np.zeros((B, H, d, d))
    W0 = np.zeros((B, H, 3, 3 * d))
    before = []
    for b in range(B):
        S0[b], W0[b] = random_state(H, d, dtype, g)
        write_object(pool, src[b], S0[b], W0[b], dtype)
        before.append(read_object_bytes(pool, src[b], nb))
    conv_w = torch.randn(H, 3 * d, 4, generator=g) * 0.5
    steps = [workloads.decode_step_tokens(B, H, d, dtype, 50, j, "cpu") for j in range(K)]
    drafts = {k: torch.stack([s[k] for s in steps]) for k in steps[0]}          # [K, B, ...]
    inter = kda.kda_verify_plan(pool, H, d, dt, B, K)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dv = {k: v.to(DEV) for k, v in drafts.items()}
    o = torch.full_like(dv["q"], float("nan"))
    kda.kda_verify_step(pool, dv["q"], dv["k"], dv["v"], dv["alpha"], dv["beta"], conv_w.to(DEV), o,
                        torch.from_numpy(src).to(DEV), torch.from_numpy(inter).to(DEV), st)
    rc, bits = kda.kda_sync_status(st)
    assert rc == kda.KDA_OK, bits
    og = o.float().cpu().numpy()
    S_ref, W_ref = S0.copy(), W0.copy()
    for j in range(K):
        t = steps[j]
        r = oracle.kda_run(t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, np.arange(B + 1),
                           S0=S_ref, win0=W_ref)
        S_ref, W_ref = r["S"], r["win"]
        for b in range(B):
            for h in range(H):
                assert_close(og[j, b, h], r["o"][b, h], TOL[dtype], f"draft {j} o req {b} head {h}",
                             name=f"speculative verify ({dtype})")
            Sg, Wg = read_object(pool, inter[j, b], H, d, dtype)
            for h in range(H):
                assert_close(Sg[h], S_ref[b, h], TOL[dtype], f"draft {j} state req {b} head {h}",
                             name=f"speculative verify ({dtype})")
            assert np.array_equal(Wg, W_ref[b])
    for b in range(B):
        assert read_object_bytes(pool, src[b], nb) == before[b]
    # accept 0, 2 and 4 tokens
    kept = [read_object_bytes(pool, src[0], nb), read_object_bytes(pool, inter[1, 1], nb),
            read_object_bytes(pool, inter[3, 2], nb)]
    act = kda.kda_verify_accept(pool, H, d, dt, [0, 2, 4], src, inter)
    assert pool.num_pages - pool.free_count() == B * P
    for b in range(B):
        assert read_object_bytes(pool, act[b], nb) == kept[b]


def _verify_case(B, H, K, seed, bad_request=None):
    """Verify step on B requests x H heads (bf16, d = 128, 64 KiB pages); returns everything the
    checks need.  bad_request: a request whose last draft object gets an out-of-pool page id."""
    dtype, d, page_bytes = "bf16", 128, 65536
    dt = kda.DTYPES[dtype]
    P = policy.object_pages(H, d, dtype, page_bytes)
    pool = kda.Pool(page_bytes, (2 * K + 2) * B * P + 8, DEV)
    src = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    g = torch.Generator().manual_seed(seed)
    S0 = np.zeros((B, H, d, d))
    W0 = np.zeros((B, H, 3, 3 * d))
    for b in range(B):
        S0[b], W0[b] = random_state(H, d, dtype, g)
        write_object(pool, src[b], S0[b], W0[b], dtype)
    conv_w = torch.randn(H, 3 * d, 4, generator=g) * 0.5
    steps = [workloads.decode_step_tokens(B, H, d, dtype, seed, j, "cpu") for j in range(K)]
    dv = {k: torch.stack([s[k] for s in steps]).to(DEV) for k in steps[0]}
    inter = kda.kda_verify_plan(pool, H, d, dt, B, K)
    inter_dev = torch.from_numpy(inter).to(DEV)
    if bad_request is not None:
        inter_dev[K - 1, bad_request, 0] = pool.num_pages + 5
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = torch.full_like(dv["q"], float("nan"))
    kda.kda_verify_step(pool, dv["q"], dv["k"], dv["v"], dv["alpha"], dv["beta"], conv_w.to(DEV), o,
                        torch.from_numpy(src).to(DEV), inter_dev, st)
    return pool, src, inter, steps, dv, conv_w, o, st, S0, W0


@pytest.mark.parametrize("K", [1, 3, 8])
def test_verify_fused_many_items_per_sm(K):
    """More (request, head) items than SMs, so every CTA of the fused kernel walks several
    items (the next record loads while the current one's draft states are stored): every
    output and every intermediate state against the oracle, and against K chained ping-pong
    decode steps of the same inputs."""
    dtype, d = "bf16", 128
    B, H = 80, 4
    pool, src, inter, steps, dv, conv_w, o, st, S0, W0 = _verify_case(B, H, K, 70 + K)
    rc, bits = kda.kda_sync_status(st)
    assert rc == kda.KDA_OK, bits
    og = o.float().cpu().numpy()
    tol = TOL[dtype]
    S_ref, W_ref = S0.copy(), W0.copy()
    for j in range(K):
        t = steps[j]
        r = oracle.kda_run(t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, np.arange(B + 1),
                           S0=S_ref, win0=W_ref)
        S_ref, W_ref = r["S"], r["win"]
        for b in range(B):
            Sg, Wg = read_object(pool, inter[j, b], H, d, dtype)
            for h in range(H):
                assert_close(og[j, b, h], r["o"][b, h], tol, f"draft {j} o req {b} head {h}",
                             name="speculative verify, fused kernel (bf16)")
                assert_close(Sg[h], S_ref[b, h], tol, f"draft {j} state req {b} head {h}",
                             name="speculative verify, fused kernel (bf16)")
            assert np.array_equal(Wg, W_ref[b])
    # the same drafts as K chained ping-pong decode steps
    dt = kda.DTYPES[dtype]
    P = inter.shape[2]
    chain = kda.kda_page_alloc(pool, K * B * P).reshape(K, B, P)
    oc = torch.full_like(o, float("nan"))
    prev = torch.from_numpy(src).to(DEV)
    for j in range(K):
        cur = torch.from_numpy(chain[j]).to(DEV)
        kda.kda_decode_step_pp(pool, dv["q"][j], dv["k"][j], dv["v"][j], dv["alpha"][j], dv["beta"][j],
                               conv_w.to(DEV), oc[j], prev, cur, st)
        prev = cur
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    ocg = oc.float().cpu().numpy()
    for j in range(K):
        for b in range(B):
            Sf, Wf = read_object(pool, inter[j, b], H, d, dtype)
            Sc, Wc = read_object(pool, chain[j, b], H, d, dtype)
            for h in range(H):
                assert_close(og[j, b, h], ocg[j, b, h], tol, f"fused vs chained o draft {j} req {b} head {h}")
                assert_close(Sf[h], Sc[h], tol, f"fused vs chained state draft {j} req {b} head {h}")
            assert np.array_equal(Wf, Wc)


def test_verify_fused_bad_page_id_skips_only_that_request():
    dtype, d, B, H, K = "bf16", 128, 40, 4, 4
    pool, src, inter, steps, dv, conv_w, o, st, S0, W0 = _verify_case(B, H, K, 90, bad_request=7)
    rc, bits = kda.kda_sync_status(st)
    assert rc == kda.KDA_EDEVICE and bits & kda.KDA_DEV_BAD_PAGE
    og = o.float().cpu().numpy()
    assert np.all(np.isnan(og[:, 7]))                      # the request was skipped, nothing written
    r = oracle.kda_run(steps[0]["q"], steps[0]["k"], steps[0]["v"], steps[0]["alpha"], steps[0]["beta"], conv_w,
                       np.arange(B + 1), S0=S0, win0=W0)
    for b in (0, 6, 8, B - 1):
        for h in range(H):
            assert_close(og[0, b, h], r["o"][b, h], TOL[dtype], f"draft 0 o req {b} head {h}")


def test_verify_beyond_fused_limit_runs_chained():
    """K above the fused kernel's limit (8) runs as chained decode steps; still exact per token."""
    dtype, d, B, H, K = "bf16", 128, 3, 2, 9
    pool, src, inter, steps, dv, conv_w, o, st, S0, W0 = _verify_case(B, H, K, 95)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    og = o.float().cpu().numpy()
    S_ref, W_ref = S0.copy(), W0.copy()
    for j in range(K):
        t = steps[j]
        r = oracle.kda_run(t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, np.arange(B + 1),
                           S0=S_ref, win0=W_ref)
        S_ref, W_ref = r["S"], r["win"]
        for b in range(B):
            Sg, _ = read_object(pool, inter[j, b], H, d, dtype)
            for h in range(H):
                assert_close(og[j, b, h], r["o"][b, h], TOL[dtype], f"draft {j} o req {b} head {h}",
                             name="speculative verify, chained decode steps (bf16)")
                assert_close(Sg[h], S_ref[b, h], TOL[dtype], f"draft {j} state req {b} head {h}",
                             name="speculative verify, chained decode steps (bf16)")
