"""GPU parity of the ping-pong decode step (kda_decode_step_pp) and of decode-interval
checkpoints taken by donation: an out-of-place step equals the in-place step bit for bit and
leaves its source object untouched; over a run, every donated object holds the state at its
position, as the oracle computes it token by token."""
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


@pytest.mark.parametrize("dtype,d,page_bytes", [("bf16", 128, 65536), ("bf16", 128, 262144), ("f32", 64, 4096)])
def test_out_of_place_step_equals_in_place_and_keeps_the_source(dtype, d, page_bytes):
    dt = kda.DTYPES[dtype]
    B, H = 5, 3
    P = policy.object_pages(H, d, dtype, page_bytes)
    pool = kda.Pool(page_bytes, 3 * B * P + 8, DEV)
    src = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    twin = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    dst = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    g = torch.Generator().manual_seed(31 + d)
    nb = policy.object_bytes(H, d, dtype)
    before = []
    for b in range(B):
        S, W = random_state(H, d, dtype, g)
        write_object(pool, src[b], S, W, dtype)
        write_object(pool, twin[b], S, W, dtype)
        before.append(read_object_bytes(pool, src[b], nb))
    conv_w = (torch.randn(H, 3 * d, 4, generator=g) * 0.5).to(DEV)
    t = workloads.decode_step_tokens(B, H, d, dtype, 31, 0, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o_in = torch.full_like(t["q"], float("nan"))
    o_pp = torch.full_like(t["q"], float("nan"))
    kda.kda_decode_step(pool, t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, o_in,
                        torch.from_numpy(twin).to(DEV), st)
    kda.kda_decode_step_pp(pool, t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, o_pp,
                           torch.from_numpy(src).to(DEV), torch.from_numpy(dst).to(DEV), st)
    rc, bits = kda.kda_sync_status(st)
    assert rc == kda.KDA_OK, bits
    assert torch.equal(o_in, o_pp)
    for b in range(B):
        assert read_object_bytes(pool, dst[b], nb) == read_object_bytes(pool, twin[b], nb)
        assert read_object_bytes(pool, src[b], nb) == before[b]


def test_decode_interval_checkpoints_by_donation_match_the_oracle():
    """Requests at different positions decode 9 tokens with a checkpoint interval of 4: each
    due step donates the request's old object, which must hold the state at that position."""
    dtype, d, H, B, steps, interval = "bf16", 128, 2, 4, 9, 4
    dt = kda.DTYPES[dtype]
    page_bytes = 65536
    P = policy.object_pages(H, d, dtype, page_bytes)
    pool = kda.Pool(page_bytes, B * P * (2 + steps) + 8, DEV)
    act = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    g = torch.Generator().manual_seed(41)
    S0 = np.zeros((B, H, d, d))
    W0 = np.zeros((B, H, 3, 3 * d))
    for b in range(B):
        S0[b], W0[b] = random_state(H, d, dtype, g)
        write_object(pool, act[b], S0[b], W0[b], dtype)
    conv_w = torch.randn(H, 3 * d, 4, generator=g) * 0.5
    pos = [1, 2, 3, 4]                         # tokens already consumed by each request
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    donated = []                               # (request, position, pages)
    toks = []
    for step in range(steps):
        t = workloads.decode_step_tokens(B, H, d, dtype, 41, step, "cpu")
        toks.append(t)
        dst, due = kda.kda_decode_pingpong_plan(pool, H, d, dt, pos, interval, act)
        assert list(due) == [r for r in range(B) if policy.decode_ckpt_due(pos[r], interval)]
        dv = {k: v.to(DEV) for k, v in t.items()}
        o = torch.empty_like(dv["q"])
        kda.kda_decode_step_pp(pool, dv["q"], dv["k"], dv["v"], dv["alpha"], dv["beta"], conv_w.to(DEV), o,
                               torch.from_numpy(act).to(DEV), torch.from_numpy(dst).to(DEV), st)
        rc, bits = kda.kda_sync_status(st)
        assert rc == kda.KDA_OK, bits
        for r in due:
            donated.append((r, pos[r], act[r].copy()))
        act = dst
        pos = [p + 1 for p in pos]
    assert len(donated) == 9                   # positions 4, 8 for requests 0-2; 4, 8, 12 for request 3
    # oracle: each request token by token from its initial state
    for r in range(B):
        S, W = S0[r][None], W0[r][None]
        states = {}
        p = [1, 2, 3, 4][r]
        for step in range(steps):
            if policy.decode_ckpt_due(p, interval):
                states[p] = (S[0].copy(), W[0].copy())
            t = toks[step]
            sl = slice(r, r + 1)
            res = oracle.kda_run(t["q"][sl], t["k"][sl], t["v"][sl], t["alpha"][sl], t["beta"][sl], conv_w,
                                 [0, 1], S0=S, win0=W)
            S, W = res["S"], res["win"]
            p += 1
        for (rr, pp, pages) in donated:
            if rr != r:
                continue
            Sg, Wg = read_object(pool, pages, H, d, dtype)
            Sref, Wref = states[pp]
            for h in range(H):
                assert_close(Sg[h], Sref[h], TOL[dtype], f"checkpoint req {r} pos {pp} head {h}",
                             name=f"ping-pong decode checkpoints ({dtype})")
            assert np.array_equal(Wg, Wref), f"window req {r} pos {pp}"
        Sg, Wg = read_object(pool, act[r], H, d, dtype)
        for h in range(H):
            assert_close(Sg[h], S[0, h], TOL[dtype], f"final req {r} head {h}",
                         name=f"ping-pong decode checkpoints ({dtype})")
        assert np.array_equal(Wg, W[0])
