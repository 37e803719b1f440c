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


@pytest.mark.parametrize("dtype,d,page_bytes", [("bf16", 128, 65536), ("f32", 64, 4096)])
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
