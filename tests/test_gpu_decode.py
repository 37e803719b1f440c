"""GPU parity of kda_decode_step and of the checkpoint copies (through the C ABI)."""
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


def _decode_case(dtype, d, B, H, steps, page_bytes, seed):
    dt = kda.DTYPES[dtype]
    P = policy.object_pages(H, d, dtype, page_bytes)
    pool = kda.Pool(page_bytes, B * P + 16, DEV)
    assert pool.object_pages(H, d, dt) == P
    # a scattered page table: claim pages in a seeded order
    table = workloads.permuted_page_table(pool.num_pages, B, P, seed)
    kda.kda_page_claim(pool, table.reshape(-1))
    g = torch.Generator().manual_seed(seed)
    S0 = np.zeros((B, H, d, d))
    W0 = np.zeros((B, H, 3, 3 * d))
    for b in range(B):
        S0[b], W0[b] = random_state(H, d, dtype, g)
        write_object(pool, table[b], S0[b], W0[b], dtype)
    conv_w = (torch.randn(H, 3 * d, 4, generator=g) * 0.5)
    pages_dev = table.to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    S_ref, W_ref = S0.copy(), W0.copy()
    for step in range(steps):
        t = workloads.decode_step_tokens(B, H, d, dtype, seed, step, "cpu")
        dev = {k: v.to(DEV) for k, v in t.items()}
        o = torch.full_like(dev["q"], float("nan"))
        kda.kda_decode_step(pool, dev["q"], dev["k"], dev["v"], dev["alpha"], dev["beta"],
                            conv_w.to(DEV), o, pages_dev, st)
        rc, bits = kda.kda_sync_status(st)
        assert rc == kda.KDA_OK, bits
        # oracle: one token per request from the reference state
        cu = np.arange(B + 1)
        r = oracle.kda_run(t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, cu,
                           S0=S_ref, win0=W_ref)
        S_ref, W_ref = r["S"], r["win"]
        og = o.float().cpu().numpy()
        for b in range(B):
            for h in range(H):
                assert_close(og[b, h], r["o"][b, h], TOL[dtype], f"step {step} o req {b} head {h}",
                             name=f"decode cases ({dtype})")
    for b in range(B):
        S, W = read_object(pool, table[b], H, d, dtype)
        for h in range(H):
            assert_close(S[h], S_ref[b, h], TOL[dtype], f"final S req {b} head {h}", name=f"decode cases ({dtype})")
        assert np.array_equal(W, W_ref[b])


@pytest.mark.parametrize("dtype,d,page_bytes", [("f32", 64, 65536), ("bf16", 128, 262144),
                                                ("bf16", 128, 65536), ("bf16", 128, 260 * 256),
                                                ("f32", 128, 4096), ("bf16", 128, 19 * 256)])
def test_decode_steps_match_oracle(dtype, d, page_bytes):
    _decode_case(dtype, d, B=6, H=3, steps=5, page_bytes=page_bytes, seed=70 + d)


def test_decode_bad_page_sets_status_and_skips():
    dtype, d, H, B = "bf16", 128, 2, 3
    dt = kda.DTYPES[dtype]
    pool = kda.Pool(65536, 64, DEV)
    P = pool.object_pages(H, d, dt)
    table = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    g = torch.Generator().manual_seed(1)
    S0, W0 = random_state(H, d, dtype, g)
    for b in range(B):
        write_object(pool, table[b], S0, W0, dtype)
    bad = table.copy()
    bad[1, 0] = 1000   # outside the pool: the kernel must skip request 1
    t = workloads.decode_step_tokens(B, H, d, dtype, 5, 0, DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = torch.zeros_like(t["q"])
    kda.kda_decode_step(pool, t["q"], t["k"], t["v"], t["alpha"], t["beta"],
                        torch.zeros(H, 3 * d, 4, device=DEV), o, torch.from_numpy(bad).to(DEV), st)
    rc, bits = kda.kda_sync_status(st)
    assert rc == kda.KDA_EDEVICE and bits & kda.KDA_DEV_BAD_PAGE
    S1, W1 = read_object(pool, table[1], H, d, dtype)
    assert np.array_equal(S1, S0.astype(np.float32).astype(np.float64)) and np.array_equal(W1, W0)
    # the status word was cleared by the sync
    assert kda.kda_sync_status(st) == (kda.KDA_OK, 0)


@pytest.mark.parametrize("dtype,d,H,page_bytes", [("bf16", 128, 32, 65536), ("f32", 64, 2, 4096),
                                                  ("bf16", 128, 5, 262144)])
def test_checkpoint_write_and_restore_are_byte_copies(dtype, d, H, page_bytes):
    dt = kda.DTYPES[dtype]
    pool = kda.Pool(page_bytes, 600, DEV)
    P = pool.object_pages(H, d, dt)
    n = 3
    nb = policy.object_bytes(H, d, dtype)
    src = kda.kda_page_alloc(pool, n * P).reshape(n, P)
    # fill whole pages with random bytes, object tails included
    g = torch.Generator(device=DEV).manual_seed(2)
    for p in src.reshape(-1):
        pool.page_view(int(p)).copy_(torch.randint(0, 256, (page_bytes,), generator=g, device=DEV,
                                                   dtype=torch.int32).to(torch.uint8))
    ws = torch.empty(kda.kda_copy_workspace_bytes(n, P), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    free0 = pool.free_count()
    dst = kda.kda_ckpt_write(pool, H, d, dt, src.reshape(-1), ws, st)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    assert pool.free_count() == free0 - n * P
    for i in range(n):
        assert read_object_bytes(pool, dst[i], nb) == read_object_bytes(pool, src[i], nb)
    act = kda.kda_page_alloc(pool, n * P).reshape(n, P)
    kda.kda_ckpt_restore(pool, H, d, dt, dst.reshape(-1), act.reshape(-1), ws, st)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    kda.kda_ckpt_release(pool, dst.reshape(-1), P)
    for i in range(n):
        assert read_object_bytes(pool, act[i], nb) == read_object_bytes(pool, src[i], nb)
    # restore onto a shared page is refused; the checkpoint stays read-only
    with pytest.raises(kda.KdaError) as e:
        kda.kda_ckpt_restore(pool, H, d, dt, dst[0], dst[0], ws, st)
    assert e.value.code == kda.KDA_EREF
