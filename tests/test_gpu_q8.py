"""GPU parity of the INT8 compressed checkpoints (kda_ckpt_write_q8 / kda_ckpt_restore_q8)
against the oracle codec: bit-exact codes, scales, windows and padding; a dequantised restore
that a decode step and a prefill continue from."""
import numpy as np
import pytest
import torch

import kda_state_chunked_gb300 as kda
from kda_state_chunked_gb300 import workloads
import oracle
from oracle import policy, q8

from kda_cases import TOL, assert_close, random_state, read_object, read_object_bytes, write_object

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _objects(pool, n, H, d, dtype, seed, scale=0.3):
    dt = kda.DTYPES[dtype]
    P = pool.object_pages(H, d, dt)
    pages = kda.kda_page_alloc(pool, n * P).reshape(n, P)
    g = torch.Generator().manual_seed(seed)
    S = np.zeros((n, H, d, d))
    W = np.zeros((n, H, 3, 3 * d))
    for i in range(n):
        S[i], W[i] = random_state(H, d, dtype, g, scale)
        S[i, :, 3] = 0.0                                   # a zero row: scale 0, codes 0
        S[i, 0, 5] *= 1e-30                                # a row of tiny values
        write_object(pool, pages[i], S[i], W[i], dtype)
    return pages, S.astype(np.float32).astype(np.float64), W


@pytest.mark.parametrize("dtype,d,H,page_bytes", [("bf16", 128, 3, 65536), ("bf16", 128, 32, 65536),
                                                  ("bf16", 128, 5, 19 * 256),   # pipeline, 70-page lists
                                                  ("f32", 64, 2, 4096), ("bf16", 64, 5, 768)])
def test_write_q8_is_the_oracle_codec_bit_for_bit(dtype, d, H, page_bytes):
    dt = kda.DTYPES[dtype]
    n = 3
    P = policy.object_pages(H, d, dtype, page_bytes)
    Pq = q8.object_pages(H, d, dtype, page_bytes)
    pool = kda.Pool(page_bytes, n * (P + Pq) + 8, DEV)
    src, S, W = _objects(pool, n, H, d, dtype, seed=11 + d + H)
    ws = torch.empty(kda.kda_copy_workspace_bytes(n, P), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dst = kda.kda_ckpt_write_q8(pool, H, d, dt, src.reshape(-1), ws, st)
    assert dst.shape == (n, Pq)
    rc, bits = kda.kda_sync_status(st)
    assert rc == kda.KDA_OK, bits
    nb = q8.object_bytes(H, d, dtype)
    for i in range(n):
        got = read_object_bytes(pool, dst[i], nb)
        assert got == q8.pack_object(S[i], W[i], dtype), f"object {i}"
    # the source objects are untouched
    for i in range(n):
        Si, Wi = read_object(pool, src[i], H, d, dtype)
        assert np.array_equal(Si, S[i]) and np.array_equal(Wi, W[i])


@pytest.mark.parametrize("dtype,d,H,page_bytes", [("bf16", 128, 4, 65536), ("bf16", 128, 5, 19 * 256),
                                                  ("f32", 64, 3, 4096), ("bf16", 64, 5, 768)])
def test_restore_q8_dequantises_bit_for_bit(dtype, d, H, page_bytes):
    dt = kda.DTYPES[dtype]
    n = 2
    P = policy.object_pages(H, d, dtype, page_bytes)
    Pq = q8.object_pages(H, d, dtype, page_bytes)
    pool = kda.Pool(page_bytes, n * (2 * P + Pq) + 8, DEV)
    src, S, W = _objects(pool, n, H, d, dtype, seed=23 + d)
    ws = torch.empty(kda.kda_copy_workspace_bytes(n, P), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ck = kda.kda_ckpt_write_q8(pool, H, d, dt, src.reshape(-1), ws, st)
    act = kda.kda_page_alloc(pool, n * P).reshape(n, P)
    # fill the private objects with garbage first: the restore must overwrite every byte
    for p in act.reshape(-1):
        pool.page_view(int(p)).fill_(0xA5)
    kda.kda_ckpt_restore_q8(pool, H, d, dt, ck.reshape(-1), act.reshape(-1), ws, st)
    rc, bits = kda.kda_sync_status(st)
    assert rc == kda.KDA_OK, bits
    kda.kda_ckpt_release(pool, ck.reshape(-1), Pq)
    nb = policy.object_bytes(H, d, dtype)
    for i in range(n):
        want = [q8.dequantize(*q8.quantize(S[i, h])) for h in range(H)]
        expect = policy.pack_object(np.stack(want).astype(np.float64), W[i], dtype)
        assert read_object_bytes(pool, act[i], nb) == expect, f"object {i}"
        # within half a quantisation step of the original state
        for h in range(H):
            sc, _ = q8.quantize(S[i, h])
            err = np.abs(want[h].astype(np.float64) - S[i, h])
            assert np.all(err <= sc[:, None] * 0.5 + np.abs(S[i, h]) * 2.0 ** -22)
    # the checkpoint pages keep their reference after the release (refcount 1 from the write)
    assert all(kda.kda_page_refcount(pool, int(p)) == 1 for p in ck.reshape(-1))


def test_decode_continues_from_an_int8_restore():
    """Snapshot to INT8, restore into a fresh private object, take decode steps: the result
    equals the oracle run from the dequantised state."""
    dtype, d, H, B, steps = "bf16", 128, 4, 3, 3
    dt = kda.DTYPES[dtype]
    page_bytes = 262144
    P = policy.object_pages(H, d, dtype, page_bytes)
    Pq = q8.object_pages(H, d, dtype, page_bytes)
    pool = kda.Pool(page_bytes, B * (2 * P + Pq) + 8, DEV)
    src, S, W = _objects(pool, B, H, d, dtype, seed=5)
    ws = torch.empty(kda.kda_copy_workspace_bytes(B, P), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    ck = kda.kda_ckpt_write_q8(pool, H, d, dt, src.reshape(-1), ws, st)
    act = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    kda.kda_ckpt_restore_q8(pool, H, d, dt, ck.reshape(-1), act.reshape(-1), ws, st)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    S_ref = np.stack([[q8.dequantize(*q8.quantize(S[b, h])) for h in range(H)] for b in range(B)]).astype(np.float64)
    W_ref = W.copy()
    g = torch.Generator().manual_seed(9)
    conv_w = torch.randn(H, 3 * d, 4, generator=g) * 0.5
    pages_dev = torch.from_numpy(act).to(DEV)
    for step in range(steps):
        t = workloads.decode_step_tokens(B, H, d, dtype, 9, step, "cpu")
        dv = {k: v.to(DEV) for k, v in t.items()}
        o = torch.full_like(dv["q"], float("nan"))
        kda.kda_decode_step(pool, dv["q"], dv["k"], dv["v"], dv["alpha"], dv["beta"], conv_w.to(DEV), o,
                            pages_dev, st)
        assert kda.kda_sync_status(st)[0] == kda.KDA_OK
        r = oracle.kda_run(t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, np.arange(B + 1),
                           S0=S_ref, win0=W_ref)
        S_ref, W_ref = r["S"], r["win"]
        og = o.float().cpu().numpy()
        for b in range(B):
            for h in range(H):
                assert_close(og[b, h], r["o"][b, h], TOL[dtype], f"step {step} o req {b} head {h}",
                             name=f"decode after INT8 restore ({dtype})")
    for b in range(B):
        Sg, Wg = read_object(pool, act[b], H, d, dtype)
        for h in range(H):
            assert_close(Sg[h], S_ref[b, h], TOL[dtype], f"S req {b} head {h}",
                         name=f"decode after INT8 restore ({dtype})")
        assert np.array_equal(Wg, W_ref[b])


def test_int8_restore_refuses_pages_outside_the_pool():
    """Page ids are checked on the host before anything is enqueued (the kernels also skip and
    flag ids outside the pool, as a second line)."""
    dtype, d, H = "bf16", 128, 2
    dt = kda.DTYPES[dtype]
    pool = kda.Pool(65536, 32, DEV)
    P = pool.object_pages(H, d, dt)
    Pq = kda.kda_object_pages_q8(pool, H, d, dt)
    src, S, W = _objects(pool, 1, H, d, dtype, seed=3)
    ws = torch.empty(kda.kda_copy_workspace_bytes(1, P), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    act = kda.kda_page_alloc(pool, P).reshape(1, P)
    free0 = pool.free_count()
    with pytest.raises(kda.KdaError) as e:
        kda.kda_ckpt_restore_q8(pool, H, d, dt, np.full(Pq, 10_000, np.int32), act.reshape(-1), ws, st)
    assert e.value.code == kda.KDA_EINVAL
    assert pool.free_count() == free0
    assert kda.kda_sync_status(st) == (kda.KDA_OK, 0)


def test_write_q8_near_rounding_ties_bit_for_bit():
    """Rows built so that S[i][j] / scale_i lies exactly on, or up to six fp32 steps beside, a
    half-integer, over scales from 1e-30 to 1e30 (the steps straddle the quantiser's 2^-16
    rounding-test band): its fast reciprocal path must take the same integer decisions as the
    IEEE division of the oracle codec on every element."""
    dtype, d, H, page_bytes = "bf16", 128, 4, 65536
    dt = kda.DTYPES[dtype]
    P = policy.object_pages(H, d, dtype, page_bytes)
    Pq = q8.object_pages(H, d, dtype, page_bytes)
    pool = kda.Pool(page_bytes, P + Pq + 8, DEV)
    src = kda.kda_page_alloc(pool, P).reshape(1, P)
    rng = np.random.default_rng(123)
    f32 = np.float32
    S = np.zeros((H, d, d), dtype=f32)
    for h in range(H):
        for i in range(d):
            amax = f32(10.0 ** rng.uniform(-30, 30))
            scale = f32(amax / f32(127))
            row = np.empty(d, dtype=f32)
            row[0] = amax
            k = rng.integers(-126, 126, d - 1).astype(f32)
            base = ((k + f32(0.5)) * scale).astype(f32)
            steps = np.arange(d - 1) % 13 - 6                  # -6 .. 6 fp32 steps away
            for u in range(1, 7):
                base = np.where(steps >= u, np.nextafter(base, f32(np.inf)), base)
                base = np.where(steps <= -u, np.nextafter(base, f32(-np.inf)), base)
            row[1:] = np.clip(base, -amax, amax)
            S[h, i] = rng.permutation(row)
    g = torch.Generator().manual_seed(5)
    _, W = random_state(H, d, dtype, g)
    write_object(pool, src[0], S.astype(np.float64), W, dtype)
    ws = torch.empty(kda.kda_copy_workspace_bytes(1, P), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dst = kda.kda_ckpt_write_q8(pool, H, d, dt, src.reshape(-1), ws, st)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    got = read_object_bytes(pool, dst[0], q8.object_bytes(H, d, dtype))
    assert got == q8.pack_object(S.astype(np.float64), W, dtype)
