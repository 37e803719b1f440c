"""GPU parity of kda_prefill_varlen (through the C ABI) against the fp64 oracle: outputs,
final states and windows, checkpoint states and windows, checkpoint positions and pages,
for single sequences that span several chunks with ragged ends, varlen batches with
restored states and unaligned starts, resume from every 512 boundary, and bit-exact
layout pins."""
import numpy as np
import pytest
import torch

import kda_state_chunked_gb300 as kda
from kda_state_chunked_gb300 import workloads
from oracle import policy

from kda_cases import (Prefill, TOL, assert_close, compare_prefill, oracle_positions, oracle_prefill,
                       random_state, read_object, read_object_bytes, write_object)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _toks(T, H, d, dtype, seed):
    t = workloads.make_tokens(T, H, d, dtype, seed, "cpu")
    return t, {k: v.to(DEV) for k, v in t.items()}


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
@pytest.mark.parametrize("T", [1, 15, 16, 63, 64, 65, 511, 512, 513, 2055])
def test_single_sequence(dtype, d, T):
    H = 2
    cpu, dev = _toks(T, H, d, dtype, 100 + T)
    pool = kda.Pool(65536, 256, DEV)
    P = pool.object_pages(H, d, kda.DTYPES[dtype])
    act = kda.kda_page_alloc(pool, P).reshape(1, P)
    cu, sp = [0, T], [0]
    run = Prefill(pool, dev, cu, sp, [0], act, stride=1, include_last=True)
    ck = oracle_positions(cu, sp, 1, True)
    ref = oracle_prefill(cpu, cu, sp, ckpt_abs=ck)
    compare_prefill(pool, run, ref, cu, act, dtype, ck, name=f"prefill cases ({dtype})")


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_varlen_batch_with_restored_states(dtype, d):
    H = 3
    lens = [700, 1, 64, 1500, 333, 0, 2100]
    starts = [0, 512, 1024, 96, 2048 + 37, 4096, 5]
    init = [0, 1, 1, 1, 1, 1, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cpu, dev = _toks(int(cu[-1]), H, d, dtype, 7)
    pool = kda.Pool(65536, 512, DEV)
    P = pool.object_pages(H, d, kda.DTYPES[dtype])
    act = kda.kda_page_alloc(pool, len(lens) * P).reshape(len(lens), P)
    g = torch.Generator().manual_seed(3)
    S0 = np.zeros((len(lens), H, d, d))
    W0 = np.zeros((len(lens), H, 3, 3 * d))
    for s in range(len(lens)):
        if init[s]:
            S0[s], W0[s] = random_state(H, d, dtype, g)
            write_object(pool, act[s], S0[s], W0[s], dtype)
    run = Prefill(pool, dev, cu, starts, init, act, stride=2, include_last=True)
    ck = oracle_positions(cu, starts, 2, True)
    ref = oracle_prefill(cpu, cu, starts, S0=S0, win0=W0, ckpt_abs=ck)
    compare_prefill(pool, run, ref, cu, act, dtype, ck, name=f"prefill cases ({dtype})")


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_resume_from_every_512_boundary(dtype, d):
    """Restore each stored checkpoint into a fresh private object and prefill the rest: the
    result equals the uninterrupted run (and the oracle)."""
    H, T = 2, 2048 + 100
    cpu, dev = _toks(T, H, d, dtype, 21)
    pool = kda.Pool(65536, 1024, DEV)
    dt = kda.DTYPES[dtype]
    P = pool.object_pages(H, d, dt)
    act = kda.kda_page_alloc(pool, P).reshape(1, P)
    full = Prefill(pool, dev, [0, T], [0], [0], act, stride=1, include_last=False)
    assert list(full.pos) == [512, 1024, 1536, 2048]
    ref_full = oracle_prefill(cpu, [0, T], [0])
    S_full, W_full = read_object(pool, act[0], H, d, dtype)
    ws = torch.empty(kda.kda_copy_workspace_bytes(1, P), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    for n, B in enumerate(full.pos):
        B = int(B)
        act2 = kda.kda_page_alloc(pool, P).reshape(1, P)
        kda.kda_ckpt_restore(pool, H, d, dt, full.pages[n], act2, ws, st)
        assert kda.kda_page_refcount(pool, int(full.pages[n][0])) == 2
        assert kda.kda_sync_status(st)[0] == kda.KDA_OK
        kda.kda_ckpt_release(pool, full.pages[n], P)
        assert kda.kda_page_refcount(pool, int(full.pages[n][0])) == 1
        # the restore is a byte copy of the checkpoint
        nb = policy.object_bytes(H, d, dtype)
        assert read_object_bytes(pool, act2[0], nb) == read_object_bytes(pool, full.pages[n], nb)
        sub = {k: (v[B:] if k != "conv_w" else v) for k, v in dev.items()}
        part = Prefill(pool, sub, [0, T - B], [B], [1], act2, stride=1, include_last=False)
        o_full = full.o[B:].float().cpu().numpy()
        o_part = part.o.float().cpu().numpy()
        S_p, W_p = read_object(pool, act2[0], H, d, dtype)
        for h in range(H):
            assert_close(o_part[:, h], o_full[:, h], TOL[dtype], f"resume {B} o head {h}")
            assert_close(o_part[:, h], ref_full["o"][B:, h], TOL[dtype], f"resume {B} o vs oracle",
                         name=f"prefill cases ({dtype})")
            assert_close(S_p[h], S_full[h], TOL[dtype], f"resume {B} S head {h}")
        assert np.array_equal(W_p, W_full)
        # checkpoints after B agree in position with the uninterrupted run
        assert [int(p) for p in part.pos] == [int(p) for p in full.pos if p > B]
        kda.kda_page_decref(pool, part.pages.reshape(-1))
        kda.kda_page_decref(pool, act2.reshape(-1))


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_identity_tokens_keep_state_bytes(dtype, d):
    """alpha = 1 and beta = 0: every checkpoint holds exactly the packed initial state."""
    H, T = 2, 1100
    cpu, dev = _toks(T, H, d, dtype, 33)
    dev["alpha"].fill_(1.0)
    dev["beta"].zero_()
    pool = kda.Pool(65536, 256, DEV)
    P = pool.object_pages(H, d, kda.DTYPES[dtype])
    act = kda.kda_page_alloc(pool, P).reshape(1, P)
    S0, W0 = random_state(H, d, dtype, torch.Generator().manual_seed(5))
    write_object(pool, act[0], S0, W0, dtype)
    run = Prefill(pool, dev, [0, T], [0], [1], act, stride=1, include_last=True)
    nS = d * d * 4
    R = policy.record_bytes(d, dtype)
    want = policy.pack_object(S0, W0, dtype)
    for n in range(len(run.pos)):
        got = read_object_bytes(pool, run.pages[n], len(want))
        for h in range(H):
            assert got[h * R:h * R + nS] == want[h * R:h * R + nS], f"S bytes ckpt {n} head {h}"
    got = read_object_bytes(pool, act[0], len(want))
    for h in range(H):
        assert got[h * R:h * R + nS] == want[h * R:h * R + nS]
    # the windows hold the raw tokens exactly
    _, W = read_object(pool, act[0], H, d, dtype)
    raw = torch.cat([cpu["q"], cpu["k"], cpu["v"]], -1)[-3:].double().numpy().transpose(1, 0, 2)
    assert np.array_equal(W, raw)


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_basis_keys_store_values_exactly(dtype, d):
    """alpha = 1, beta = 1, distinct standard-basis keys, zero state, identity conv:
    S^T e_i returns v_i bit for bit."""
    H, T = 1, d
    cpu, dev = _toks(T, H, d, dtype, 44)
    perm = torch.randperm(d, generator=torch.Generator().manual_seed(9))
    k = torch.zeros(T, H, d)
    k[torch.arange(T), 0, perm[:T]] = 1.0
    dev["k"] = k.to(dev["k"].dtype).to(DEV)
    dev["alpha"].fill_(1.0)
    dev["beta"].fill_(1.0)
    w = torch.zeros(H, 3 * d, 4)
    w[..., 3] = 1.0
    dev["conv_w"] = w.to(DEV)
    pool = kda.Pool(65536, 64, DEV)
    P = pool.object_pages(H, d, kda.DTYPES[dtype])
    act = kda.kda_page_alloc(pool, P).reshape(1, P)
    Prefill(pool, dev, [0, T], [0], [0], act, stride=1, include_last=False)
    S, _ = read_object(pool, act[0], H, d, dtype)
    v = dev["v"].double().cpu().numpy()
    for t in range(T):
        assert np.array_equal(S[0][int(perm[t])], v[t, 0]), f"token {t}"


def test_bad_checkpoint_page_is_reported_not_faulted():
    """A checkpoint page id that the pool does not hold is rejected on the host."""
    H, d, T = 2, 64, 600
    _, dev = _toks(T, H, d, "f32", 55)
    pool = kda.Pool(65536, 16, DEV)
    P = pool.object_pages(H, d, kda.KDA_F32)
    act = kda.kda_page_alloc(pool, P).reshape(1, P)
    ws = torch.empty(4096, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = torch.empty_like(dev["q"])
    with pytest.raises(kda.KdaError) as e:
        kda.kda_prefill_varlen(pool, [0, T], [0], [0], dev["q"], dev["k"], dev["v"], dev["alpha"],
                               dev["beta"], dev["conv_w"], o, act, [0], [512], [[99]], ws, st)
    assert e.value.code == kda.KDA_EINVAL


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_decay_outside_the_factored_range_is_reported(dtype, d):
    """A forget gate of exactly 0 (a full reset of one key channel) puts its chunk's decay
    product below the 2^-100 the chunked kernels factor exactly: the call reports
    KDA_DEV_RANGE, and the (sequence, head) pairs it does not touch still match the oracle.
    A strong decay inside the range (a gate of about 0.377 over a whole chunk, product about
    2^-90) reports nothing and matches the oracle everywhere."""
    H, lens = 2, [300, 200]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    starts = [0, 0]
    cpu, dev = _toks(int(cu[-1]), H, d, dtype, 41)
    pool = kda.Pool(65536, 256, DEV)
    P = pool.object_pages(H, d, kda.DTYPES[dtype])

    # a gate of 0 in sequence 0, head 1, channel 5, token 70 (its second chunk)
    cz, dz = {k: v.clone() for k, v in cpu.items()}, {k: v.clone() for k, v in dev.items()}
    cz["alpha"][70, 1, 5] = 0.0
    dz["alpha"][70, 1, 5] = 0.0
    act = kda.kda_page_alloc(pool, 2 * P).reshape(2, P)
    ws = kda.prefill_workspace(dz["q"], cu, starts, 0, P)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    o = torch.full_like(dz["q"], float("nan"))
    kda.kda_prefill_varlen(pool, cu, starts, [0, 0], dz["q"], dz["k"], dz["v"], dz["alpha"], dz["beta"],
                           dz["conv_w"], o, act, workspace=ws, status=st)
    rc, bits = kda.kda_sync_status(st)
    assert rc == kda.KDA_EDEVICE and bits == kda.KDA_DEV_RANGE
    ref = oracle_prefill(cz, cu, starts)
    on = o.float().cpu().numpy()
    for s, h in ((0, 0), (1, 0), (1, 1)):
        a, b = int(cu[s]), int(cu[s + 1])
        assert_close(on[a:b, h], ref["o"][a:b, h], TOL[dtype], f"gate 0: o seq {s} head {h}")
        S, W = read_object(pool, act[s], H, d, dtype)
        assert_close(S[h], ref["S"][s, h], TOL[dtype], f"gate 0: final S seq {s} head {h}")
    kda.kda_page_decref(pool, act.reshape(-1))

    # the same channel decaying by 0.377 per token over the whole second chunk
    g = torch.tensor(0.377).to(cpu["alpha"].dtype)
    cs, ds = {k: v.clone() for k, v in cpu.items()}, {k: v.clone() for k, v in dev.items()}
    cs["alpha"][64:128, 1, 5] = g
    ds["alpha"][64:128, 1, 5] = g.to(DEV)
    assert float(g) ** 64 > 2.0 ** -100
    act = kda.kda_page_alloc(pool, 2 * P).reshape(2, P)
    run = Prefill(pool, ds, cu, starts, [0, 0], act, stride=1, include_last=True)
    ck = oracle_positions(cu, starts, 1, True)
    ref = oracle_prefill(cs, cu, starts, ckpt_abs=ck)
    compare_prefill(pool, run, ref, cu, act, dtype, ck, name=f"prefill cases ({dtype})")


@pytest.mark.parametrize("dtype,d", [("f32", 64), ("bf16", 128)])
def test_scattered_pages_of_a_non_power_of_two_size(dtype, d):
    """Pages of 19 x 256 bytes, every object's pages three ids apart in a fragmented pool: page
    translation without a power-of-two shift, and state records that cross non-adjacent pages
    (the kernels' contiguous-run fast path cannot apply)."""
    H = 3
    lens = [700, 1, 64, 1500, 333, 0, 2100]
    starts = [0, 512, 1024, 96, 2048 + 37, 4096, 5]
    init = [0, 1, 1, 1, 1, 1, 1]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cpu, dev = _toks(int(cu[-1]), H, d, dtype, 17)
    page_bytes = 19 * 256
    pool = kda.Pool(page_bytes, 3000, DEV)
    held = kda.kda_page_alloc(pool, 3000)
    kda.kda_page_decref(pool, held[1::3])          # later allocations get ids 1, 4, 7, ...
    P = pool.object_pages(H, d, kda.DTYPES[dtype])
    act = kda.kda_page_alloc(pool, len(lens) * P).reshape(len(lens), P)
    assert np.all(np.diff(act.reshape(-1)) == 3)
    g = torch.Generator().manual_seed(19)
    S0 = np.zeros((len(lens), H, d, d))
    W0 = np.zeros((len(lens), H, 3, 3 * d))
    for s in range(len(lens)):
        if init[s]:
            S0[s], W0[s] = random_state(H, d, dtype, g)
            write_object(pool, act[s], S0[s], W0[s], dtype)
    run = Prefill(pool, dev, cu, starts, init, act, stride=2, include_last=True)
    ck = oracle_positions(cu, starts, 2, True)
    ref = oracle_prefill(cpu, cu, starts, S0=S0, win0=W0, ckpt_abs=ck)
    compare_prefill(pool, run, ref, cu, act, dtype, ck, name=f"prefill cases ({dtype})")
