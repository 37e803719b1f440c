"""CPU tests of libkda.so's host side: the library loads without a GPU, exports every
symbol include/kda.h declares, and its allocator / checkpoint policy / sizes agree bit for
bit with the oracle's independent Python version.  No kernel is launched here."""
import ctypes
import os
import re

import numpy as np
import pytest

import kda_state_chunked_gb300 as kda
from kda_state_chunked_gb300 import build as kbuild
from oracle import policy

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    kbuild.build()


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = _declared_functions()
    assert len(names) >= 20
    L = ctypes.CDLL(kda.library_path())
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # the binding declares a signature for each of them, under the same name
    assert sorted(kda._SIGS) == names
    for n in names:
        assert callable(getattr(kda, n, None)) or n in ("kda_pool_create", "kda_pool_destroy",
                                                       "kda_pool_page_bytes", "kda_pool_num_pages",
                                                       "kda_pool_free_count", "kda_status_string")


def test_header_documents_every_call():
    """Each declaration in include/kda.h sits under a comment: directly, or as part of a run
    of declarations that one comment introduces (no blank line between them)."""
    lines = open(os.path.join(ROOT, "include", "kda.h")).read().splitlines()
    undocumented = []
    for i, ln in enumerate(lines):
        m = re.match(r"^(?:int|int32_t|int64_t|void|const char \*)\s*\**\s*(kda_\w+)\s*\(", ln)
        if not m:
            continue
        j = i - 1
        # walk back over the run of declarations (and their continuation lines) above
        while j >= 0 and lines[j].strip() and not lines[j].rstrip().endswith("*/"):
            j -= 1
        if j < 0 or not lines[j].rstrip().endswith("*/"):
            undocumented.append(m.group(1))
    assert len(_declared_functions()) >= 30
    assert undocumented == []


@pytest.mark.parametrize("H,d,dt", [(16, 128, "bf16"), (32, 128, "bf16"), (2, 64, "f32"),
                                    (3, 64, "bf16"), (5, 128, "f32")])
def test_sizes_match_oracle(H, d, dt):
    assert kda.kda_record_bytes(d, kda.DTYPES[dt]) == policy.record_bytes(d, dt)
    assert kda.kda_object_bytes(H, d, kda.DTYPES[dt]) == policy.object_bytes(H, d, dt)
    for pb in (256, 4096, 65536, 262144):
        pool = kda.Pool(pb, 8)
        assert pool.object_pages(H, d, kda.DTYPES[dt]) == policy.object_pages(H, d, dt, pb)


def test_bad_shapes_rejected():
    L = kda.lib()
    assert L.kda_record_bytes(96, 0) == kda.KDA_EINVAL
    assert L.kda_record_bytes(64, 7) == kda.KDA_EINVAL
    assert L.kda_object_bytes(0, 64, 0) == kda.KDA_EINVAL
    h = ctypes.c_void_p()
    assert L.kda_pool_create(1000, 4, ctypes.byref(h)) == kda.KDA_EINVAL   # not a 256 multiple
    assert L.kda_pool_create(4096, 0, ctypes.byref(h)) == kda.KDA_EINVAL


def test_positions_match_oracle():
    rng = np.random.default_rng(11)
    for _ in range(400):
        start = int(rng.integers(0, 1 << 21))
        end = start + int(rng.integers(0, 50000))
        hb = int(rng.choice([64, 128, 512]))
        stride = int(rng.integers(1, 8))
        last = bool(rng.integers(0, 2))
        assert kda.kda_ckpt_positions(start, end, hb, stride, last) == \
            policy.ckpt_positions(start, end, hb, stride, last)
    assert kda.kda_ckpt_positions(0, 1048576, 512, 4, True)[-1] == 1048576
    # truncated output still reports the full count
    out = np.zeros(2, dtype=np.int64)
    n = kda.lib().kda_ckpt_positions(0, 8192, 512, 1, 0, out.ctypes.data_as(ctypes.c_void_p), 2)
    assert n == 16 and list(out) == [512, 1024]
    assert kda.lib().kda_ckpt_positions(10, 5, 512, 1, 0, None, 0) == kda.KDA_EINVAL


def test_allocator_matches_oracle_under_random_traffic():
    rng = np.random.default_rng(12)
    N = 64
    pool = kda.Pool(4096, N)
    sim = policy.PoolSim(N)
    for _ in range(3000):
        op = int(rng.integers(0, 4))
        if op == 0:
            n = int(rng.integers(0, 9))
            try:
                want = sim.alloc(n)
            except policy.AllocError:
                want = None
            try:
                got = list(kda.kda_page_alloc(pool, n))
            except kda.KdaError as e:
                assert e.code == kda.KDA_ENOPAGES
                got = None
            assert got == want
        else:
            ids = [int(x) for x in rng.integers(0, N, int(rng.integers(1, 4)))]
            fn_sim = {1: sim.claim, 2: sim.incref, 3: sim.decref}[op]
            fn_lib = {1: kda.kda_page_claim, 2: kda.kda_page_incref, 3: kda.kda_page_decref}[op]
            try:
                fn_sim(ids)
                ok_sim = True
            except policy.AllocError:
                ok_sim = False
            try:
                fn_lib(pool, ids)
                ok_lib = True
            except kda.KdaError as e:
                assert e.code in (kda.KDA_EREF, kda.KDA_EINVAL)
                ok_lib = False
            assert ok_lib == ok_sim, (op, ids)
        assert pool.free_count() == sim.free_count()
    assert [kda.kda_page_refcount(pool, i) for i in range(N)] == sim.ref


def test_allocator_error_codes():
    pool = kda.Pool(4096, 8)
    assert list(kda.kda_page_alloc(pool, 3)) == [0, 1, 2]
    with pytest.raises(kda.KdaError) as e:
        kda.kda_page_alloc(pool, 6)
    assert e.value.code == kda.KDA_ENOPAGES and pool.free_count() == 5
    with pytest.raises(kda.KdaError) as e:
        kda.kda_page_decref(pool, [5])
    assert e.value.code == kda.KDA_EREF
    with pytest.raises(kda.KdaError) as e:
        kda.kda_page_claim(pool, [1])
    assert e.value.code == kda.KDA_EREF
    with pytest.raises(kda.KdaError) as e:
        kda.kda_page_claim(pool, [9])
    assert e.value.code == kda.KDA_EINVAL
    with pytest.raises(kda.KdaError) as e:
        kda.kda_page_claim(pool, [4, 4])
    assert e.value.code == kda.KDA_EREF
    assert kda.kda_page_refcount(pool, 4) == 0


@pytest.mark.parametrize("stride,last", [(1, False), (4, True), (2, False)])
def test_plan_matches_oracle(stride, last):
    rng = np.random.default_rng(13 + stride)
    H, d, dt, PB = 4, 64, "bf16", 8192
    P = policy.object_pages(H, d, dt, PB)
    pool = kda.Pool(PB, 4000)
    sim = policy.PoolSim(4000)
    lens = [int(x) for x in rng.integers(0, 5000, 6)]
    starts = [int(512 * x) for x in rng.integers(0, 8, 6)]
    act = kda.kda_page_alloc(pool, 6 * P)
    assert list(act) == sim.alloc(6 * P)
    cu = np.concatenate([[0], np.cumsum(lens)])
    seq, pos, pages = kda.kda_ckpt_plan(pool, H, d, kda.DTYPES[dt], cu, starts, 512, stride, last)
    want = policy.plan_checkpoints(sim, [(s, s + L) for s, L in zip(starts, lens)], P, 512, stride, last)
    assert [(int(a), int(b)) for a, b in zip(seq, pos)] == [(s, p) for s, p, _ in want]
    assert [list(map(int, row)) for row in pages] == [pg for _, _, pg in want]
    assert pool.free_count() == sim.free_count()


def test_plan_all_or_nothing():
    pool = kda.Pool(65536, 10)
    P = pool.object_pages(16, 128, kda.KDA_BF16)   # 17 pages: cannot fit
    with pytest.raises(kda.KdaError) as e:
        kda.kda_ckpt_plan(pool, 16, 128, kda.KDA_BF16, [0, 4096], [0], 512, 4, True)
    assert e.value.code == kda.KDA_ENOPAGES and pool.free_count() == 10 and P == 17


def test_gpu_calls_reject_bad_arguments_before_touching_the_device():
    """Host validation returns KDA_EINVAL without any CUDA call (safe on a CPU machine)."""
    L = kda.lib()
    pool = kda.Pool(65536, 64)
    fake = ctypes.c_void_p(256)
    cu = np.array([0, 10], dtype=np.int32)
    sp = np.array([0], dtype=np.int64)
    hi = np.array([0], dtype=np.uint8)
    act = np.arange(2, dtype=np.int32)
    args = [pool.handle, 2, 64, kda.KDA_F32, 1, kda._ptr(cu), kda._ptr(sp), kda._ptr(hi),
            fake, fake, fake, fake, fake, fake, fake, fake, kda._ptr(act), 0, None, None, None,
            fake, 1 << 20, fake, None]
    # active pages are not allocated -> reference error
    assert L.kda_prefill_varlen(*args) == kda.KDA_EINVAL or L.kda_prefill_varlen(*args) == kda.KDA_EREF
    bad = list(args)
    bad[2] = 96                     # d not supported
    assert L.kda_prefill_varlen(*bad) == kda.KDA_EINVAL
    bad = list(args)
    bad[4] = 0                      # no sequences
    assert L.kda_prefill_varlen(*bad) == kda.KDA_EINVAL
    kda.kda_page_alloc(pool, 1)
    ok = list(args)
    ok[16] = kda._ptr(np.array([0], dtype=np.int32))
    ok[22] = 16                     # workspace too small
    assert L.kda_prefill_varlen(*ok) == kda.KDA_EINVAL
    # checkpoint position not on a chunk boundary
    ck = list(ok)
    ck[22] = 1 << 20
    kda.kda_page_alloc(pool, 1)
    ck[17] = 1
    ck[18] = kda._ptr(np.array([0], dtype=np.int32))
    ck[19] = kda._ptr(np.array([5], dtype=np.int64))
    ck[20] = kda._ptr(np.array([1], dtype=np.int32))
    assert L.kda_prefill_varlen(*ck) == kda.KDA_EINVAL
    # a shared (refcount 2) page may not be written
    kda.kda_page_incref(pool, [0])
    assert L.kda_prefill_varlen(*ok[:22], 1 << 20, *ok[23:]) == kda.KDA_EREF
    assert L.kda_decode_step(pool.handle, 2, 80, 0, 4, *([fake] * 10), None) == kda.KDA_EINVAL
    assert L.kda_ckpt_write(pool.handle, 2, 64, 0, 1, None, None, fake, fake, 0, fake, None) == kda.KDA_EINVAL


def test_split_prefill_plan_launches_and_workspace():
    """bf16 d=128 runs as waves of chunk preparation + chains (the preparation of a wave beside
    the chains of the one before); the host plan decides the wave split, the launch count and
    the operand-image workspace."""
    cu = [0, 8192, 16384, 24576, 32768]
    st = [0, 0, 0, 0]
    bf, f32 = kda.KDA_BF16, kda.KDA_F32
    unit = 82432
    b = kda.kda_prefill_waves(16, 128, bf, cu, st)
    W = len(b) - 1
    # the waves tile the 128 chunks of every chain, each wave's images fit one 512 MiB slot
    assert W >= 2 and b[0] == 0 and b[-1] == 128 and np.all(np.diff(b) > 0)
    assert np.max(np.diff(b)) * 4 * 16 * unit <= 512 << 20
    assert kda.kda_prefill_kernel_launches(16, 128, bf, cu, st) == 2 * W
    assert kda.kda_prefill_kernel_launches(16, 128, f32, cu, st) == 1
    assert kda.kda_prefill_kernel_launches(16, 64, bf, cu, st) == 1
    assert kda.kda_prefill_kernel_launches(16, 128, bf, [0, 0], [5]) == 1     # empty sequence only
    assert len(kda.kda_prefill_waves(16, 128, bf, [0, 0], [5])) == 0
    assert len(kda.kda_prefill_waves(16, 128, f32, cu, st)) == 0
    assert kda.kda_prefill_kernel_launches(2, 128, bf, [0, 100], [0]) == 2     # one wave
    ws = kda.kda_prefill_workspace_bytes(16, 128, bf, cu, st, 16, 17)
    images = 2 * int(np.max(np.diff(b))) * 4 * 16 * unit     # two slots of the largest wave
    scratch = 4 * 16 * 128 * 128 * 4 + 4 * 16 * 9 * 128 * 2
    assert images + scratch <= ws <= images + scratch + (1 << 20)
    # metadata only on the fp32 path
    assert kda.kda_prefill_workspace_bytes(16, 128, f32, cu, st, 16, 17) < (1 << 20)
    with pytest.raises(kda.KdaError):
        kda.kda_prefill_kernel_launches(16, 128, bf, [0, 10, 5], [0, 0])      # decreasing offsets


@pytest.mark.parametrize("H,lens,starts", [
    (32, [65536], [0]),                                  # one long chain per head
    (32, [1 << 20], [0]),                                # the 1M-token sequence: many waves
    (16, [8192, 100, 0, 5000], [0, 30, 7, 64 * 9 + 3]),  # ragged, an empty one, unaligned starts
    (4, [64 * 3 + 1], [63]),
    (32, [20000 + 397 * i for i in range(32)], [512 * (i % 5) for i in range(32)]),   # 1024 chains
])
def test_wave_split_covers_every_chunk_within_the_slot(H, lens, starts):
    """Whatever split the cost model picks: ascending bounds from 0 to the longest chain's
    chunk count, no empty wave, every wave's images (all chains' chunks in it) within one
    slot: 512 MiB while the chains fit on the 152 SMs at once, 2 GiB beyond."""
    bf = kda.KDA_BF16
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    b = kda.kda_prefill_waves(H, 128, bf, cu, starts)
    nch = [0 if n == 0 else (s + n - 1) // 64 - s // 64 + 1 for n, s in zip(lens, starts)]
    assert b[0] == 0 and b[-1] == max(nch) and np.all(np.diff(b) > 0)
    cap = (2048 << 20) if sum(n > 0 for n in nch) * H > 152 else (512 << 20)
    for w in range(len(b) - 1):
        chunks = sum(max(0, min(n, b[w + 1]) - b[w]) for n in nch)
        assert chunks * H * 82432 <= cap
    assert kda.kda_prefill_kernel_launches(H, 128, bf, cu, starts) == 2 * (len(b) - 1)


def test_q8_sizes_match_oracle_and_bad_arguments_are_refused():
    from oracle import q8
    for d, dt in [(128, "bf16"), (64, "f32"), (128, "f32"), (64, "bf16")]:
        assert kda.kda_record_bytes_q8(d, kda.DTYPES[dt]) == q8.record_bytes(d, dt)
        assert kda.kda_object_bytes_q8(5, d, kda.DTYPES[dt]) == q8.object_bytes(5, d, dt)
    pool = kda.Pool(65536, 64)
    assert kda.kda_object_pages_q8(pool, 32, 128, kda.KDA_BF16) == q8.object_pages(32, 128, "bf16", 65536) == 10
    L = kda.lib()
    dummy = ctypes.c_void_p(16)
    ids = np.zeros(64, dtype=np.int32)
    out = np.zeros(64, dtype=np.int32)
    # bad shape, missing buffers, short workspace: refused before anything is enqueued
    assert L.kda_ckpt_write_q8(pool.handle, 2, 96, kda.KDA_BF16, 1, kda._ptr(ids), kda._ptr(out), dummy, dummy,
                               1 << 20, dummy, None) == kda.KDA_EINVAL
    assert L.kda_ckpt_write_q8(pool.handle, 2, 128, kda.KDA_BF16, 1, None, kda._ptr(out), dummy, dummy,
                               1 << 20, dummy, None) == kda.KDA_EINVAL
    assert L.kda_ckpt_write_q8(pool.handle, 2, 128, kda.KDA_BF16, 1, kda._ptr(ids), kda._ptr(out), dummy, dummy,
                               8, dummy, None) == kda.KDA_EINVAL
    # unallocated source pages: refcount error, nothing allocated
    free0 = pool.free_count()
    assert L.kda_ckpt_write_q8(pool.handle, 2, 128, kda.KDA_BF16, 1, kda._ptr(ids), kda._ptr(out), dummy, dummy,
                               1 << 20, dummy, None) == kda.KDA_EREF
    assert pool.free_count() == free0
    # restore onto pages that are not private
    assert L.kda_ckpt_restore_q8(pool.handle, 2, 128, kda.KDA_BF16, 1, kda._ptr(ids), kda._ptr(ids), dummy, dummy,
                                 1 << 20, dummy, None) in (kda.KDA_EREF, kda.KDA_EINVAL)


def test_pingpong_plan_matches_oracle_under_random_positions():
    rng = np.random.default_rng(7)
    H, d, dt = 4, 64, kda.KDA_F32
    for trial in range(20):
        pool = kda.Pool(8192, 400)
        sim = policy.PoolSim(400)
        P = pool.object_pages(H, d, dt)
        B = int(rng.integers(1, 12))
        # some noise in the pool first, mirrored in the simulation
        noise = int(rng.integers(0, 30))
        kda.kda_page_alloc(pool, noise)
        sim.alloc(noise)
        act = kda.kda_page_alloc(pool, B * P).reshape(B, P)
        act_sim = [sim.alloc(P) for _ in range(B)]
        assert [list(a) for a in act] == act_sim
        interval = int(rng.integers(1, 9))
        pos = [int(x) for x in rng.integers(0, 40, size=B)]
        dst, don = kda.kda_decode_pingpong_plan(pool, H, d, dt, pos, interval, act)
        dst_sim, due = policy.pingpong_plan(sim, pos, interval, act_sim, P)
        assert list(don) == due
        assert [list(x) for x in dst] == dst_sim
        assert pool.free_count() == sim.free_count()


def test_pingpong_plan_is_all_or_nothing_and_checks_ownership():
    H, d, dt = 2, 64, kda.KDA_F32
    pool = kda.Pool(65536, 3)                      # one page per object, one page free
    P = pool.object_pages(H, d, dt)
    assert P == 1
    act = kda.kda_page_alloc(pool, 2 * P).reshape(2, P)
    free0 = pool.free_count()
    with pytest.raises(kda.KdaError) as e:
        kda.kda_decode_pingpong_plan(pool, H, d, dt, [8, 8], 4, act)      # needs 2 objects, 1 fits
    assert e.value.code == kda.KDA_ENOPAGES and pool.free_count() == free0
    kda.kda_page_incref(pool, act[0])                                     # shared: not private
    with pytest.raises(kda.KdaError) as e:
        kda.kda_decode_pingpong_plan(pool, H, d, dt, [1, 1], 4, act)
    assert e.value.code == kda.KDA_EREF


def test_offload_and_prefetch_refuse_bad_arguments():
    pool = kda.Pool(65536, 16)
    L = kda.lib()
    dummy = ctypes.c_void_p(16)
    ids = kda.kda_page_alloc(pool, 2)
    H, d, dt = 1, 128, kda.KDA_BF16
    nb = kda.kda_object_bytes(H, d, dt)
    # host buffer too small, misaligned, or missing: refused before anything is enqueued
    assert L.kda_ckpt_offload(pool.handle, H, d, dt, 1, kda._ptr(ids), dummy, nb - 16, dummy, dummy, 1 << 20,
                              dummy, None) == kda.KDA_EINVAL
    assert L.kda_ckpt_offload(pool.handle, H, d, dt, 1, kda._ptr(ids), ctypes.c_void_p(24), nb, dummy, dummy,
                              1 << 20, dummy, None) == kda.KDA_EINVAL
    assert L.kda_ckpt_offload(pool.handle, H, d, dt, 1, kda._ptr(ids), None, nb, dummy, dummy, 1 << 20,
                              dummy, None) == kda.KDA_EINVAL
    out = np.zeros(4, dtype=np.int32)
    free0 = pool.free_count()
    assert L.kda_ckpt_prefetch(pool.handle, H, d, dt, 1, dummy, nb - 16, kda._ptr(out), dummy, dummy, 1 << 20,
                               dummy, None) == kda.KDA_EINVAL
    assert pool.free_count() == free0


def test_verify_plan_and_accept_keep_one_object_per_request():
    H, d, dt = 2, 64, kda.KDA_F32
    pool = kda.Pool(65536, 64)
    P = pool.object_pages(H, d, dt)
    B, K = 3, 4
    src = kda.kda_page_alloc(pool, B * P).reshape(B, P)
    inter = kda.kda_verify_plan(pool, H, d, dt, B, K)
    assert inter.shape == (K, B, P)
    # lowest free first, token-major
    assert list(inter.reshape(-1)) == list(range(B * P, B * P + K * B * P))
    used = pool.num_pages - pool.free_count()
    act = kda.kda_verify_accept(pool, H, d, dt, [0, 2, 4], src, inter)
    assert list(act[0]) == list(src[0]) and list(act[1]) == list(inter[1, 1]) and list(act[2]) == list(inter[3, 2])
    assert pool.num_pages - pool.free_count() == B * P == used - B * K * P
    for b in range(B):
        assert all(kda.kda_page_refcount(pool, int(p)) == 1 for p in act[b])
    with pytest.raises(kda.KdaError) as e:
        kda.kda_verify_accept(pool, H, d, dt, [5, 0, 0], src, kda.kda_verify_plan(pool, H, d, dt, B, K))
    assert e.value.code == kda.KDA_EINVAL
    with pytest.raises(kda.KdaError) as e:
        kda.kda_verify_plan(pool, H, d, dt, B, 64)      # more than the pool holds
    assert e.value.code == kda.KDA_ENOPAGES


def test_prefill_waves_arguments():
    """kda_prefill_waves returns the wave count and writes at most `cap` bounds; bad shapes,
    decreasing offsets, negative starts and a NULL array with cap > 0 are refused."""
    L = kda.lib()
    bf = kda.KDA_BF16
    cu = np.array([0, 8192, 16384, 24576, 32768], dtype=np.int32)
    st = np.zeros(4, dtype=np.int64)
    W = L.kda_prefill_waves(16, 128, bf, 4, kda._ptr(cu), kda._ptr(st), None, 0)
    assert W >= 1
    full = np.full(W + 3, -7, dtype=np.int32)
    assert L.kda_prefill_waves(16, 128, bf, 4, kda._ptr(cu), kda._ptr(st), kda._ptr(full), W + 3) == W
    assert full[0] == 0 and full[W] == 128 and np.all(full[W + 1:] == -7)   # W + 1 bounds written
    part = np.full(2, -7, dtype=np.int32)
    assert L.kda_prefill_waves(16, 128, bf, 4, kda._ptr(cu), kda._ptr(st), kda._ptr(part), 2) == W
    assert list(part) == list(full[:2])
    assert L.kda_prefill_waves(16, 128, bf, 4, kda._ptr(cu), kda._ptr(st), None, 2) == kda.KDA_EINVAL
    assert L.kda_prefill_waves(16, 128, bf, 4, kda._ptr(cu), kda._ptr(st), kda._ptr(part), -1) == kda.KDA_EINVAL
    assert L.kda_prefill_waves(16, 96, bf, 4, kda._ptr(cu), kda._ptr(st), None, 0) == kda.KDA_EINVAL
    bad = np.array([0, 10, 5], dtype=np.int32)
    assert L.kda_prefill_waves(16, 128, bf, 2, kda._ptr(bad), kda._ptr(st), None, 0) == kda.KDA_EINVAL
    neg = np.array([-1, 0, 0, 0], dtype=np.int64)
    assert L.kda_prefill_waves(16, 128, bf, 4, kda._ptr(cu), kda._ptr(neg), None, 0) == kda.KDA_EINVAL
    # shapes that do not take the split path have no waves
    assert L.kda_prefill_waves(16, 64, bf, 4, kda._ptr(cu), kda._ptr(st), None, 0) == 0
    assert L.kda_prefill_waves(16, 128, kda.KDA_F32, 4, kda._ptr(cu), kda._ptr(st), None, 0) == 0
