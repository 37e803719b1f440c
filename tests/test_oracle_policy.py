"""Pins of the oracle's host policy: checkpoint positions, the resume boundary, page
allocation order and the paged byte layout.  The worked numbers come from
tests/golden/page_examples.json (each entry cites its page and section)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import policy

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_examples.json")))


# ------------------------------------------------------------------ positions
def test_positions_tiny_workload():
    # one sequence of 1024 tokens, a checkpoint at every hash-block end: 512 and 1024
    assert policy.ckpt_positions(0, 1024, 512, 1, False) == [512, 1024]


def test_positions_batched_workload():
    # every 4th 512-token hash-block end of an 8192-token sequence
    assert policy.ckpt_positions(0, 8192, 512, 4, True) == [2048, 4096, 6144, 8192]
    assert policy.ckpt_positions(0, 8192, 512, 4, False) == [2048, 4096, 6144, 8192]


def test_positions_long_workload():
    pos = policy.ckpt_positions(0, 1048576, 512, 4, True)
    assert len(pos) == 512 and pos[0] == 2048 and pos[-1] == 1048576
    assert all(b - a == 2048 for a, b in zip(pos, pos[1:]))


def test_positions_resume_with_last_aligned():
    # resume at 2560, prefill to 7000: stride-4 ends 4096, 6144, plus the last hash end 6656
    assert policy.ckpt_positions(2560, 7000, 512, 4, True) == [4096, 6144, 6656]
    assert policy.ckpt_positions(2560, 7000, 512, 4, False) == [4096, 6144]
    # nothing at or before the start; the start itself is never re-emitted
    assert policy.ckpt_positions(4096, 4100, 512, 1, True) == []
    assert policy.ckpt_positions(4096, 4608, 512, 1, False) == [4608]
    assert policy.ckpt_positions(100, 500, 512, 1, True) == []


def test_positions_are_hash_multiples_in_range():
    rng = np.random.default_rng(5)
    for _ in range(500):
        start = int(rng.integers(0, 20000))
        end = start + int(rng.integers(0, 20000))
        stride = int(rng.integers(1, 6))
        last = bool(rng.integers(0, 2))
        pos = policy.ckpt_positions(start, end, 512, stride, last)
        assert pos == sorted(set(pos))
        assert all(start < p <= end and p % 512 == 0 for p in pos)
        brute = [p for p in range(start + 1, end + 1) if p % (512 * stride) == 0]
        if last and (end // 512) * 512 > start:
            brute = sorted(set(brute + [(end // 512) * 512]))
        assert pos == brute


# ------------------------------------------------------------------ worked examples
def test_hit_2800_resumes_at_2560():
    g = GOLDEN["hit_2800"]
    stored = policy.ckpt_positions(0, g["physical_block"], g["hash_block"], 1, False)
    assert policy.hit_boundary(stored, g["matched"]) == g["resume"]
    assert g["resume"] % g["hash_block"] == 0 and g["resume"] < g["physical_block"]


def test_rollback_6000_to_4096():
    g = GOLDEN["rollback_6000"]
    B = policy.hit_boundary(g["stored"], g["matched"])
    assert B == g["resume"] and g["matched"] - B == g["replay"]


def test_hit_exactly_at_a_stored_position_replays_nothing():
    """A checkpoint at p holds the state after tokens [0, p) (the oracle's resume test shows
    that state continues the uninterrupted run), so a match of exactly p tokens resumes at p
    with nothing to replay; one token fewer falls back to the previous checkpoint.  Stored
    positions as in the 6000-token rollback example."""
    g = GOLDEN["rollback_6000"]
    assert policy.hit_boundary(g["stored"], 4096) == 4096
    assert policy.hit_boundary(g["stored"], 8192) == 8192
    assert policy.hit_boundary(g["stored"], 4095) == 0


def test_rollback_15k_to_10k():
    g = GOLDEN["rollback_15k"]
    stored = list(range(g["interval"], 10 * g["interval"], g["interval"]))
    B = policy.hit_boundary(stored, g["matched"])
    assert B == g["resume"] and g["matched"] - B == g["replay"]


def test_rollback_905k():
    g = GOLDEN["rollback_905k"]
    for case in g["cases"]:
        assert g["matched"] - policy.hit_boundary(case["stored"], g["matched"]) == case["replay"]


def test_dense_checkpoint_cost_arithmetic():
    g = GOLDEN["state_size_217"]
    per_req = g["layers"] * g["heads"] * g["d_k"] * g["d_v"] * g["bytes_per_elem"]
    assert per_req == 217_055_232 and round(per_req / 1e6) == g["approx_MB"]
    n = len(policy.ckpt_positions(0, g["context"], g["hash_block"], 1, False))
    assert n == g["checkpoints"]
    assert n * per_req > g["over_GiB"] * 2 ** 30


# ------------------------------------------------------------------ layout
def test_record_sizes():
    assert policy.record_bytes(128, "bf16") == 67840
    assert policy.record_bytes(64, "f32") == 18688
    assert policy.object_pages(16, 128, "bf16", 65536) == 17
    assert policy.object_pages(32, 128, "bf16", 65536) == 34
    assert policy.object_pages(32, 128, "bf16", 262144) == 9
    assert policy.object_pages(2, 64, "f32", 65536) == 1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_record_round_trip_and_byte_positions(dtype):
    rng = np.random.default_rng(7)
    d = 8
    S = rng.standard_normal((d, d)).astype(np.float32).astype(np.float64)
    win = torch.randn(3, 3 * d).to(torch.bfloat16 if dtype == "bf16" else torch.float32)
    win = win.double().numpy()
    buf = policy.pack_record(S, win, dtype)
    assert len(buf) == policy.record_bytes(d, dtype)
    # S first, fp32 row-major: element (i, j) at byte 4 (i d + j)
    i, j = 3, 5
    assert np.frombuffer(buf[4 * (i * d + j):4 * (i * d + j) + 4], np.float32)[0] == S[i, j]
    # window next: token 0 (oldest) first, channels q | k | v
    es = policy.DTYPE_SIZE[dtype]
    off = d * d * 4 + es * (2 * 3 * d + d + 1)   # newest token, channel k[1]
    raw = buf[off:off + es]
    if dtype == "f32":
        val = np.frombuffer(raw, np.float32)[0]
    else:
        val = torch.from_numpy(np.frombuffer(raw, np.int16).copy()).view(torch.bfloat16).item()
    assert val == win[2, d + 1]
    S2, W2 = policy.unpack_record(buf, d, dtype)
    assert np.array_equal(S2, S) and np.array_equal(W2, win)
    assert buf[d * d * 4 + 9 * d * es:] == b"\0" * (len(buf) - d * d * 4 - 9 * d * es)


def test_object_pages_straddle_and_round_trip():
    rng = np.random.default_rng(8)
    H, d, dtype, PB = 5, 8, "f32", 1024
    R = policy.record_bytes(d, dtype)  # 768: records straddle the 1024-byte pages
    assert R == 768
    S = rng.standard_normal((H, d, d)).astype(np.float32).astype(np.float64)
    W = rng.standard_normal((H, 3, 3 * d)).astype(np.float32).astype(np.float64)
    obj = policy.pack_object(S, W, dtype)
    assert len(obj) == H * R
    pool = np.zeros(40 * PB, dtype=np.uint8)
    pages = [33, 2, 17, 9]
    assert len(pages) == (len(obj) + PB - 1) // PB
    policy.scatter_object(pool, pages, PB, obj)
    back = policy.gather_object(pool, pages, PB, len(obj))
    assert back == obj
    S2, W2 = policy.unpack_object(back, H, d, dtype)
    assert np.array_equal(S2, S) and np.array_equal(W2, W)
    # logical byte x of the object sits in page list[x // PB] at x % PB
    x = 3 * R + 100
    assert pool[pages[x // PB] * PB + x % PB] == obj[x]


# ------------------------------------------------------------------ allocator
def test_lowest_free_first_and_refcounts():
    p = policy.PoolSim(10)
    assert p.alloc(3) == [0, 1, 2]
    p.claim([7, 5])
    assert p.alloc(2) == [3, 4]
    p.decref([1])
    assert p.alloc(2) == [1, 6]
    p.incref([7])
    p.decref([7])
    assert p.ref[7] == 1
    p.decref([7])
    assert p.ref[7] == 0 and p.free_count() == 3   # 7, 8, 9
    with pytest.raises(policy.AllocError):
        p.alloc(4)              # only 3 free: nothing allocated
    assert p.free_count() == 3
    with pytest.raises(policy.AllocError):
        p.decref([7])           # already free
    with pytest.raises(policy.AllocError):
        p.claim([0])            # in use
    with pytest.raises(policy.AllocError):
        p.incref([8, 9])        # 8 is free
    with pytest.raises(policy.AllocError):
        p.decref([5, 5])        # refcount 1, two decrefs
    assert p.ref[5] == 1


def test_plan_allocates_in_sequence_then_position_order():
    p = policy.PoolSim(100)
    active = p.alloc(2 * 3)      # active objects first, 3 pages each
    plan = policy.plan_checkpoints(p, [(0, 2048), (512, 1600)], 3, 512, 1, True)
    assert [(s, pos) for s, pos, _ in plan] == [(0, 512), (0, 1024), (0, 1536), (0, 2048),
                                               (1, 1024), (1, 1536)]
    assert plan[0][2] == [6, 7, 8] and plan[-1][2] == [21, 22, 23]
    assert active == [0, 1, 2, 3, 4, 5]
    small = policy.PoolSim(5)
    with pytest.raises(policy.AllocError):
        policy.plan_checkpoints(small, [(0, 2048)], 2, 512, 1, False)
    assert small.free_count() == 5


def test_decode_checkpoint_interval():
    """Decode keeps a checkpoint every `interval` tokens: the state a step starts from is kept
    when its position is a positive multiple of the interval."""
    assert not policy.decode_ckpt_due(0, 64)
    assert policy.decode_ckpt_due(64, 64) and policy.decode_ckpt_due(128, 64)
    assert not policy.decode_ckpt_due(65, 64) and not policy.decode_ckpt_due(63, 64)
    assert [p for p in range(1, 20) if policy.decode_ckpt_due(p, 5)] == [5, 10, 15]


def test_pingpong_plan_allocates_only_for_due_requests():
    pool = policy.PoolSim(20)
    active = [pool.alloc(2) for _ in range(4)]            # pages 0..7
    dst, due = policy.pingpong_plan(pool, [3, 4, 8, 0], 4, active, 2)
    assert due == [1, 2]
    assert dst[0] == active[0] and dst[3] == active[3]
    assert dst[1] == [8, 9] and dst[2] == [10, 11]        # lowest free first, request order
    with pytest.raises(policy.AllocError):
        policy.pingpong_plan(pool, [4, 4, 4, 4], 4, active, 4)   # 16 pages needed, 8 free
    assert pool.free_count() == 8                          # nothing taken
