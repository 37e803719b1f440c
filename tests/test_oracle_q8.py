"""Pins of the oracle's INT8 checkpoint codec (per key-channel symmetric max-abs scale along
the value channels; "KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제", §0x05 5.3, §0x06 6.6)."""
import numpy as np
import pytest

from oracle import policy, q8


def test_record_sizes():
    assert q8.record_bytes(128, "bf16") == 19200          # 512 + 16384 + 2304
    assert q8.record_bytes(64, "f32") == 6656              # 256 + 4096 + 2304
    assert q8.record_bytes(128, "f32") == 512 + 16384 + 4608
    # the recurrent state shrinks 4x, the window does not
    assert policy.record_bytes(128, "bf16") / q8.record_bytes(128, "bf16") == pytest.approx(3.533, abs=1e-3)


def test_power_of_two_grid_is_exact():
    """Rows whose max is 127 * 2^k and whose entries are integers times 2^k quantise with no
    error: the scale is exactly 2^k and every code is the integer itself."""
    rng = np.random.default_rng(0)
    d = 64
    k = rng.integers(-20, 10, size=d)
    ints = rng.integers(-127, 128, size=(d, d))
    ints[np.arange(d), rng.integers(0, d, size=d)] = 127 * rng.choice([-1, 1], size=d)
    S = (ints * np.ldexp(1.0, k)[:, None]).astype(np.float32)
    scale, codes = q8.quantize(S)
    assert np.array_equal(scale, np.ldexp(1.0, k).astype(np.float32))
    assert np.array_equal(codes.astype(np.int64), ints)
    assert np.array_equal(q8.dequantize(scale, codes), S)


def test_error_is_at_most_half_a_step():
    rng = np.random.default_rng(1)
    S = (rng.standard_normal((128, 128)) * rng.lognormal(0, 2, size=(128, 1))).astype(np.float32)
    scale, codes = q8.quantize(S)
    err = np.abs(q8.dequantize(scale, codes).astype(np.float64) - S.astype(np.float64))
    # half a quantisation step, plus the fp32 rounding of the division and the product
    bound = scale.astype(np.float64)[:, None] * (0.5 + 1e-6) + np.abs(S) * 2.0 ** -22
    assert np.all(err <= bound)
    # the max-abs entry of every row maps to +-127
    i = np.arange(128)
    j = np.argmax(np.abs(S), axis=1)
    assert np.array_equal(np.abs(codes[i, j]).astype(np.int64), np.full(128, 127))
    assert codes.min() >= -127


def test_symmetric_and_zero_rows():
    rng = np.random.default_rng(2)
    S = rng.standard_normal((32, 32)).astype(np.float32)
    S[5] = 0.0
    s1, c1 = q8.quantize(S)
    s2, c2 = q8.quantize(-S)
    assert np.array_equal(s1, s2) and np.array_equal(c1, -c2)
    assert s1[5] == 0 and not c1[5].any() and not q8.dequantize(s1, c1)[5].any()


def test_ties_round_to_even():
    # scale 1 (max 127): x = 2.5 -> 2, 3.5 -> 4, -2.5 -> -2
    S = np.zeros((1, 8), dtype=np.float32)
    S[0, :4] = [127.0, 2.5, 3.5, -2.5]
    scale, codes = q8.quantize(S)
    assert scale[0] == 1.0
    assert codes[0, :4].tolist() == [127, 2, 4, -2]


@pytest.mark.parametrize("d,dtype", [(128, "bf16"), (64, "f32")])
def test_record_layout_and_round_trip(d, dtype):
    rng = np.random.default_rng(3)
    H = 3
    S = rng.standard_normal((H, d, d)).astype(np.float32).astype(np.float64)
    win = rng.standard_normal((H, 3, 3 * d))
    win = np.asarray(policy.unpack_object(policy.pack_object(S, win, dtype), H, d, dtype)[1])  # exact in dtype
    buf = q8.pack_object(S, win, dtype)
    R = q8.record_bytes(d, dtype)
    assert len(buf) == H * R
    sc, codes, w2 = q8.unpack_object(buf, H, d, dtype)
    assert np.array_equal(w2, win)
    for h in range(H):
        s_ref, c_ref = q8.quantize(S[h])
        assert np.array_equal(sc[h], s_ref) and np.array_equal(codes[h], c_ref)
        # byte positions: scales, then codes row-major, then the window, then zero padding
        rec = buf[h * R:(h + 1) * R]
        assert rec[:4 * d] == s_ref.tobytes()
        assert rec[4 * d:4 * d + d * d] == c_ref.tobytes()
        assert rec[4 * d + d * d + 9 * d * policy.DTYPE_SIZE[dtype]:] == bytes(R - 4 * d - d * d - 9 * d * policy.DTYPE_SIZE[dtype])
