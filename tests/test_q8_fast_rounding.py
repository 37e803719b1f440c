"""The error bound behind the INT8 quantiser's reciprocal path, checked in fp32 on the host.

The codec's code is rint(RN(x / s)) with s = RN(m / 127) and |x| <= m ("KIMI K3 경량 복제에서
본 KDA의 AI 인프라 과제", §0x05 5.3).  The kernel computes y = RN(x RN(1/s)) instead and keeps
rint(y) unless y lies within 2^-16 of a half-integer.  That is sound if |y - RN(x/s)| < 2^-16
for every such x and s: then RN(x/s) sits strictly on the same side of the nearest
half-integer as y.  The bound follows from |x/s| <= 127 (1 + 2^-23): the reciprocal's relative
error 2^-24 moves x rs by less than 2^-17, and the two roundings near 64..128 add 2^-18 each.
These tests draw many (x, s) pairs, adversarial ones beside the half-integers included, and
check the bound and the decisions in numpy's IEEE fp32 arithmetic."""
import numpy as np

f32 = np.float32
BAND = f32(0.5) - f32(2.0 ** -16)


def _pairs(seed, n_rows=4096, d=128):
    """Rows of one max-abs m each, scales 1e-30 .. 1e30; half the entries placed within +-8
    fp32 steps of (k + 1/2) s, the rest uniform in [-m, m]."""
    rng = np.random.default_rng(seed)
    m = (10.0 ** rng.uniform(-30, 30, n_rows)).astype(f32)
    s = (m / f32(127)).astype(f32)
    x = (rng.uniform(-1, 1, (n_rows, d)) * m[:, None]).astype(f32)
    k = rng.integers(-127, 127, (n_rows, d // 2)).astype(f32)
    near = ((k + f32(0.5)) * s[:, None]).astype(f32)
    steps = rng.integers(-8, 9, (n_rows, d // 2))
    for u in range(1, 9):
        near = np.where(steps >= u, np.nextafter(near, f32(np.inf)), near)
        near = np.where(steps <= -u, np.nextafter(near, f32(-np.inf)), near)
    x[:, : d // 2] = np.clip(near, -m[:, None], m[:, None])
    x[:, -1] = m                                      # the row's max-abs entry itself
    return x, np.broadcast_to(s[:, None], x.shape)


def _fast(x, s):
    rs = (f32(1) / s).astype(f32)
    return (x * rs).astype(f32)


def test_reciprocal_product_within_two_to_minus_16_of_the_quotient():
    for seed in range(4):
        x, s = _pairs(seed)
        q = (x / s).astype(f32)
        y = _fast(x, s)
        err = np.abs(y.astype(np.float64) - q.astype(np.float64))
        assert err.max() < 2.0 ** -16
        assert np.all(np.abs(q) <= 127 * (1 + 2.0 ** -23))


def test_decisions_outside_the_band_match_the_division():
    total = in_band = 0
    for seed in range(4, 8):
        x, s = _pairs(seed)
        y = _fast(x, s)
        r = np.rint(y)
        keep = np.abs(y - r) <= BAND
        ref = np.rint((x / s).astype(f32))
        assert np.array_equal(r[keep], ref[keep])
        total += y.size
        in_band += int((~keep).sum())
    # only the adversarial half (entries within eight fp32 steps of a half-integer) can land
    # in the band, and not all of it does
    assert 0 < in_band < total // 2


def test_a_planted_wider_error_is_caught():
    """The check has teeth: a product rounded once more (to bf16-like precision) breaks it."""
    x, s = _pairs(9, n_rows=512)
    y = _fast(x, s)
    coarse = (y.view(np.uint32) & np.uint32(0xFFFF0000)).view(f32)
    q = (x / s).astype(f32)
    assert np.abs(coarse.astype(np.float64) - q.astype(np.float64)).max() >= 2.0 ** -16
