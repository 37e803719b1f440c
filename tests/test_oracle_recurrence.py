"""Pins of the fp64 oracle's recurrence and conv against what the sources and the
mathematics fix.  None of these re-types the oracle's own loop: each checks a closed form,
an invariant, a library routine or brute force.

Sources: "Lesson 01 · Architecture map" §两种 Attention，两种状态 (decay, delta write, read);
"KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제" §0x01 1.3 (segment map, composition,
non-commutativity) and §0x09 9.1 (closed form); "Cache de préfixe hybride KDA–MLA"
§Le fonctionnement du prefill (resume from a checkpoint).
"""
import itertools

import numpy as np
import pytest

import oracle

RNG_SEED = 20261202


def _rand_seq(T, d, rng, alpha_lo=0.4):
    q = rng.standard_normal((T, d))
    k = rng.standard_normal((T, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, d))
    alpha = rng.uniform(alpha_lo, 1.0, (T, d))
    beta = rng.uniform(0.05, 1.0, T)
    return q, k, v, alpha, beta


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# ------------------------------------------------------------------ affine segment maps
def test_composition_law_matches_scan():
    """F_C2(F_C1(S)) = M2 M1 S + M2 b1 + b2 equals the sequential scan."""
    rng = np.random.default_rng(RNG_SEED)
    T, d, B = 24, 5, 9
    q, k, v, a, b = _rand_seq(T, d, rng)
    S0 = rng.standard_normal((d, d))
    _, S_scan = oracle.scan(q, k, v, a, b, S0)
    M1, b1 = oracle.segment_affine(k[:B], v[:B], a[:B], b[:B])
    M2, b2 = oracle.segment_affine(k[B:], v[B:], a[B:], b[B:])
    M, bb = oracle.segment_affine(k, v, a, b)
    assert _rel(M2 @ (M1 @ S0 + b1) + b2, S_scan) < 1e-12
    assert _rel(M2 @ M1 @ S0 + M2 @ b1 + b2, S_scan) < 1e-12
    assert _rel(M2 @ M1, M) < 1e-12
    assert _rel(M2 @ b1 + b2, bb) < 1e-12
    assert _rel(M @ S0 + bb, S_scan) < 1e-12


def test_closed_form_product_and_sum():
    """S_n = M_n..M_1 S_0 + sum_i M_n..M_{i+1} b_i, with per-token (M_t, b_t)."""
    rng = np.random.default_rng(RNG_SEED + 1)
    T, d = 11, 4
    q, k, v, a, b = _rand_seq(T, d, rng)
    S0 = rng.standard_normal((d, d))
    maps = [oracle.segment_affine(k[t:t + 1], v[t:t + 1], a[t:t + 1], b[t:t + 1]) for t in range(T)]
    # single-token map is (I - beta k k^T) Diag(alpha) and beta k v^T
    for t, (Mt, bt) in enumerate(maps):
        assert _rel(Mt, (np.eye(d) - b[t] * np.outer(k[t], k[t])) @ np.diag(a[t])) < 1e-15
        assert _rel(bt, b[t] * np.outer(k[t], v[t])) < 1e-15
    prod = np.eye(d)
    for Mt, _ in maps:
        prod = Mt @ prod
    acc = prod @ S0
    for i in range(T):
        P = np.eye(d)
        for Mt, _ in maps[i + 1:]:
            P = Mt @ P
        acc = acc + P @ maps[i][1]
    _, S_scan = oracle.scan(q, k, v, a, b, S0)
    assert _rel(acc, S_scan) < 1e-12


@pytest.mark.parametrize("T,d", [(16, 2), (10, 4)])
def test_bruteforce_all_segmentations(T, d):
    """Every split of [0, T) into contiguous segments composes to the sequential scan."""
    rng = np.random.default_rng(RNG_SEED + T * 7 + d)
    q, k, v, a, b = _rand_seq(T, d, rng)
    S0 = rng.standard_normal((d, d))
    _, S_scan = oracle.scan(q, k, v, a, b, S0)
    seg = {}
    for i in range(T):
        for j in range(i + 1, T + 1):
            seg[(i, j)] = oracle.segment_affine(k[i:j], v[i:j], a[i:j], b[i:j])
    worst = 0.0
    for mask in range(1 << (T - 1)):
        cuts = [0] + [t + 1 for t in range(T - 1) if mask >> t & 1] + [T]
        S = S0
        for i, j in zip(cuts[:-1], cuts[1:]):
            M, bb = seg[(i, j)]
            S = M @ S + bb
        worst = max(worst, _rel(S, S_scan))
    assert worst < 1e-12


def test_segments_do_not_commute():
    """Swapping the order of two segments changes the state."""
    rng = np.random.default_rng(RNG_SEED + 3)
    T, d = 12, 4
    q, k, v, a, b = _rand_seq(T, d, rng)
    S0 = rng.standard_normal((d, d))
    M1, b1 = oracle.segment_affine(k[:6], v[:6], a[:6], b[:6])
    M2, b2 = oracle.segment_affine(k[6:], v[6:], a[6:], b[6:])
    fwd = M2 @ (M1 @ S0 + b1) + b2
    rev = M1 @ (M2 @ S0 + b2) + b1
    assert _rel(rev, fwd) > 1e-3


# ------------------------------------------------------------------ special cases
def test_alpha_one_beta_zero_leaves_state_unchanged():
    rng = np.random.default_rng(RNG_SEED + 4)
    T, H, d = 37, 2, 8
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, H, d))
    v = rng.standard_normal((T, H, d))
    alpha = np.ones((T, H, d))
    beta = np.zeros((T, H))
    w = rng.standard_normal((H, 3 * d, 4)) * 0.5
    S0 = rng.standard_normal((1, H, d, d))
    win0 = rng.standard_normal((1, H, 3, 3 * d))
    r = oracle.kda_run(q, k, v, alpha, beta, w, [0, T], S0=S0, win0=win0, want_xbar=True)
    assert np.array_equal(r["S"], S0)
    for h in range(H):
        qbar = r["xbar"][:, h, :d]
        assert _rel(r["o"][:, h], qbar @ S0[0, h]) < 1e-13


def test_standard_basis_keys_return_values_exactly():
    """alpha = 1, beta = 1, distinct basis keys, zero state, identity conv: S^T e_i = v_i."""
    rng = np.random.default_rng(RNG_SEED + 5)
    d, T = 16, 16
    perm = rng.permutation(d)
    k = np.zeros((T, 1, d))
    k[np.arange(T), 0, perm[:T]] = 1.0
    q = rng.standard_normal((T, 1, d))
    v = rng.standard_normal((T, 1, d))
    w = np.zeros((1, 3 * d, 4))
    w[..., 3] = 1.0
    r = oracle.kda_run(q, k, v, np.ones((T, 1, d)), np.ones((T, 1)), w, [0, T])
    S = r["S"][0, 0]
    for t in range(T):
        assert np.array_equal(S.T @ k[t, 0], v[t, 0])
        assert np.array_equal(S[perm[t]], v[t, 0])


def test_orthonormal_keys_return_values():
    rng = np.random.default_rng(RNG_SEED + 6)
    d = 12
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    k = Qm.T.copy()  # rows orthonormal
    v = rng.standard_normal((d, d))
    q = rng.standard_normal((d, d))
    _, S = oracle.scan(q, k, v, np.ones((d, d)), np.ones(d))
    for t in range(d):
        assert _rel(S.T @ k[t], v[t]) < 1e-12


def test_delta_write_is_exact_after_decay():
    """Unit key, beta = 1, any decay and any prior state: right after the write, reading
    with that key returns the written value (the state was decayed before the write)."""
    rng = np.random.default_rng(RNG_SEED + 7)
    T, d = 20, 6
    q, k, v, a, _ = _rand_seq(T, d, rng, alpha_lo=0.2)
    b = np.ones(T)
    S0 = rng.standard_normal((d, d))
    for t in range(1, T + 1):
        _, S = oracle.scan(q[:t], k[:t], v[:t], a[:t], b[:t], S0)
        assert _rel(S.T @ k[t - 1], v[t - 1]) < 1e-12


def test_printed_formula_differs_only_when_decaying():
    """The printed variant S_t = (I - beta k k^T Diag(alpha)) S + beta k v^T agrees with the
    adopted prose order when alpha = 1 and differs otherwise."""
    rng = np.random.default_rng(RNG_SEED + 8)
    T, d = 15, 5
    q, k, v, a, b = _rand_seq(T, d, rng)
    S0 = rng.standard_normal((d, d))

    def printed(alpha):
        S = S0.copy()
        for t in range(T):
            S = (np.eye(d) - b[t] * np.outer(k[t], k[t]) @ np.diag(alpha[t])) @ S \
                + b[t] * np.outer(k[t], v[t])
        return S

    ones = np.ones_like(a)
    _, S1 = oracle.scan(q, k, v, ones, b, S0)
    assert _rel(printed(ones), S1) < 1e-12
    _, Sa = oracle.scan(q, k, v, a, b, S0)
    assert _rel(printed(a), Sa) > 1e-2


def test_first_step_from_zero_is_outer_product():
    rng = np.random.default_rng(RNG_SEED + 9)
    d = 7
    q, k, v, a, b = _rand_seq(1, d, rng)
    o, S = oracle.scan(q, k, v, a, b)
    assert _rel(S, b[0] * np.outer(k[0], v[0])) < 1e-15
    assert _rel(o[0], S.T @ q[0]) < 1e-15


def test_scalar_recurrence_closed_form():
    """d = 1: s_t = (1 - beta k^2) alpha s_{t-1} + beta k v, o_t = s_t q_t."""
    rng = np.random.default_rng(RNG_SEED + 10)
    T = 60
    q = rng.standard_normal((T, 1))
    k = rng.uniform(-1.2, 1.2, (T, 1))
    v = rng.standard_normal((T, 1))
    a = rng.uniform(0.3, 1.0, (T, 1))
    b = rng.uniform(0.0, 1.0, T)
    o, S = oracle.scan(q, k, v, a, b, np.array([[0.7]]))
    s = 0.7
    for t in range(T):
        s = (1.0 - b[t] * k[t, 0] ** 2) * a[t, 0] * s + b[t] * k[t, 0] * v[t, 0]
        assert abs(o[t, 0] - s * q[t, 0]) <= 1e-13 * max(1.0, abs(s * q[t, 0]))
    assert abs(S[0, 0] - s) < 1e-13


def test_decay_only_is_diagonal_product():
    rng = np.random.default_rng(RNG_SEED + 11)
    T, d = 30, 6
    q, k, v, a, _ = _rand_seq(T, d, rng)
    S0 = rng.standard_normal((d, d))
    _, S = oracle.scan(q, k, v, a, np.zeros(T), S0)
    assert _rel(S, np.diag(np.prod(a, axis=0)) @ S0) < 1e-14


def test_linear_in_values_and_affine_in_initial_state():
    rng = np.random.default_rng(RNG_SEED + 12)
    T, d = 25, 5
    q, k, v1, a, b = _rand_seq(T, d, rng)
    v2 = rng.standard_normal((T, d))
    o1, S1 = oracle.scan(q, k, v1, a, b)
    o2, S2 = oracle.scan(q, k, v2, a, b)
    o3, S3 = oracle.scan(q, k, v1 + v2, a, b)
    assert _rel(S1 + S2, S3) < 1e-12 and _rel(o1 + o2, o3) < 1e-12
    S0 = rng.standard_normal((d, d))
    _, Sx = oracle.scan(q, k, v1, a, b, S0)
    M, _ = oracle.segment_affine(k, v1, a, b)
    # measured against the state's own scale: M S0 is small after 25 decays
    assert np.max(np.abs((Sx - S1) - M @ S0)) < 1e-12 * np.max(np.abs(Sx))


# ------------------------------------------------------------------ short conv
def _run_conv(x, w, win0=None):
    """Drive the full path with beta = 0 so only the conv output (xbar) matters."""
    T, H, C = x.shape
    d = C // 3
    r = oracle.kda_run(x[..., :d], x[..., d:2 * d], x[..., 2 * d:], np.ones((T, H, d)),
                       np.zeros((T, H)), w, [0, T], win0=win0, want_xbar=True)
    return r


def test_conv_identity_weights_pass_through():
    rng = np.random.default_rng(RNG_SEED + 13)
    T, H, d = 9, 2, 4
    x = rng.standard_normal((T, H, 3 * d))
    w = np.zeros((H, 3 * d, 4))
    w[..., 3] = 1.0
    r = _run_conv(x, w, win0=rng.standard_normal((1, H, 3, 3 * d)))
    assert np.array_equal(r["xbar"], x)


def test_conv_impulse_returns_weights():
    rng = np.random.default_rng(RNG_SEED + 14)
    T, H, d = 10, 1, 3
    w = rng.standard_normal((H, 3 * d, 4))
    for c in range(3 * d):
        x = np.zeros((T, H, 3 * d))
        t0 = 4
        x[t0, 0, c] = 1.0
        xb = _run_conv(x, w)["xbar"][:, 0, c]
        expect = np.zeros(T)
        for j in range(4):
            expect[t0 + j] = w[0, c, 3 - j]
        assert np.array_equal(xb, expect)


def test_conv_matches_numpy_convolve_with_window():
    rng = np.random.default_rng(RNG_SEED + 15)
    T, H, d = 23, 2, 4
    x = rng.standard_normal((T, H, 3 * d))
    w = rng.standard_normal((H, 3 * d, 4)) * 0.5
    win0 = rng.standard_normal((1, H, 3, 3 * d))
    xb = _run_conv(x, w, win0)["xbar"]
    for h in range(H):
        for c in range(3 * d):
            y = np.concatenate([win0[0, h, :, c], x[:, h, c]])
            ref = np.convolve(y, w[h, c][::-1], mode="valid")
            assert np.max(np.abs(xb[:, h, c] - ref)) < 1e-13


@pytest.mark.parametrize("T", [1, 2, 3, 8])
def test_conv_window_holds_last_three_raw_tokens(T):
    rng = np.random.default_rng(RNG_SEED + 16 + T)
    H, d = 2, 4
    x = rng.standard_normal((T, H, 3 * d))
    w = rng.standard_normal((H, 3 * d, 4))
    win0 = rng.standard_normal((1, H, 3, 3 * d))
    r = _run_conv(x, w, win0)
    full = np.concatenate([win0[0].transpose(1, 0, 2), x], axis=0)  # [3+T, H, 3d]
    assert np.array_equal(r["win"][0], full[-3:].transpose(1, 0, 2))


# ------------------------------------------------------------------ checkpoints / resume
def test_resume_from_every_checkpoint_equals_uninterrupted_run():
    rng = np.random.default_rng(RNG_SEED + 17)
    T, H, d, blk = 40, 2, 4, 8
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, H, d))
    v = rng.standard_normal((T, H, d))
    a = rng.uniform(0.5, 1.0, (T, H, d))
    b = rng.uniform(0.0, 1.0, (T, H))
    w = rng.standard_normal((H, 3 * d, 4)) * 0.5
    cks = list(range(blk, T + 1, blk))
    full = oracle.kda_run(q, k, v, a, b, w, [0, T], ckpt_counts=[cks])
    for n, B in enumerate(cks):
        part = oracle.kda_run(q[B:], k[B:], v[B:], a[B:], b[B:], w, [0, T - B],
                              S0=full["ck_S"][0][n][None], win0=full["ck_win"][0][n][None])
        assert np.array_equal(part["o"], full["o"][B:])
        assert np.array_equal(part["S"], full["S"])
        assert np.array_equal(part["win"], full["win"])


def test_varlen_batch_equals_separate_runs():
    rng = np.random.default_rng(RNG_SEED + 18)
    H, d = 2, 4
    lens = [5, 1, 17, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    a = rng.uniform(0.5, 1.0, (T, H, d))
    b = rng.uniform(0.0, 1.0, (T, H))
    w = rng.standard_normal((H, 3 * d, 4))
    S0 = rng.standard_normal((len(lens), H, d, d))
    win0 = rng.standard_normal((len(lens), H, 3, 3 * d))
    batch = oracle.kda_run(q, k, v, a, b, w, cu, S0=S0, win0=win0)
    for s in range(len(lens)):
        sl = slice(cu[s], cu[s + 1])
        one = oracle.kda_run(q[sl], k[sl], v[sl], a[sl], b[sl], w, [0, lens[s]],
                             S0=S0[s:s + 1], win0=win0[s:s + 1])
        assert np.array_equal(one["o"], batch["o"][sl])
        assert np.array_equal(one["S"][0], batch["S"][s])


def test_full_path_is_conv_then_recurrence_per_head():
    """The full path is the conv followed by the recurrence, each (sequence, head) on its own
    slices: its outputs, final states and checkpoints equal the plain scan (pinned above) run
    on that pair's post-conv values (pinned against numpy's convolution above) with that
    pair's own decay and beta, from that pair's initial state.  This pins the packed
    [T][H][d] indexing of every input and the token count at which a checkpoint is taken."""
    rng = np.random.default_rng(RNG_SEED + 19)
    H, d = 3, 5
    lens = [7, 12, 3]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    q, k, v = (rng.standard_normal((T, H, d)) for _ in range(3))
    a = rng.uniform(0.3, 1.0, (T, H, d))
    b = rng.uniform(0.05, 1.0, (T, H))
    w = rng.standard_normal((H, 3 * d, 4)) * 0.5
    S0 = rng.standard_normal((len(lens), H, d, d))
    win0 = rng.standard_normal((len(lens), H, 3, 3 * d))
    cks = [[2, 7], [1, 5, 12], [3]]
    r = oracle.kda_run(q, k, v, a, b, w, cu, S0=S0, win0=win0, ckpt_counts=cks, want_xbar=True)
    xb = r["xbar"]
    for s in range(len(lens)):
        sl = slice(cu[s], cu[s + 1])
        for h in range(H):
            qb, kb, vb = xb[sl, h, :d], xb[sl, h, d:2 * d], xb[sl, h, 2 * d:]
            o, S = oracle.scan(qb, kb, vb, a[sl, h], b[sl, h], S0[s, h])
            assert _rel(r["o"][sl, h], o) < 1e-13
            assert _rel(r["S"][s, h], S) < 1e-13
            for n, p in enumerate(cks[s]):
                _, Sp = oracle.scan(qb[:p], kb[:p], vb[:p], a[sl, h][:p], b[sl, h][:p], S0[s, h])
                assert _rel(r["ck_S"][s][n][h], Sp) < 1e-13
