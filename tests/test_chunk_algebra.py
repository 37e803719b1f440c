"""The chunk algebra of the tensor-core prefill, written out in fp64 the way the kernels group
it, checked against the oracle's token recurrence.

Chunk preparation builds one operand image per chunk: Gamma_C [-WK' | Qt'] (the decay of the
chunk folded into the first operand: [-WK' Gamma_C | q gamma_r]), [P^T | Kb], V, T and gamma_C.
The chain then applies four steps per chunk:
  1. U^T = V^T T^T;
  2. [W^T | O^T] = [U^T | 0] + S^T (Gamma_C [-WK' | Qt'])^T;
  3. [O^T | S^T] = [O^T | (Gamma_C S)^T] + W^T [P^T | Kb];
  4. the output of the chunk is O.
A sign, transpose or grouping error in that design fails here on the CPU. The GPU tests check
the kernels themselves against the oracle.

Source of the chunked form: "KIMI K3 경량 복제에서 본 KDA의 AI 인프라 과제" §0x01 1.3 (a chunk
acts on S as one affine map); recurrence: "Lesson 01 · Architecture map" §两种 Attention，两种状态.
"""
import numpy as np
import pytest

import oracle


def _image(qb, kb, vb, al, beta):
    """Operand image of one chunk of C rows (post-conv q, k, v; per-key decay al; beta)."""
    C, d = kb.shape
    gam = np.cumprod(al, axis=0)                 # gamma_r, per key channel
    gC = gam[-1]
    Kt = kb * gam / gC                           # Kt' = k gamma_r / gamma_C
    Qt = qb * gam / gC                           # Qt' = q gamma_r / gamma_C
    Kb = kb * gC / gam                           # Kb  = k gamma_C / gamma_r
    G = Kt @ Kb.T
    P = np.tril(Qt @ Kb.T, -1) + np.diag(np.sum(qb * kb, axis=1))   # exact diagonal q . k
    A = np.diag(beta) @ np.tril(G, -1)
    T = np.linalg.inv(np.eye(C) + A) @ np.diag(beta)
    WK = T @ Kt                                  # WK' = T Kt'  (C x d)
    # N rows of the first group's B operand, key columns scaled by gamma_C
    return {"WQ": np.concatenate([-WK, Qt]) * gC[None, :],
            "PK": np.concatenate([P.T, Kb], axis=1),   # [j][i | key]: the second group's B
            "V": vb, "T": T, "gC": gC}


def _chain_step(ST, img):
    """One chunk on S^T (lane = value channel, column = key): returns (O [C][d_v], new S^T)."""
    C = img["T"].shape[0]
    GST = ST * img["gC"][None, :]                # (Gamma_C S)^T, keys scaled
    UT = img["V"].T @ img["T"].T                 # U^T = V^T T^T
    WO = np.concatenate([UT, np.zeros_like(UT)], axis=1) + ST @ img["WQ"].T
    WT, OT = WO[:, :C], WO[:, C:]
    OS = np.concatenate([OT, GST], axis=1) + WT @ img["PK"]
    return OS[:, :C].T, OS[:, C:]


def _chunked(q, k, v, a, b, S0, C):
    """Token rows run in chunks of C; a ragged last chunk is padded with inert rows
    (q = k = v = 0, alpha = 1, beta = 0), which is how the kernels mask rows past the end."""
    T, d = k.shape
    n = -(-T // C) * C
    pad = n - T
    zq = np.zeros((pad, d))
    q, k, v = (np.concatenate([x, zq]) for x in (q, k, v))
    a = np.concatenate([a, np.ones((pad, d))])
    b = np.concatenate([b, np.zeros(pad)])
    ST = S0.T.copy()
    outs = []
    for c0 in range(0, n, C):
        sl = slice(c0, c0 + C)
        o, ST = _chain_step(ST, _image(q[sl], k[sl], v[sl], a[sl], b[sl]))
        outs.append(o)
    return np.concatenate(outs)[:T], ST.T


@pytest.mark.parametrize("T,d,C,seed", [(48, 8, 16, 1), (37, 6, 16, 2), (130, 16, 64, 3), (5, 4, 8, 4)])
def test_kernel_grouping_equals_the_token_recurrence(T, d, C, seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((T, d))
    k = rng.standard_normal((T, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, d))
    a = rng.uniform(0.4, 1.0, (T, d))
    b = rng.uniform(0.05, 1.0, T)
    S0 = rng.standard_normal((d, d))
    o_ref, S_ref = oracle.scan(q, k, v, a, b, S0)
    o, S = _chunked(q, k, v, a, b, S0, C)
    scale_o = max(np.max(np.abs(o_ref)), 1.0)
    assert np.max(np.abs(o - o_ref)) / scale_o < 1e-10
    assert np.max(np.abs(S - S_ref)) / max(np.max(np.abs(S_ref)), 1.0) < 1e-10


def test_a_wrong_sign_in_the_first_group_is_caught():
    """The check has teeth: the same algebra with +WK' instead of -WK' does not match."""
    rng = np.random.default_rng(9)
    T, d, C = 32, 6, 16
    q = rng.standard_normal((T, d))
    k = rng.standard_normal((T, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, d))
    a = rng.uniform(0.4, 1.0, (T, d))
    b = rng.uniform(0.05, 1.0, T)
    S0 = rng.standard_normal((d, d))
    o_ref, _ = oracle.scan(q, k, v, a, b, S0)
    img = _image(q[:C], k[:C], v[:C], a[:C], b[:C])
    img["WQ"] = np.concatenate([-img["WQ"][:C], img["WQ"][C:]])
    o, _ = _chain_step(S0.T.copy(), img)
    assert np.max(np.abs(o - o_ref[:C])) > 1e-3


def _series_solve(A, beta, skip=True):
    """T = (I + A)^{-1} Diag(beta) as chunk prep forms it: 16 x 16 diagonal block inverses
    (Binv), E = Binv N with N the strictly block-lower part of I + A, then the products
    E^2, E Binv and E^2 G (G = Binv - E Binv) over 16-deep K-steps, skipping the steps the
    block structure makes zero (E = Binv N: K-blocks 1-3; E^2: 1-2; E Binv: 0-2; E^2 G: 0-1)."""
    C = A.shape[0]
    L = np.eye(C) + A
    blk = [slice(i, i + 16) for i in range(0, C, 16)]
    Binv = np.zeros_like(L)
    for s in blk:
        Binv[s, s] = np.linalg.inv(L[s, s])
    N = L - sum(np.pad(L[s, s], ((s.start, C - s.stop), (s.start, C - s.stop))) for s in blk)

    def prod(X, Y, ks):
        ks = ks if skip else range(len(blk))
        return sum(X[:, blk[k]] @ Y[blk[k], :] for k in ks)

    E = prod(Binv, N, (1, 2, 3))
    E2 = prod(E, E, (1, 2))
    G = Binv - prod(E, Binv, (0, 1, 2))
    return np.tril(G + prod(E2, G, (0, 1))) @ np.diag(beta)


def test_block_series_solve_equals_the_inverse():
    rng = np.random.default_rng(11)
    for _ in range(5):
        C = 64
        K = rng.standard_normal((C, 32)) / np.sqrt(32)
        beta = 1 / (1 + np.exp(-rng.standard_normal(C)))
        A = np.diag(beta) @ np.tril(K @ K.T, -1)
        ref = np.linalg.inv(np.eye(C) + A) @ np.diag(beta)
        got = _series_solve(A, beta)
        assert np.allclose(got, ref, rtol=0, atol=1e-11)
        # the skipped K-steps contribute nothing
        assert np.allclose(got, _series_solve(A, beta, skip=False), rtol=0, atol=1e-14)


def test_a_dropped_series_term_is_caught():
    """Without the E^2 G term (or with E^2 summed over too few K-steps) the result is wrong."""
    rng = np.random.default_rng(12)
    C = 64
    K = rng.standard_normal((C, 32)) / np.sqrt(32)
    beta = np.full(C, 0.9)
    A = np.diag(beta) @ np.tril(K @ K.T, -1)
    ref = np.linalg.inv(np.eye(C) + A) @ np.diag(beta)
    L = np.eye(C) + A
    mask = np.kron(np.eye(4), np.ones((16, 16)))
    Binv = np.linalg.inv(L * mask)
    E = Binv @ (L * (1 - mask))
    G = Binv - E @ Binv
    assert not np.allclose(np.tril(G) @ np.diag(beta), ref, atol=1e-6)
    E2_short = E[:, 16:32] @ E[16:32, :]           # K-block 2 dropped
    assert not np.allclose(np.tril(G + E2_short @ G) @ np.diag(beta), ref, atol=1e-6)
    assert np.allclose(np.tril(G + E @ E @ G) @ np.diag(beta), ref, atol=1e-11)


def _factored_gram_fp32(k, al):
    """G = Kt' Kb^T with the kernels' fp32 factors: gamma_r by running products, the row scale
    gamma_r / gamma_C through the reciprocal of gamma_C, and Kb's scale as its reciprocal."""
    f32 = np.float32
    k, al = k.astype(f32), al.astype(f32)
    gam = np.cumprod(al, axis=0, dtype=f32)
    gC = gam[-1]
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        s = gam * (f32(1) / gC)
        Kt, Kb = k * s, k * (f32(1) / s)
        G = (Kt @ Kb.T).astype(f32)
    return G, gC


def _exact_gram_lower(k, al):
    """Strictly lower G in fp64 from the per-pair decay prod_{s<u<=r} alpha_u, no factoring."""
    C = k.shape[0]
    G = np.zeros((C, C))
    for r in range(C):
        for s in range(r):
            G[r, s] = np.sum(k[r] * k[s] * np.prod(al[s + 1:r + 1], axis=0))
    return G


def test_factored_decay_is_exact_down_to_the_range_limit():
    """With a channel decaying to about 2^-99.5 over the chunk (just inside the 2^-100 the
    prefill kernels accept), the fp32 factors stay finite, every sum of the Gram matrix
    (the upper triangle's large ones included) stays finite, and the strictly lower part
    the solve uses matches the unfactored per-pair decay to fp32 rounding.  A gate of 0
    puts gamma_C below the limit and the factored form produces non-finite values, which is
    why the kernels report such a chunk."""
    rng = np.random.default_rng(21)
    C, d = 64, 128
    k = rng.standard_normal((C, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    al = rng.uniform(0.4, 1.0, (C, d))
    al[:, :4] = 2.0 ** (-99.5 / 64)                  # four channels at the edge of the range
    al = al.astype(np.float32).astype(np.float64)
    G, gC = _factored_gram_fp32(k, al)
    assert np.min(gC) >= np.float32(2.0 ** -100)
    assert np.all(np.isfinite(G))
    ref = _exact_gram_lower(k.astype(np.float32).astype(np.float64), al)
    low = np.tril(G.astype(np.float64), -1)
    assert np.max(np.abs(low - ref)) <= 1e-5 * np.max(np.abs(ref))

    al0 = al.copy()
    al0[30, 0] = 0.0
    G0, gC0 = _factored_gram_fp32(k, al0)
    assert not gC0[0] >= np.float32(2.0 ** -100)
    assert not np.all(np.isfinite(G0))


def _block_anchored_products_fp32(a, b, al, blk=16):
    """sum_i a_ri b_si prod_{s<u<=r} al_ui for s <= r, in fp32, with every decay factor <= 1:
    an earlier key block is reached through the start b of the row's block,
    (prod_{b<u<=r} al)(prod_{s<u<=b} al); inside a diagonal block the per-pair product is
    taken directly.  (The form chunk prep would need to cover every gate in [0, 1].)"""
    f32 = np.float32
    a, b, al = a.astype(f32), b.astype(f32), al.astype(f32)
    C = a.shape[0]
    out = np.zeros((C, C), dtype=f32)
    for R in range(C // blk):
        r0 = R * blk
        rows = slice(r0, r0 + blk)
        # row factor prod_{r0<u<=r} al (1 at the block start)
        f1 = np.ones((blk, a.shape[1]), dtype=f32)
        for j in range(1, blk):
            f1[j] = f1[j - 1] * al[r0 + j]
        ar = a[rows] * f1
        if r0 > 0:
            # key factor prod_{s<u<=r0} al for every earlier key s, a suffix product
            f2 = np.ones((r0, a.shape[1]), dtype=f32)
            f2[r0 - 1] = al[r0]
            for s in range(r0 - 2, -1, -1):
                f2[s] = f2[s + 1] * al[s + 1]
            out[rows, :r0] = (ar @ (b[:r0] * f2).T).astype(f32)
        for r in range(blk):
            dec = np.ones(a.shape[1], dtype=f32)
            for s in range(r, -1, -1):
                out[r0 + r, r0 + s] = np.sum(a[r0 + r] * b[r0 + s] * dec, dtype=f32)
                dec = dec * al[r0 + s]
    return out


def test_block_anchored_decay_covers_a_zero_gate():
    """The block-anchored form stays finite and exact to fp32 rounding where the chunk-end
    anchoring breaks: a gate of exactly 0 in some channels and gates near 0 in others."""
    rng = np.random.default_rng(22)
    C, d = 64, 32
    q = rng.standard_normal((C, d))
    k = rng.standard_normal((C, d))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    al = rng.uniform(0.4, 1.0, (C, d))
    al[30, 0] = 0.0                                  # a full reset of channel 0
    al[:, 1] = 1e-3                                  # a channel decaying to 1e-192 over the chunk
    al = al.astype(np.float32).astype(np.float64)
    ref = np.zeros((C, C))
    for r in range(C):
        for s in range(r + 1):
            ref[r, s] = np.sum(q[r].astype(np.float32) * k[s].astype(np.float32) * np.prod(al[s + 1:r + 1], axis=0))
    got = _block_anchored_products_fp32(q, k, al)
    assert np.all(np.isfinite(got))
    assert np.max(np.abs(np.tril(got) - ref)) <= 1e-5 * np.max(np.abs(ref))
    # the chunk-end anchoring on the same chunk does not survive
    G, gC = _factored_gram_fp32(k, al)
    assert not np.all(np.isfinite(G))
