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
