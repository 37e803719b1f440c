"""Helpers for the GPU parity tests: run the library through its Python binding (which
calls the C ABI), read objects back from the device pool, run the oracle on the same
inputs, and compare.  Error metric: max |x - ref| / max |ref| per (sequence, head) block."""
from __future__ import annotations

import os

import numpy as np
import torch

import kda_state_chunked_gb300 as kda
import oracle
from oracle import policy

TOL = {"f32": 1e-4, "bf16": 2e-2}

# Worst max-relative error seen per named case in this process, with its tolerance; printed
# at the end of the pytest run (tests/conftest.py) so that the margin to the limit is visible.
MARGINS: dict = {}


def record_margin(name: str, err: float, tol: float, what: str = "") -> float:
    """Keep the worst error under `name`, with its limit, the test and the block it came from."""
    old = MARGINS.get(name, (0.0, tol, "", ""))
    if float(err) >= old[0]:
        test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0].split("::")[-1]
        MARGINS[name] = (float(err), tol, test, what)
    return err


def rel_err(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    num = np.max(np.abs(x - ref)) if x.size else 0.0
    if den == 0:
        return float(num)
    return float(num / den)


def assert_close(x, ref, tol, what, name=None):
    """Max-relative-error check of one block; the error is recorded under `name` if given."""
    e = rel_err(x, ref)
    assert np.all(np.isfinite(np.asarray(x, dtype=np.float64))), f"{what}: non-finite values"
    assert e <= tol, f"{what}: max relative error {e:.3e} > {tol:.1e}"
    if name:
        record_margin(name, e, tol, what)
    return e


def read_object(pool: kda.Pool, pages, H, d, dtype):
    pages = [int(p) for p in np.asarray(pages).reshape(-1)]
    nb = policy.object_bytes(H, d, dtype)
    PB = pool.page_bytes
    parts = [pool.base[p * PB:(p + 1) * PB] for p in pages]
    buf = torch.cat(parts).cpu().numpy().tobytes()[:nb]
    return policy.unpack_object(buf, H, d, dtype)


def read_object_bytes(pool: kda.Pool, pages, nbytes: int) -> bytes:
    pages = [int(p) for p in np.asarray(pages).reshape(-1)]
    PB = pool.page_bytes
    return torch.cat([pool.base[p * PB:(p + 1) * PB] for p in pages]).cpu().numpy().tobytes()[:nbytes]


def write_object(pool: kda.Pool, pages, S, win, dtype):
    obj = policy.pack_object(S, win, dtype)
    PB = pool.page_bytes
    pages = [int(p) for p in np.asarray(pages).reshape(-1)]
    t = torch.frombuffer(bytearray(obj), dtype=torch.uint8)
    for i, p in enumerate(pages):
        n = min(PB, len(obj) - i * PB)
        if n <= 0:
            break
        pool.base[p * PB:p * PB + n].copy_(t[i * PB:i * PB + n].to(pool.base.device))


def random_state(H, d, dtype, gen, scale=0.3):
    """A random initial (S, window) whose values are exact in the storage types.  The window
    holds three raw tokens drawn like the workload's: q and k parts unit-norm per token, v part
    N(0, 1) (a window is the raw q | k | v of the last three tokens, and the input recipe
    normalises q and k per token).  Un-normalised q, k rows would put beta |k_bar|^2 far above 2,
    a regime no workload input reaches, where the recurrence amplifies every rounding."""
    S = (torch.randn(H, d, d, generator=gen) * scale).float().double().numpy()
    wdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    w = torch.randn(H, 3, 3 * d, generator=gen)
    for part in (0, 1):
        blk = w[:, :, part * d:(part + 1) * d]
        w[:, :, part * d:(part + 1) * d] = blk / blk.norm(dim=-1, keepdim=True)
    win = w.to(wdt).double().numpy()
    return S, win


class Prefill:
    """One prefill call through the binding, with its checkpoint plan."""

    def __init__(self, pool, toks, cu, start_pos, has_init, active_pages, stride=1,
                 include_last=True, hash_block=512, checkpoints=True):
        q = toks["q"]
        T_tot, H, d = q.shape
        dt = kda.dtype_of(q)
        self.H, self.d = H, d
        if checkpoints:
            self.seq, self.pos, self.pages = kda.kda_ckpt_plan(pool, H, d, dt, cu, start_pos, hash_block,
                                                               stride, include_last)
        else:
            P0 = pool.object_pages(H, d, dt)
            self.seq = np.zeros(0, np.int32)
            self.pos = np.zeros(0, np.int64)
            self.pages = np.zeros((0, P0), np.int32)
        P = pool.object_pages(H, d, dt)
        ws = kda.prefill_workspace(q, cu, start_pos, len(self.seq), P)
        self.status = torch.zeros(1, dtype=torch.int32, device=q.device)
        self.o = torch.full_like(q, float("nan"))
        kda.kda_prefill_varlen(pool, cu, start_pos, has_init, q, toks["k"], toks["v"], toks["alpha"],
                               toks["beta"], toks["conv_w"], self.o, active_pages, self.seq, self.pos,
                               self.pages, ws, self.status)
        rc, bits = kda.kda_sync_status(self.status)
        assert rc == kda.KDA_OK, f"device status bits {bits}"


def oracle_prefill(toks, cu, start_pos, S0=None, win0=None, ckpt_abs=None):
    """Oracle on the same tokens; ckpt_abs: per-sequence absolute checkpoint positions."""
    nseq = len(cu) - 1
    counts = None
    if ckpt_abs is not None:
        counts = [[int(p) - int(start_pos[s]) for p in ckpt_abs[s]] for s in range(nseq)]
    return oracle.kda_run(toks["q"], toks["k"], toks["v"], toks["alpha"], toks["beta"],
                          toks["conv_w"], cu, S0=S0, win0=win0, ckpt_counts=counts)


def oracle_positions(cu, start_pos, stride=1, include_last=True, hash_block=512):
    """Checkpoint positions per sequence from the oracle's own policy."""
    return [policy.ckpt_positions(int(start_pos[s]), int(start_pos[s]) + int(cu[s + 1] - cu[s]),
                                  hash_block, stride, include_last) for s in range(len(cu) - 1)]


def compare_prefill(pool, run: Prefill, ref, cu, active_pages, dtype, ck_abs, tol=None, name=None):
    """Compare outputs, final states / windows and every checkpoint with the oracle.
    ck_abs: the oracle policy's positions, which the library's plan must equal exactly.
    Returns the worst max-relative error (recorded under `name` when given)."""
    tol = TOL[dtype] if tol is None else tol
    H, d = run.H, run.d
    nseq = len(cu) - 1
    assert ckpt_lists(run, nseq) == [list(x) for x in ck_abs], "checkpoint positions differ"
    o = run.o.float().cpu().numpy()
    worst = 0.0
    for s in range(nseq):
        a, b = int(cu[s]), int(cu[s + 1])
        for h in range(H):
            if b > a:
                worst = max(worst, assert_close(o[a:b, h], ref["o"][a:b, h], tol, f"o seq {s} head {h}", name))
        S, W = read_object(pool, active_pages[s], H, d, dtype)
        for h in range(H):
            worst = max(worst, assert_close(S[h], ref["S"][s, h], tol, f"final S seq {s} head {h}", name))
        assert np.array_equal(W, ref["win"][s]), f"final window seq {s}"
    for n, (s, p) in enumerate(zip(run.seq, run.pos)):
        S, W = read_object(pool, run.pages[n], H, d, dtype)
        idx = _ck_index(run, n)
        for h in range(H):
            worst = max(worst, assert_close(S[h], ref["ck_S"][s][idx][h], tol,
                                            f"checkpoint {p} seq {s} head {h}", name))
        assert np.array_equal(W, ref["ck_win"][s][idx]), f"checkpoint window {p} seq {s}"
    return worst


def _ck_index(run: Prefill, n: int) -> int:
    s = run.seq[n]
    return int(sum(1 for m in range(n) if run.seq[m] == s))


def ckpt_lists(run: Prefill, nseq: int):
    out = [[] for _ in range(nseq)]
    for s, p in zip(run.seq, run.pos):
        out[int(s)].append(int(p))
    return out
