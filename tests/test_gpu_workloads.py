"""Full-size parity on the five benchmark workloads (through the C ABI), against the fp64
oracle run from token 0 on the same seeded inputs.

  tiny            1 x 1024 tokens, H = 2, d = 64, fp32, checkpoints at 512 and 1024: everything
  batched         4 x 8192, H = 16, d = 128, bf16, checkpoints every 2048: every sequence and head
  varlen resume   32 sequences, lengths U[512, 32768], H = 32: setup prefill with a checkpoint at
                  every 512 end, restore a random stored checkpoint (bit-exact copy checked for all
                  32), prefill the suffix with new sparse checkpoints; oracle from token 0 on every
                  (sequence, head) pair: outputs, final states and windows, every new checkpoint
  decode          256 requests x 32 heads, 512-token setup prefill then 64 decode steps through a
                  permuted page table of 256 KiB pages; oracle on every request and head
  long            1 x 1,048,576 tokens, H = 32, 512 checkpoints; oracle on four heads in full
Error metric: max |x - ref| / max |ref| per (sequence, head) block; 1e-4 for fp32 inputs, 2e-2
for bf16 inputs.  Checkpoint positions and page ids are compared exactly."""
import numpy as np
import pytest
import torch

import kda_state_chunked_gb300 as kda
from kda_state_chunked_gb300 import workloads
import oracle
from oracle import policy

from kda_cases import (Prefill, TOL, assert_close, compare_prefill, ckpt_lists, oracle_positions,
                       oracle_prefill, read_object, read_object_bytes, record_margin)

pytestmark = pytest.mark.gpu
DEV = "cuda"
# names under which the worst errors are reported
NM_VARLEN = "varlen resume workload prefill (bf16)"
NM_DECODE = "decode workload, 64 steps (bf16)"
NM_LONG = "long workload prefill, 4 heads (bf16)"


def _cpu_heads(toks, rows, heads):
    """Exact CPU copies of the token tensors for a row slice and a list of heads."""
    out = {}
    for k in ("q", "k", "v", "alpha"):
        out[k] = toks[k][rows][:, heads].cpu()
    out["beta"] = toks["beta"][rows][:, heads].cpu()
    out["conv_w"] = toks["conv_w"][heads].cpu()
    return out


def test_tiny_workload():
    w = workloads.WORKLOADS["tiny"]
    cpu = workloads.make_tokens(w.T, w.H, w.d, w.dtype, w.seed, "cpu")
    dev = {k: v.to(DEV) for k, v in cpu.items()}
    pool = kda.Pool(w.page_bytes, 64, DEV)
    P = pool.object_pages(w.H, w.d, kda.DTYPES[w.dtype])
    act = kda.kda_page_alloc(pool, P).reshape(1, P)
    cu, sp = [0, w.T], [0]
    run = Prefill(pool, dev, cu, sp, [0], act, stride=w.stride, include_last=w.include_last)
    ck = oracle_positions(cu, sp, w.stride, w.include_last)
    assert ck == [[512, 1024]]
    ref = oracle_prefill(cpu, cu, sp, ckpt_abs=ck)
    compare_prefill(pool, run, ref, cu, act, w.dtype, ck, name="tiny workload prefill (f32)")


def test_batched_workload_all_heads():
    w = workloads.WORKLOADS["batched"]
    T_tot = w.nseq * w.T
    toks = workloads.make_tokens(T_tot, w.H, w.d, w.dtype, w.seed, DEV)
    pool = kda.Pool(w.page_bytes, 1024, DEV)
    dt = kda.DTYPES[w.dtype]
    P = pool.object_pages(w.H, w.d, dt)
    assert P == 17
    act = kda.kda_page_alloc(pool, w.nseq * P).reshape(w.nseq, P)
    cu = [i * w.T for i in range(w.nseq + 1)]
    sp = [0] * w.nseq
    run = Prefill(pool, toks, cu, sp, [0] * w.nseq, act, stride=w.stride, include_last=w.include_last)
    ck = oracle_positions(cu, sp, w.stride, w.include_last)
    assert ck == [[2048, 4096, 6144, 8192]] * 4
    cpu = {k: v.cpu() for k, v in toks.items()}
    ref = oracle_prefill(cpu, cu, sp, ckpt_abs=ck)
    compare_prefill(pool, run, ref, cu, act, w.dtype, ck, name="batched workload prefill (bf16)")
    # checkpoint pages: lowest free first after the active objects, in (sequence, position) order
    sim = policy.PoolSim(1024)
    sim.alloc(w.nseq * P)
    want = policy.plan_checkpoints(sim, [(0, w.T)] * w.nseq, P, 512, w.stride, w.include_last)
    assert [list(map(int, r)) for r in run.pages] == [pg for _, _, pg in want]


def test_varlen_resume_workload():
    w = workloads.WORKLOADS["varlen_resume"]
    H, d, dt = w.H, w.d, kda.DTYPES[w.dtype]
    L = workloads.varlen_lengths(w.seed, w.nseq)
    B = workloads.resume_points(L, w.seed)
    cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int64)
    toks = workloads.make_tokens(int(cu[-1]), H, d, w.dtype, w.seed, DEV)
    P = policy.object_pages(H, d, w.dtype, w.page_bytes)
    n_setup = sum(len(policy.ckpt_positions(0, x, 512, 1, False)) for x in L)
    n_new = sum(len(policy.ckpt_positions(b, x, 512, w.stride, w.include_last)) for b, x in zip(B, L))
    pool = kda.Pool(w.page_bytes, (2 * w.nseq + n_setup + n_new) * P + 64, DEV)
    # setup: every sequence in full, a checkpoint at every 512 end
    act0 = kda.kda_page_alloc(pool, w.nseq * P).reshape(w.nseq, P)
    setup = Prefill(pool, toks, cu, [0] * w.nseq, [0] * w.nseq, act0, stride=1, include_last=False)
    where = {(int(s), int(p)): i for i, (s, p) in enumerate(zip(setup.seq, setup.pos))}
    # restore each sequence's resume checkpoint into a fresh private object
    act = kda.kda_page_alloc(pool, w.nseq * P).reshape(w.nseq, P)
    rs = [s for s in range(w.nseq) if B[s] > 0]
    ck_pages = np.stack([setup.pages[where[(s, B[s])]] for s in rs])
    ws = torch.empty(kda.kda_copy_workspace_bytes(len(rs), P), dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kda.kda_ckpt_restore(pool, H, d, dt, ck_pages.reshape(-1), act[rs].reshape(-1), ws, st)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    kda.kda_ckpt_release(pool, ck_pages.reshape(-1), P)
    nb = policy.object_bytes(H, d, w.dtype)
    for i, s in enumerate(rs):
        assert read_object_bytes(pool, act[s], nb) == read_object_bytes(pool, ck_pages[i], nb)
    # resumed prefill of the suffixes
    suf_rows = [torch.arange(int(cu[s]) + B[s], int(cu[s + 1]), device=DEV) for s in range(w.nseq)]
    idx = torch.cat(suf_rows)
    suf = {k: (v[idx] if k != "conv_w" else v) for k, v in toks.items()}
    cu2 = np.concatenate([[0], np.cumsum([x - b for x, b in zip(L, B)])])
    run = Prefill(pool, suf, cu2, B, [1 if b > 0 else 0 for b in B], act, stride=w.stride,
                  include_last=w.include_last)
    ck = oracle_positions(cu2, B, w.stride, w.include_last)
    assert ckpt_lists(run, w.nseq) == [list(x) for x in ck]
    # oracle from token 0 on every (sequence, head) pair, one sequence (all heads) at a time
    tol = TOL[w.dtype]
    worst = 0.0
    o = run.o
    for s in range(w.nseq):
        rows = slice(int(cu[s]), int(cu[s + 1]))
        cpu = _cpu_heads(toks, rows, list(range(H)))
        ref = oracle.kda_run(cpu["q"], cpu["k"], cpu["v"], cpu["alpha"], cpu["beta"], cpu["conv_w"],
                             [0, L[s]], ckpt_counts=[list(ck[s])])
        got_o = o[int(cu2[s]):int(cu2[s + 1])].float().cpu().numpy()
        S, W = read_object(pool, act[s], H, d, w.dtype)
        mine = [i for i, q in enumerate(run.seq) if int(q) == s]
        cks = [read_object(pool, run.pages[i], H, d, w.dtype) for i in mine]
        for h in range(H):
            worst = max(worst, assert_close(got_o[:, h], ref["o"][B[s]:, h], tol, f"o seq {s} head {h}", name=NM_VARLEN))
            worst = max(worst, assert_close(S[h], ref["S"][0, h], tol, f"final S seq {s} head {h}", name=NM_VARLEN))
            for n, i in enumerate(mine):
                worst = max(worst, assert_close(cks[n][0][h], ref["ck_S"][0][n][h], tol,
                                                f"ckpt {run.pos[i]} seq {s} head {h}", name=NM_VARLEN))
        assert np.array_equal(W, ref["win"][0]), f"final window seq {s}"
        for n in range(len(mine)):
            assert np.array_equal(cks[n][1], ref["ck_win"][0][n]), f"checkpoint window seq {s}"


def test_decode_workload():
    w = workloads.WORKLOADS["decode"]
    Bq, H, d, dt = w.nseq, w.H, w.d, kda.DTYPES[w.dtype]
    pool = kda.Pool(w.page_bytes, 4096, DEV)
    P = pool.object_pages(H, d, dt)
    assert P == 9
    table = workloads.permuted_page_table(4096, Bq, P, w.seed)
    kda.kda_page_claim(pool, table.reshape(-1))
    setup_T, steps = 512, 64
    toks = workloads.make_tokens(Bq * setup_T, H, d, w.dtype, w.seed, DEV)
    cu = [i * setup_T for i in range(Bq + 1)]
    Prefill(pool, toks, cu, [0] * Bq, [0] * Bq, table.numpy(), checkpoints=False)
    conv_w = toks["conv_w"]
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    td = table.to(DEV)
    outs, step_toks = [], []
    for s in range(steps):
        t = workloads.decode_step_tokens(Bq, H, d, w.dtype, w.seed, s, DEV)
        o = torch.full_like(t["q"], float("nan"))
        kda.kda_decode_step(pool, t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, o, td, st)
        outs.append(o.float().cpu())
        step_toks.append({k: v.cpu() for k, v in t.items()})
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    got_all = torch.stack(outs).numpy()                                   # [steps, B, H, d]
    tol = TOL[w.dtype]
    worst = 0.0
    # oracle on every request (all heads), 32 requests per call: setup tokens then the steps
    group = 32
    for r0 in range(0, Bq, group):
        reqs = list(range(r0, min(r0 + group, Bq)))
        seq = {}
        for k in ("q", "k", "v", "alpha", "beta"):
            parts = []
            for r in reqs:
                parts.append(toks[k][r * setup_T:(r + 1) * setup_T].cpu())
                parts.append(torch.stack([step_toks[s][k][r] for s in range(steps)]))
            seq[k] = torch.cat(parts)
        n_tok = setup_T + steps
        ref = oracle.kda_run(seq["q"], seq["k"], seq["v"], seq["alpha"], seq["beta"], conv_w.cpu(),
                             [i * n_tok for i in range(len(reqs) + 1)])
        for i, r in enumerate(reqs):
            got = got_all[:, r]                                           # [steps, H, d]
            want = ref["o"][i * n_tok + setup_T:(i + 1) * n_tok]
            S, W = read_object(pool, table[r], H, d, w.dtype)
            for h in range(H):
                worst = max(worst, assert_close(got[:, h], want[:, h], tol, f"decode o req {r} head {h}", name=NM_DECODE))
                worst = max(worst, assert_close(S[h], ref["S"][i, h], tol, f"decode state req {r} head {h}", name=NM_DECODE))
            assert np.array_equal(W, ref["win"][i]), f"decode window req {r}"


@pytest.mark.slow
def test_long_workload_four_heads():
    w = workloads.WORKLOADS["long"]
    H, d, dt = w.H, w.d, kda.DTYPES[w.dtype]
    toks = workloads.make_tokens(w.T, H, d, w.dtype, w.seed, DEV)
    P = policy.object_pages(H, d, w.dtype, w.page_bytes)
    pool = kda.Pool(w.page_bytes, 513 * P + 64, DEV)
    act = kda.kda_page_alloc(pool, P).reshape(1, P)
    run = Prefill(pool, toks, [0, w.T], [0], [0], act, stride=w.stride, include_last=w.include_last)
    ck = oracle_positions([0, w.T], [0], w.stride, w.include_last)
    assert len(ck[0]) == 512 and [int(p) for p in run.pos] == ck[0]
    heads = [0, 11, 22, 31]
    cpu = _cpu_heads(toks, slice(0, w.T), heads)
    import concurrent.futures as cf

    # conv weights differ per head: one oracle call per head, run in parallel threads
    def one(i):
        h = heads[i]
        return oracle.kda_run(cpu["q"][:, i:i + 1], cpu["k"][:, i:i + 1], cpu["v"][:, i:i + 1],
                              cpu["alpha"][:, i:i + 1], cpu["beta"][:, i:i + 1], toks["conv_w"][h:h + 1].cpu(),
                              [0, w.T], ckpt_counts=[ck[0]])

    with cf.ThreadPoolExecutor(4) as ex:
        refs = list(ex.map(one, range(4)))
    S, W = read_object(pool, act[0], H, d, w.dtype)
    tol = TOL[w.dtype]
    worst = 0.0
    for i, h in enumerate(heads):
        worst = max(worst, assert_close(run.o[:, h].float().cpu().numpy(), refs[i]["o"][:, 0], tol,
                                        f"long o head {h}", name=NM_LONG))
        worst = max(worst, assert_close(S[h], refs[i]["S"][0, 0], tol, f"long final S head {h}", name=NM_LONG))
        assert np.array_equal(W[h], refs[i]["win"][0, 0])
    for n in range(512):
        Sc, Wc = read_object(pool, run.pages[n], H, d, w.dtype)
        for i, h in enumerate(heads):
            worst = max(worst, assert_close(Sc[h], refs[i]["ck_S"][0][n][0], tol, f"long ckpt {n} head {h}", name=NM_LONG))
            assert np.array_equal(Wc[h], refs[i]["ck_win"][0][n][0])
