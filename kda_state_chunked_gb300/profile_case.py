"""Run one kernel of the library on a named workload a few times (for ncu captures).

python -m kda_state_chunked_gb300.profile_case prefill-batched --launches 2
python -m kda_state_chunked_gb300.profile_case decode --launches 3
python -m kda_state_chunked_gb300.profile_case ckpt-restore --launches 2
python -m kda_state_chunked_gb300.profile_case ckpt-write-q8 --launches 2
python -m kda_state_chunked_gb300.profile_case prefill-long-slice --launches 1

Cases
  prefill-batched     4 x 8192 tokens, H = 16, d = 128, bf16, checkpoints every 2048
  prefill-long-slice  one 65536-token slice of the long workload (H = 32), same layout
  prefill-tiny        the tiny fp32 workload: 1 x 1024 tokens, H = 2, d = 64 (CUDA-core kernel)
  decode              256 requests x 32 heads, 256 KiB pages, permuted page table
  ckpt-restore        256 objects x 32 heads copied checkpoint -> private, 64 KiB pages
  ckpt-write-q8       the same objects quantised into INT8 checkpoints
  ckpt-restore-q8     INT8 checkpoints dequantised into the private objects
  verify              speculative verify, 4 draft tokens for 256 requests x 32 heads
"""
from __future__ import annotations

import argparse

import torch

import kda_state_chunked_gb300 as kda
from kda_state_chunked_gb300 import workloads


def prefill(T_seq, nseq, H, seed, launches, dev):
    d, dt = 128, kda.KDA_BF16
    toks = workloads.make_tokens(nseq * T_seq, H, d, "bf16", seed, dev)
    pool = kda.Pool(65536, 64 + (nseq * (T_seq // 2048 + 1) + nseq) * 34, dev)
    P = pool.object_pages(H, d, dt)
    act = kda.kda_page_alloc(pool, nseq * P).reshape(nseq, P)
    cu = [i * T_seq for i in range(nseq + 1)]
    o = torch.empty_like(toks["q"])
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(launches):
        seq, pos, pages = kda.kda_ckpt_plan(pool, H, d, dt, cu, [0] * nseq, 512, 4, True)
        ws = kda.prefill_workspace(toks["q"], cu, [0] * nseq, len(seq), P)
        kda.kda_prefill_varlen(pool, cu, [0] * nseq, [0] * nseq, toks["q"], toks["k"], toks["v"],
                               toks["alpha"], toks["beta"], toks["conv_w"], o, act, seq, pos, pages, ws, st)
        torch.cuda.synchronize()
        kda.kda_page_decref(pool, pages.reshape(-1))
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK


def prefill_tiny(launches, dev):
    """The tiny fp32 workload: 1 sequence x 1024 tokens, H = 2, d = 64, checkpoints every 512."""
    w = workloads.WORKLOADS["tiny"]
    dt = kda.DTYPES[w.dtype]
    toks = workloads.make_tokens(w.nseq * w.T, w.H, w.d, w.dtype, w.seed, dev)
    pool = kda.Pool(w.page_bytes, 256, dev)
    P = pool.object_pages(w.H, w.d, dt)
    act = kda.kda_page_alloc(pool, w.nseq * P).reshape(w.nseq, P)
    cu = [i * w.T for i in range(w.nseq + 1)]
    o = torch.empty_like(toks["q"])
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(launches):
        seq, pos, pages = kda.kda_ckpt_plan(pool, w.H, w.d, dt, cu, [0] * w.nseq, 512, w.stride, w.include_last)
        ws = kda.prefill_workspace(toks["q"], cu, [0] * w.nseq, len(seq), P)
        kda.kda_prefill_varlen(pool, cu, [0] * w.nseq, [0] * w.nseq, toks["q"], toks["k"], toks["v"],
                               toks["alpha"], toks["beta"], toks["conv_w"], o, act, seq, pos, pages, ws, st)
        torch.cuda.synchronize()
        kda.kda_page_decref(pool, pages.reshape(-1))
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK


def decode(launches, dev):
    w = workloads.WORKLOADS["decode"]
    dt = kda.DTYPES[w.dtype]
    pool = kda.Pool(w.page_bytes, 4096, dev)
    P = pool.object_pages(w.H, w.d, dt)
    table = workloads.permuted_page_table(4096, w.nseq, P, w.seed)
    kda.kda_page_claim(pool, table.reshape(-1))
    conv_w = workloads.make_tokens(1, w.H, w.d, w.dtype, w.seed, dev)["conv_w"]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    td = table.to(dev)
    for s in range(launches):
        t = workloads.decode_step_tokens(w.nseq, w.H, w.d, w.dtype, w.seed, s, dev)
        o = torch.empty_like(t["q"])
        kda.kda_decode_step(pool, t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, o, td, st)
    torch.cuda.synchronize()
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK


def verify(launches, dev, K=4):
    """Speculative verify: K = 4 draft tokens for 256 requests x 32 heads (256 KiB pages)."""
    w = workloads.WORKLOADS["decode"]
    dt = kda.DTYPES[w.dtype]
    P = 9
    pool = kda.Pool(w.page_bytes, (K + 1) * w.nseq * P + 8, dev)
    assert pool.object_pages(w.H, w.d, dt) == P
    torch.manual_seed(7)
    pool.base.view(torch.float32).normal_(0.0, 0.3)
    src = torch.from_numpy(kda.kda_page_alloc(pool, w.nseq * P).reshape(w.nseq, P)).to(dev)
    inter = torch.from_numpy(kda.kda_verify_plan(pool, w.H, w.d, dt, w.nseq, K)).to(dev)
    conv_w = workloads.make_tokens(1, w.H, w.d, w.dtype, w.seed, dev)["conv_w"]
    steps = [workloads.decode_step_tokens(w.nseq, w.H, w.d, w.dtype, w.seed, j, dev) for j in range(K)]
    dr = {k: torch.stack([x[k] for x in steps]) for k in steps[0]}
    o = torch.empty_like(dr["q"])
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(launches):
        kda.kda_verify_step(pool, dr["q"], dr["k"], dr["v"], dr["alpha"], dr["beta"], conv_w, o, src, inter, st)
    torch.cuda.synchronize()
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK


def ckpt_restore(launches, dev, n=256):
    H, d, dt = 32, 128, kda.KDA_BF16
    pool = kda.Pool(65536, 2 * n * 34 + 64, dev)
    P = pool.object_pages(H, d, dt)
    src = kda.kda_page_alloc(pool, n * P)
    act = kda.kda_page_alloc(pool, n * P)
    ws = torch.empty(kda.kda_copy_workspace_bytes(n, P), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(launches):
        kda.kda_ckpt_restore(pool, H, d, dt, src, act, ws, st)
        torch.cuda.synchronize()
        kda.kda_ckpt_release(pool, src, P)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK


def ckpt_q8(launches, dev, n=256, restore=False):
    H, d, dt = 32, 128, kda.KDA_BF16
    pool = kda.Pool(65536, (launches + 3) * n * 34 + 64, dev)
    P = pool.object_pages(H, d, dt)
    Pq = kda.kda_object_pages_q8(pool, H, d, dt)
    src = kda.kda_page_alloc(pool, n * P)
    torch.manual_seed(7)
    pool.base.view(torch.float32).normal_(0.0, 0.3)     # every row has a nonzero scale
    ws = torch.empty(kda.kda_copy_workspace_bytes(n, P), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ck = kda.kda_ckpt_write_q8(pool, H, d, dt, src, ws, st).reshape(-1)
    torch.cuda.synchronize()
    for _ in range(launches):
        if restore:
            kda.kda_ckpt_restore_q8(pool, H, d, dt, ck, src, ws, st)
            torch.cuda.synchronize()
            kda.kda_ckpt_release(pool, ck, Pq)
        else:
            made = kda.kda_ckpt_write_q8(pool, H, d, dt, src, ws, st)
            torch.cuda.synchronize()
            kda.kda_page_decref(pool, made.reshape(-1))
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["prefill-batched", "prefill-long-slice", "prefill-tiny", "decode", "ckpt-restore",
                                     "ckpt-write-q8", "ckpt-restore-q8", "verify"])
    ap.add_argument("--launches", type=int, default=2)
    a = ap.parse_args()
    from kda_state_chunked_gb300.build import build
    build()
    dev = "cuda:0"
    if a.case == "prefill-batched":
        prefill(8192, 4, 16, 1, a.launches, dev)
    elif a.case == "prefill-long-slice":
        prefill(65536, 1, 32, 4, a.launches, dev)
    elif a.case == "prefill-tiny":
        prefill_tiny(a.launches, dev)
    elif a.case == "decode":
        decode(a.launches, dev)
    elif a.case == "ckpt-write-q8":
        ckpt_q8(a.launches, dev)
    elif a.case == "ckpt-restore-q8":
        ckpt_q8(a.launches, dev, restore=True)
    elif a.case == "verify":
        verify(a.launches, dev)
    else:
        ckpt_restore(a.launches, dev)
    print("ok")


if __name__ == "__main__":
    main()
