"""Benchmark of the KDA state path on GB300.

One step = one pass of the prefill path over the batched workload (4 sequences x 8192
tokens, H = 16, d = 128, bf16 inputs, fp32 state, chunk 64, checkpoints at every 4th
512-token hash-block end into a pool of 64 KiB pages): host checkpoint plan and page
allocation, one prefill launch (conv, chunked recurrence, outputs, checkpoint streaming,
final-state write), then the checkpoint pages are released for the next step.  The decode
step (256 requests x 32 heads through a permuted page table), checkpoint write/restore
copies, the plain CPU-GPU link copy rate, the 1M-token long-context prefill and the
varlen-resume prefill are measured in the same run and reported beside the headline number,
and the oracle is timed on bounded samples of each workload on the host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch under torch.distributed.run: each rank runs its own batch on its own GPU
(weak scaling, no data-path collective); timings are maxed over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KDA prefill tokens/s and decode step µs at B=256; % of tensor/HBM roofline"
WORKLOAD = "batched"
# sources of the dominant (prefill) kernel, for matching committed ncu traffic to the code
PREFILL_SOURCES = ["kernels/prefill_split.cu", "kernels/tc_common.cuh", "kernels/sm100_ptx.cuh",
                   "kernels/common.cuh", "kda_internal.h", "host/split_plan.cpp"]


# --------------------------------------------------------------------------- helpers
def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def _kernel_source_hash(files):
    """Hash of the kernel's sources with comments and blank lines removed (a comment edit
    does not change the kernel the counters were taken on)."""
    import re
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "kda_state_chunked_gb300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


def _traffic(kernel: str, source_files, scale: float):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)[kernel]
    except Exception:
        return None
    if t.get("source_hash") != _kernel_source_hash(source_files):
        return None
    return float(t["dram_bytes_per_unit"]) * scale


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        import torch
        try:
            uuid = "GPU-" + str(torch.cuda.get_device_properties(self.dev).uuid)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", uuid, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------- workload
class BatchedPrefill:
    """The batched prefill workload resident on one GPU."""

    def __init__(self, dev, seed_offset: int = 0):
        import torch
        import kda_state_chunked_gb300 as kda
        from kda_state_chunked_gb300 import workloads
        self.kda = kda
        self.w = w = workloads.WORKLOADS[WORKLOAD]
        self.dev = dev
        self.T_tot = w.nseq * w.T
        self.toks = workloads.make_tokens(self.T_tot, w.H, w.d, w.dtype, w.seed + seed_offset, dev)
        self.cu = [i * w.T for i in range(w.nseq + 1)]
        self.start = [0] * w.nseq
        self.dt = kda.DTYPES[w.dtype]
        self.pool = kda.Pool(w.page_bytes, 1024, dev)
        self.P = self.pool.object_pages(w.H, w.d, self.dt)
        self.active = kda.kda_page_alloc(self.pool, w.nseq * self.P).reshape(w.nseq, self.P)
        self.o = torch.empty_like(self.toks["q"])
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        n_ck = sum(len(kda.kda_ckpt_positions(0, w.T, w.hash_block, w.stride, w.include_last))
                   for _ in range(w.nseq))
        self.n_ckpt = n_ck
        self.ws = kda.prefill_workspace(self.toks["q"], self.cu, self.start, n_ck, self.P)
        self.rec = kda.kda_record_bytes(w.d, self.dt)
        self.launches_per_step = kda.kda_prefill_kernel_launches(w.H, w.d, self.dt, self.cu, self.start)

    def step(self, toks=None, o=None):
        kda, w = self.kda, self.w
        t = toks or self.toks
        seq, pos, pages = kda.kda_ckpt_plan(self.pool, w.H, w.d, self.dt, self.cu, self.start,
                                            w.hash_block, w.stride, w.include_last)
        kda.kda_prefill_varlen(self.pool, self.cu, self.start, [0] * w.nseq, t["q"], t["k"], t["v"],
                               t["alpha"], t["beta"], t["conv_w"], o if o is not None else self.o,
                               self.active, seq, pos, pages, self.ws, self.status)
        kda.kda_page_decref(self.pool, pages.reshape(-1))

    def algorithmic_bytes(self) -> int:
        w = self.w
        es = 2 if w.dtype == "bf16" else 4
        th = self.T_tot * w.H
        tokens = th * (4 * w.d * es + es + w.d * es)     # q, k, v, alpha, beta in; o out
        states = (self.n_ckpt + w.nseq) * w.H * self.rec  # checkpoints + final states
        return tokens + states

    def algorithmic_flops(self) -> int:
        w = self.w
        C, d = 64, w.d
        return self.T_tot * w.H * (6 * d * d + 4 * C * d + C * C // 3)


def _time_steps(fn, steps, warmup, stream, min_warm_s=0.0):
    """Run `warmup` untimed steps (and keep warming for at least min_warm_s, so that the
    clock sampler has samples under load), then time exactly `steps` steps with CUDA events
    on `stream`.  Returns (total ms, per-step ms list)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < min_warm_s:
        for _ in range(max(1, warmup)):
            fn()
        torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    per = [a.elapsed_time(b) for a, b in ev]
    return start.elapsed_time(end), per


def _decode_phase(dev, steps=64, warmup=3):
    """Decode workload: 256 requests x 32 heads, states in a 4096-page pool of 256 KiB pages
    addressed through a permuted page table; states come from a 512-token setup prefill."""
    import torch
    import kda_state_chunked_gb300 as kda
    from kda_state_chunked_gb300 import workloads
    w = workloads.WORKLOADS["decode"]
    dt = kda.DTYPES[w.dtype]
    pool = kda.Pool(w.page_bytes, 4096, dev)
    P = pool.object_pages(w.H, w.d, dt)
    table = workloads.permuted_page_table(4096, w.nseq, P, w.seed)
    kda.kda_page_claim(pool, table.reshape(-1))
    setup_T = 512
    toks = workloads.make_tokens(w.nseq * setup_T, w.H, w.d, w.dtype, w.seed, dev)
    cu = [i * setup_T for i in range(w.nseq + 1)]
    ws = kda.prefill_workspace(toks["q"], cu, [0] * w.nseq, 0, P)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    o = torch.empty_like(toks["q"])
    kda.kda_prefill_varlen(pool, cu, [0] * w.nseq, [0] * w.nseq, toks["q"], toks["k"], toks["v"],
                           toks["alpha"], toks["beta"], toks["conv_w"], o, table.numpy(), [], [], None,
                           ws, st)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    del toks, o
    step_toks = [workloads.decode_step_tokens(w.nseq, w.H, w.d, w.dtype, w.seed, s, dev)
                 for s in range(steps)]
    conv_w = workloads.make_tokens(1, w.H, w.d, w.dtype, w.seed, dev)["conv_w"]
    table_dev = table.to(dev)
    od = torch.empty_like(step_toks[0]["q"])
    stream = torch.cuda.current_stream()
    it = iter(range(10 ** 9))

    def one():
        t = step_toks[next(it) % steps]
        kda.kda_decode_step(pool, t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, od,
                            table_dev, st)

    total, per = _time_steps(one, steps, warmup, stream)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    es = 2
    bytes_per = w.nseq * w.H * (2 * w.d * w.d * 4 + 2 * 3 * 3 * w.d * es + 4 * w.d * es + es + w.d * es)
    us = statistics.median(per) * 1e3
    del pool
    # ping-pong: every request writes its new state to its second object (all of them at a
    # decode-checkpoint boundary), alternating between two permuted page tables
    pool2 = kda.Pool(w.page_bytes, 2 * w.nseq * P, dev)
    pool2.base.zero_()
    both = workloads.permuted_page_table(2 * w.nseq * P, 2 * w.nseq, P, w.seed)
    kda.kda_page_claim(pool2, both.reshape(-1))
    ta, tb = both[:w.nseq].to(dev), both[w.nseq:].to(dev)
    it2 = iter(range(10 ** 9))

    def one_pp():
        i = next(it2)
        t = step_toks[i % steps]
        src, dst = (ta, tb) if i % 2 == 0 else (tb, ta)
        kda.kda_decode_step_pp(pool2, t["q"], t["k"], t["v"], t["alpha"], t["beta"], conv_w, od, src, dst, st)

    _, per_pp = _time_steps(one_pp, steps, warmup, stream)
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    us_pp = statistics.median(per_pp) * 1e3
    del pool2
    # speculative verify: K = 4 draft tokens per request, the state after each kept
    K = 4
    pool3 = kda.Pool(w.page_bytes, (K + 1) * w.nseq * P, dev)
    pool3.base.zero_()
    src3 = kda.kda_page_alloc(pool3, w.nseq * P).reshape(w.nseq, P)
    inter3 = torch.from_numpy(kda.kda_verify_plan(pool3, w.H, w.d, dt, w.nseq, K)).to(dev)
    src3_dev = torch.from_numpy(src3).to(dev)
    drafts = {k: torch.stack([step_toks[j][k] for j in range(K)]) for k in step_toks[0]}
    ov = torch.empty_like(drafts["q"])

    def one_verify():
        kda.kda_verify_step(pool3, drafts["q"], drafts["k"], drafts["v"], drafts["alpha"], drafts["beta"], conv_w,
                            ov, src3_dev, inter3, st)

    _, per_v = _time_steps(one_verify, steps, warmup, stream)
    rec = kda.kda_record_bytes(w.d, dt)
    verify_bytes = w.nseq * w.H * ((K + 1) * rec + K * (4 * w.d * es + es + w.d * es))
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    us_v = statistics.median(per_v) * 1e3
    return {"step_us": us, "mean_step_us": total * 1e3 / steps, "steps": steps, "B": w.nseq, "H": w.H,
            "bytes_per_step": bytes_per, "achieved_gbs": bytes_per / (us * 1e-6) / 1e9,
            "l2": "state set 1.1 GB per step > L2",
            "pingpong": {"step_us": us_pp, "achieved_gbs": bytes_per / (us_pp * 1e-6) / 1e9,
                         "note": "every request writes its next state to a second object (a decode checkpoint "
                                 "by donation at every step)"},
            "verify": {"draft_tokens": K, "step_us": us_v, "draft_tokens_per_s": w.nseq * K / (us_v * 1e-6),
                       "algorithmic_bytes": verify_bytes, "achieved_gbs": verify_bytes / (us_v * 1e-6) / 1e9,
                       "note": "one fused kernel: each source record read once, the record after every draft "
                               "token written to its own object (bytes: one record read, K record writes, the "
                               "draft tokens in and their outputs out)"}}


def _ckpt_io_phase(dev, n=256, reps=5):
    """Checkpoint write (snapshot) and restore of 256 objects of 32 heads, 64 KiB pages,
    timed over `reps` back-to-back calls each (host staging overlaps the previous copy)."""
    import torch
    import kda_state_chunked_gb300 as kda
    H, d, dt = 32, 128, kda.KDA_BF16
    P = 34
    pool = kda.Pool(65536, (2 + reps + 3) * n * P + 64, dev)
    assert pool.object_pages(H, d, dt) == P
    src = kda.kda_page_alloc(pool, n * P)
    act = kda.kda_page_alloc(pool, n * P)
    # states of realistic magnitude (N(0, 0.3^2) fp32 everywhere), so that the INT8 quantiser
    # divides every element as it does on real checkpoints (an all-zero row skips its divisions)
    torch.manual_seed(7)
    pool.base.view(torch.float32).normal_(0.0, 0.3)
    ws = [torch.empty(kda.kda_copy_workspace_bytes(n, P), dtype=torch.uint8, device=dev) for _ in range(4)]
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    nb = kda.kda_object_bytes(H, d, dt) * n * 2
    stream = torch.cuda.current_stream()
    res = {}
    for name in ("write", "restore"):
        for warm in (True, False):
            count = 2 if warm else reps
            dsts = []
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(count):
                if name == "write":
                    dsts.append(kda.kda_ckpt_write(pool, H, d, dt, src, ws[i % 4], st))
                else:
                    kda.kda_ckpt_restore(pool, H, d, dt, src, act, ws[i % 4], st)
            b.record(stream)
            torch.cuda.synchronize()
            for dst in dsts:
                kda.kda_page_decref(pool, dst.reshape(-1))
            if name == "restore":
                for _ in range(count):
                    kda.kda_ckpt_release(pool, src, P)
            ms = a.elapsed_time(b) / count
        res[name] = {"ms": ms, "gbs": nb / (ms * 1e-3) / 1e9, "calls_timed": reps}
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    res["objects"] = n
    res["bytes_moved"] = nb
    # INT8 checkpoints: quantise the same objects into new INT8 checkpoints, and dequantise
    # them back into the private objects (bytes: one full and one INT8 object each way)
    Pq = kda.kda_object_pages_q8(pool, H, d, dt)
    nbq = (kda.kda_object_bytes(H, d, dt) + kda.kda_object_bytes_q8(H, d, dt)) * n
    for name in ("write_q8", "restore_q8"):
        for warm in (True, False):
            count = 2 if warm else reps
            made = []
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(count):
                if name == "write_q8":
                    made.append(kda.kda_ckpt_write_q8(pool, H, d, dt, src, ws[i % 4], st))
                else:
                    kda.kda_ckpt_restore_q8(pool, H, d, dt, q8_ck, act, ws[i % 4], st)
            b.record(stream)
            torch.cuda.synchronize()
            if name == "write_q8":
                q8_ck = made[-1].reshape(-1)
                for m in made[:-1]:
                    kda.kda_page_decref(pool, m.reshape(-1))
                if not warm:
                    keep = q8_ck
                else:
                    kda.kda_page_decref(pool, q8_ck)
            else:
                for _ in range(count):
                    kda.kda_ckpt_release(pool, q8_ck, Pq)
            ms = a.elapsed_time(b) / count
        if name == "write_q8":
            q8_ck = keep
        res[name] = {"ms": ms, "gbs": nbq / (ms * 1e-3) / 1e9, "calls_timed": reps}
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    res["bytes_moved_q8"] = nbq
    res["q8_compression"] = kda.kda_object_bytes(H, d, dt) / kda.kda_object_bytes_q8(H, d, dt)
    # write-back host offload and prefetch of the same objects through pinned, device-mapped
    # host memory (CPU-GPU link; one object size per call)
    nbo = kda.kda_object_bytes(H, d, dt) * n
    host = torch.empty(nbo, dtype=torch.uint8).pin_memory()
    for name in ("offload", "prefetch"):
        for warm in (True, False):
            count = 2 if warm else reps
            made = []
            torch.cuda.synchronize()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for i in range(count):
                if name == "offload":
                    kda.kda_ckpt_offload(pool, H, d, dt, src, host, ws[i % 4], st)
                else:
                    made.append(kda.kda_ckpt_prefetch(pool, H, d, dt, n, host, ws[i % 4], st))
            b.record(stream)
            torch.cuda.synchronize()
            for m in made:
                kda.kda_page_decref(pool, m.reshape(-1))
            ms = a.elapsed_time(b) / count
        res[name] = {"ms": ms, "gbs": nbo / (ms * 1e-3) / 1e9, "calls_timed": reps,
                     "bytes": nbo, "link": "CPU-GPU (pinned host memory)"}
    assert kda.kda_sync_status(st)[0] == kda.KDA_OK
    return res


def _prefill_algorithmic_bytes(token_heads: int, objects: int, H: int, rec: int) -> int:
    """q, k, v, alpha, beta in and o out (bf16, d = 128) per token-head, plus whole records."""
    return token_heads * (4 * 256 + 2 + 256) + objects * H * rec


def _long_phase(dev, steps=3, warmup=3):
    """Long-context prefill at its full size: one sequence of 1,048,576 tokens, H = 32, chunk
    64, checkpoints at every 4th 512-token hash-block end (512 checkpoints of 32 head records,
    1.11 GB streamed to the pool during the prefill), final state into the active object."""
    import torch
    import kda_state_chunked_gb300 as kda
    from kda_state_chunked_gb300 import workloads
    w = workloads.WORKLOADS["long"]
    T = w.T
    dt = kda.DTYPES[w.dtype]
    toks = workloads.make_tokens(T, w.H, w.d, w.dtype, w.seed, dev)
    n_ck = len(kda.kda_ckpt_positions(0, T, w.hash_block, w.stride, w.include_last))
    pool = kda.Pool(w.page_bytes, 64 + (n_ck + 2) * 34, dev)
    P = pool.object_pages(w.H, w.d, dt)
    act = kda.kda_page_alloc(pool, P).reshape(1, P)
    cu, st0 = [0, T], [0]
    ws = kda.prefill_workspace(toks["q"], cu, st0, n_ck, P)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    o = torch.empty_like(toks["q"])

    def one():
        seq, pos, pages = kda.kda_ckpt_plan(pool, w.H, w.d, dt, cu, st0, w.hash_block, w.stride, w.include_last)
        kda.kda_prefill_varlen(pool, cu, st0, [0], toks["q"], toks["k"], toks["v"], toks["alpha"], toks["beta"],
                               toks["conv_w"], o, act, seq, pos, pages, ws, status)
        kda.kda_page_decref(pool, pages.reshape(-1))

    total, per = _time_steps(one, steps, warmup, torch.cuda.current_stream())
    assert kda.kda_sync_status(status)[0] == kda.KDA_OK
    ms = statistics.median(per)
    ab = _prefill_algorithmic_bytes(T * w.H, n_ck + 1, w.H, kda.kda_record_bytes(w.d, dt))
    launches = kda.kda_prefill_kernel_launches(w.H, w.d, dt, cu, st0)
    del toks, o, ws, pool
    torch.cuda.empty_cache()
    return {"workload": f"long context: 1 sequence x {T:,} tokens, H={w.H}, d=128, bf16, chunk 64, "
                        f"{n_ck} checkpoints (every 4th 512-token hash-block end), 64 KiB pages",
            "tokens": T, "checkpoints": n_ck, "ms_per_step": ms, "tokens_per_s": T / (ms * 1e-3),
            "algorithmic_bytes": ab, "achieved_gbs": ab / (ms * 1e-3) / 1e9, "steps": steps,
            "launches_per_step": launches}


def _varlen_phase(dev, steps=5, warmup=3):
    """Varlen resume: 32 sequences (lengths uniform in [512, 32768], seed 2), H = 32; each
    step restores every resumed sequence's checkpoint into its private object and prefills
    the suffixes with new checkpoints (stride 4 + last), then releases the new pages."""
    import numpy as np
    import torch
    import kda_state_chunked_gb300 as kda
    from kda_state_chunked_gb300 import workloads
    w = workloads.WORKLOADS["varlen_resume"]
    H, d, dt = w.H, w.d, kda.DTYPES[w.dtype]
    L = workloads.varlen_lengths(w.seed, w.nseq)
    B = workloads.resume_points(L, w.seed)
    cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int64)
    toks = workloads.make_tokens(int(cu[-1]), H, d, w.dtype, w.seed, dev)
    rec = kda.kda_record_bytes(d, dt)
    n_setup = sum(len(kda.kda_ckpt_positions(0, x, 512, 1, False)) for x in L)
    n_new = sum(len(kda.kda_ckpt_positions(b, x, 512, w.stride, w.include_last)) for b, x in zip(B, L))
    pool = kda.Pool(w.page_bytes, 64 + (2 * w.nseq + n_setup + n_new) * 34, dev)
    P = pool.object_pages(H, d, dt)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # setup (untimed): every sequence in full with a checkpoint at every 512-token end
    act0 = kda.kda_page_alloc(pool, w.nseq * P).reshape(w.nseq, P)
    cu_l = [int(x) for x in cu]
    seq0, pos0, pages0 = kda.kda_ckpt_plan(pool, H, d, dt, cu_l, [0] * w.nseq, 512, 1, False)
    ws0 = kda.prefill_workspace(toks["q"], cu_l, [0] * w.nseq, len(seq0), P)
    o0 = torch.empty_like(toks["q"])
    kda.kda_prefill_varlen(pool, cu_l, [0] * w.nseq, [0] * w.nseq, toks["q"], toks["k"], toks["v"], toks["alpha"],
                           toks["beta"], toks["conv_w"], o0, act0, seq0, pos0, pages0, ws0, status)
    assert kda.kda_sync_status(status)[0] == kda.KDA_OK
    del o0, ws0
    where = {(int(s), int(p)): i for i, (s, p) in enumerate(zip(seq0, pos0))}
    rs = [s for s in range(w.nseq) if B[s] > 0]
    ck = np.stack([pages0[where[(s, B[s])]] for s in rs]).reshape(-1)
    act = kda.kda_page_alloc(pool, w.nseq * P).reshape(w.nseq, P)
    act_rs = act[rs].reshape(-1)
    cws = torch.empty(kda.kda_copy_workspace_bytes(len(rs), P), dtype=torch.uint8, device=dev)
    idx = torch.cat([torch.arange(int(cu[s]) + B[s], int(cu[s + 1]), device=dev) for s in range(w.nseq)])
    suf = {k: (v[idx] if k != "conv_w" else v) for k, v in toks.items()}
    del toks
    cu2 = [int(x) for x in np.concatenate([[0], np.cumsum([x - b for x, b in zip(L, B)])])]
    has = [1 if b > 0 else 0 for b in B]
    ws = kda.prefill_workspace(suf["q"], cu2, B, n_new, P)
    o = torch.empty_like(suf["q"])

    def one():
        kda.kda_ckpt_restore(pool, H, d, dt, ck, act_rs, cws, status)
        seq, pos, pages = kda.kda_ckpt_plan(pool, H, d, dt, cu2, B, 512, w.stride, w.include_last)
        kda.kda_prefill_varlen(pool, cu2, B, has, suf["q"], suf["k"], suf["v"], suf["alpha"], suf["beta"],
                               suf["conv_w"], o, act, seq, pos, pages, ws, status)
        kda.kda_page_decref(pool, pages.reshape(-1))
        kda.kda_ckpt_release(pool, ck, P)

    total, per = _time_steps(one, steps, warmup, torch.cuda.current_stream())
    assert kda.kda_sync_status(status)[0] == kda.KDA_OK
    ms = statistics.median(per)
    T_suf = cu2[-1]
    ab = _prefill_algorithmic_bytes(T_suf * H, n_new + w.nseq, H, rec) + 2 * len(rs) * H * rec
    return {"workload": "varlen resume: 32 sequences (lengths U[512, 32768], seed 2), H=32, restore of each "
                        "resume checkpoint + suffix prefill with stride-4 + last checkpoints",
            "suffix_tokens": T_suf, "restored_objects": len(rs), "new_checkpoints": n_new, "ms_per_step": ms,
            "tokens_per_s": T_suf / (ms * 1e-3), "algorithmic_bytes": ab,
            "achieved_gbs": ab / (ms * 1e-3) / 1e9, "steps": steps}


def _oracle_sample(toks_cpu_fn, gpu_o=None):
    """Time the oracle (as it stands) on one sequence of the batched workload.  With gpu_o
    (the library's output for that sequence, [T, H, d] on the host) the result also holds the
    worst max-relative error of the library's output per head against the oracle's."""
    import numpy as np
    import oracle
    from kda_state_chunked_gb300 import workloads
    w = workloads.WORKLOADS[WORKLOAD]
    t = toks_cpu_fn()
    ck = [[p for p in range(2048, w.T + 1, 2048)]]
    t0 = time.perf_counter()
    ref = oracle.kda_run(t["q"], t["k"], t["v"], t["alpha"], t["beta"], t["conv_w"], [0, w.T], ckpt_counts=ck)
    sec = time.perf_counter() - t0
    out = {"value": w.T / sec, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"sequence 0 of the batched workload: {w.T} tokens x {w.H} heads, conv + "
                     f"fp64 token recurrence + 4 checkpoints ({sec:.2f} s wall)"}
    if gpu_o is not None:
        worst = 0.0
        for h in range(w.H):
            r = ref["o"][:, h]
            worst = max(worst, float(np.max(np.abs(gpu_o[:, h] - r)) / np.max(np.abs(r))))
        out["parity"] = {"o_max_rel_err": worst, "tol": 2e-2,
                         "of": f"the timed step's output for sequence 0, all {w.H} heads, max |x - ref| / "
                               f"max |ref| per head against the oracle on the same inputs"}
    return out


def _oracle_workloads():
    """The oracle (as it stands, on the host cores) on bounded samples of the other workloads:
    one whole decode step (256 requests x 32 heads from random resident states), and 4,096-token
    samples x 32 heads shaped like the varlen-resume suffixes (resumed from a state) and the
    long-context sequence (checkpoints every 2,048 tokens)."""
    import numpy as np
    import oracle
    from kda_state_chunked_gb300 import workloads
    out = {}
    w = workloads.WORKLOADS["decode"]
    t = workloads.decode_step_tokens(w.nseq, w.H, w.d, w.dtype, w.seed, 0, "cpu")
    cw = workloads.make_tokens(1, w.H, w.d, w.dtype, w.seed, "cpu")["conv_w"]
    rng = np.random.default_rng(w.seed)
    S0 = rng.standard_normal((w.nseq, w.H, w.d, w.d)) * 0.3
    W0 = rng.standard_normal((w.nseq, w.H, 3, 3 * w.d))
    t0 = time.perf_counter()
    oracle.kda_run(t["q"], t["k"], t["v"], t["alpha"], t["beta"], cw, list(range(w.nseq + 1)), S0=S0, win0=W0)
    sec = time.perf_counter() - t0
    out["decode"] = {"value": sec * 1e6, "unit": "us per decode step", "kind": "oracle",
                     "sample": f"one whole step: {w.nseq} requests x {w.H} heads, one token each, from resident "
                               f"states ({sec:.3f} s wall)"}
    del S0, W0
    T = 4096
    for name, seed, init, ck in (("varlen_resume", workloads.WORKLOADS["varlen_resume"].seed, True, []),
                                  ("long", workloads.WORKLOADS["long"].seed, False, [2048, 4096])):
        ww = workloads.WORKLOADS[name]
        t = workloads.make_tokens(T, ww.H, ww.d, ww.dtype, seed, "cpu")
        S0 = rng.standard_normal((1, ww.H, ww.d, ww.d)) * 0.3 if init else None
        W0 = rng.standard_normal((1, ww.H, 3, 3 * ww.d)) if init else None
        t0 = time.perf_counter()
        oracle.kda_run(t["q"], t["k"], t["v"], t["alpha"], t["beta"], t["conv_w"], [0, T], S0=S0, win0=W0,
                       ckpt_counts=[ck])
        sec = time.perf_counter() - t0
        out[name] = {"value": T / sec, "unit": "tokens/s", "kind": "oracle",
                     "sample": f"{T} tokens x {ww.H} heads of a {'resumed suffix' if init else 'fresh sequence'}"
                               f" ({sec:.2f} s wall)"}
    return out


def _link_phase(dev, nbytes=1 << 29, reps=9):
    """Plain copy rate of the CPU-GPU link: one cudaMemcpyAsync of 512 MiB per call between
    pinned host memory and the device, each direction timed call by call (CUDA events on the
    copying stream) over `reps` calls after two untimed ones; the median call gives the rate."""
    import torch
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    res = {}
    for name in ("h2d", "d2h"):
        times = []
        for i in range(2 + reps):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            if name == "h2d":
                d.copy_(host, non_blocking=True)
            else:
                host.copy_(d, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                times.append(a.elapsed_time(b))
        times.sort()
        res[name + "_gbs"] = nbytes / (times[len(times) // 2] * 1e-3) / 1e9
        res[name + "_gbs_range"] = [nbytes / (times[-1] * 1e-3) / 1e9, nbytes / (times[0] * 1e-3) / 1e9]
    res["bytes_per_copy"] = nbytes
    res["how"] = f"pinned host <-> device cudaMemcpyAsync, 512 MiB per call, median of {reps} calls"
    del host, d
    return res


# --------------------------------------------------------------------------- replicas
def _max_over_ranks(x: float, world: int, device="cpu") -> float:
    """Max of a per-rank number over all ranks (NCCL wants the tensor on the GPU)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0].item())


def _aggregate(units_per_rank_step: int, steps: int, total_ms_max: float, world: int):
    """Whole-job throughput: all ranks' units over the slowest rank's time (weak scaling)."""
    ms = total_ms_max / steps
    return ms, units_per_rank_step * world / (ms * 1e-3)


# --------------------------------------------------------------------------- end to end
def _e2e_pipelined(bench, steps: int, warmup: int, stream, world: int):
    """End-to-end steps through the public API from pinned host memory: every step copies its
    inputs host -> device, runs the prefill, and copies its output device -> host.  Steps are
    pipelined the way a serving loop would run them: the input copies of step i + 1 (four copy
    streams, one per large input: concurrent copies keep more of the link busy than one or two
    streams do) and the output copy of step i - 1 (a fifth stream) overlap the prefill of step i,
    with double-buffered device inputs and outputs ordered by events.  Returns (h2d bytes per
    step, d2h bytes per step, total ms of the `steps` timed steps, every copy included)."""
    import torch
    import torch.distributed as dist
    host = {k: v.cpu().pin_memory() for k, v in bench.toks.items()}
    o_host = [torch.empty(bench.o.shape, dtype=bench.o.dtype).pin_memory() for _ in range(2)]
    dtoks = [{k: torch.empty_like(v) for k, v in bench.toks.items()} for _ in range(2)]
    dout = [torch.empty_like(bench.o) for _ in range(2)]
    s_in = [torch.cuda.Stream() for _ in range(4)]
    s_out = torch.cuda.Stream()
    ev_in = [[torch.cuda.Event() for _ in s_in] for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]
    keys = sorted(host, key=lambda k: -host[k].numel())

    def step(i):
        b = i & 1
        for j, s in enumerate(s_in):
            if used[b]:
                s.wait_event(ev_comp[b])          # step i - 2 has read these inputs
            with torch.cuda.stream(s):
                for k in keys[j::len(s_in)]:
                    dtoks[b][k].copy_(host[k], non_blocking=True)
                ev_in[b][j].record(s)
            stream.wait_event(ev_in[b][j])
        if used[b]:
            stream.wait_event(ev_out[b])          # step i - 2's output has been copied out
        bench.step(dtoks[b], dout[b])
        ev_comp[b].record(stream)
        s_out.wait_event(ev_comp[b])
        with torch.cuda.stream(s_out):
            o_host[b].copy_(dout[b], non_blocking=True)
            ev_out[b].record(s_out)
        used[b] = True

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for s in s_in + [s_out]:
        s.wait_event(start)
    for i in range(steps):
        step(warmup + i)
    stream.wait_event(ev_out[(warmup + steps - 1) & 1])   # the last output is on the host
    end.record(stream)
    torch.cuda.synchronize()
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = o_host[0].numel() * o_host[0].element_size()
    return h2d, d2h, start.elapsed_time(end)


# --------------------------------------------------------------------------- arms
def run_ours(args, rank, world, dev):
    import torch
    import torch.distributed as dist
    torch.cuda.set_device(dev)
    peaks = _peaks()
    bench = BatchedPrefill(dev, seed_offset=rank * 1000)
    stream = torch.cuda.current_stream()
    w = bench.w

    # device-resident timed region
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        total_ms, per = _time_steps(bench.step, args.steps, args.warmup, stream, min_warm_s=1.0)
    rc, bits = bench.kda.kda_sync_status(bench.status)
    assert rc == bench.kda.KDA_OK, f"device status {bits}"
    # the last timed step's output for sequence 0, read back after the timed region
    o_seq0 = bench.o[:w.T].double().cpu().numpy() if rank == 0 and world == 1 and not args.no_cpu else None
    total_ms = _max_over_ranks(total_ms, world, dev)
    if world > 1:
        dist.barrier()
    ms_per_step, value = _aggregate(bench.T_tot, args.steps, total_ms, world)
    launch_ms = statistics.mean(per)
    ab = bench.algorithmic_bytes()
    achieved = ab / (launch_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
            "kernel": "prefill", "algorithmic_bytes_per_launch": ab,
            "launch_ms": launch_ms,
            "traffic": _traffic("prefill_batched", PREFILL_SOURCES, 1.0),
            "tensor": {"flops_per_launch": bench.algorithmic_flops(),
                       "achieved_tflops": bench.algorithmic_flops() / (launch_ms * 1e-3) / 1e12,
                       "peak_tflops": peaks["bf16_tflops"]}}
    roof["tensor"]["frac"] = roof["tensor"]["achieved_tflops"] / peaks["bf16_tflops"]

    # end to end through the public API with host buffers
    h2d, d2h, e2e_ms = _e2e_pipelined(bench, args.steps, args.warmup, stream, world)
    _, e2e_value = _aggregate(bench.T_tot, args.steps, _max_over_ranks(e2e_ms, world, dev), world)

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; q,k unit-norm N(0,1), v N(0,1), beta=sigmoid(N(0,1)), "
                    "alpha=sigmoid(N(3,1)), conv w N(0,0.5^2))",
            "config": {"workload": "batched prefill: 4 sequences x 8192 tokens, H=16, d_k=d_v=128, "
                                   "bf16 inputs, fp32 state, chunk 64, conv width 4, checkpoints at "
                                   "every 4th 512-token hash-block end, 64 KiB pages",
                       "nseq": w.nseq, "seq_len": w.T, "H": w.H, "d": w.d, "chunk": 64, "stride": w.stride,
                       "page_bytes": w.page_bytes, "checkpoints_per_step": bench.n_ckpt,
                       "l2": f"inputs larger than L2 ({ab / 1e6:.0f} MB per step, no flush)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "clocks": clk.summary(),
            "gpu_launches": args.steps * bench.launches_per_step}
    if rank == 0 and not args.no_extras:
        dec = _decode_phase(dev)
        dec["roofline"] = {"bound": "hbm", "achieved": dec["achieved_gbs"], "peak": peaks["hbm_gbs"],
                           "unit": "GB/s", "frac": dec["achieved_gbs"] / peaks["hbm_gbs"]}
        line["decode"] = dec
        io = _ckpt_io_phase(dev)
        for k in ("write", "restore", "write_q8", "restore_q8"):
            io[k]["frac"] = io[k]["gbs"] / peaks["hbm_gbs"]
        link = _link_phase(dev)
        line["link"] = link
        for k, direction in (("offload", "d2h_gbs"), ("prefetch", "h2d_gbs")):
            io[k]["link_frac"] = io[k]["gbs"] / link[direction]
        e2e_in_gbs = h2d / (e2e_ms / args.steps * 1e-3) / 1e9
        line["e2e"]["h2d_gbs"] = e2e_in_gbs
        line["e2e"]["link_frac"] = e2e_in_gbs / link["h2d_gbs"]
        line["ckpt_io"] = io
        for name, fn in (("long_prefill", _long_phase), ("varlen_resume", _varlen_phase)):
            r = fn(dev)
            r["roofline"] = {"bound": "hbm", "achieved": r["achieved_gbs"], "peak": peaks["hbm_gbs"], "unit": "GB/s",
                             "frac": r["achieved_gbs"] / peaks["hbm_gbs"]}
            line[name] = r
        line["gpu_launches"] = args.steps * bench.launches_per_step   # headline timed region
    if rank == 0 and world == 1 and not args.no_cpu:
        def cpu_toks():
            return {k: (v[:w.T] if k != "conv_w" else v).cpu() for k, v in bench.toks.items()}
        line["cpu_baseline"] = _oracle_sample(cpu_toks, gpu_o=o_seq0)
        line["parity"] = line["cpu_baseline"].pop("parity")
        if not args.no_extras:
            line["cpu_baseline"]["workloads"] = _oracle_workloads()
    return line


def run_reference(args, rank, world):
    """The oracle as it stands, on the host cores, over a bounded sample per step."""
    if rank != 0:
        return None
    import torch
    from kda_state_chunked_gb300 import workloads
    w = workloads.WORKLOADS[WORKLOAD]
    toks = workloads.make_tokens(w.T, w.H, w.d, w.dtype, w.seed, "cpu")
    samples = []
    for i in range(args.warmup + args.steps):
        r = _oracle_sample(lambda: toks)
        if i >= args.warmup:
            samples.append(r)
    sec = statistics.mean(w.T / s["value"] for s in samples)
    value = w.T / sec
    cb = dict(samples[-1])
    cb["value"] = value
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded, same distributions as the GPU arm)",
            "config": {"workload": "batched prefill (one 8192-token sequence x 16 heads per step: "
                                   "bounded sample of the 4-sequence workload)",
                       "nseq": 1, "seq_len": w.T, "H": w.H, "d": w.d},
            "cpu_baseline": cb,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the decode and copy phases")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch
    from kda_state_chunked_gb300.build import build
    build()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    line = run_ours(args, rank, world, f"cuda:{local}")
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
