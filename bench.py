"""Benchmark of the paged MLA decode path on one GB300 (or N replicas).

One step = one ``mla_decode_run`` (the CTA-pair decode kernel, then the
merge kernel for split requests) over one batch of the workload, inputs
resident in HBM.  Default workload: DeepSeek-V3-shaped decode, batch 64, 128
heads, kv_len 4096 per request, page size 64, bf16 cache, pages randomly
permuted over the pool.  Other modes (``--config``): ragged, long_b1,
long_b4, fp8, deepseek_mtp2 (two query tokens per request), long_b4_mtp4
(four query tokens per request of 16 heads, packed into one request's
rows), deepseek_absorbed (W_UK absorb + decode + W_UV projection),
deepseek_cascade (shared prefix + own suffix + state merge).

Prints one JSON line.  ``value`` is microseconds per batch (device time of
the timed steps, CUDA events on the launching stream).  The inputs are larger
than L2, and L2 is flushed between steps: a buffer larger than it is written,
then another read, so the next step finds neither its inputs nor dirty lines
in L2.  ``roofline`` reports the decode
kernel alone (timed with events recorded by the library around it) against
the measured HBM bandwidth; ``e2e`` is the same step through the host-buffer
entry point with the q / out / lse copies inside the timed region;
``cpu_baseline`` is the float64 oracle on a bounded sample of the batch.

``--impl reference`` times that oracle alone (the slow CPU reference of this
method) on the same workload, metric and unit.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MLA decode µs/batch, KV GB/s and % of HBM/bf16 roofline on 1 GB300"
UNIT = "us/batch"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FLOP_PER_TOKEN_HEAD = 2 * 576 + 2 * 512          # QK^T over 576 + PV over 512


def workload_config(x) -> dict:
    qtok = f", {x.q_len} query tokens per request (causal in the block)" if x.q_len > 1 else ""
    cfg = {"workload": f"paged MLA decode {x.name}: batch {x.batch}, heads {x.num_heads}, "
                       f"kv_len {'mixed' if len(set(x.kv_len.tolist())) > 1 else int(x.kv_len[0])}, "
                       f"page {x.page_size}, {x.kv_dtype} cache, kv_lora_rank 512, rope 64{qtok}",
           "batch": x.batch, "num_heads": x.num_heads, "page_size": x.page_size,
           "total_kv_tokens": x.total_tokens, "kv_dtype": x.kv_dtype,
           "sm_scale": x.sm_scale, "l2": L2_NOTE}
    if x.q_len > 1:
        cfg["q_len"] = x.q_len
    return cfg


def algorithmic(x) -> tuple[float, float]:
    """(bytes, flops) one batch must move / compute, pad rows not counted.
    With Q query tokens per request the cache is still needed once; query j
    of a request attends to kv_len - Q + 1 + j tokens."""
    tok = float(x.total_tokens)
    kv_bytes_per_tok = 576 * (2 if x.kv_dtype == "bf16" else 1)
    H, B, Q = x.num_heads, x.batch, x.q_len
    rows = B * Q * H
    nbytes = (tok * kv_bytes_per_tok + rows * (576 * 2 + 512 * 2 + 4)
              + 4 * len(x.kv_indices) + 8 * B)
    seen = float(Q * x.kv_len.astype(np.int64).sum() - B * Q * (Q - 1) // 2)
    flops = seen * H * FLOP_PER_TOKEN_HEAD
    return nbytes, flops


def pct(ms: list[float]) -> list[float]:
    """p10, p50, p90 of a list of millisecond times, in microseconds."""
    return [float(np.percentile(ms, q) * 1000) for q in (10, 50, 90)]


def peaks() -> tuple[float, float, float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            p = json.load(open(path))
            hbm = float(p.get("hbm_gbs") or p.get("hbm_GBps"))
            bf = float(p.get("bf16_tflops"))
            bfs = float(p.get("bf16_tflops_sustained", bf))
            return hbm, bf, bfs, "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


L2_NOTE = ("inputs larger than L2, and L2 flushed between steps: 256 MiB written, then "
           "256 MiB read, so no kernel input and no dirty line is left in it")


class L2Flush:
    """Between timed steps: write a 256 MiB buffer (evicting every kernel
    input from the 129 MB L2), then read another, so the write-backs of the
    dirty lines happen here and not inside the next timed step."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(256 << 20, dtype=torch.uint8, device=dev)

    def zero_(self):
        import torch
        self.w.zero_()
        self.r.view(torch.float32).sum()   # the read pass, reduced as fp32 words: no widened copy


# DRAM traffic of the dominant kernel per launch on the deepseek workload, from
# the committed ncu summaries: (summary, the sources the figure was taken of)
PAIR_SOURCES = ["decode_pair.cu", "tc_utils.cuh", "device_utils.cuh", "kernels.h", "mla_internal.h"]
PROFILES = {   # (kernel, workload) -> committed ncu figures and the sources they were taken from
    ("pair", "deepseek"): ("decode_pair_deepseek.json", PAIR_SOURCES),
    ("pair", "fp8"): ("decode_pair_fp8.json", PAIR_SOURCES),
    ("tcgen05", "deepseek"): ("decode_tc_deepseek.json",
                              ["decode_tc.cu", "tc_utils.cuh", "device_utils.cuh", "kernels.h", "mla_internal.h"]),
}
KERNEL_NAMES = {1: "tcgen05", 2: "mma_sync", 3: "pair"}   # mla_kernel_t values
# kernels one mla_decode_run launches per plan kernel: the one-CTA tcgen05
# kernel merges split requests itself, the others are followed by the merge
RUN_LAUNCHES = {1: 1, 2: 2, 3: 2}


def kernel_run(plan_kernel: int, requested: str, kv_dtype: str, page_size: int) -> str:
    """The decode kernel a run launches: a DEFAULT plan is made for the
    CTA-pair kernel and runs an fp8 cache with 16-token pages on the one-CTA
    kernel."""
    if requested == "default" and kv_dtype != "bf16" and page_size < 32:
        return "tcgen05"
    return KERNEL_NAMES[plan_kernel]


def profiled_traffic(workload: str, kernel: str) -> float | None:
    """DRAM bytes per launch of the decode kernel from the committed ncu
    summary, or None when there is none for this kernel and workload or the
    kernel sources changed since it was taken (hash recorded beside the
    figure)."""
    import hashlib
    if (kernel, workload) not in PROFILES:
        return None
    name, sources = PROFILES[(kernel, workload)]
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    h = hashlib.sha256()
    for f in sources:
        h.update(f.encode())
        with open(os.path.join(ROOT, "paged_mla_decode_02_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    vals = json.load(open(path))
    if vals.get("source_sha256") != h.hexdigest() or "dram_bytes_per_launch" not in vals:
        return None
    return float(vals["dram_bytes_per_launch"])


def oracle_sample(x, budget_s: float):
    """Float64 oracle on as many requests as fit in ~budget_s; returns (us per batch, n, secs)."""
    from oracle import mla_oracle as O
    order = list(range(x.batch))
    done, t0 = 0, time.perf_counter()
    for b in order:
        if x.q_len > 1:
            O.mla_decode_multi(x.q_nope, x.q_pe, x.ckv, x.kpe, x.kv_indptr, x.kv_indices,
                               x.kv_len, x.page_size, x.sm_scale, requests=[b])
        else:
            O.mla_decode_inputs(x, requests=[b])
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    secs = time.perf_counter() - t0
    tok_done = float(x.kv_len[:done].astype(np.int64).sum())
    us_per_batch = secs / max(tok_done, 1.0) * float(x.total_tokens) * 1e6
    return us_per_batch, done, secs


class ClockSampler:
    """SM clock and throttle reasons sampled through NVML (read-only queries)
    by a background thread, as fast as NVML answers, during the timed region."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap"}

    def __init__(self, index: int):
        import ctypes
        import threading
        self.samples, self.reasons, self.max_mhz, self.err = [], 0, None, None
        self._stop = threading.Event()
        try:
            nvml = ctypes.CDLL("libnvidia-ml.so.1")
            nvml.nvmlInit_v2()
            h = ctypes.c_void_p()
            nvml.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(h))
            mx = ctypes.c_uint()
            if nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:   # NVML_CLOCK_SM
                self.max_mhz = mx.value
            self._nvml, self._h = nvml, h
        except Exception as e:  # no driver library: report it, do not fail the bench
            self._nvml, self.err = None, str(e)
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()

    def _run(self):
        import ctypes
        if self._nvml is None:
            return
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self._nvml.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self._nvml.nvmlDeviceGetCurrentClocksEventReasons(self._h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(0.0005)

    def stop(self) -> dict:
        self._stop.set()
        self._t.join(timeout=5)
        names = sorted(n for bit, n in self.REASONS.items() if self.reasons & bit)
        out = {"sm_mhz": statistics.median(self.samples) if self.samples else None,
               "sm_max_mhz": self.max_mhz, "samples": len(self.samples), "reasons": names,
               "source": "nvml"}
        if self.err:
            out["error"] = self.err
        return out


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def job_us_per_batch(total_ms: float, steps: int, world: int, device=None) -> float:
    """Whole-job microseconds per batch for N replicas: each rank ran one
    batch per step, so the job did steps x world batches in the time of the
    slowest rank (max over ranks of its total)."""
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms * 1000.0 / steps / world


def run_reference(args, x) -> None:
    """Oracle-only arm: each step is a bounded sample of the batch on host cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    per_step = []
    for i in range(args.warmup + args.steps):
        us, n, secs = oracle_sample(x, args.ref_step_budget)
        if i >= args.warmup:
            per_step.append(us)
    value = statistics.mean(per_step)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": value / 1000.0, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(x),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"requests in ~{args.ref_step_budget:.0f}s per step, "
                                       f"scaled to the whole batch by token count"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


CASCADE_PREFIX, CASCADE_SUFFIX, CASCADE_BATCH = 2048, 2048, 64


def cascade_inputs():
    """64 requests of 128 heads over 64-token pages: a 2048-token prefix that
    every request shares, then 2048 tokens of each request's own.  Request 0
    of the generated batch holds the prefix pages; requests 1.. hold the
    suffixes and the queries."""
    from paged_mla_decode_02_gb300 import inputs as I
    return I.make_inputs("deepseek_cascade", [CASCADE_PREFIX] + [CASCADE_SUFFIX] * CASCADE_BATCH,
                         128, 64, seed=0)


def run_cascade(args) -> None:
    """Two-level decode step: the shared prefix (once per request) and the own
    suffixes as two planned batches, combined by mla_merge_states."""
    import torch
    from paged_mla_decode_02_gb300 import build as B
    from paged_mla_decode_02_gb300 import mla
    x = cascade_inputs()
    Bq, H, P = CASCADE_BATCH, x.num_heads, x.page_size
    torch.cuda.set_device(0)
    B.build()
    dev = torch.device("cuda", 0)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    qn, qp = bf16(x.q_nope[1:]), bf16(x.q_pe[1:])
    ckv, kpe = bf16(x.ckv), bf16(x.kpe)
    pre_pages = x.kv_indices[x.kv_indptr[0]:x.kv_indptr[1]]
    npre = len(pre_pages)
    pre_idx = torch.from_numpy(np.tile(pre_pages, Bq).astype(np.int32)).to(dev)
    suf_idx = torch.from_numpy(x.kv_indices[x.kv_indptr[1]:].astype(np.int32)).to(dev)
    stream = torch.cuda.Stream(device=dev)
    d_pre = mla.MLADecoder(Bq, H)
    d_suf = mla.MLADecoder(Bq, H)
    o0 = torch.empty((Bq, H, 512), dtype=torch.float32, device=dev)
    o1 = torch.empty_like(o0)
    l0 = torch.empty((Bq, H), dtype=torch.float32, device=dev)
    l1 = torch.empty_like(l0)
    out = torch.empty((Bq, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty_like(l0)
    flush = L2Flush(dev)
    with torch.cuda.stream(stream):
        d_pre.plan(np.arange(Bq + 1, dtype=np.int32) * npre, pre_idx,
                   np.full(Bq, CASCADE_PREFIX, np.int32), P, x.sm_scale)
        d_suf.plan(x.kv_indptr[1:] - x.kv_indptr[1], suf_idx, x.kv_len[1:], P, x.sm_scale)

    def step(q_nope, q_pe):
        d_pre.run(q_nope, q_pe, ckv, kpe, o0, l0, stream=stream)
        d_suf.run(q_nope, q_pe, ckv, kpe, o1, l1, stream=stream)
        mla.mla_merge_states(o0, l0, o1, l1, out, lse, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            step(qn, qp)
    stream.synchronize()
    d_pre.check_status()
    d_suf.check_status()
    # the three launches replayed from a CUDA graph: the timed region holds
    # the device work, not the host's tensor-map encoding between launches
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step(qn, qp)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(0)
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    d_pre.check_status()
    d_suf.check_status()
    us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1000.0

    # end to end: queries from pinned host memory in, output and lse back
    qn_h, qp_h = qn.cpu().pin_memory(), qp.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    qn_d, qp_d = torch.empty_like(qn), torch.empty_like(qp)
    e2e = []
    for i in range(args.steps + 2):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            qn_d.copy_(qn_h, non_blocking=True)
            qp_d.copy_(qp_h, non_blocking=True)
            step(qn_d, qp_d)
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
        stream.synchronize()
        if i >= 2:
            e2e.append((time.perf_counter() - t0) * 1e6)

    tok = float(CASCADE_PREFIX + Bq * CASCADE_SUFFIX)            # distinct cached tokens
    rows = Bq * H
    nbytes = (tok * 1152 + rows * (576 * 2 + 512 * 2 + 4)
              + 4 * (npre + len(suf_idx)) + 8 * Bq)
    flops = float(Bq) * (CASCADE_PREFIX + CASCADE_SUFFIX) * H * FLOP_PER_TOKEN_HEAD
    hbm, bf, _, peak_src = peaks()
    t_hbm, t_tc = nbytes / (hbm * 1e9) * 1e6, flops / (bf * 1e12) * 1e6
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    achieved = nbytes / (us * 1e-6) / 1e9 if bound == "hbm" else flops / (us * 1e-6) / 1e12
    peak = hbm if bound == "hbm" else bf
    line = {"metric": METRIC, "value": us, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": us / 1000.0, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"two-level (cascade) MLA decode: {Bq} requests, 128 heads, "
                                   f"a {CASCADE_PREFIX}-token prefix shared by all plus "
                                   f"{CASCADE_SUFFIX} own tokens each, page 64, bf16 cache; "
                                   f"prefix decode + suffix decode + state merge per step",
                       "batch": Bq, "num_heads": H, "page_size": P,
                       "l2": L2_NOTE},
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak,
                         "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": achieved / peak,
                         "traffic": None, "peak_source": peak_src,
                         "kernel": "whole step (two decode launches + merge)",
                         "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                         "roofline_time_us": max(t_hbm, t_tc)},
            "clocks": clk,
            "e2e": {"value": statistics.mean(e2e), "unit": UNIT,
                    "h2d_bytes_per_step": int((qn.numel() + qp.numel()) * 2),
                    "d2h_bytes_per_step": int(out.numel() * 2 + lse.numel() * 4)},
            "gpu_launches": (RUN_LAUNCHES[d_pre.info()["kernel"]] + RUN_LAUNCHES[d_suf.info()["kernel"]] + 1)
                            * args.steps,
            "cuda_graph": True}
    if not args.no_cpu_baseline:
        # the oracle on the concatenated pages of as many requests as fit the budget
        from oracle import mla_oracle as O
        t0, done = time.perf_counter(), 0
        for b in range(Bq):
            own = x.kv_indices[x.kv_indptr[b + 1]:x.kv_indptr[b + 2]]
            pages = np.concatenate([pre_pages, own]).astype(np.int32)
            O.mla_decode(x.q_nope[b + 1:b + 2], x.q_pe[b + 1:b + 2], x.ckv, x.kpe,
                         np.array([0, len(pages)], np.int32), pages,
                         np.array([CASCADE_PREFIX + CASCADE_SUFFIX], np.int32), P, x.sm_scale)
            done += 1
            if time.perf_counter() - t0 > args.cpu_budget:
                break
        secs = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": secs / done * Bq * 1e6, "unit": UNIT,
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{done} of {Bq} requests over their concatenated "
                                          f"pages ({secs:.1f}s float64 numpy), scaled to the batch"}
    print(json.dumps(line), flush=True)
    d_pre.close()
    d_suf.close()


def run_absorbed(args) -> None:
    """The absorbed decode layer: a head's no-rope query taken into the latent
    space (mla_absorb_q), the latent decode, and its output taken back to the
    head's value width (mla_project_out), on the deepseek decode shape with
    qk_nope_head_dim = v_head_dim = 128 (random weights)."""
    import torch
    from paged_mla_decode_02_gb300 import build as B
    from paged_mla_decode_02_gb300 import inputs as I
    from paged_mla_decode_02_gb300 import mla
    x = I.make_config("deepseek")
    Bq, H, P, dn, dv = x.batch, x.num_heads, x.page_size, 128, 128
    torch.cuda.set_device(0)
    B.build()
    dev = torch.device("cuda", 0)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    g = torch.Generator(device="cpu").manual_seed(0)
    q_raw = torch.randn((Bq, H, dn), generator=g).to(torch.bfloat16).to(dev)
    w_uk = (torch.randn((H, 512, dn), generator=g) / math.sqrt(dn)).to(torch.bfloat16).to(dev)
    w_uv = (torch.randn((H, 512, dv), generator=g) / math.sqrt(512)).to(torch.bfloat16).to(dev)
    q_pe, ckv, kpe = bf16(x.q_pe), bf16(x.ckv), bf16(x.kpe)
    idx = torch.from_numpy(x.kv_indices).to(dev)
    q_nope = torch.empty((Bq, H, 512), dtype=torch.bfloat16, device=dev)
    out = torch.empty((Bq, H, 512), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((Bq, H), dtype=torch.float32, device=dev)
    o = torch.empty((Bq, H, dv), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.Stream(device=dev)
    dec = mla.MLADecoder(Bq, H)
    with torch.cuda.stream(stream):
        dec.plan(x.kv_indptr, idx, x.kv_len, P, x.sm_scale)

    def step(qr):
        mla.mla_absorb_q(qr, w_uk, q_nope, stream=stream)
        dec.run(q_nope, q_pe, ckv, kpe, out, lse, stream=stream)
        mla.mla_project_out(out, w_uv, o, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            step(q_raw)
    stream.synchronize()
    dec.check_status()
    # the step: the chain's launches replayed from one CUDA graph (the host's
    # tensor-map encoding stays out of the timed region), L2 flushed before
    # each replay outside the events
    chain = torch.cuda.CUDAGraph()
    with torch.cuda.graph(chain, stream=stream):
        step(q_raw)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            chain.replay()
    stream.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(0)
    with torch.cuda.stream(stream):
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            chain.replay()
            e1.record(stream)
    stream.synchronize()
    clk = clocks.stop()
    dec.check_status()
    us = statistics.mean(a.elapsed_time(b) for a, b in ev) * 1000.0
    # the parts: each launch replayed from its own CUDA graph, events between
    graphs = []
    for fn in (lambda: mla.mla_absorb_q(q_raw, w_uk, q_nope, stream=stream),
               lambda: dec.run(q_nope, q_pe, ckv, kpe, out, lse, stream=stream),
               lambda: mla.mla_project_out(out, w_uv, o, stream=stream)):
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_, stream=stream):
            fn()
        graphs.append(g_)
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    with torch.cuda.stream(stream):
        for e in pev:
            flush.zero_()
            e[0].record(stream)
            for k, g_ in enumerate(graphs):
                g_.replay()
                e[k + 1].record(stream)
    stream.synchronize()
    dec.check_status()
    part = [statistics.mean(e[k].elapsed_time(e[k + 1]) for e in pev) * 1000.0 for k in range(3)]
    dec_us = part[1]

    qr_h = q_raw.cpu().pin_memory()
    qr_d = torch.empty_like(q_raw)
    o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    e2e = []
    for i in range(args.steps + 2):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            qr_d.copy_(qr_h, non_blocking=True)
            step(qr_d)
            o_h.copy_(o, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)
        stream.synchronize()
        if i >= 2:
            e2e.append((time.perf_counter() - t0) * 1e6)

    dec_bytes, dec_flops = algorithmic(x)
    rows = Bq * H
    # the chain's own inputs and outputs: q_raw in, o out, the two weights;
    # the latent q_nope / out between the launches are not counted
    nbytes = (dec_bytes - rows * (512 * 2 + 512 * 2) + rows * (dn * 2 + dv * 2)
              + H * 512 * (dn + dv) * 2)
    flops = dec_flops + 2.0 * rows * 512 * (dn + dv)
    hbm, bf, _, peak_src = peaks()
    t_hbm, t_tc = nbytes / (hbm * 1e9) * 1e6, flops / (bf * 1e12) * 1e6
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    achieved = nbytes / (us * 1e-6) / 1e9 if bound == "hbm" else flops / (us * 1e-6) / 1e12
    peak = hbm if bound == "hbm" else bf
    line = {"metric": METRIC, "value": us, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": us / 1000.0, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"absorbed MLA decode layer on the deepseek shape: {Bq} requests "
                                   f"x 4096 tokens, 128 heads, page 64; q_raw (dn {dn}) -> W_UK "
                                   f"absorb -> latent decode -> W_UV projection (dv {dv})",
                       "batch": Bq, "num_heads": H, "page_size": P,
                       "l2": L2_NOTE},
            "roofline": {"bound": bound, "achieved": achieved, "peak": peak,
                         "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": achieved / peak,
                         "traffic": None, "peak_source": peak_src,
                         "kernel": "whole step (absorb + decode + project launches)",
                         "decode_us": dec_us, "absorb_us": part[0], "project_us": part[2],
                         "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
                         "roofline_time_us": max(t_hbm, t_tc)},
            "clocks": clk,
            "e2e": {"value": statistics.mean(e2e), "unit": UNIT,
                    "h2d_bytes_per_step": int(qr_h.numel() * 2),
                    "d2h_bytes_per_step": int(o_h.numel() * 2 + lse_h.numel() * 4)},
            "gpu_launches": (2 + RUN_LAUNCHES[dec.info()["kernel"]]) * args.steps,
            "cuda_graph": True,
            "timing": {"method": "step: absorb, decode and project replayed from one CUDA graph; parts "
                                 "(absorb_us, decode_us, project_us): each launch replayed from its own "
                                 "graph, events between; L2 flushed before each replay, outside the events"}}
    print(json.dumps(line), flush=True)
    dec.close()


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="deepseek")
    ap.add_argument("--kernel", default="default", choices=["default", "tcgen05", "mma_sync", "pair"])
    ap.add_argument("--cpu-budget", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--ref-step-budget", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.config == "deepseek_absorbed":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the oracle arm is timed on the single-level configs"}))
            return
        run_absorbed(args)
        return
    if args.config == "deepseek_cascade":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the oracle arm is timed on the single-level configs"}))
            return
        run_cascade(args)
        return
    from paged_mla_decode_02_gb300 import inputs as I
    x = I.make_config(args.config)
    if args.impl == "reference":
        run_reference(args, x)
        return

    import torch
    import torch.distributed as dist
    from paged_mla_decode_02_gb300 import build as B
    from paged_mla_decode_02_gb300 import mla

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    B.build()
    dev = torch.device("cuda", local)

    def bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    def cache(a):
        if x.kv_dtype == "bf16":
            return bf16(a)
        return torch.from_numpy(np.ascontiguousarray(a)).to(dev).view(torch.float8_e4m3fn)

    q_nope, q_pe, ckv, kpe = bf16(x.q_nope), bf16(x.q_pe), cache(x.ckv), cache(x.kpe)
    idx = torch.from_numpy(x.kv_indices).to(dev)
    out = torch.empty(tuple(q_nope.shape[:-1]) + (512,), dtype=torch.bfloat16, device=dev)
    lse = torch.empty(tuple(q_nope.shape[:-1]), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)

    multi = x.q_nope.ndim == 4          # several query tokens per request
    dec = mla.MLADecoder(x.batch * x.q_len, x.num_heads, args.kernel)
    stream = torch.cuda.Stream(device=dev)
    t_plan = time.perf_counter()
    with torch.cuda.stream(stream):
        dec.plan(x.kv_indptr, idx, x.kv_len, x.page_size, x.sm_scale,
                 q_len=x.q_len if multi else 0)
    stream.synchronize()
    plan_us = (time.perf_counter() - t_plan) * 1e6
    info = dec.info()

    def step():
        dec.run(q_nope, q_pe, ckv, kpe, out, lse, kv_scale=x.kv_scale, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    dec.check_status()
    K = args.steps
    ev = lambda n: [torch.cuda.Event(enable_timing=True) for _ in range(n)]   # noqa: E731
    k0, k1, s0, s1, h0 = ev(K), ev(K), ev(K), ev(K), ev(K + 1)
    # torch creates an event lazily at its first record: create all of them
    # here, before the library is handed their handles
    with torch.cuda.stream(stream):
        for e in k0 + k1 + s0 + s1 + h0:
            e.record(stream)
        for _ in range(args.warmup):
            flush.zero_()
            step()
    stream.synchronize()

    # (1) the decode kernel alone: K eager runs, events the library records
    # immediately around its kernel launch (roofline.kernel_us)
    with torch.cuda.stream(stream):
        for i in range(K):
            flush.zero_()
            mla.mla_plan_set_profile_events(dec.handle, k0[i], k1[i])
            step()
    stream.synchronize()
    mla.mla_plan_set_profile_events(dec.handle, None, None)
    dec.check_status()
    kern_ms = [a.elapsed_time(b) for a, b in zip(k0, k1)]

    # (2) the timed steps: the run replayed from a CUDA graph, L2 flushed
    # before each replay (outside the events)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush.zero_()
            graph.replay()
    stream.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    wall0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush.zero_()
            s0[i].record(stream)
            graph.replay()
            s1[i].record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    dec.check_status()
    step_ms = [a.elapsed_time(b) for a, b in zip(s0, s1)]
    us_per_batch = job_us_per_batch(sum(step_ms), K, world, dev)

    # (3) hot: K replays back to back, nothing flushed (the inputs exceed L2,
    # so most of them still come from DRAM)
    with torch.cuda.stream(stream):
        h0[0].record(stream)
        for i in range(K):
            graph.replay()
            h0[i + 1].record(stream)
    stream.synchronize()
    dec.check_status()
    hot_ms = [h0[i].elapsed_time(h0[i + 1]) for i in range(K)]

    # end to end through the host-buffer entry point (q in, out / lse back)
    qn_h = q_nope.cpu().pin_memory()
    qp_h = q_pe.cpu().pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    for _ in range(3):
        mla.mla_decode_run_host(dec.handle, qn_h, qp_h, ckv, kpe, out_h, lse_h, x.kv_scale, stream)
    e2e = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        mla.mla_decode_run_host(dec.handle, qn_h, qp_h, ckv, kpe, out_h, lse_h, x.kv_scale, stream)
        e2e.append((time.perf_counter() - t0) * 1e6)
    e2e_us = job_us_per_batch(sum(e2e) / 1000.0, args.steps, world, dev)

    nbytes, flops = algorithmic(x)
    hbm, bf, bfs, peak_src = peaks()
    run_kernel = kernel_run(info["kernel"], args.kernel, x.kv_dtype, x.page_size)
    kern_us = statistics.mean(kern_ms) * 1000.0
    achieved_gbs = nbytes / (kern_us * 1e-6) / 1e9
    achieved_tf = flops / (kern_us * 1e-6) / 1e12
    t_hbm = nbytes / (hbm * 1e9) * 1e6
    t_tc = flops / (bf * 1e12) * 1e6
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    roof = {"bound": bound,
            "achieved": achieved_gbs if bound == "hbm" else achieved_tf,
            "peak": hbm if bound == "hbm" else bf,
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "peak_source": peak_src,
            "traffic": profiled_traffic(args.config, run_kernel),
            "traffic_unit": "bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum)",
            "kernel": f"mla_decode ({run_kernel} decode kernel)",
            "kernel_us": kern_us,
            "algorithmic_bytes": nbytes, "algorithmic_flops": flops,
            "achieved_tflops": achieved_tf, "achieved_gbs": achieved_gbs,
            "roofline_time_us": max(t_hbm, t_tc),
            "frac_of_roofline_time_step": max(t_hbm, t_tc) / us_per_batch}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if x.kv_dtype != "bf16" and run_kernel == "pair":
        # the pair kernel multiplies e4m3 codes (kind::f8f6f4) with two e4m3
        # terms for the query and for P: two e4m3 products per product of
        # the method, at twice the bf16 rate
        roof["tensor_accounting"] = (
            "e4m3 MMAs with two-term (hi + lo) query and P: 2 e4m3 products per algorithmic "
            "product, so the algorithmic flops are set against the measured bf16 peak (the same "
            "as the executed e4m3 flops against the e4m3 peak, measured bf16 x the nominal 2)")
        roof["frac_of_e4m3_peak_algorithmic_flops"] = achieved_tf / (2.0 * bf)
        roof["frac_of_hbm"] = achieved_gbs / hbm

    if rank != 0:
        return
    line = {"metric": METRIC, "value": us_per_batch, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": us_per_batch / 1000.0,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
            "dtype": ("bf16" if x.kv_dtype == "bf16" else
                      "fp8-e4m3 cache, e4m3 mma (hi + lo query and P)" if run_kernel == "pair" else
                      "fp8-e4m3 cache, bf16 mma"),
            "data": "synthetic", "config": workload_config(x),
            "kv_gbs": float(x.total_tokens) * 576 * (2 if x.kv_dtype == "bf16" else 1)
                      / (us_per_batch * 1e-6) / 1e9,
            "tflops": flops / (us_per_batch * 1e-6) / 1e12,
            "roofline": roof, "clocks": clk,
            "e2e": {"value": e2e_us, "unit": UNIT,
                    "h2d_bytes_per_step": int(qn_h.numel() * 2 + qp_h.numel() * 2),
                    "d2h_bytes_per_step": int(out_h.numel() * out_h.element_size()
                                              + lse_h.numel() * 4)},
            # tcgen05: one kernel per step (split requests merged in its epilogue);
            # CTA pair and mma.sync: decode + merge
            "gpu_launches": (1 if run_kernel == "tcgen05" else 2) * args.steps,
            "wall_s_timed": wall, "plan_us": plan_us,
            "kernel": run_kernel, "plan": info,
            "timing": {"method": "each timed step replays the run from a CUDA graph; CUDA events "
                                 "on the launching stream around each replay; L2 flushed before "
                                 "each cold replay, outside the events",
                       "cold_us_mean": us_per_batch,
                       "cold_us_p10_p50_p90": pct(step_ms),
                       "hot_us_mean": statistics.mean(hot_ms) * 1000.0,
                       "hot_us_p10_p50_p90": pct(hot_ms),
                       "kernel_us_p10_p50_p90": pct(kern_ms)}}
    if not args.no_cpu_baseline and world == 1:
        us, n, secs = oracle_sample(x, args.cpu_budget)
        line["cpu_baseline"] = {"value": us, "unit": UNIT, "cores": os.cpu_count(),
                                "kind": "oracle",
                                "sample": f"{n} of {x.batch} requests ({secs:.1f}s float64 numpy), "
                                          f"scaled to the batch by token count"}
    print(json.dumps(line), flush=True)
    dec.close()


if __name__ == "__main__":
    main()
