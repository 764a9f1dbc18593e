#!/usr/bin/env python3
"""Benchmark of the DCP decode hot path on one GB300 (or N replicas).

One step = one decode token per request through the whole path:
per-rank context lengths, slot mapping of the B new tokens, owner-masked
cache write, per-rank split-KV partial attention and the exact LSE merge
(``dcp_local_seq_lens`` + ``dcp_slot_mapping`` + ``dcp_cache_write_*`` +
``dcp_decode_*``), on the GQA workload B=32, Hq=32, Hkv=8, d=128, bf16,
bimodal 1k-256k contexts, dcp=8, block_size 16 (other workloads with
--config).  The KV cache is resident state, built once before timing.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config NAME] [--no-extra] [--no-cpu-baseline] [--no-graph]

Prints one JSON line (rank 0).  ``value`` is KV-read GB/s of the step
(KV bytes the step must read / device time).  After the headline workload
the default run measures the other workloads (MLA B=64, SFA B=32, long-tail
GQA and MLA) in the same process, each with its own clock record, and
reports them under ``configs`` (``--no-extra`` skips them).  The timed steps replay the
step captured once as a CUDA graph, as a serving loop would (``--no-graph``
launches the kernels one by one).  ``e2e`` is the same metric through the
public calls with the per-step inputs copied from pinned host memory and the
output copied back inside the timed region; the step and its copies are
captured as one graph too (eager calls with ``--no-graph``).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KV-read GB/s & decode tok/s of sharded attn + LSE merge, % of roofline (1 GB300)"
FALLBACK_HBM_GBS = 6800.0
# nominal HBM3e rate of a GB300 (the figure the ">= 75% of HBM peak" target
# is stated against); the roofline fraction is also given against the
# measured copy rate, which a streaming-read kernel can exceed
NOMINAL_HBM_GBS = 7900.0
EXTRA_CONFIGS = ("mla_bf16_b64", "sfa_bf16_b32", "longtail_gqa", "longtail_mla")


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


FALLBACK_BF16_TFLOPS = 1900.0

# DRAM traffic of the dominant kernel from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum), taken on a smaller case of the same workload and
# scaled to a full launch by the KV bytes processed (traffic grows in
# proportion: the kernel reads each KV byte once).  Valid only while the
# kernel source is the one captured (sha256 prefix); otherwise null.
NCU_TRAFFIC = {
    "gqa_bf16_b32": {"source": "context_paged_decode_gb300/csrc/dcp_gqa.cu",
                     "sha256_16": "e99da6e59345a4eb", "dram_bytes": 1159464704 + 6609152,
                     "kv_bytes": 282732 * 4096,
                     "capture": "profiles/gqa_tma_kernel_gqa_bf16_b32.md"},
    "mla_bf16_b64": {"source": "context_paged_decode_gb300/csrc/dcp_mla_tc.cu",
                     "sha256_16": "3fdb673daa322567", "dram_bytes": 251370240 + 5882112,
                     "kv_bytes": 216885 * 1152,
                     "capture": "profiles/mla_tc_kernel_mla_bf16_b64.md"},
    "sfa_bf16_b32": {"source": "context_paged_decode_gb300/csrc/dcp_sfa_tc.cu",
                     "sha256_16": "14ff0928b47b9535", "dram_bytes": 78460672 + 2981376,
                     "kv_bytes": 32 * 2048 * 1152,
                     "capture": "profiles/sfa_tc_kernel_sfa_bf16_b32.md"},
}
# the long-tail workloads run the same kernels
NCU_TRAFFIC["longtail_gqa"] = NCU_TRAFFIC["gqa_bf16_b32"]
NCU_TRAFFIC["longtail_mla"] = NCU_TRAFFIC["mla_bf16_b64"]


def traffic_per_launch(name, kv_bytes):
    import hashlib
    e = NCU_TRAFFIC.get(name)
    if not e:
        return None
    with open(os.path.join(ROOT, e["source"]), "rb") as f:
        if hashlib.sha256(f.read()).hexdigest()[:16] != e["sha256_16"]:
            return None
    return int(e["dram_bytes"] * kv_bytes / e["kv_bytes"])


def peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def step_flops(cfg, lens, B):
    """Algorithmic tensor flops of one decode step (Q.K^T + P.V, all heads)."""
    import numpy as np
    if cfg.kind == "sfa":
        tokens = B * cfg.topk
    else:
        tokens = int(np.asarray(lens, dtype=np.int64).sum())
    return tokens * cfg.Hq * (2 * cfg.dk + 2 * cfg.dv)


class Clocks:
    """nvidia-smi samples (every 100 ms) around the timed region.

    Samples taken inside [begin, end] are used; a region shorter than the
    sampling interval is represented by the last sample before it and the
    first after it ("bracketing")."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.samples = []          # (time, sm, max, reasons)
        self.t0 = self.t1 = None

    def _reader(self):
        for line in self.proc.stdout:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm, mx = float(f[1]), float(f[2])
            except ValueError:
                continue
            rs = {n for n, v in zip(self.NAMES, f[5:9]) if v.lower().startswith("active")}
            self.samples.append((time.monotonic(), sm, mx, rs))

    def start(self):
        """Start sampling and wait (up to 3 s) for the first sample."""
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._reader, daemon=True).start()
        t_end = time.monotonic() + 3.0
        while not self.samples and time.monotonic() < t_end:
            time.sleep(0.01)

    def begin(self):
        self.t0 = time.monotonic()

    def end(self):
        self.t1 = time.monotonic()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        t_end = time.monotonic() + 1.0  # one sample after the region
        while time.monotonic() < t_end and not (self.samples and self.samples[-1][0] > self.t1):
            time.sleep(0.01)
        self.proc.terminate()
        try:
            self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [x for x in self.samples if self.t0 <= x[0] <= self.t1]
        how = "inside the timed region"
        if not inside:
            before = [x for x in self.samples if x[0] < self.t0][-1:]
            after = [x for x in self.samples if x[0] > self.t1][:1]
            inside, how = before + after, "bracketing the timed region (shorter than the 100 ms interval)"
        sm = [x[1] for x in inside]
        reasons = set().union(*[x[3] for x in inside]) if inside else set()
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(x[2] for x in inside) if inside else None,
                "reasons": sorted(reasons), "samples": len(inside), "sampled": how}


# ---------------------------------------------------------------------------
# whole-job aggregation over ranks (replicas)
# ---------------------------------------------------------------------------

def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings over the default process group
    (identity without one).  Every rank gets the result."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_value(units_per_rank, world, seconds):
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return world * units_per_rank / seconds


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def workload_config(cfg, lens, world):
    """The workload a line measures (the same dict in both arms)."""
    import numpy as np
    kv = step_bytes(cfg, lens, len(lens))[0]
    if cfg.kind == "sfa":
        kv = cfg.B * cfg.topk * cfg.dk * 2
    return {"workload": cfg.description, "name": cfg.name, "batch": cfg.B,
            "context_tokens": int(np.asarray(lens, dtype=np.int64).sum()),
            "kv_bytes_per_step": int(kv),
            "parallelism": f"dcp{cfg.dcp} virtual ranks on 1 GPU" +
                           (f" x {world} replicas" if world > 1 else "")}


def step_bytes(cfg, lens, B):
    """(KV bytes, total algorithmic bytes) of one decode step."""
    import numpy as np
    es = 2 if cfg.dtype == "bf16" else 4
    tokens = int(np.asarray(lens, dtype=np.int64).sum())
    if cfg.kind == "gqa":
        kv = tokens * cfg.Hkv * cfg.dk * 2 * es
        new_tok = B * cfg.Hkv * cfg.dk * 2 * es * 2          # read + write of the new k/v rows
    else:
        kv = tokens * cfg.dk * es
        new_tok = B * cfg.dk * es * 2
    q = B * cfg.Hq * cfg.dk * es
    out = B * cfg.Hq * cfg.dv * es + B * cfg.Hq * 4
    partial = 2 * cfg.dcp * B * cfg.Hq * (cfg.dv + 1) * 4    # per-rank partials written + read
    nvb = (np.asarray(lens, dtype=np.int64) + cfg.bs * cfg.dcp - 1) // (cfg.bs * cfg.dcp)
    bt = int(nvb.sum()) * cfg.dcp * 4
    return kv, kv + new_tok + q + out + partial + bt


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def staged(tensors, dev):
    """One device byte buffer holding copies of `tensors` (None entries kept
    as None) at 256-byte offsets; returns (buffer, views in the same order)."""
    import torch
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        if t is not None:
            total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(tensors, offs):
        if t is None:
            views.append(None)
            continue
        v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


def measure(cfg, args, world, dev, local_rank, with_e2e=True):
    """Time one workload: the step (replayed as a CUDA graph unless
    --no-graph), the decode call alone (roofline), and the end-to-end step
    with its host copies.  Returns (result dict, host context lengths)."""
    import torch

    import context_paged_decode_gb300 as dcp
    import workloads as W
    from workloads import device as D

    t0 = time.time()
    wl = D.build(cfg, device=dev)
    torch.cuda.synchronize()
    setup_s = time.time() - t0
    B = cfg.B
    lay = wl.layout
    tdt = D.torch_dtype(cfg.dtype)
    stream = torch.cuda.current_stream()

    # per-step inputs: the new token of every request sits at position L_b - 1
    req = torch.arange(B, dtype=torch.int32, device=dev)
    pos = (wl.seq_lens.to(torch.int64) - 1).contiguous()
    if cfg.kind == "gqa":
        newk = torch.empty((B, cfg.Hkv, cfg.dk), dtype=tdt, device=dev)
        newv = torch.empty_like(newk)
        row = cfg.Hkv * cfg.dk
        for b in range(B):
            x = int(wl.seq_lens_host[b]) - 1
            D.fill(newk[b], cfg.seed, W.T_K, b, x * row, cfg.dtype)
            D.fill(newv[b], cfg.seed, W.T_V, b, x * row, cfg.dtype)
    else:
        newk = torch.empty((B, cfg.dk), dtype=tdt, device=dev)
        newv = None
        for b in range(B):
            x = int(wl.seq_lens_host[b]) - 1
            D.fill(newk[b], cfg.seed, W.T_LATENT, b, x * cfg.dk, cfg.dtype)
    kind = {"gqa": dcp.KIND_GQA, "mla": dcp.KIND_MLA, "sfa": dcp.KIND_SFA}[cfg.kind]
    ws = torch.empty(dcp.decode_workspace_size(lay, kind, B, cfg.Hq, cfg.Hkv, cfg.dv),
                     dtype=torch.uint8, device=dev)
    out = torch.empty((B, cfg.Hq, cfg.dv), dtype=tdt, device=dev)
    out_lse = torch.empty((B, cfg.Hq), dtype=torch.float32, device=dev)
    # A step's inputs (q, the new token's rows, positions, lengths) and its
    # results (output, LSE) each live in one device buffer, at 256-byte
    # offsets, so the end-to-end step moves them with one copy per direction.
    in_buf, in_views = staged([wl.q, newk, newv, pos, wl.seq_lens], dev)
    wl.q, newk, newv, pos, wl.seq_lens = in_views
    out_buf, (out, out_lse) = staged([out, out_lse], dev)
    local = torch.empty((B, cfg.dcp), dtype=torch.int32, device=dev)
    o_rank = torch.empty(B, dtype=torch.int32, device=dev)
    o_slot = torch.empty((cfg.dcp, B), dtype=torch.int64, device=dev)
    kv = wl.kv

    def decode():
        if cfg.kind == "gqa":
            dcp.decode_gqa(lay, wl.q, kv, local, cfg.scale, sink=wl.sink, out=out,
                           out_lse=out_lse, workspace=ws)
        elif cfg.kind == "mla":
            dcp.decode_mla(lay, wl.q, kv, local, cfg.scale, cfg.dv, sink=wl.sink, out=out,
                           out_lse=out_lse, workspace=ws)
        else:
            dcp.sfa_decode(lay, wl.q, kv, wl.topk, wl.seq_lens, cfg.scale, cfg.dv, sink=wl.sink,
                           out=out, out_lse=out_lse, workspace=ws)

    def step():
        dcp.local_seq_lens(lay, wl.seq_lens, out=local)
        dcp.slot_mapping(lay, req, pos, wl.block_table, wl.num_blocks, out_rank=o_rank,
                         out_slot=o_slot)
        if cfg.kind == "gqa":
            dcp.cache_write_gqa(lay, newk, newv, o_slot, wl.k_pools, wl.v_pools, wl.num_blocks)
        else:
            dcp.cache_write_mla(lay, newk, o_slot, wl.k_pools, wl.num_blocks)
        decode()

    # lengths, slot mapping and cache write, then the decode call's three
    # kernels (plan or remap, partials, merge)
    launches_per_step = 3 + 3
    kv_bytes, alg_bytes = step_bytes(cfg, wl.seq_lens_host, B)
    if cfg.kind == "sfa":
        kv_bytes = B * cfg.topk * cfg.dk * 2
        alg_bytes = kv_bytes + B * cfg.Hq * cfg.dk * 2 + 2 * cfg.dcp * B * cfg.Hq * (cfg.dv + 1) * 4 \
            + B * cfg.topk * 4 + B * cfg.Hq * (cfg.dv * 2 + 4)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # warm-up
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    run_step = step
    graph = e2e_graph = None
    if not args.no_graph:
        # the step as one CUDA graph: every call reads its sizes from device
        # memory and allocates nothing, so the launches capture as they are
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        run_step = graph.replay

    # A working set that fits in L2 (the SFA rows a step gathers) would be
    # served from L2 by the next step: flush it before every timed call by
    # writing a buffer four times the L2 size, outside the timed interval.
    flush = kv_bytes <= 512 << 20
    l2buf = torch.empty(512 << 20, dtype=torch.uint8, device=dev) if flush else None

    def timed(fn, k):
        """Mean device ms per call of fn over k calls (CUDA events on `stream`)."""
        if not flush:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(k):
                fn()
            b.record(stream)
            b.synchronize()
            return a.elapsed_time(b) / k
        tot = 0.0
        for i in range(k):
            l2buf.fill_(i & 0xff)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            tot += a.elapsed_time(b)
        return tot / k

    # timed steps (device time, CUDA events on the launching stream)
    clk = Clocks(local_rank)
    clk.start()
    barrier()
    torch.cuda.synchronize()
    clk.begin()
    step_ms = timed(run_step, args.steps)
    torch.cuda.synchronize()
    barrier()

    # the dominant call alone: per-launch durations of the decode call
    dec_ms = [timed(decode, 1) for _ in range(args.steps)]

    e2e_ms = None
    h2d = in_buf.numel()
    d2h = out_buf.numel()
    if with_e2e:
        # end to end: host inputs (pinned) -> device, step, output -> host,
        # one copy per direction of the staged buffers
        h_in = torch.empty(in_buf.shape, dtype=torch.uint8, pin_memory=True)
        h_in.copy_(in_buf)
        h_res = torch.empty(out_buf.shape, dtype=torch.uint8, pin_memory=True)

        def e2e_step():
            in_buf.copy_(h_in, non_blocking=True)
            step()
            h_res.copy_(out_buf, non_blocking=True)

        for _ in range(max(1, args.warmup)):
            e2e_step()
        torch.cuda.synchronize()
        run_e2e = e2e_step
        if not args.no_graph:
            # the same step with its host copies (pinned inputs in, result
            # out), captured once and replayed: every replay moves the bytes
            e2e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graph):
                e2e_step()
            torch.cuda.synchronize()
            e2e_graph.replay()
            torch.cuda.synchronize()
            run_e2e = e2e_graph.replay
        barrier()
        e2e_ms = timed(run_e2e, args.steps)
        torch.cuda.synchronize()
        barrier()
    # the clock record spans the step, decode-call and end-to-end timings
    clk.end()
    clocks = clk.stop()

    step_ms, e2e_ms_all, dec_avg = max_over_ranks(
        [step_ms, e2e_ms if e2e_ms is not None else 0.0, statistics.mean(dec_ms)],
        device=dev if world > 1 else None)
    if e2e_ms is not None:
        e2e_ms = e2e_ms_all

    hbm_peak, tc_peak, peak_src = peaks()
    flops = step_flops(cfg, wl.seq_lens_host, B)
    t_hbm = alg_bytes / (hbm_peak * 1e9)
    t_tc = flops / (tc_peak * 1e12)
    tensor_bound = cfg.kind != "gqa" and t_tc > t_hbm
    achieved = alg_bytes / (dec_avg * 1e-3) / 1e9
    value = job_value(kv_bytes, world, step_ms * 1e-3) / 1e9
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": round(flops / (dec_avg * 1e-3) / 1e12, 1),
                "peak": tc_peak, "peak_source": f"{peak_src} bf16_tflops", "unit": "TFLOP/s",
                "frac": round(flops / (dec_avg * 1e-3) / 1e12 / tc_peak, 4), "traffic": None}
    else:
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                "peak_source": f"{peak_src} hbm_gbs", "unit": "GB/s",
                "frac": round(achieved / hbm_peak, 4),
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "nominal_peak": NOMINAL_HBM_GBS,
                "traffic": traffic_per_launch(cfg.name if not args.reqs else "", kv_bytes)}
    res = {
        "value": round(value, 2),
        "unit": "GB/s",
        "ms_per_step": round(step_ms, 4),
        "decode_tok_per_s": round(job_value(B, world, step_ms * 1e-3), 1),
        "config": workload_config(cfg, wl.seq_lens_host, world),
        "timing": {"l2": "inputs larger than L2 (KV >> 129 MB)" if not flush
                   else "L2 flushed before every timed call (512 MB write)",
                   "launch": "step kernels launched one by one" if args.no_graph
                   else "step replayed as one CUDA graph (e2e: the step and its host copies "
                        "replayed as one graph)"},
        "roofline": roof,
        "roofline_detail": {"kernel": f"dcp_decode_{cfg.kind} (plan + split + merge)",
                            "alg_bytes_per_launch": alg_bytes, "alg_flops_per_launch": flops,
                            "launch_ms": round(dec_avg, 4),
                            "roofline_ms": round(1e3 * max(t_hbm, t_tc), 4),
                            "hbm_ms": round(1e3 * t_hbm, 4), "tensor_ms": round(1e3 * t_tc, 4),
                            "tensor_tflops": round(flops / (dec_avg * 1e-3) / 1e12, 1),
                            "roofline_frac": round(1e3 * max(t_hbm, t_tc) / dec_avg, 4)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "setup_s": round(setup_s, 2),
    }
    if e2e_ms is not None:
        res["e2e"] = {"value": round(job_value(kv_bytes, world, e2e_ms * 1e-3) / 1e9, 2),
                      "unit": "GB/s", "ms_per_step": round(e2e_ms, 4),
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    lens = wl.seq_lens_host.copy()
    # release the workload before the next one is built
    del graph, e2e_graph, wl, kv, ws, in_buf, out_buf, l2buf
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res, lens


def run_ours(args, rank, world, local_rank):
    import torch

    import __graft_entry__
    import workloads as W

    __graft_entry__.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    cfg = W.CONFIGS[args.config]
    if args.reqs:
        import dataclasses
        cfg = dataclasses.replace(cfg, B=args.reqs,
                                  lengths=[int(x) for x in W.make_seq_lens(cfg)[:args.reqs]])
    head, lens = measure(cfg, args, world, dev, local_rank)
    res = {
        "metric": METRIC,
        "value": head["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded N(0,1) values; context lengths from the trace statistics)",
        "config": head["config"],
        "timing": head["timing"],
        "decode_tok_per_s": head["decode_tok_per_s"],
        "e2e": head["e2e"],
        "roofline": head["roofline"],
        "gpu_launches": head["gpu_launches"],
        "roofline_detail": head["roofline_detail"],
        "clocks": head["clocks"],
        "setup_s": head["setup_s"],
    }
    if not args.no_extra and not args.reqs:
        # every other workload, after the headline, in the same process: the
        # step, the decode call's roofline, e2e and clocks of each
        extra = {}
        for name in EXTRA_CONFIGS:
            if name == cfg.name:
                continue
            r, _ = measure(W.CONFIGS[name], args, world, dev, local_rank)
            extra[name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "decode_tok_per_s",
                                             "roofline", "roofline_detail", "e2e", "clocks",
                                             "gpu_launches")}
            extra[name]["config"] = r["config"]
            extra[name]["timing"] = r["timing"]
        res["configs"] = extra
    return res, cfg, lens


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm, and the cpu_baseline of our arm)
# ---------------------------------------------------------------------------

def blas_threads():
    """Threads numpy's BLAS runs with (the oracle's matmuls), else the host's
    CPU count: threadpoolctl when installed, else the OpenBLAS that numpy
    loaded, found in this process's memory map."""
    try:
        from threadpoolctl import threadpool_info
        n = sum(i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas")
        if n > 0:
            return n
    except Exception:
        pass
    try:
        import ctypes
        import re
        import numpy as np
        np.dot(np.ones((64, 64)), np.ones((64, 64)))        # make sure the BLAS is loaded
        with open("/proc/self/maps") as f:
            paths = {m.group(1) for m in (re.search(r"(/\S*openblas\S*\.so\S*)", ln) for ln in f) if m}
        for path in sorted(paths):
            lib = ctypes.CDLL(path)
            for name in ("openblas_get_num_threads", "openblas_get_num_threads64_",
                         "scipy_openblas_get_num_threads64_", "scipy_openblas_get_num_threads"):
                fn = getattr(lib, name, None)
                if fn is not None:
                    n = int(fn())
                    if n > 0:
                        return n
    except Exception:
        pass
    return os.cpu_count()


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in r.stdout.splitlines():
            if line.strip().lower().startswith("model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_baseline(cfg, lens, budget_s, seed=0, kind="oracle"):
    """The fp64 oracle timed on a bounded sample of the workload, with the
    host it ran on and the sample's share of one full step's KV bytes."""
    b, s, what = oracle_sample(cfg, lens, budget_s, seed=seed)
    kv_step = step_bytes(cfg, lens, len(lens))[0]
    return {"value": round(b / s / 1e9, 4), "unit": "GB/s", "cores": blas_threads(),
            "kind": kind, "cpu_model": cpu_model(), "nproc": os.cpu_count(),
            "sample": what + f", {s:.1f} s",
            "sample_kv_bytes": int(b), "step_kv_bytes": int(kv_step),
            "sample_fraction_of_step": round(b / kv_step, 5)}


def oracle_sample(cfg, lens, budget_s, seed=0):
    """Time the fp64 oracle on whole (request, head) problems until budget_s of
    oracle compute; returns (KV bytes covered, seconds, description)."""
    import numpy as np

    import oracle as O
    from tests import ref

    rng = np.random.default_rng(seed)
    order = rng.permutation(len(lens))
    done_bytes, spent, n = 0.0, 0.0, 0
    G = cfg.Hq // cfg.Hkv if cfg.kind == "gqa" else cfg.Hq
    es = 2 if cfg.dtype == "bf16" else 4
    for b in order:
        L = int(lens[b])
        if cfg.kind == "gqa":
            g = int(rng.integers(cfg.Hkv))
            K, V = ref.gqa_kv(cfg, b, g, L)
            heads = [g * G + i for i in range(G)]
            unit_bytes = L * cfg.dk * 2 * es          # one kv head's K and V, read once per group
        else:
            K, V = ref.latent_kv(cfg, b, L)
            heads = list(range(cfg.Hq))
            unit_bytes = L * cfg.dk * es
        qs = [ref.q_vec(cfg, b, h) for h in heads]
        t0 = time.perf_counter()
        for i, q in enumerate(qs):
            O.sharded_attention(q, K, V, cfg.scale, L, cfg.dcp, cfg.bs, cfg.I)
            if cfg.kind != "gqa" and time.perf_counter() - t0 + spent > budget_s:
                unit_bytes *= (i + 1) / len(qs)
                break
        spent += time.perf_counter() - t0
        done_bytes += unit_bytes
        n += 1
        if spent > budget_s:
            break
    what = (f"{n} requests x one kv head group ({G} q heads), full context, fp64 oracle"
            if cfg.kind == "gqa" else f"{n} requests x all {cfg.Hq} heads (last partial), fp64")
    return done_bytes, spent, what


def run_reference(args, rank, world):
    """Reference arm: the CPU oracle (no reference implementation exists)."""
    import workloads as W

    cfg = W.CONFIGS[args.config]
    lens = W.make_seq_lens(cfg)
    per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    for i in range(args.warmup):
        oracle_sample(cfg, lens, per_step, seed=100 + i)
    tot_b, tot_s, what = 0.0, 0.0, ""
    for i in range(args.steps):
        b, s, what = oracle_sample(cfg, lens, per_step, seed=i)
        tot_b += b
        tot_s += s
    v = tot_b / tot_s / 1e9
    kv_step = step_bytes(cfg, lens, len(lens))[0]
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_s / max(1, args.steps), 2), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(cfg, lens, world),
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": blas_threads(),
                         "kind": "oracle", "cpu_model": cpu_model(), "nproc": os.cpu_count(),
                         "sample": f"per step: {what}",
                         "sample_fraction_of_step": round(tot_b / max(1, args.steps) / kv_step,
                                                          5)},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="gqa_bf16_b32")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="measure only the --config workload (not the other four)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the step's kernels one by one instead of replaying a CUDA graph")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--reqs", type=int, default=0,
                    help="keep only the first N requests of the workload (profiling cases)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    if world > 1:
        import torch
        torch.distributed.init_process_group("nccl")
    res, cfg, lens = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(cfg, lens, args.cpu_budget)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
