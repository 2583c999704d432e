#!/usr/bin/env python3
"""Throughput benchmark of the attention hot path on GB300.

A step is one pass of the whole hot path on one batch of synthetic input:
one prefill forward on the long-context causal workload (B=2, H=32, N=8192,
d=128, inputs x0.5) followed by one paged decode (B=32, H=32, d=128, contexts
U[512, 8192] in 16-token pages).  Both inputs are larger than the 129 MB L2, so
no flush is needed between steps (and the 2.3 GB decode pass evicts the prefill
data anyway).

Output: one JSON line.  `value` is the prefill rate in TFLOP/s (FLOPs =
4*B*H*N^2*d / 2 for causal) summed over ranks; the `decode` object carries the
paged-decode rate in GB/s of algorithmic HBM traffic.  Each carries a roofline
against the measured peaks of this GPU type.  The default run adds `configs`:
one sub-line for each of the three small prefill workloads (a single 128x64
tile, a BERT-large-like encoder with key padding, a GPT-2-small-like causal
decoder), timed on their own after the main region with L2 flushed between
steps, each with its roofline and the oracle timed on the whole workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the fp64 CPU oracle on the host cores
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from attn_fwd_02_gb300 import metrics, workloads  # noqa: E402

METRIC = "attention TFLOP/s (prefill) and HBM GB/s (paged decode), % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
# Traffic entries of profiles/ncu_traffic.txt: key -> source files whose hash the entry was taken on.
# Each key stands for one kernel on the workload its bench line times.
KERNEL_SOURCES = {
    "prefill_kernel": ["attn_fwd_02_gb300/csrc/prefill.cu", "attn_fwd_02_gb300/csrc/sm103_ptx.cuh"],
    "decode_split_kernel": ["attn_fwd_02_gb300/csrc/decode.cu", "attn_fwd_02_gb300/csrc/sm103_ptx.cuh"],
    "decode_split_kernel_e4m3": ["attn_fwd_02_gb300/csrc/decode.cu", "attn_fwd_02_gb300/csrc/sm103_ptx.cuh"],
    "decode_gqa_mma_kernel": ["attn_fwd_02_gb300/csrc/decode.cu", "attn_fwd_02_gb300/csrc/sm103_ptx.cuh"],
    "decode_gqa_mma_kernel_e4m3": ["attn_fwd_02_gb300/csrc/decode.cu", "attn_fwd_02_gb300/csrc/sm103_ptx.cuh"],
}

PREFILL_BY_NAME = {
    "tile": workloads.TILE_128x64,
    "encoder": workloads.ENCODER_PAD,
    "decoder": workloads.DECODER_CAUSAL,
    "long": workloads.LONG_CAUSAL,
}


# ----------------------------------------------------------------------------- helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_sha(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current source."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    want = source_sha(kernel)
    with open(PROFILE_TRAFFIC) as f:
        for line in f:
            parts = line.split()
            # "<kernel> <source sha> <dram bytes per launch> ..."
            if len(parts) >= 3 and parts[0] == kernel and parts[1] == want:
                try:
                    return float(parts[2])
                except ValueError:
                    return None
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, FileNotFoundError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, begin: bool):
        if begin:
            self.t_start = time.time()
        else:
            self.t_stop = time.time()

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            if self.t_start is None or not (self.t_start - 0.05 <= t <= (self.t_stop or t) + 0.15):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append(parts)
        if not rows:  # timed region shorter than the sampling period: use everything sampled
            rows = [[p.strip() for p in l.split(",")] for _, l in self.lines if len(l.split(",")) >= 9]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()), default=None)}


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier_sync(world):
    import torch
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        torch.cuda.synchronize()


def max_over_ranks(x: float, world: int) -> float:
    """Slowest rank's value: the job is done when the last rank is done."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms_max: float, scale: float) -> float:
    """Whole-job throughput: every rank processes units_per_rank (weak scaling, replicas),
    the job takes the slowest rank's time.  `scale` converts units/s to the reported unit."""
    return units_per_rank * world / (ms_max * 1e-3) / scale


# ----------------------------------------------------------------------------- GPU arm

class PrefillCase:
    def __init__(self, shape, torch, A):
        self.shape, self.A = shape, A
        inp = workloads.prefill_inputs(shape)
        self.host = {k: (v.pin_memory() if v is not None else None) for k, v in inp.items()}
        self.dev = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
        self.o = torch.empty_like(self.dev["q"])
        self.lse = torch.empty(self.dev["q"].shape[:3], dtype=torch.float32, device="cuda")
        kl = inp["kv_lens"]
        self.kv_lens = None if kl is None else [int(x) for x in kl]
        s = shape
        if kl is None:
            self.flops = metrics.prefill_flops(s.B, s.H, s.Nq, s.Nkv, s.d, s.causal)
        else:
            self.flops = metrics.prefill_flops_kvlen(s.H, s.Nq, s.d, self.kv_lens)
        self.flops_nominal = metrics.prefill_flops(s.B, s.H, s.Nq, s.Nkv, s.d, s.causal)
        self.bytes = metrics.prefill_bytes(s.B, s.H, s.Nq, s.Nkv, s.d, kv_lens=self.kv_lens)
        self.launches = 1
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in self.host.values() if v is not None)
        self.d2h_bytes = self.o.numel() * 2 + self.lse.numel() * 4
        self.out_names = ("o", "lse")

    def run(self):
        s, d = self.shape, self.dev
        if d["kv_lens"] is None:
            self.A.attn_fwd(d["q"], d["k"], d["v"], s.causal, s.scale, out=self.o, lse=self.lse)
        else:
            self.A.attn_fwd_kvlen(d["q"], d["k"], d["v"], s.causal, s.scale, kv_lens=d["kv_lens"], out=self.o,
                                  lse=self.lse)


class DecodeCase:
    def __init__(self, shape, torch, A, kv_heads=None):
        self.shape, self.A = shape, A
        self.kv_heads = kv_heads
        inp = workloads.decode_inputs(shape, kv_heads=kv_heads)
        self.host = {k: v.pin_memory() for k, v in inp.items()}
        self.dev = {k: v.cuda() for k, v in inp.items()}
        d = self.dev
        self.o = torch.empty_like(d["q"])
        self.lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device="cuda")
        need = A.paged_attn_decode_workspace_size(shape.B, shape.H, shape.d, d["page_table"].shape[1],
                                                  shape.page_size)
        self.ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
        self.ctx = [int(x) for x in inp["ctx_lens"]]
        self.bytes = metrics.decode_bytes(shape.H, shape.d, self.ctx, shape.page_size, kv_heads=kv_heads)
        self.launches = 2
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in self.host.values())
        self.d2h_bytes = self.o.numel() * 2 + self.lse.numel() * 4
        self.out_names = ("o", "lse")

    def run(self):
        d = self.dev
        fn = self.A.paged_attn_decode if self.kv_heads is None else self.A.paged_attn_decode_gqa
        fn(d["q"], d["k_pages"], d["v_pages"], d["page_table"], d["ctx_lens"], self.shape.scale, out=self.o,
           lse=self.lse, workspace=self.ws)


class DecodeFp8Case(DecodeCase):
    """Paged decode over an e4m3 cache: the bf16 pages of the workload converted on the GPU
    with kv_quantize_fp8 (per-tensor scale 6/448), then decoded with paged_attn_decode_fp8."""
    SCALE = 6.0 / 448

    def __init__(self, shape, torch, A, kv_heads=None):
        super().__init__(shape, torch, A, kv_heads=kv_heads)
        d = self.dev
        for n in ("k_pages", "v_pages"):
            codes = A.kv_quantize_fp8(d[n], self.SCALE)
            d[n] = codes
            self.host[n] = codes.cpu().pin_memory()
        torch.cuda.synchronize()
        self.bytes = metrics.decode_bytes(shape.H, shape.d, self.ctx, shape.page_size, kv_heads=kv_heads, kv_elem=1)
        self.h2d_bytes = sum(v.numel() * v.element_size() for v in self.host.values())

    def run(self):
        d = self.dev
        self.A.paged_attn_decode_fp8(d["q"], d["k_pages"], d["v_pages"], self.SCALE, self.SCALE, d["page_table"],
                                     d["ctx_lens"], self.shape.scale, out=self.o, lse=self.lse, workspace=self.ws)


class PagedPrefillCase:
    """Chunked prefill over the paged cache (queries = the last Nq cached positions)."""

    def __init__(self, shape, kv_heads, nq, torch, A):
        self.shape, self.A, self.Nq = shape, A, nq
        inp = workloads.decode_inputs(shape, kv_heads=kv_heads)
        g = torch.Generator().manual_seed(shape.seed + 1)
        q = torch.randn(shape.B, shape.H, nq, shape.d, generator=g).to(torch.bfloat16)
        self.dev = {k: v.cuda() for k, v in inp.items()}
        self.q = q.cuda()
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty(self.q.shape[:3], dtype=torch.float32, device="cuda")
        self.ctx = [int(x) for x in inp["ctx_lens"]]
        self.flops = metrics.paged_prefill_flops(shape.H, nq, shape.d, self.ctx, causal=True)
        self.bytes = metrics.paged_prefill_bytes(shape.H, nq, shape.d, self.ctx, shape.page_size, kv_heads=kv_heads)
        self.launches = 1

    def run(self):
        d = self.dev
        self.A.paged_attn_prefill(self.q, d["k_pages"], d["v_pages"], d["page_table"], d["ctx_lens"], True,
                                  self.shape.scale, out=self.o, lse=self.lse)


class PagedPrefillFp8Case(PagedPrefillCase):
    """The chunked prefill over an e4m3 copy of the same cache (kv_quantize_fp8, per-tensor
    scale 6/448), with paged_attn_prefill_fp8."""
    SCALE = 6.0 / 448

    def __init__(self, shape, kv_heads, nq, torch, A):
        super().__init__(shape, kv_heads, nq, torch, A)
        d = self.dev
        for n in ("k_pages", "v_pages"):
            d[n] = A.kv_quantize_fp8(d[n], self.SCALE)
        torch.cuda.synchronize()

    def run(self):
        d = self.dev
        self.A.paged_attn_prefill_fp8(self.q, d["k_pages"], d["v_pages"], self.SCALE, self.SCALE, d["page_table"],
                                      d["ctx_lens"], True, self.shape.scale, out=self.o, lse=self.lse)


L2_BYTES = 129e6
FLUSH_BYTES = 512 << 20


def step_flushes_l2(parts) -> bool:
    """Flush L2 between steps when one step's inputs would otherwise stay resident in it."""
    return sum(getattr(p, "bytes", 0) for p in parts) < 2 * L2_BYTES


class BackwardCase:
    """Backward of a prefill workload (the forward runs once, untimed, for O and LSE)."""

    def __init__(self, shape, torch, A):
        self.shape, self.A = shape, A
        inp = workloads.prefill_inputs(shape)
        do = workloads.backward_upstream(shape)
        q, k, v = inp["q"], inp["k"], inp["v"]
        self.dev = {"q": q.cuda(), "k": k.cuda(), "v": v.cuda(), "do": do.cuda()}
        d = self.dev
        o, lse = A.attn_fwd(d["q"], d["k"], d["v"], shape.causal, shape.scale)
        d["o"], d["lse"] = o, lse
        self.host = {n: t.cpu().pin_memory() for n, t in d.items()}
        self.dq, self.dk, self.dv = (torch.empty_like(d[n]) for n in ("q", "k", "v"))
        self.ws = torch.empty(max(A.attn_bwd_workspace_size(shape.B, shape.H, shape.Nq), 16), dtype=torch.uint8,
                              device="cuda")
        s = shape
        self.flops = metrics.backward_flops(s.B, s.H, s.Nq, s.Nkv, s.d, s.causal)
        self.flops_executed = metrics.backward_flops_executed(s.B, s.H, s.Nq, s.Nkv, s.d, s.causal)
        # read q, k, v, o, dO once, LSE; write dQ, dK, dV and D
        qkv = 2.0 * s.B * s.H * s.Nq * s.d
        self.bytes = 8 * qkv + 8.0 * s.B * s.H * s.Nq
        self.launches = 3
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in self.host.values())
        self.d2h_bytes = sum(t.numel() * t.element_size() for t in (self.dq, self.dk, self.dv))
        self.out_names = ("dq", "dk", "dv")

    def run(self):
        d, s = self.dev, self.shape
        self.A.attn_bwd(d["q"], d["k"], d["v"], d["o"], d["lse"], d["do"], s.causal, s.scale, dq=self.dq,
                        dk=self.dk, dv=self.dv, workspace=self.ws)


def backward_arm(args, torch, A, rank, world, peaks, peak_kind):
    """Backward of the long-context causal prefill, timed alone (not part of the default step)."""
    case = BackwardCase(workloads.LONG_CAUSAL, torch, A)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.5)
    region_ms, part_ms = time_parts(torch, [case], args.steps, args.warmup, world, sampler, graphs=args.graphs)
    clocks = sampler.stop() if sampler else None
    if A.attn_check_device_status() != 0:
        raise RuntimeError("device status error after the timed region")
    ms = part_ms[0]
    achieved = case.flops / (ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    e2e_ms = time_e2e(torch, case, max(3, min(args.steps, 10)), 1, world)
    s = case.shape
    out = {"metric": METRIC, "value": round(job_rate(case.flops, world, ms, 1e12), 2), "unit": "TFLOP/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(region_ms / args.steps, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded torch.randn -> bf16)",
           "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(achieved / peak, 4), "traffic": None,
                        "kernel": "attn_bwd (row term + dK/dV + dQ kernels)",
                        "executed_tflops": round(case.flops_executed / (ms * 1e-3) / 1e12, 2),
                        "peak_source": f"{peak_kind} bf16_tflops"},
           "e2e": {"value": round(job_rate(case.flops, world, e2e_ms, 1e12), 2), "unit": "TFLOP/s",
                   "schedule": E2E_SCHEDULE, "h2d_bytes_per_step": int(case.h2d_bytes), "d2h_bytes_per_step": int(case.d2h_bytes),
                   "ms_per_step": round(e2e_ms, 3)},
           "config": {"workload": "backward of " + s.name, "B": s.B, "H": s.H, "Nq": s.Nq, "Nkv": s.Nkv, "d": s.d,
                      "causal": s.causal, "flops_per_call": case.flops, "flops_executed_per_call": case.flops_executed,
                      "flops_accounting": "5 products of the forward's size (2.5 x forward); the dQ kernel recomputes "
                                          "S and dP (3.5 x forward executed)",
                      "ms_per_call": round(ms, 4), "l2": "inputs larger than L2 (no flush)",
                      "launch": "CUDA graph replay per call (captured through the API)" if args.graphs
                      else "direct calls"},
           "gpu_launches": case.launches * args.steps}
    if clocks is not None:
        out["clocks"] = clocks
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


def time_parts(torch, parts, steps, warmup, world, sampler=None, graphs=False):
    """Warm up, then time `steps` steps; each step runs every part once.  Returns the
    region time (max over ranks) and each part's mean per-call device time (ms).

    With graphs, each part's call (all its kernels) is captured once into a CUDA graph
    after the warm-up and the timed steps replay the graphs: the host's per-call launch
    cost, which exceeds the device time of the smallest workloads, stays out of the
    device-throughput figure (the end-to-end figure keeps it)."""
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        for p in parts:
            p.run()
    barrier_sync(world)
    runners = [p.run for p in parts]
    if graphs:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        captured = []
        for p in parts:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                p.run()
            captured.append(g)
        stream.wait_stream(side)
        runners = [g.replay for g in captured]
        for r in runners:  # one untimed replay each
            r()
        barrier_sync(world)
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in parts]
           for _ in range(steps)]
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device="cuda") if step_flushes_l2(parts) else None
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark(True)
    t0.record(stream)
    for s in range(steps):
        if flush is not None:  # outside the per-call events; inside the step's region time
            flush.zero_()
        for i, run in enumerate(runners):
            evs[s][i][0].record(stream)
            run()
            evs[s][i][1].record(stream)
    t1.record(stream)
    barrier_sync(world)
    if sampler:
        sampler.mark(False)
    region_ms = max_over_ranks(t0.elapsed_time(t1), world)
    part_ms = [max_over_ranks(sum(evs[s][i][0].elapsed_time(evs[s][i][1]) for s in range(steps)) / steps, world)
               for i in range(len(parts))]
    return region_ms, part_ms


E2E_SCHEDULE = ("every step copies its inputs from pinned host memory and its outputs back; steps pipelined "
                "(double-buffered device inputs/outputs, copies on two streams overlapping neighbouring steps)")


def time_e2e(torch, part, steps, warmup, world):
    """End to end through the public API with host buffers: every step copies its inputs from
    pinned host memory to the device, runs the call, and copies its outputs back to pinned host
    memory; all of it inside the timed region.  Steps are pipelined the way a serving loop runs
    them: step s+1's inputs travel on a copy stream into a second set of device buffers while
    step s computes, and step s's outputs travel back on a third stream from a second set of
    output buffers, so copies in both directions overlap the compute of neighbouring steps."""
    cmp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    names = [n for n, t in part.host.items() if t is not None]
    ins = [dict(part.dev), {n: (torch.empty_like(t) if t is not None else None) for n, t in part.dev.items()}]
    outs = [{n: getattr(part, n) for n in part.out_names}, {n: torch.empty_like(getattr(part, n)) for n in part.out_names}]
    host_out = {n: torch.empty(getattr(part, n).shape, dtype=getattr(part, n).dtype, pin_memory=True)
                for n in part.out_names}
    ev = lambda: torch.cuda.Event()
    in_ready, cmp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    saved_dev, saved_out = part.dev, {n: getattr(part, n) for n in part.out_names}

    def step(s):
        i = s % 2
        with torch.cuda.stream(h2d):
            if s >= 2:
                h2d.wait_event(cmp_done[i])  # step s-2 has finished reading this input set
            for n in names:
                ins[i][n].copy_(part.host[n], non_blocking=True)
            in_ready[i].record(h2d)
        cmp.wait_event(in_ready[i])
        if s >= 2:
            cmp.wait_event(out_done[i])  # step s-2's outputs have left this output set
        part.dev = ins[i]
        for n in part.out_names:
            setattr(part, n, outs[i][n])
        part.run()
        cmp_done[i].record(cmp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(cmp_done[i])
            for n in part.out_names:
                host_out[n].copy_(outs[i][n], non_blocking=True)
            out_done[i].record(d2h)

    try:
        for s in range(max(2, warmup)):
            step(s)
        torch.cuda.synchronize()
        barrier_sync(world)
        t0, t1, start = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True), ev()
        t0.record(cmp)
        start.record(cmp)
        h2d.wait_event(start)
        for s in range(steps):
            step(s)
        cmp.wait_event(out_done[(steps - 1) % 2])
        t1.record(cmp)
        barrier_sync(world)
    finally:
        part.dev = saved_dev
        for n, t in saved_out.items():
            setattr(part, n, t)
    return max_over_ranks(t0.elapsed_time(t1), world) / steps


def roofline_prefill(case, ms, peaks, peak_kind):
    achieved = case.flops / (ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    traffic = ncu_traffic("prefill_kernel") if case.shape is workloads.LONG_CAUSAL else None
    # attainable = min(peak, arithmetic intensity x HBM bandwidth) over the algorithmic bytes
    ai = case.flops / case.bytes
    attainable = min(peak, ai * hbm / 1e3)
    return {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": "prefill_kernel",
            "arithmetic_intensity": round(ai, 1), "attainable": round(attainable, 1),
            "frac_attainable": round(achieved / attainable, 4),
            "peak_source": f"{peak_kind} bf16_tflops (burst: the kernel is timed in sub-second steps)"}


def roofline_decode(case, ms_split, ms_total, peaks, peak_kind):
    achieved = case.bytes / (ms_split * 1e-3) / 1e9
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    fp8 = isinstance(case, DecodeFp8Case)
    if case.kv_heads is not None and case.kv_heads < case.shape.H:
        kernel = "decode_gqa_mma_kernel"
        key = (kernel + "_e4m3" if fp8 else kernel) if case.shape is workloads.PAGED_DECODE_GQA else None
    else:
        kernel = "decode_split_kernel"
        key = ("decode_split_kernel_e4m3" if fp8 else "decode_split_kernel") \
            if case.shape is workloads.PAGED_DECODE else None
    traffic = ncu_traffic(key) if key else None
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "traffic": traffic,
            "kernel": kernel + (" (e4m3 cache)" if fp8 else ""), "peak_source": f"{peak_kind} hbm_gbs"}


def gpu_arm(args):
    import torch

    import attn_fwd_02_gb300 as A
    rank, world, local = dist_setup()
    A.load_library()
    peaks, peak_kind = load_peaks()

    if args.workload == "default":
        pre = PrefillCase(workloads.LONG_CAUSAL, torch, A)
        dec = DecodeCase(workloads.PAGED_DECODE, torch, A)
        parts = [pre, dec]
    elif args.workload in ("decode", "decode_small", "decode_gqa", "decode_fp8", "decode_gqa_fp8") or \
            args.workload.startswith("decode_d"):
        if args.workload.startswith("decode_d"):  # decode_d32, decode_d80_fp8, ...
            d = int(args.workload[len("decode_d"):].split("_")[0])
            shape = workloads.PAGED_DECODE_BY_DIM[d]
            dec = DecodeFp8Case(shape, torch, A) if args.workload.endswith("_fp8") else DecodeCase(shape, torch, A)
        elif args.workload == "decode_gqa":
            dec = DecodeCase(workloads.PAGED_DECODE_GQA, torch, A, kv_heads=workloads.PAGED_DECODE_GQA_KV_HEADS)
        elif args.workload == "decode_fp8":
            dec = DecodeFp8Case(workloads.PAGED_DECODE, torch, A)
        elif args.workload == "decode_gqa_fp8":
            dec = DecodeFp8Case(workloads.PAGED_DECODE_GQA, torch, A, kv_heads=workloads.PAGED_DECODE_GQA_KV_HEADS)
        else:
            shape = workloads.PAGED_DECODE if args.workload == "decode" else workloads.PAGED_DECODE_SMALL
            dec = DecodeCase(shape, torch, A)
        pre = None
        parts = [dec]
    elif args.workload.startswith("prefill_paged"):
        return paged_prefill_arm(args, torch, A, rank, world, peaks, peak_kind)
    elif args.workload == "backward":
        return backward_arm(args, torch, A, rank, world, peaks, peak_kind)
    else:
        pre, dec = PrefillCase(PREFILL_BY_NAME[args.workload], torch, A), None
        parts = [pre]

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.5)
    region_ms, part_ms = time_parts(torch, parts, args.steps, args.warmup, world, sampler, graphs=args.graphs)
    clocks = sampler.stop() if sampler else None
    status = A.attn_check_device_status()
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")

    # end-to-end through the public API with host buffers (copies inside the timed region)
    e2e_steps = max(3, min(args.steps, 20))
    out = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(region_ms / args.steps, 4), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded torch.randn -> bf16)"}
    cfg = {"l2": "L2 flushed between steps (512 MiB write, outside the per-call events)"
           if step_flushes_l2(parts) else "inputs larger than L2 (no flush)",
           "parallelism": "replicas" if world > 1 else "single GPU",
           "launch": "CUDA graph replay per call (captured through the API)" if args.graphs else "direct calls"}
    launches = 0
    if pre is not None:
        i = parts.index(pre)
        ms = part_ms[i]
        out["value"] = round(job_rate(pre.flops, world, ms, 1e12), 2)
        out["unit"] = "TFLOP/s"
        out["roofline"] = roofline_prefill(pre, ms, peaks, peak_kind)
        e2e_ms = time_e2e(torch, pre, e2e_steps, 1, world)
        out["e2e"] = {"value": round(job_rate(pre.flops, world, e2e_ms, 1e12), 2), "unit": "TFLOP/s",
                      "schedule": E2E_SCHEDULE, "h2d_bytes_per_step": int(pre.h2d_bytes), "d2h_bytes_per_step": int(pre.d2h_bytes),
                      "ms_per_step": round(e2e_ms, 3), "part": "prefill"}
        cfg["workload"] = pre.shape.name
        s = pre.shape
        cfg["prefill"] = {"B": s.B, "H": s.H, "Nq": s.Nq, "Nkv": s.Nkv, "d": s.d, "causal": s.causal,
                          "scale": s.scale, "value_scale": s.value_scale, "kv_len_range": s.kv_len_range,
                          "flops_per_call": pre.flops, "flops_nominal": pre.flops_nominal,
                          "ms_per_call": round(ms, 4), "bytes_per_call": pre.bytes}
        launches += pre.launches * args.steps
    if dec is not None:
        i = parts.index(dec)
        ms = part_ms[i]
        dec_val = job_rate(dec.bytes, world, ms, 1e9)
        e2e_ms = time_e2e(torch, dec, e2e_steps, 1, world)
        dec_obj = {"value": round(dec_val, 1), "unit": "GB/s", "ms_per_call": round(ms, 4),
                   "bytes_per_call": dec.bytes,
                   "roofline": roofline_decode(dec, ms, ms, peaks, peak_kind),
                   "e2e": {"value": round(job_rate(dec.bytes, world, e2e_ms, 1e9), 1), "unit": "GB/s",
                           "schedule": E2E_SCHEDULE, "h2d_bytes_per_step": int(dec.h2d_bytes), "d2h_bytes_per_step": int(dec.d2h_bytes),
                           "ms_per_step": round(e2e_ms, 3)}}
        s = dec.shape
        cfg["decode"] = {"workload": s.name, "B": s.B, "H": s.H, "d": s.d, "page_size": s.page_size,
                         "ctx_range": s.ctx_range, "ctx_total": sum(dec.ctx)}
        if dec.kv_heads is not None:
            cfg["decode"]["Hkv"] = dec.kv_heads
        if isinstance(dec, DecodeFp8Case):
            cfg["decode"]["kv_cache"] = f"e4m3 codes, per-tensor scale {dec.SCALE:.6g} (kv_quantize_fp8)"
        if pre is None:
            out["value"], out["unit"] = dec_obj["value"], "GB/s"
            out["roofline"] = dec_obj["roofline"]
            out["e2e"] = dec_obj["e2e"]
            cfg["workload"] = s.name
        else:
            out["decode"] = dec_obj
            cfg["workload"] = f"{pre.shape.name} + {s.name}"
        launches += dec.launches * args.steps
    out["config"] = cfg
    out["gpu_launches"] = launches
    if clocks is not None:
        out["clocks"] = clocks
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(pre, dec, args.cpu_seconds)
    if args.workload == "default" and not args.no_configs:
        out["configs"] = small_prefill_lines(args, torch, A, rank, world, peaks, peak_kind)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


SMALL_PREFILL = (workloads.TILE_128x64, workloads.ENCODER_PAD, workloads.DECODER_CAUSAL)


def oracle_whole_prefill(shape, min_seconds=0.3):
    """The oracle on the whole prefill workload, repeated until at least min_seconds have passed.
    Returns (seconds per call, calls)."""
    from oracle import oracle
    inp = workloads.prefill_inputs(shape)
    calls, t_all = 0, 0.0
    while t_all < min_seconds or calls == 0:
        t = time.perf_counter()
        oracle.attn_fwd(inp["q"], inp["k"], inp["v"], shape.causal, shape.scale, kv_lens=inp["kv_lens"])
        t_all += time.perf_counter() - t
        calls += 1
    return t_all / calls, calls


def small_prefill_lines(args, torch, A, rank, world, peaks, peak_kind):
    """Sub-lines of the default run for the three small prefill workloads (the single 128x64 tile,
    the BERT-large-like encoder with key padding, the GPT-2-small-like causal decoder): each timed
    on its own after the main region, L2 flushed between steps, as CUDA-graph replays of the call
    (the host's per-call issue time exceeds the device time of the smallest ones), with its
    roofline and the oracle timed on the whole workload on the host cores."""
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    cases = [PrefillCase(shape, torch, A) for shape in SMALL_PREFILL]
    if sampler:
        sampler.start()
        time.sleep(0.5)
        sampler.mark(True)
    timed = []
    for case in cases:
        _, part_ms = time_parts(torch, [case], args.steps, args.warmup, world, None, graphs=True)
        timed.append(part_ms[0])
    if sampler:
        sampler.mark(False)
    clocks = sampler.stop() if sampler else None
    if A.attn_check_device_status() != 0:
        raise RuntimeError("device status set after the small-workload timing")
    lines = []
    for case, ms in zip(cases, timed):
        s = case.shape
        line = {"workload": s.name, "value": round(job_rate(case.flops, world, ms, 1e12), 3), "unit": "TFLOP/s",
                "ms_per_call": round(ms, 5), "flops_per_call": case.flops, "flops_nominal": case.flops_nominal,
                "bytes_per_call": case.bytes,
                "l2": "L2 flushed between steps (512 MiB write, outside the per-call events)",
                "launch": "CUDA graph replay per call (captured through the API)", "steps": args.steps,
                "roofline": roofline_prefill(case, ms, peaks, peak_kind),
                "prefill": {"B": s.B, "H": s.H, "Nq": s.Nq, "Nkv": s.Nkv, "d": s.d, "causal": s.causal,
                            "scale": s.scale, "kv_len_range": s.kv_len_range}}
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            from oracle import oracle
            sec, calls = oracle_whole_prefill(s)
            line["cpu_baseline"] = {"kind": "oracle", "cores": oracle.num_threads(),
                                    "value": round(case.flops / sec / 1e12, 6), "unit": "TFLOP/s",
                                    "sample": f"the whole workload, {calls} call(s) of fp64 C (OpenMP), "
                                              f"{sec * 1e3:.1f} ms per call"}
        lines.append(line)
    return {"lines": lines, "clocks": clocks,
            "gpu_launches": len(cases) * args.steps}


def paged_prefill_shape(workload: str):
    """prefill_paged[_dNN][_fp8] -> the chunked-prefill shape (d = 128 unless _dNN)."""
    rest = workload[len("prefill_paged"):]
    if rest.startswith("_d"):
        return workloads.PAGED_PREFILL_BY_DIM[int(rest[2:].split("_")[0])]
    return workloads.PAGED_PREFILL


def paged_prefill_arm(args, torch, A, rank, world, peaks, peak_kind):
    """Chunked prefill over the paged cache, timed alone (not part of the default step)."""
    cls = PagedPrefillFp8Case if args.workload.endswith("_fp8") else PagedPrefillCase
    case = cls(paged_prefill_shape(args.workload), workloads.PAGED_PREFILL_KV_HEADS, workloads.PAGED_PREFILL_NQ, torch,
               A)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
        time.sleep(0.5)
    region_ms, part_ms = time_parts(torch, [case], args.steps, args.warmup, world, sampler, graphs=args.graphs)
    clocks = sampler.stop() if sampler else None
    if A.attn_check_device_status() != 0:
        raise RuntimeError("device status error after the timed region")
    ms = part_ms[0]
    achieved = case.flops / (ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    s = case.shape
    out = {"metric": METRIC, "value": round(job_rate(case.flops, world, ms, 1e12), 2), "unit": "TFLOP/s",
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(region_ms / args.steps, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded torch.randn -> bf16)",
           "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(achieved / peak, 4), "traffic": None, "kernel": "prefill_kernel (paged)",
                        "peak_source": f"{peak_kind} bf16_tflops"},
           "config": {"workload": s.name + (" (e4m3 cache)" if cls is PagedPrefillFp8Case else ""), "B": s.B,
                      "H": s.H, "Hkv": workloads.PAGED_PREFILL_KV_HEADS, "d": s.d,
                      "Nq": case.Nq, "ctx_total": sum(case.ctx), "flops_per_call": case.flops,
                      "ms_per_call": round(ms, 4), "l2": "inputs larger than L2 (no flush)"},
           "gpu_launches": case.launches * args.steps}
    if clocks is not None:
        out["clocks"] = clocks
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


# ----------------------------------------------------------------------------- CPU oracle arm

def oracle_prefill_sample(shape, inp, budget_s, rng_seed=0):
    """Time the oracle on seeded random query rows until about budget_s seconds of work."""
    import numpy as np

    from oracle import oracle
    B, H, Nq, Nkv, d = shape.B, shape.H, shape.Nq, shape.Nkv, shape.d
    kl = inp["kv_lens"]
    rows_all = np.random.default_rng(rng_seed).permutation(B * H * Nq)
    done, flops, t_used, chunk = 0, 0.0, 0.0, 64
    while done < len(rows_all) and t_used < budget_s:
        rows = rows_all[done:done + chunk]
        t = time.perf_counter()
        oracle.attn_rows(inp["q"], inp["k"], inp["v"], shape.causal, shape.scale, rows, kv_lens=kl)
        t_used += time.perf_counter() - t
        for r in rows:  # FLOPs of these rows, counted as the metric counts them (4*d per valid key)
            i, b = int(r % Nq), int(r // (H * Nq))
            n = Nkv if kl is None else min(int(kl[b]), Nkv)
            if shape.causal:
                n = max(0, min(n, i + Nkv - Nq + 1))
            flops += 4.0 * d * n
        done += len(rows)
        chunk = min(4096, chunk * 2)
    return flops, t_used, done


def cpu_baseline(pre, dec, budget_s):
    from oracle import oracle
    cores = oracle.num_threads()
    out = {"kind": "oracle", "cores": cores}
    if pre is not None:
        inp = workloads.prefill_inputs(pre.shape)
        flops, t, rows = oracle_prefill_sample(pre.shape, inp, budget_s)
        out.update(value=round(flops / t / 1e12, 6), unit="TFLOP/s",
                   sample=f"{rows} seeded random query rows of {pre.shape.name} ({t:.1f} s of fp64 C, OpenMP)")
    if dec is not None:
        inp = workloads.decode_inputs(dec.shape, kv_heads=dec.kv_heads)
        t = time.perf_counter()
        if isinstance(dec, DecodeFp8Case):  # timing only: the codes the benchmark decodes
            oracle.paged_decode_fp8_gqa(inp["q"], dec.host["k_pages"], dec.host["v_pages"], dec.SCALE, dec.SCALE,
                                        inp["page_table"], inp["ctx_lens"], dec.shape.scale)
        else:
            oracle.paged_decode_gqa(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"], inp["ctx_lens"],
                                    dec.shape.scale)
        t = time.perf_counter() - t
        dobj = {"value": round(dec.bytes / t / 1e9, 3), "unit": "GB/s",
                "sample": f"the whole {dec.shape.name} ({t:.1f} s)"}
        if pre is None:
            out.update(dobj)
        else:
            out["decode"] = dobj
    return out


def time_oracle_decode(oracle, dshape, inp, steps, max_calls=10):
    """Seconds per whole oracle paged decode: one untimed call, then min(steps, max_calls) timed
    ones (each is the full workload, so a few calls give a stable mean)."""
    times = []
    for s in range(1 + max(1, min(steps, max_calls))):
        t = time.perf_counter()
        oracle.paged_decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["page_table"], inp["ctx_lens"], dshape.scale)
        if s >= 1:
            times.append(time.perf_counter() - t)
    return times


def reference_sampled_calls(oracle, args):
    """The oracle on the chunked prefill or the backward, one bounded call per step: for the chunked
    prefill one sequence's query-head group (query heads 0 .. group-1 over cache head 0) of the
    workload, over the same cache (e4m3 codes from the oracle's own quantiser for the _fp8 forms); for
    the backward one head of the long-context workload.  Returns (TFLOP/s, unit, sample, config, ms)."""
    import torch
    steps = []
    if args.workload == "backward":
        s = workloads.LONG_CAUSAL
        inp = workloads.prefill_inputs(s)
        do = workloads.backward_upstream(s)
        for i in range(args.warmup + args.steps):
            b, h = i % s.B, (i // s.B) % s.H
            sl = lambda t: t[b:b + 1, h:h + 1].contiguous()
            t0 = time.perf_counter()
            oracle.attn_bwd_gqa(sl(inp["q"]), sl(inp["k"]), sl(inp["v"]), sl(do), s.causal, s.scale)
            if i >= args.warmup:
                steps.append((metrics.backward_flops(1, 1, s.Nq, s.Nkv, s.d, s.causal), time.perf_counter() - t0))
        sample = f"one (sequence, head) of the backward of {s.name} per step (fp64 C, OpenMP)"
        cfgname = "backward of " + s.name
    else:
        s = paged_prefill_shape(args.workload)
        fp8 = args.workload.endswith("_fp8")
        hkv, nq = workloads.PAGED_PREFILL_KV_HEADS, workloads.PAGED_PREFILL_NQ
        group = s.H // hkv
        inp = workloads.decode_inputs(s, kv_heads=hkv)
        q = torch.randn(s.B, s.H, nq, s.d, generator=torch.Generator().manual_seed(s.seed + 1)).to(torch.bfloat16)
        kp, vp = inp["k_pages"][:, 0:1].contiguous(), inp["v_pages"][:, 0:1].contiguous()
        scale8 = PagedPrefillFp8Case.SCALE
        if fp8:
            kp, vp = oracle.e4m3_quantize(kp, scale8), oracle.e4m3_quantize(vp, scale8)
        ctx = [int(x) for x in inp["ctx_lens"]]
        for i in range(args.warmup + args.steps):
            b = i % s.B
            args_b = (q[b:b + 1, 0:group].contiguous(), kp, vp, inp["page_table"][b:b + 1].contiguous(),
                      inp["ctx_lens"][b:b + 1].contiguous())
            t0 = time.perf_counter()
            if fp8:
                oracle.paged_prefill_fp8_gqa(args_b[0], args_b[1], args_b[2], scale8, scale8, args_b[3], args_b[4],
                                             True, s.scale)
            else:
                oracle.paged_prefill_gqa(*args_b, True, s.scale)
            if i >= args.warmup:
                steps.append((metrics.paged_prefill_flops(group, nq, s.d, [ctx[b]], causal=True),
                              time.perf_counter() - t0))
        sample = (f"one sequence's query-head group ({group} query heads over one cache head) of {s.name}"
                  f"{' (e4m3 cache)' if fp8 else ''} per step (fp64 C, OpenMP)")
        cfgname = s.name + (" (e4m3 cache)" if fp8 else "")
    rate = sum(f for f, _ in steps) / sum(t for _, t in steps) / 1e12
    return rate, "TFLOP/s", sample, cfgname, statistics.mean(t for _, t in steps) * 1e3


def reference_arm(args):
    """The oracle, as it stands, on the host cores: same metric, unit and config."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import oracle
    oracle.build()
    cores = oracle.num_threads()
    shape = workloads.LONG_CAUSAL if args.workload in ("default", "long") else PREFILL_BY_NAME.get(args.workload)
    # about a minute of oracle work in all: each step is a seeded sample of query rows (at least one
    # block of 64) sized to its share of the minute
    budget = min(10.0, 60.0 / max(1, args.steps + args.warmup))
    if args.workload.startswith("prefill_paged") or args.workload == "backward":
        val, unit, sample, cfgname, ms = reference_sampled_calls(oracle, args)
    elif shape is None:  # decode only: the decode workload the GPU arm would time (its bf16 cache)
        dshape = workloads.PAGED_DECODE
        if args.workload.startswith("decode_d"):
            dshape = workloads.PAGED_DECODE_BY_DIM[int(args.workload[len("decode_d"):].split("_")[0])]
        inp = workloads.decode_inputs(dshape)
        bytes_ = metrics.decode_bytes(dshape.H, dshape.d, [int(x) for x in inp["ctx_lens"]], dshape.page_size)
        times = time_oracle_decode(oracle, dshape, inp, args.steps)
        val, unit = bytes_ / statistics.mean(times) / 1e9, "GB/s"
        sample = f"the whole {dshape.name} per call, {len(times)} timed calls after one untimed"
        cfgname = dshape.name
        ms = statistics.mean(times) * 1e3
    else:
        inp = workloads.prefill_inputs(shape)
        rates, ms_l = [], []
        for s in range(args.warmup + args.steps):
            flops, t, rows = oracle_prefill_sample(shape, inp, budget, rng_seed=s)
            if s >= args.warmup:
                rates.append(flops / t)
                ms_l.append(t * 1e3)
        val, unit = statistics.mean(rates) / 1e12, "TFLOP/s"
        sample = (f"per step, seeded random query rows of {shape.name} (blocks of 64 rows or more) for about "
                  f"{budget:.2g} s of fp64 C")
        cfgname = shape.name
        ms = statistics.mean(ms_l)
    cfg = {"workload": cfgname, "l2": "n/a (CPU)"}
    if shape is not None:
        cfg["prefill"] = {"B": shape.B, "H": shape.H, "Nq": shape.Nq, "Nkv": shape.Nkv, "d": shape.d,
                          "causal": shape.causal, "scale": shape.scale, "value_scale": shape.value_scale,
                          "kv_len_range": shape.kv_len_range}
    decode = None
    if args.workload == "default":
        # the default step is the prefill plus the paged decode: the decode leg, one whole oracle
        # decode per step (about 0.1 s), is reported beside the prefill as the GPU arm reports it
        dshape = workloads.PAGED_DECODE
        dinp = workloads.decode_inputs(dshape)
        ctx = [int(x) for x in dinp["ctx_lens"]]
        dbytes = metrics.decode_bytes(dshape.H, dshape.d, ctx, dshape.page_size)
        times = time_oracle_decode(oracle, dshape, dinp, args.steps)
        decode = {"value": round(dbytes / statistics.mean(times) / 1e9, 3), "unit": "GB/s",
                  "ms_per_call": round(statistics.mean(times) * 1e3, 1), "bytes_per_call": dbytes,
                  "sample": f"the whole {dshape.name} per call, {len(times)} timed calls after one untimed"}
        cfg["workload"] = f"{shape.name} + {dshape.name}"
        cfg["decode"] = {"workload": dshape.name, "B": dshape.B, "H": dshape.H, "d": dshape.d,
                         "page_size": dshape.page_size, "ctx_range": list(dshape.ctx_range), "ctx_total": sum(ctx)}
    out = {"impl": "reference", "metric": METRIC, "value": round(val, 6), "unit": unit, "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 1), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded torch.randn -> bf16)",
           "config": cfg,
           "cpu_baseline": {"kind": "oracle", "cores": cores, "sample": sample, "value": round(val, 6),
                            "unit": unit},
           "e2e": {"value": round(val, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    if decode is not None:
        out["decode"] = decode
    print(json.dumps(out), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["default", "decode", "decode_small", "decode_gqa", "decode_fp8", "decode_gqa_fp8",
                                           *[f"decode_d{d}{s}" for d in (32, 64, 80, 96) for s in ("", "_fp8")],
                                           "prefill_paged", "prefill_paged_fp8",
                                           *[f"prefill_paged_d{d}{s}" for d in (32, 64, 80, 96) for s in ("", "_fp8")],
                                           "backward",
                                           *PREFILL_BY_NAME], default="default")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-baseline oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="default run: skip the sub-lines of the three small prefill workloads")
    ap.add_argument("--graphs", action="store_true", help="time CUDA graph replays of each call instead of direct calls")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps, always
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
