#!/usr/bin/env python3
"""Benchmark of the GB300 routed-MoE layer: prints ONE JSON line on rank 0.

Default workload: single-token decode of a GLM-5.2-shaped layer (E=256
experts, top-8, d=6144, f=2048, shared expert 2048, Q8_0 weights, s=2.5,
Zipf-skewed router logits), one token per step, token seeds 0..99.  A step is
one moe_layer call (route -> permute -> quantise -> expert FFN -> shared
expert -> combine), launched eagerly (--graph: a CUDA graph per step; its
GPU-side launch adds ~1.5 us to the decode step).  Inputs and weights are
resident in HBM; between steps, outside the per-step CUDA-event timing, L2
(129 MB) is flushed by writing a 2x-L2 buffer and reading it back (the read
pass evicts the written lines, so the timed step does not pay for writing the
flush buffer's dirty lines back to HBM; the write-only figure is reported too).

--gpus N (under torchrun) runs N replicas: each rank decodes its own tokens on
its own copy of the weights with no data-path collective (token-parallel
decode, weak scaling).  ``value`` = all ranks' tokens / max over ranks of the
device time.

--impl reference times the CPU oracle (plain C, one host core) on bounded
samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and achieved HBM GB/s (% of GB300 roofline) at T=1/16/512"
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_t1")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="budget of the oracle CPU-baseline sample")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the T=2/16/512 and 2-bit side measurements")
    ap.add_argument("--graph", action="store_true",
                    help="time each step as a replay of a CUDA graph of its moe_layer call "
                         "(default: eager moe_layer calls)")
    ap.add_argument("--no-graph", action="store_true", help="no CUDA graphs anywhere (e2e too)")
    ap.add_argument("--flags", type=int, default=0, help="moe_desc.flags for the timed calls")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(torch, dist, value: float, device) -> float:
    """MAX of a per-rank float over the process group (the value itself on one
    rank): the job's time is its slowest replica's."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, max_ms: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return units_per_rank * world / (max_ms / 1e3)


def rank_seeds(seeds, rank: int):
    """Token seeds of one replica: rank 0 keeps the workload's seeds, rank r
    shifts them by 1000*r so that replicas decode different tokens."""
    return tuple(s + 1000 * rank for s in seeds)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


FALLBACK_TENSOR_TFLOPS = 1900.0  # dense 16-bit, one earlier GB300 measurement
SM_MHZ_MAX = 2070.0              # the GB300's maximum SM clock


def load_tensor_peak() -> float:
    """Dense 16-bit tensor peak (TFLOP/s) of a kernel timed alone: the measured
    bf16 burst figure (fp16 runs at the same dense rate), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            p = json.load(fh)
        if p.get("bf16_tflops"):
            return float(p["bf16_tflops"])
    return FALLBACK_TENSOR_TFLOPS


# ------------------------------------------------------------------ bytes model
def row_bytes(fmt: int, K: int) -> int:
    """Bytes of one quantised weight row of K weights: codes + fp16 block scales."""
    return {0: K, 1: K // 4, 2: K // 2}[fmt] + (K // 32) * 2


def tc_tiles(spec, T: int, counts, tc_rows) -> int:
    """Gate/up tiles (128 features x 64 rows) the row rule sends to the tensor
    cores: routed experts with more than tc_rows rows, and the shared expert when
    its width equals f."""
    n = sum((spec.f // 128) * ((int(c) + 63) // 64) for c in counts if int(c) > tc_rows)
    if spec.f_shared and spec.f_shared == spec.f and T > tc_rows:
        n += (spec.f_shared // 128) * ((T + 63) // 64)
    return n


def stage_bytes(spec, T: int, counts, tc_rows=None, sm_count=None):
    """Algorithmic HBM bytes per stage: each selected expert's weights and the
    shared expert's, read once.  counts: rows per routed expert; experts with
    more than tc_rows rows (None: no tensor path) are charged to the
    tensor-core stages -- unless their gate/up tiles number fewer than sm_count,
    when the library runs every expert on the GEMV."""
    if tc_rows is not None and sm_count is not None and tc_tiles(spec, T, counts, tc_rows) < sm_count:
        tc_rows = None
    out = {"gateup": 0, "down": 0, "gateup_tc": 0, "down_tc": 0}

    def add(rows, fmt, f):
        tc = "_tc" if tc_rows is not None and rows > tc_rows else ""
        out["gateup" + tc] += 2 * f * row_bytes(fmt, spec.d)
        out["down" + tc] += spec.d * row_bytes(fmt, f)

    for c in counts:
        if c > 0:
            add(int(c), spec.fmt, spec.f)
    if spec.f_shared:
        add(T, 0, spec.f_shared)
    out["total"] = sum(out.values())
    out["decode_fused"] = out["total"]
    return out


ROOFLINE_STAGES = ("gateup", "down", "gateup_tc", "down_tc", "decode_fused")

FMT_NAMES = {0: "Q8_0", 1: "Q2S", 2: "E2M1"}


def workload_desc(name: str, spec, T: int) -> str:
    """The workload as both arms name it in config.workload."""
    return (f"{name}: T={T}, E={spec.E}, top_k={spec.k}, d={spec.d}, f={spec.f}, "
            f"f_shared={spec.f_shared}, fmt={FMT_NAMES[spec.fmt]}, s={spec.s}, "
            f"zipf_beta={spec.zipf_beta}")

# dp4a issue rate of one SM per clock: half the 128 fp32 lanes (a probe kernel
# of independent dp4a chains measured 60.2 per SM per clock on this GB300)
DP4A_PER_SM_CLK = 64


def stage_macs(spec, T: int, counts, tc_rows=None, sm_count=None):
    """int8 (or 2-bit x int8) multiply-adds of the gate/up and down stages: each
    selected expert's rows times its weights, split like stage_bytes between the
    dp4a GEMV and the tensor cores."""
    if tc_rows is not None and sm_count is not None and tc_tiles(spec, T, counts, tc_rows) < sm_count:
        tc_rows = None
    out = {"gateup": 0, "down": 0, "gateup_tc": 0, "down_tc": 0}

    def add(rows, f):
        tc = "_tc" if tc_rows is not None and rows > tc_rows else ""
        out["gateup" + tc] += 2 * f * spec.d * rows
        out["down" + tc] += spec.d * f * rows

    for c in counts:
        if c > 0:
            add(int(c), spec.f)
    if spec.f_shared:
        add(T, spec.f_shared)
    return out


def unit_fractions(macs, stage_ms, sm_count, sm_mhz, tensor_tflops):
    """Which unit binds each expert stage: the dp4a stages' dp4a issue rate
    against SMs x 64 / clock x SM clock, the tensor-core stages' fp16 MMA rate
    (2 flops a multiply-add) against the measured dense 16-bit peak."""
    out = {}
    dp4a_peak = sm_count * DP4A_PER_SM_CLK * sm_mhz * 1e6
    for st in ("gateup", "down"):
        if st in stage_ms and macs[st]:
            out[st + "_dp4a_frac"] = round(macs[st] / 4 / (stage_ms[st] / 1e3) / dp4a_peak, 4)
    for st in ("gateup_tc", "down_tc"):
        if st in stage_ms and macs[st] and tensor_tflops:
            out[st + "_tensor_frac"] = round(2 * macs[st] / (stage_ms[st] / 1e3) /
                                            (tensor_tflops * 1e12), 4)
    return out


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm
def source_hash(paths):
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(kernel_stage: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as fh:
        rec = json.load(fh)
    for r in rec.get("records", []):
        if r.get("stage") == kernel_stage and r.get("workload") == workload:
            if r.get("source_hash") != source_hash(r.get("sources", [])):
                return None
            return float(r["dram_bytes_per_launch"])
    return None


class L2Flush:
    """Evicts the previous step's data from L2 between timed steps: write a
    2x-L2 buffer, then read it back.  Writing alone leaves up to a full L2 of
    dirty lines whose write-back to HBM would then land inside the next timed
    step; the read pass evicts them (and the written data) before the timer
    starts.  ``write_only`` is the plain write flush, kept for the side
    measurement that shows the difference."""

    def __init__(self, torch, dev):
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
        self.words = self.buf.view(torch.int64)
        self.acc = torch.zeros(1, dtype=torch.int64, device=dev)
        self.torch = torch

    def __call__(self):
        self.buf.zero_()
        self.torch.sum(self.words, dim=0, out=self.acc[0])

    def write_only(self):
        self.buf.zero_()


def run_ours(args):
    import torch
    import torch.distributed as dist

    import synth
    import __graft_entry__ as ge
    from routed_expert_decode_gb300 import moe

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    ge.build()
    spec, T, seeds = synth.WORKLOADS[args.workload]
    seeds = rank_seeds(seeds, rank)
    K, W = args.steps, args.warmup

    weights = synth.fill_layer_device(spec, dev)
    layer = moe.Layer(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s, weights,
                      dev)
    desc = layer.desc(args.flags)
    ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=dev)
    bias = torch.from_numpy(synth.bias(spec)).to(dev)
    host_in = {s: synth.token_inputs(spec, s, T) for s in seeds}
    dev_in = {s: (torch.from_numpy(host_in[s][1]).to(dev), torch.from_numpy(host_in[s][0]).to(dev))
              for s in seeds}
    y = torch.empty((T, spec.d), dtype=torch.float32, device=dev)
    flush = L2Flush(torch, dev)

    # unique routed experts per seed (setup pass through the library's router)
    U_of, counts_of = {}, {}
    off = torch.empty(spec.E + 1, dtype=torch.int32, device=dev)
    idx = torch.empty((T, spec.k), dtype=torch.int32, device=dev)
    wts = torch.empty((T, spec.k), dtype=torch.float32, device=dev)
    perm = torch.empty(T * spec.k, dtype=torch.int32, device=dev)
    pos = torch.empty(T * spec.k, dtype=torch.int32, device=dev)
    for s in seeds:
        moe.route(desc, dev_in[s][1], bias, idx, wts, off, perm, pos)
        counts_of[s] = (off[1:] - off[:-1]).cpu().tolist()
        U_of[s] = sum(1 for c in counts_of[s] if c > 0)
    tc_rows = moe.tc_min_rows(desc, T)

    names = moe.stage_names(desc, T)
    path = moe.layer_path(desc, T)
    nst = len(names)
    step_seed = [seeds[i % len(seeds)] for i in range(K)]
    stage_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst + 1)] for _ in range(K)]
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    stream = torch.cuda.current_stream(dev)

    # the timed steps are plain moe_layer calls (what a user runs); a second set
    # of steps with per-stage events (moe_layer_timed) gives the stage split
    def plain(i, s):
        x_d, l_d = dev_in[s]
        moe.layer(desc, layer.weights, x_d, l_d, bias, y, ws)

    def staged(i, s):
        x_d, l_d = dev_in[s]
        moe.layer_timed(desc, layer.weights, x_d, l_d, bias, y, ws, stage_ev[i])

    for evs in stage_ev:  # create every CUDA event before any capture
        for ev in evs:
            ev.record()
    for i in range(W):  # warm-up
        plain(i % K, step_seed[i % K])
        staged(i % K, step_seed[i % K])
    torch.cuda.synchronize()

    graphs = staged_graphs = None
    graphed = args.graph and not args.no_graph
    if graphed:
        graphs, staged_graphs = [], []
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for i in range(K):
                for fn, out in ((plain, graphs), (staged, staged_graphs)):
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=cap):
                        fn(i, step_seed[i])
                    out.append(g)
        stream.wait_stream(cap)
        for i in range(min(W, K)):
            graphs[i].replay()
            staged_graphs[i].replay()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    # untimed GPU work ahead of the first step (~0.7 ms of flushes) lets the host
    # enqueue several steps before the GPU reaches the first one, so no step's
    # events bracket an idle GPU waiting for the host's next launch
    for _ in range(8):
        flush()
    torch.cuda.nvtx.range_push("timed_steps")  # lets a profiler select these launches
    for i in range(K):
        flush()  # evict the previous step's weights from L2 (not timed)
        ev0[i].record()
        if graphs is not None:
            graphs[i].replay()
        else:
            plain(i, step_seed[i])
        ev1[i].record()
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    if world > 1:
        dist.barrier()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()

    # stage split (not part of the timed steps)
    for i in range(K):
        flush()
        if staged_graphs is not None:
            staged_graphs[i].replay()
        else:
            staged(i, step_seed[i])
    torch.cuda.synchronize()

    step_ms = [ev0[i].elapsed_time(ev1[i]) for i in range(K)]

    # side check (not the reported number): the same steps after a write-only
    # flush, whose dirty lines are written back inside the step, and with no
    # flush at all (the weights alone exceed L2)
    flush_check = {}
    for mode, fl in (("write_only_flush", flush.write_only), ("no_flush", lambda: None)):
        n = min(K, 20)
        for i in range(n):
            fl()
            ev0[i].record()
            if graphs is not None:
                graphs[i].replay()
            else:
                plain(i, step_seed[i])
            ev1[i].record()
        torch.cuda.synchronize()
        flush_check[mode + "_ms_per_step"] = round(
            statistics.mean(ev0[i].elapsed_time(ev1[i]) for i in range(n)), 5)
    stage_ms = {n: [stage_ev[i][j].elapsed_time(stage_ev[i][j + 1]) for i in range(K)]
                for j, n in enumerate(names)}
    if nst == 1:  # a single kernel: its duration is the timed step
        stage_ms = {names[0]: list(step_ms)}
    total_ms = max_over_ranks(torch, dist, sum(step_ms), dev)
    ms_per_step = total_ms / K
    tokens = T * K * world
    value = job_throughput(T * K, world, total_ms)

    # roofline of the dominant kernel
    peak, peak_src = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    bytes_steps = [stage_bytes(spec, T, counts_of[s], tc_rows, sms) for s in step_seed]
    mean_stage = {n: statistics.mean(v) for n, v in stage_ms.items()}
    dom = max(mean_stage, key=mean_stage.get)
    dom_bytes = sum(b.get(dom, 0) for b in bytes_steps) / K
    achieved = (dom_bytes / (mean_stage[dom] / 1e3) / 1e9
                if dom in ROOFLINE_STAGES and dom_bytes > 0 else None)
    layer_gbs = sum(b["total"] for b in bytes_steps) / (sum(step_ms) / 1e3) / 1e9

    # end-to-end through the C ABI with host buffers: every step copies its inputs
    # in from pinned host memory and its result out, K steps back to back with the
    # copies in and the copies out on two more streams (step i+1's inputs and
    # step i-1's result move while layer i computes; double-buffered device
    # buffers; one copy stream for both directions would queue step i+1's inputs
    # behind step i's result, between the two layers).  The K steps run as one
    # CUDA graph (the steps as eager calls are reported beside it).  No L2 flush
    # here: a step reads 361 MB of weights, far more than L2.
    pin_in = {s: (torch.from_numpy(host_in[s][1]).pin_memory(),
                  torch.from_numpy(host_in[s][0]).pin_memory()) for s in seeds}
    x_d = [torch.empty((T, spec.d), dtype=torch.float32, device=dev) for _ in range(2)]
    l_d = [torch.empty((T, spec.E), dtype=torch.float32, device=dev) for _ in range(2)]
    y_d = [torch.empty((T, spec.d), dtype=torch.float32, device=dev) for _ in range(2)]
    y_h = [torch.empty((T, spec.d), dtype=torch.float32).pin_memory() for _ in range(2)]
    cs_in, cs_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    n_ev = max(W, K)
    in_ok, done, out_ok = ([torch.cuda.Event() for _ in range(n_ev)] for _ in range(3))

    def run_steps(n, comp):
        cs_in.wait_stream(comp)  # brings the copy streams into a capture on comp
        cs_out.wait_stream(comp)
        for i in range(n):
            b = i % 2
            s_ = step_seed[i % K]
            with torch.cuda.stream(cs_in):
                if i >= 2:
                    cs_in.wait_event(done[i - 2])  # layer i-2 has read x_d[b], l_d[b]
                x_d[b].copy_(pin_in[s_][0], non_blocking=True)
                l_d[b].copy_(pin_in[s_][1], non_blocking=True)
                in_ok[i].record(cs_in)
            comp.wait_event(in_ok[i])
            if i >= 2:
                comp.wait_event(out_ok[i - 2])  # y_d[b] of step i-2 is copied out
            moe.layer(desc, layer.weights, x_d[b], l_d[b], bias, y_d[b], ws)
            done[i].record(comp)
            with torch.cuda.stream(cs_out):
                cs_out.wait_event(done[i])
                y_h[b].copy_(y_d[b], non_blocking=True)
                out_ok[i].record(cs_out)
        comp.wait_event(in_ok[n - 1])  # joins both copy streams
        comp.wait_event(out_ok[n - 1])

    def timed_ms(go):
        ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ea.record()
        go()
        eb.record()
        torch.cuda.synchronize()
        return ea.elapsed_time(eb)

    main = torch.cuda.current_stream(dev)
    run_steps(W, main)
    torch.cuda.synchronize()
    eager_ms = max_over_ranks(torch, dist, timed_ms(lambda: run_steps(K, main)), dev)
    e2e_ms, e2e_how = eager_ms, "eager moe_layer calls"
    if not args.no_graph:
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(main)
        g_e2e = []
        with torch.cuda.stream(cap):
            for n in (W, K):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    run_steps(n, cap)
                g_e2e.append(g)
        main.wait_stream(cap)
        g_e2e[0].replay()
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(torch, dist, timed_ms(g_e2e[1].replay), dev)
        e2e_how = "the K steps captured as one CUDA graph"
    # what a user reads back: the last two steps' y in pinned host memory equal
    # an eager call on the same inputs (the same kernels, so bit for bit)
    torch.cuda.synchronize()
    for i in range(max(K - 2, 0), K):
        s_ = step_seed[i]
        y_ref = torch.empty_like(y_d[0])
        moe.layer(desc, layer.weights, pin_in[s_][0].to(dev), pin_in[s_][1].to(dev), bias,
                  y_ref, ws)
        torch.cuda.synchronize()
        if not torch.equal(y_h[i % 2], y_ref.cpu()):
            raise RuntimeError(f"end-to-end step {i}: y read back differs from an eager call")
    e2e = {"value": round(job_throughput(T * K, world, e2e_ms), 2), "unit": "tokens/s",
           "h2d_bytes_per_step": T * spec.d * 4 + T * spec.E * 4,
           "d2h_bytes_per_step": T * spec.d * 4,
           "method": e2e_how + "; per step x and router logits in from pinned host memory, "
                     "moe_layer, y out to pinned host memory (copies in and copies out on "
                     "two more streams, double-buffered device buffers)",
           "checked": "the last two steps' y as read back equal an eager call bit for bit",
           "eager_calls_value": round(job_throughput(T * K, world, eager_ms), 2)}
    assert moe.check_device_error(ws) == 0

    sweep = None
    if not args.no_sweep and world == 1 and args.workload == "decode_t1":
        del graphs
        sweep = run_sweep(torch, moe, synth, dev, layer, flush, peak)

    cpu = None
    if rank == 0 and world == 1:
        cpu = cpu_baseline(args.workload, args.cpu_seconds)

    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return None
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_per_step, 5),
        "ms_per_step_median": round(statistics.median(step_ms), 5),
        "ms_per_step_p90": round(percentile(step_ms, 90), 5),
        "ms_per_step_max": round(max(step_ms), 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8 x int8 -> int32 block dots, fp32 scales/accumulation",
        "data": "synthetic (seeded counter-based generator; random Q8_0 weights of the layer's shape)",
        "config": {
            "workload": workload_desc(args.workload, spec, T),
            "token_seeds": seeds_run(step_seed),
            "tokens_per_step": T,
            "l2": "flushed between steps (2x L2 write, then read back), outside the per-step "
                  "CUDA-event time; e2e: K steps back to back, each reading 361 MB of weights "
                  "(> L2), no flush",
            "timing": ("one CUDA graph of one moe_layer call per step" if graphed
                       else "eager moe_layer calls (the flush kernels between steps keep the "
                            "launches ahead of the GPU)")
                      + "; CUDA events around each step; stage split from a second, "
                        "untimed pass with per-stage events",
            "parallelism": f"replicas x{world} (token-parallel decode, no collective)",
            "host": f"{platform.machine()}, {os.cpu_count()} cores",
        },
        "hbm": {"algorithmic_bytes_per_step": round(statistics.mean(b["total"] for b in bytes_steps)),
                "achieved_gbs": round(layer_gbs, 1), "peak_gbs": peak,
                "frac_of_measured": round(layer_gbs / peak, 4),
                "frac_of_8tbs_nominal": round(layer_gbs / 8000.0, 4)},
        "stage_us": {n: round(v * 1e3, 2) for n, v in mean_stage.items()},
        "roofline": {"bound": "hbm", "kernel": dom,
                     "achieved": round(achieved, 1) if achieved else None,
                     "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4) if achieved else None,
                     "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": round(dom_bytes),
                     "traffic": traffic_for(dom, args.workload)},
        "gpu_launches": K * (1 if path == "fused_decode" else nst),
        "path": path,
        "clocks": clk,
        "e2e": e2e,
        "l2_flush_check": flush_check,
        "cpu_baseline": cpu,
        "wall_s_timed_region": round(t_wall, 4),
    }
    if sweep:
        line["sweep"] = sweep
    return line


def seeds_run(step_seed) -> str:
    """The token seeds the timed steps used (each step takes the next seed)."""
    u = sorted(set(step_seed))
    if u == list(range(u[0], u[-1] + 1)):
        return f"{u[0]}..{u[-1]} ({len(u)} seeds)"
    return ",".join(str(v) for v in u)


def percentile(v, q: float) -> float:
    """q-th percentile by linear interpolation between order statistics."""
    a = sorted(v)
    if len(a) == 1:
        return a[0]
    x = (len(a) - 1) * q / 100.0
    i = int(x)
    j = min(i + 1, len(a) - 1)
    return a[i] + (a[j] - a[i]) * (x - i)


def run_sweep(torch, moe, synth, dev, layer, flush, peak):
    """Side measurements at T=2/16/512 on the same layer and T=64 on the 2-bit
    and the e2m1 layers: 10 eager moe_layer calls each after 3 warm-ups, L2 flushed between,
    CUDA events around each call (ms_per_step); then 10 more calls with events
    between the stages (stage_us)."""
    out = {}
    cases = [("batch_t2", layer), ("batch_t16", layer), ("prefill_t512", layer), ("q2_t64", None),
             ("fp4_t64", None)]
    for name, lay in cases:
        spec, T, seeds = synth.WORKLOADS[name]
        if lay is None:
            w = synth.fill_layer_device(spec, dev)
            lay = moe.Layer(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s, w, dev)
        desc = lay.desc()
        ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=dev)
        bias = torch.from_numpy(synth.bias(spec)).to(dev)
        logits, x = synth.token_inputs(spec, seeds[0], T)
        x_d, l_d = torch.from_numpy(x).to(dev), torch.from_numpy(logits).to(dev)
        y = torch.empty((T, spec.d), dtype=torch.float32, device=dev)
        names = moe.stage_names(desc, T)
        n = 10
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)]
               for _ in range(n)]
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for i in range(3):
            moe.layer(desc, lay.weights, x_d, l_d, bias, y, ws)
            moe.layer_timed(desc, lay.weights, x_d, l_d, bias, y, ws, evs[0])
        torch.cuda.synchronize()
        for i in range(n):
            flush()
            e0[i].record()
            moe.layer(desc, lay.weights, x_d, l_d, bias, y, ws)
            e1[i].record()
        torch.cuda.synchronize()
        step = [e0[i].elapsed_time(e1[i]) for i in range(n)]
        for i in range(n):
            flush()
            moe.layer_timed(desc, lay.weights, x_d, l_d, bias, y, ws, evs[i])
        torch.cuda.synchronize()
        stage = {nm: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(n))
                 for j, nm in enumerate(names)}
        lay_off = lay.views(ws, T)["off"].cpu()
        counts = (lay_off[1:] - lay_off[:-1]).tolist()
        U = sum(1 for c in counts if c > 0)
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        b = stage_bytes(spec, T, counts, moe.tc_min_rows(desc, T), sms)
        macs = stage_macs(spec, T, counts, moe.tc_min_rows(desc, T), sms)
        ms = statistics.mean(step)
        out[name] = {"T": T, "unique_experts": U, "ms_per_step": round(ms, 4),
                     "tokens_per_s": round(T / (ms / 1e3), 1),
                     "algorithmic_bytes": b["total"],
                     "hbm_gbs": round(b["total"] / (ms / 1e3) / 1e9, 1),
                     "frac_of_measured": round(b["total"] / (ms / 1e3) / 1e9 / peak, 4),
                     "stage_us": {k: round(v * 1e3, 1) for k, v in stage.items()},
                     "stage_gbs": {k: round(b[k] / (stage[k] / 1e3) / 1e9, 1)
                                   for k in ROOFLINE_STAGES if k in stage and b[k] > 0},
                     "stage_hbm_frac": {k: round(b[k] / (stage[k] / 1e3) / 1e9 / peak, 4)
                                        for k in ROOFLINE_STAGES if k in stage and b[k] > 0},
                     "stage_unit_frac": unit_fractions(macs, stage, sms, SM_MHZ_MAX,
                                                       load_tensor_peak()),
                     "ms_per_step_median": round(statistics.median(step), 4)}
        assert moe.check_device_error(ws) == 0
    out.update(run_router_sweep(torch, moe, synth, dev, layer, flush, peak))
    out.update(run_stream_sweep(torch, moe, synth, dev, layer))
    return out


def run_router_sweep(torch, moe, synth, dev, layer, flush, peak):
    """The router front end at T=1: x -> router logits GEMM (fp32 W_r [E][d]) ->
    layer, on the sigmoid layer and on the DeepSeek-scored 384-expert layer.
    Three CUDA graphs per case -- the logits GEMM kernel alone, that kernel
    followed by moe_layer, and moe_layer_from_x (the GEMM inside the decode
    kernel) -- each replayed 10 times after 3 warm-ups with L2 flushed before
    every replay.  ms_per_step is moe_layer_from_x."""
    out = {}
    cases = [("router_decode_t1", synth.GLM_LAYER, layer), ("ds_router_decode_t1", synth.DS_LAYER, None)]
    stream = torch.cuda.current_stream(dev)
    for name, spec, lay in cases:
        if lay is None:
            w = synth.fill_layer_device(spec, dev)
            lay = moe.Layer(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s, w, dev,
                            score=spec.score)
        T = 1
        desc = lay.desc()
        ws = torch.zeros(moe.workspace_size(desc, T), dtype=torch.uint8, device=dev)
        bias = torch.from_numpy(synth.bias(spec)).to(dev)
        w_r = torch.from_numpy(synth.router_weights(spec)).to(dev)
        _, x = synth.token_inputs(spec, 0, T)
        x_d = torch.from_numpy(x).to(dev)
        l_d = torch.empty((T, spec.E), dtype=torch.float32, device=dev)
        y = torch.empty((T, spec.d), dtype=torch.float32, device=dev)

        def router_only():
            moe.router_logits(desc, w_r, x_d, l_d)

        def separate():
            moe.router_logits(desc, w_r, x_d, l_d)
            moe.layer(desc, lay.weights, x_d, l_d, bias, y, ws)

        def from_x():
            moe.layer_from_x(desc, lay.weights, w_r, x_d, bias, l_d, y, ws)

        for _ in range(3):
            separate()
            from_x()
        torch.cuda.synchronize()
        graphs = []
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            for fn in (router_only, separate, from_x):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=cap):
                    fn()
                graphs.append(g)
        stream.wait_stream(cap)
        n = 10
        times = []
        for g in graphs:
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(n)]
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
            for a, b in ev:
                flush()
                a.record()
                g.replay()
                b.record()
            torch.cuda.synchronize()
            times.append(statistics.mean(a.elapsed_time(b) for a, b in ev))
        r_ms, sep_ms, ms = times
        off = lay.views(ws, T)["off"].cpu()
        counts = (off[1:] - off[:-1]).tolist()
        b = stage_bytes(spec, T, counts, None)["total"] + spec.E * spec.d * 4
        out[name] = {"T": T, "E": spec.E, "top_k": spec.k,
                     "score": "sqrt_softplus" if spec.score else "sigmoid",
                     "ms_per_step": round(ms, 4), "router_us": round(r_ms * 1e3, 1),
                     "separate_kernels_ms": round(sep_ms, 4),
                     "router_gbs": round(spec.E * spec.d * 4 / (r_ms / 1e3) / 1e9, 1),
                     "tokens_per_s": round(T / (ms / 1e3), 1), "algorithmic_bytes": b,
                     "hbm_gbs": round(b / (ms / 1e3) / 1e9, 1),
                     "frac_of_measured": round(b / (ms / 1e3) / 1e9 / peak, 4)}
        assert moe.check_device_error(ws) == 0
    return out


def h2d_peak_gbs(torch, dev, nbytes=1 << 30):
    """Pinned host -> HBM copy bandwidth (one cudaMemcpyAsync of 1 GiB, best of 5)."""
    src = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dst = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    best = None
    for _ in range(6):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    del src, dst
    return nbytes / (best / 1e3) / 1e9


def run_stream_sweep(torch, moe, synth, dev, layer, n_layers=8, n_slots=512, warm=24, timed=40):
    """Host-tier expert streaming: a decode stack of n_layers layers of the headline
    shape whose routed experts live in pinned host memory (every layer reuses the
    headline layer's routed weights: the cache keys (layer, expert) differ, so each
    miss is a real 40 MB copy), an HBM cache of n_slots expert slots, resident
    shared experts.  Per token and layer: router GEMM on rmsnorm(x) plus the
    layer's popularity offset -> moe_stream_layer -> x += y.  With lookahead the
    next layer's router also runs on this layer's input and its picks are
    prefetched on a side stream.  Cold cache, `warm` tokens, then `timed` tokens
    timed with CUDA events; weights far exceed L2 (no flush needed)."""
    import dataclasses
    import numpy as np

    spec = synth.GLM_LAYER
    out = {}
    t = layer.tensors
    host_t = {}
    for n in ("gate", "up", "down"):
        for sfx in ("_q", "_s"):
            host_t[n + sfx] = t[n + sfx].cpu().pin_memory()
    host_w = moe.MoeWeights()
    for n in ("gate", "up", "down"):
        setattr(host_w, n, moe.MoeMat(host_t[n + "_q"].data_ptr(), host_t[n + "_s"].data_ptr()))
    arena_t = {k: torch.empty((n_slots,) + tuple(v.shape[1:]), dtype=v.dtype, device=dev)
               for k, v in host_t.items()}
    arena = moe.MoeWeights()
    for n in ("gate", "up", "down"):
        setattr(arena, n, moe.MoeMat(arena_t[n + "_q"].data_ptr(), arena_t[n + "_s"].data_ptr()))
    shared = moe.MoeWeights()
    for n in ("s_gate", "s_up", "s_down"):
        setattr(shared, n, getattr(layer.weights, n))
    desc = layer.desc()
    specs = [dataclasses.replace(spec, layer_seed=1000 + l) for l in range(n_layers)]
    w_r = [torch.from_numpy(synth.router_weights(s)).to(dev) for s in specs]
    offs = [torch.from_numpy(synth.zipf_offset(s.layer_seed, synth.STREAM_ZIPF, s.E,
                                               s.zipf_beta)).to(dev) for s in specs]
    bias = [torch.from_numpy(synth.bias(s)).to(dev) for s in specs]
    ws = torch.zeros(moe.workspace_size(desc, 1), dtype=torch.uint8, device=dev)
    peak = h2d_peak_gbs(torch, dev)
    # the link rate from where the expert tier itself sits in host memory (its
    # pinned pages may land on another NUMA node than the 1 GiB probe's): 16
    # experts' gate codes, one copy each, best of 3
    n_probe = 16
    src_rows = host_t["gate_q"].view(spec.E, -1)
    dst_probe = torch.empty((n_probe, src_rows.shape[1]), dtype=torch.int8, device=dev)
    tier_gbs = None
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(n_probe):
            dst_probe[i].copy_(src_rows[(37 * i) % spec.E], non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        gbs = n_probe * src_rows.shape[1] / (a.elapsed_time(b) / 1e3) / 1e9
        tier_gbs = gbs if tier_gbs is None else max(tier_gbs, gbs)
    del dst_probe
    expert_bytes = spec.f * spec.d * 2 * 1.0625 + spec.d * spec.f * 1.0625
    side = torch.cuda.Stream(dev)

    def logits_of(l, xn):
        lg = torch.empty((1, spec.E), dtype=torch.float32, device=dev)
        moe.router_logits(desc, w_r[l], xn, lg)
        return lg + offs[l]

    for lookahead in (False, True):
        table = torch.full((n_layers, spec.E), -1, dtype=torch.int32, device=dev)
        cache = moe.ExpertCache(desc, [host_w] * n_layers, arena, n_slots, table.data_ptr())
        evs = []
        y = torch.empty((1, spec.d), dtype=torch.float32, device=dev)
        for tok in range(warm + timed):
            if tok == warm:
                torch.cuda.synchronize()
                s0 = cache.stats()
            _, x0 = synth.token_inputs(spec, 7000 + tok, 1)
            x = torch.from_numpy(x0).to(dev)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            for l in range(n_layers):
                xn = x * torch.rsqrt((x * x).mean(dim=1, keepdim=True) + 1e-6)
                lg = logits_of(l, xn)
                nl = logits_of(l + 1, xn) if lookahead and l + 1 < n_layers else None
                moe.stream_layer(cache, l, desc, shared, xn, lg, bias[l], y, ws, next_logits=nl,
                                 next_bias=bias[l + 1] if nl is not None else None,
                                 prefetch_stream=side)
                x = x + y
            b.record()
            if tok >= warm:
                evs.append((a, b))
        torch.cuda.synchronize()
        assert moe.check_device_error(ws) == 0
        s1 = cache.stats()
        cache.close()
        ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
        d = {k: s1[k] - s0[k] for k in s1}
        link = d["bytes_h2d"] / timed
        name = "stream_decode_t1" + ("_lookahead" if lookahead else "")
        out[name] = {
            "layers": n_layers, "cache_slots": n_slots,
            "cache_fraction": round(n_slots / (n_layers * spec.E), 4),
            "ms_per_token": round(ms, 4), "tokens_per_s": round(1e3 / ms, 2),
            "hit_rate": round(d["hits"] / max(d["lookups"], 1), 4),
            "misses_per_token": round(d["misses"] / timed, 2),
            "prefetch_loads_per_token": round(d["prefetch_loads"] / timed, 2),
            "prefetch_hit_rate": round(d["prefetch_hits"] / max(d["prefetch_loads"], 1), 4),
            "h2d_bytes_per_token": int(link),
            "h2d_gbs": round(link / (ms / 1e3) / 1e9, 1),
            "h2d_peak_gbs": round(peak, 1),
            "h2d_expert_tier_gbs": round(tier_gbs, 1),
            "h2d_frac_of_measured": round(link / (ms / 1e3) / 1e9 / peak, 4),
            "hbm_bytes_per_token": int(n_layers * 9 * expert_bytes),
        }
    del arena_t, host_t
    torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------ CPU oracle
_HOST_EXPERTS = {}


def _host_expert(spec, e):
    key = (spec.name, e)
    if key not in _HOST_EXPERTS:
        if len(_HOST_EXPERTS) > 64:
            _HOST_EXPERTS.clear()
        import synth

        _HOST_EXPERTS[key] = synth.expert_host(spec, e)
    return _HOST_EXPERTS[key]


def oracle_tokens(workload: str, seconds: float, max_tokens=None, start=0):
    """Time the oracle on successive tokens of the workload (from sample number
    `start`) until `seconds` of oracle time have been spent or `max_tokens` are
    done.  Returns (tokens, oracle_seconds, description)."""
    import oracle
    import synth

    spec, T, seeds = synth.WORKLOADS[workload]
    bias = synth.bias(spec)
    shared = _host_expert(spec, spec.E) if spec.f_shared else None
    done = 0
    spent = 0.0
    while True:
        sample = start + done
        s = seeds[sample % len(seeds)]
        logits, x = synth.token_inputs(spec, s, T)
        # one token of the batch per sample (tokens are independent given the routing)
        t_pick = (sample * 37) % T
        idx, _ = oracle.route(logits, bias, spec.k, spec.s)
        cache = {int(e): _host_expert(spec, int(e)) for e in idx[t_pick]}
        t0 = time.perf_counter()
        oracle.layer(spec.E, spec.k, spec.d, spec.f, spec.f_shared, spec.fmt, spec.s, cache,
                     shared, x, logits, bias, want=[t_pick])
        spent += time.perf_counter() - t0
        done += 1
        if spent >= seconds or (max_tokens and done >= max_tokens):
            break
    desc = (f"{done} token(s) of {workload} (T={T} batch routed, one token's experts + shared "
            f"expert run through the oracle per sample)")
    return done, spent, desc


def cpu_baseline(workload: str, seconds: float):
    n, spent, desc = oracle_tokens(workload, seconds)
    return {"value": round(n / spent, 4), "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": desc, "oracle_seconds": round(spent, 2)}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import synth

    spec, T, seeds = synth.WORKLOADS[args.workload]
    K, W = args.steps, args.warmup
    for i in range(W):
        oracle_tokens(args.workload, 0.0, max_tokens=1, start=i)
    per = []
    total_tokens = 0
    t0 = time.perf_counter()
    for i in range(K):
        n, spent, desc = oracle_tokens(args.workload, 0.0, max_tokens=1, start=i)
        per.append(spent)
        total_tokens += n
    wall = time.perf_counter() - t0
    value = total_tokens / sum(per)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(1e3 * sum(per) / K, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int8 x int8 -> int32 block dots, fp64 sums (CPU oracle)",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": workload_desc(args.workload, spec, T), "tokens_per_step": 1,
                   "host": f"{platform.machine()}, {os.cpu_count()} cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": 1,
                         "kind": "oracle", "sample": f"{K} steps x 1 token of {args.workload}"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 2),
    }


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        line = run_reference(args)
    else:
        line = run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
