"""Benchmark of the GB300 routed-expert MoE block (one JSON line on stdout).

Headline workload (the default): the long prefill, 8,192 tokens through 48 residual MoE layers
(512 Q2_0 experts per layer, 33,973,862,400 bytes of blobs resident in HBM, top-10 routing with a
Zipf prior reseeded per layer, seed 0).  A step is one strata_moe_stack call over the chunk (router
GEMM, top-10, grouping, Q2_0 SwiGLU experts on the tensor cores, combine, rmsnorm + residual, for
every layer) on inputs resident in HBM; the step streams far more than the 129 MB L2, so no flush is
needed.  The line's "configs" record measures the other workloads of the block the same way, each with
its own roofline, end-to-end figure and oracle baseline:
  0  one token, one layer            (HBM-bound decode; L2 flushed between steps)
  1  4-token verify window, one layer (HBM-bound decode; L2 flushed between steps)
  2  one token through 48 layers      (HBM-bound decode stack)
  3  2,048 tokens, one layer          (tensor-core prefill; reports the per-expert load)

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl reference]
                  [--no-cpu-baseline] [--no-subconfigs] [--layers L]

--config picks the headline workload (default 4); --impl reference times the CPU oracle (plain C,
double precision) on the host cores on a bounded sample of the headline workload; --layers limits a
stack workload to its first L layers (for profiling one layer's kernels; such a line is not a bench
figure).  Under torchrun each rank runs an independent replica (the block shards by requests; no
collective on the data path).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gen  # noqa: E402

METRIC = "MoE-layer tokens/s at 1 GB300; achieved HBM GB/s (decode) / TC util (prefill)"
E = 512
H = 2560
BLOB = 1382400
ROUTER_BYTES = E * H * 2
HEADLINE = 4
SUBCONFIGS = (0, 1, 2, 3)
# timed steps per workload: the headline's default, and the sub-records' (each about a second or less)
DEFAULT_STEPS = {0: 2000, 1: 2000, 2: 100, 3: 50, 4: 10}
SUB_STEPS = {0: 1000, 1: 1000, 2: 60, 3: 30, 4: 3}
# expert FLOPs per (token, expert) pair: gate/up two 640 x 2560 products, down one 2560 x 640
FLOPS_PER_PAIR = {"TC_GATEUP": 2 * 2 * 2560 * 640, "TC_DOWN": 2 * 640 * 2560}
ROUTER_FLOPS_PER_TOKEN = 2 * E * H


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=HEADLINE)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-subconfigs", action="store_true")
    ap.add_argument("--layers", type=int, default=None)
    return ap.parse_args(argv)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), d.get("bf16_tflops_sustained", 1700.0), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi samples during the timed region (median SM clock, throttle reasons)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
# workload set-up
# ------------------------------------------------------------------------------------------------
class Arena:
    """Packed blobs of layers 0..n_layers-1 (seed `seed`), generated and packed on the device, shared by
    every workload (they all draw layer l's experts from the same seed)."""

    def __init__(self, qre, seed, dev, n_layers):
        import torch
        self.n_layers = n_layers
        table = torch.from_numpy(gen.SCALE_TABLE.view(np.int16)).to(dev)
        self.blobs = torch.empty(n_layers * E * BLOB, dtype=torch.uint8, device=dev)
        tmp = torch.empty(E * BLOB, dtype=torch.uint8, device=dev)
        s = torch.cuda.current_stream().cuda_stream
        for l in range(n_layers):
            gen.device_canonical_blobs(seed, l, 0, E, table.data_ptr(), tmp.data_ptr(), BLOB, s)
            qre.strata_pack_q2_0_device(tmp, BLOB, self.blobs[l * E * BLOB:], BLOB, E)
        del tmp
        torch.cuda.synchronize()
        self.exs = [qre.experts(self.blobs[l * E * BLOB:], E, 1) for l in range(n_layers)]


def workload(cfg_id, seed, layers=None):
    c = gen.CONFIGS[cfg_id]
    L = c["L"] if layers is None or c["L"] == 1 else min(layers, c["L"])
    return gen.config_inputs(cfg_id, seed, L=L)


def run_step(qre, cfg, exs, wr, bias, x_in, x_work, out, ids, ids_all, ws):
    """One pass of the whole hot path over the batch (x_in is never modified)."""
    T, L = cfg["T"], cfg["L"]
    if L == 1:
        qre.strata_moe_layer(exs[0], wr[0], None if bias is None else bias[0], x_in, T, 0, out, ids, None, ws)
        return out
    x_work.copy_(x_in)
    qre.strata_moe_stack(exs, wr, bias, L, x_work, T, ids_all, None, ws)
    return x_work


# Kernels timed with the library's own event hooks: the whole decode layer for T <= 8; for prefill
# every kernel of the step (the dominant one is picked by total time).
PREFILL_KERNELS = ("ROUTER_PREP", "ROUTER_TC", "TOP_K", "GROUP_HIST", "GROUP_SCAN", "GROUP_SCATTER", "TC_PREPARE",
                   "TC_GATHER", "TC_GATEUP", "TC_DOWN", "COMBINE")
CSRC = os.path.join(ROOT, "quantized_routed_expert_top10_gb300", "csrc")
KERNEL_SOURCES = {
    "DECODE_LAYER": ("decode_fused.cu", "common.cuh", "device_common.cuh"),
    "TC_GATEUP": ("experts_tc.cu", "tc_common.cuh", "common.cuh", "device_common.cuh"),
    "TC_DOWN": ("experts_tc.cu", "tc_common.cuh", "common.cuh", "device_common.cuh"),
}
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch from one ncu capture (summaries
# under profiles/), keyed by (workload, kernel), with the SHA-256 of the kernel's sources at capture
# time: once a source changes the figure no longer describes the kernel (null).  A stack workload's
# per-launch figure is one layer's launch, captured on its first layer (--layers 1).
NCU_TRAFFIC = {
    # profiles/decode_layer_kernel_verify_4tok_1layer.md: mean of 3 launches
    ("verify_4tok_1layer", "DECODE_LAYER"): (29646336, "e149b7c83497eb48"),
    ("decode_1tok_1layer", "DECODE_LAYER"): (16677120, "e149b7c83497eb48"),
    # profiles/decode_layer_kernel_verify_4tok_1layer.md: mean over the 48 launches of one step
    ("decode_1tok_48layer_stack", "DECODE_LAYER"): (19518325, "e149b7c83497eb48"),
    # profiles/tc_expert_kernel_prefill_2048tok_1layer.md: one launch of each expert kernel
    ("prefill_2048tok_1layer", "TC_GATEUP"): (299194112, "86eb6d87c4faf3a8"),
    ("prefill_2048tok_1layer", "TC_DOWN"): (132272640, "86eb6d87c4faf3a8"),
    # profiles/tc_expert_kernel_prefill_8192tok_48layer_stack.md: mean over the 48 launches of each
    # expert kernel in one step (a single-pass capture of the full workload)
    ("prefill_8192tok_48layer_stack", "TC_GATEUP"): (554060512, "86eb6d87c4faf3a8"),
    ("prefill_8192tok_48layer_stack", "TC_DOWN"): (259167040, "86eb6d87c4faf3a8"),
}


def source_digest(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(kernel, ()):
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_name, kernel):
    rec = NCU_TRAFFIC.get((workload_name, kernel))
    if rec is None or rec[1] != source_digest(kernel):
        return None
    return rec[0]


def max_over_ranks(ms, device):
    """The slowest rank's time, on every rank (all-reduce MAX, then a barrier): replicas run the same
    work, so the job's time is its slowest replica's."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def whole_job_rate(tokens_per_step, steps, world, total_ms):
    """Tokens per second of the whole job: every rank processes tokens_per_step per step."""
    return world * tokens_per_step * steps / (total_ms / 1e3)


def measure_workload(qre, arena, cfg_id, args, K, W, world, dev, local_rank, e2e_calls):
    """Time K steps of one workload (after W warm-up steps) and return its record."""
    import torch
    cfg = workload(cfg_id, args.seed, args.layers)
    T, L = cfg["T"], cfg["L"]
    wr = torch.from_numpy(np.stack(cfg["wr"]).view(np.int16)).to(dev)
    bias = None if cfg["bias"][0] is None else torch.from_numpy(np.stack(cfg["bias"])).to(dev)
    exs = arena.exs[:L]
    x_host = cfg["x"]
    x_in = torch.from_numpy(x_host).to(dev)
    x_work = torch.empty_like(x_in)
    out = torch.empty_like(x_in)
    ids = torch.empty(T, 10, dtype=torch.int32, device=dev)
    ids_all = torch.empty(L, T, 10, dtype=torch.int32, device=dev) if L > 1 else None
    ws = torch.empty(qre.strata_moe_workspace_bytes(T), dtype=torch.uint8, device=dev)
    qre.strata_moe_workspace_init(ws)
    need_flush = L == 1 and T <= 8  # one decode layer's working set fits the L2; everything else streams past it
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if need_flush else None
    stream = torch.cuda.current_stream()
    step_args = (qre, cfg, exs, wr, bias, x_in, x_work, out, ids, ids_all, ws)

    for _ in range(W):
        run_step(*step_args)
    torch.cuda.synchronize()
    check_status(qre, ws)

    # Decode steps (T <= 8: one cooperative launch per layer) would be bound by the host's launch rate,
    # so the step is captured once in a CUDA graph and replayed; prefill steps run eagerly.
    graph, graph_launches, graph_note = None, None, "eager launches"
    if T <= 8:
        try:
            n0 = qre.strata_moe_launch_count()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                run_step(*step_args)
            graph_launches = qre.strata_moe_launch_count() - n0
            for _ in range(W):
                graph.replay()
            torch.cuda.synchronize()
            check_status(qre, ws)
            graph_note = "CUDA graph replay of the step"
        except Exception as exc:  # capture refused: fall back to eager launches, and say so
            graph, graph_launches = None, None
            graph_note = f"eager launches (graph capture failed: {str(exc)[:120]})"
            torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    # Dominant-kernel timing inside the timed region: T <= 8 and one layer -> the step is exactly one
    # launch of the decode layer kernel (its events are the step's); T <= 8 stacks replayed as a graph ->
    # the step time over its L launches (an upper bound on the kernel's duration), or, run eagerly,
    # library event hooks around one layer per step; prefill -> every launch of the two tensor-core
    # expert kernels.
    timed = () if (T <= 8 and (L == 1 or graph is not None)) else ("DECODE_LAYER",) if T <= 8 \
        else ("TC_GATEUP", "TC_DOWN")
    per_step = 1 if T <= 8 else L
    kev = {}
    for k in timed:
        kev[k] = ([torch.cuda.Event(enable_timing=True) for _ in range(K * per_step)],
                  [torch.cuda.Event(enable_timing=True) for _ in range(K * per_step)])
        for e in kev[k][0] + kev[k][1]:
            e.record(stream)  # creates the CUDA event behind the torch object
    torch.cuda.synchronize()
    armed = {}
    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.25)
    wall0 = time.perf_counter()
    launches0 = qre.strata_moe_launch_count()
    for i in range(K):
        if need_flush:
            flush.fill_(i & 0xFF)
        for k in timed:
            if T <= 8:  # layer i % L of this step
                armed[k] = qre.strata_moe_profile_arm(k, kev[k][0][i:i + 1], kev[k][1][i:i + 1], skip=i % L)
            elif i == 0:
                armed[k] = qre.strata_moe_profile_arm(k, *kev[k])
        starts[i].record(stream)
        if graph is not None:
            graph.replay()
        else:
            run_step(*step_args)
        ends[i].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    n_launches = graph_launches * K if graph is not None else qre.strata_moe_launch_count() - launches0
    kernel_ms = {}
    for k in timed:
        kernel_ms[k] = [a.elapsed_time(b) for a, b in zip(*kev[k])]
        qre.strata_moe_profile_arm(k, [], [])
    del armed
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    if T <= 8 and L == 1:
        kernel_ms["DECODE_LAYER"] = list(step_ms)
    elif T <= 8 and graph is not None:
        kernel_ms["DECODE_LAYER"] = [m / L for m in step_ms for _ in range(L)]
    if wall < 1.0:
        time.sleep(0.3)
    clk = clocks.stop()
    total_ms = float(np.sum(step_ms))
    if world > 1:
        total_ms = max_over_ranks(total_ms, dev)
    check_status(qre, ws)
    ids_layers = ids_all.cpu().numpy() if L > 1 else ids.cpu().numpy()[None]

    roof = kernel_roofline(cfg, kernel_ms, ids_layers, graph_stack=T <= 8 and L > 1 and graph is not None)
    rec = {
        "value": whole_job_rate(T, K, world, total_ms),
        "unit": "tokens/s",
        "steps": K,
        "warmup": W,
        "ms_per_step": total_ms / K,
        "dtype": path_dtype(T),
        "config": dict(workload_config(cfg, args.seed, world, need_flush), launch=graph_note),
        "roofline": roof,
        "clocks": clk,
        "gpu_launches": n_launches,
    }
    if T > 8:
        rec["kernel_ms_per_step"] = step_breakdown(qre, step_args, stream, L)
        rec["step_tc"] = step_tensor_fraction(cfg, total_ms / K)
        rec["expert_load"] = expert_load(ids_layers)
        rec["expert_roofline"] = expert_roofline(cfg, ids_layers, roof)
    else:
        rec["distinct_experts_per_layer"] = float(np.mean([len(np.unique(l)) for l in ids_layers]))
    rec["e2e"] = measure_e2e(qre, cfg, exs, wr, bias, x_host, ws, flush, dev, e2e_calls, world)
    del ws, flush
    torch.cuda.empty_cache()
    return rec


def check_status(qre, ws):
    st = qre.strata_poll_status(ws)
    if st != 0:
        raise RuntimeError(f"device status {qre.STATUS.get(st, st)}")


def step_breakdown(qre, step_args, stream, L, steps=2):
    """Per-kernel device time of a step (ms), from a separate untimed pass with every prefill kernel's
    launches bracketed by events (the extra event records are kept out of the timed region)."""
    import torch
    evs, armed = {}, {}
    for k in PREFILL_KERNELS:
        evs[k] = ([torch.cuda.Event(enable_timing=True) for _ in range(steps * L)],
                  [torch.cuda.Event(enable_timing=True) for _ in range(steps * L)])
        for e in evs[k][0] + evs[k][1]:
            e.record(stream)
    torch.cuda.synchronize()
    for k in PREFILL_KERNELS:
        armed[k] = qre.strata_moe_profile_arm(k, *evs[k])
    for _ in range(steps):
        run_step(*step_args)
    torch.cuda.synchronize()
    out = {}
    for k in PREFILL_KERNELS:
        n = qre.strata_moe_profile_recorded(k)
        if n:
            out[k] = round(sum(a.elapsed_time(b) for a, b in zip(evs[k][0][:n], evs[k][1][:n])) / steps, 5)
        qre.strata_moe_profile_arm(k, [], [])
    del armed
    return dict(sorted(out.items(), key=lambda kv: -kv[1]))


def path_dtype(T):
    """Arithmetic of the path: one token = dp4a on 2-bit codes x int16-split activations (int32 partial
    sums, fp32 accumulation); 2-8 tokens = fp16 x fp16 warp MMA (mma.sync) with fp32 accumulation;
    prefill = fp16 x fp16 tcgen05 products with fp32 accumulation."""
    if T <= 1:
        return "s8 dp4a (q2 x int16-split x), fp32 acc"
    return "f16 mma.sync, fp32 acc" if T <= 8 else "f16 tcgen05, fp32 acc"


def workload_config(cfg, seed, world, need_flush):
    return {
        "workload": cfg["name"],
        "tokens": cfg["T"],
        "layers": cfg["L"],
        "experts": E,
        "top_k": 10,
        "hidden": 2560,
        "ffn": 640,
        "q2_offset": 1,
        "seed": seed,
        "l2": "256 MB buffer written between timed steps (flush excluded)" if need_flush
        else "working set larger than L2 (no flush)",
        "parallelism": f"replicas x{world}",
    }


def kernel_roofline(cfg, kernel_ms, ids_layers, graph_stack=False):
    """Roofline of the dominant kernel from the per-launch event times taken in the timed region.

    decode layer (T <= 8): HBM-bound; algorithmic bytes per launch = router rows (512 x 2560 bf16) +
      D distinct experts x 1,382,400 B, D from that layer's ids.
    prefill (T > 8): tensor-bound; algorithmic flops per launch = T*10 pairs x 6,553,600 (gate/up:
      two 640 x 2560 products) or x 3,276,800 (down: 2560 x 640).  fp16 operands run at the bf16 rate,
      so the peak is the measured bf16 figure: burst for a single layer, sustained for 48-layer stacks.
    """
    hbm, tc_burst, tc_sust, how = load_peaks()
    T, L = cfg["T"], cfg["L"]
    totals = {k: float(np.sum(v)) for k, v in kernel_ms.items() if v}
    if not totals:
        return None
    dom = max(totals, key=totals.get)
    ms = kernel_ms[dom]
    avg_ms = float(np.mean(ms))
    src = f"{how} (MEASURED_PEAKS.json)" if how == "measured" else "fallback"
    if dom == "DECODE_LAYER":
        d = [len(np.unique(ids_layers[l])) for l in range(ids_layers.shape[0])]
        per_launch = ROUTER_BYTES + float(np.mean(d)) * BLOB
        achieved = per_launch / (avg_ms / 1e3) / 1e9
        return {"kernel": "decode_layer_kernel (router + top-10 + grouping + Q2_0 experts + combine)",
                "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "frac_of": f"hbm_gbs, {src}", "traffic": ncu_traffic(cfg["name"], dom),
                "algorithmic_bytes_per_launch": per_launch, "distinct_experts_per_layer": float(np.mean(d)),
                "avg_launch_ms": avg_ms, "launches_timed": len(ms),
                "timing": "step events (one launch per step)" if L == 1 else
                "step events / layers (graph replay of the layer launches; includes the gaps between them)"
                if graph_stack else "library event hooks around one layer per step (layer = step % layers)"}
    peak = tc_burst if L == 1 else tc_sust
    flops = T * 10 * FLOPS_PER_PAIR[dom]
    achieved = flops / (avg_ms / 1e3) / 1e12
    other = "TC_DOWN" if dom == "TC_GATEUP" else "TC_GATEUP"
    o_ms = float(np.mean(kernel_ms[other])) if kernel_ms.get(other) else None
    return {"kernel": f"tc_expert_kernel ({'gate/up + SwiGLU' if dom == 'TC_GATEUP' else 'down + combine'}, "
                      f"tcgen05 fp16)",
            "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "frac_of": f"{'bf16_tflops' if L == 1 else 'bf16_tflops_sustained'}, {src}",
            "traffic": ncu_traffic(cfg["name"], dom), "algorithmic_flops_per_launch": flops,
            "avg_launch_ms": avg_ms, "launches_timed": len(ms),
            "other_expert_kernel": None if o_ms is None else {
                "kernel": other, "avg_launch_ms": o_ms,
                "achieved_tflops": T * 10 * FLOPS_PER_PAIR[other] / (o_ms / 1e3) / 1e12,
                "frac": T * 10 * FLOPS_PER_PAIR[other] / (o_ms / 1e3) / 1e12 / peak},
            "timing": "library event hooks around every launch of the two expert kernels"}


def step_tensor_fraction(cfg, step_ms):
    """The whole step's algorithmic tensor work (expert gate/up and down, and the router GEMM) over the
    step time, against the same peak as the dominant kernel."""
    _, tc_burst, tc_sust, how = load_peaks()
    T, L = cfg["T"], cfg["L"]
    flops = L * T * (10 * (FLOPS_PER_PAIR["TC_GATEUP"] + FLOPS_PER_PAIR["TC_DOWN"]) + ROUTER_FLOPS_PER_TOKEN)
    peak = tc_burst if L == 1 else tc_sust
    achieved = flops / (step_ms / 1e3) / 1e12
    return {"flops_per_step": flops, "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "frac_of": f"{'bf16_tflops' if L == 1 else 'bf16_tflops_sustained'}, {how}"}


def expert_roofline(cfg, ids_layers, roof):
    """The expert kernels against a roofline that takes each touched expert as it is: an expert with
    n tokens needs n x 9,830,400 flops on the tensor cores but also its 1,382,400-byte blob from HBM, so
    its ideal time is max(flops / tensor peak, bytes / HBM peak); the layer's ideal is the sum over its
    touched experts (tiny experts are bound by their weight bytes, big ones by their flops).  Compared
    with the measured gate/up + down time per layer."""
    hbm, tc_burst, tc_sust, how = load_peaks()
    tc = tc_burst if cfg["L"] == 1 else tc_sust
    per_pair = FLOPS_PER_PAIR["TC_GATEUP"] + FLOPS_PER_PAIR["TC_DOWN"]
    ideal = []
    for l in ids_layers:
        c = np.bincount(l.reshape(-1), minlength=E)
        c = c[c > 0].astype(np.float64)
        ideal.append(float(np.sum(np.maximum(c * per_pair / (tc * 1e12), BLOB / (hbm * 1e9)))) * 1e3)
    other = roof.get("other_expert_kernel", {})
    measured = roof.get("avg_launch_ms", 0.0) + other.get("avg_launch_ms", 0.0)
    ideal_ms = float(np.mean(ideal))
    return {"ideal_ms_per_layer": ideal_ms, "expert_kernels_ms_per_layer": measured,
            "frac": ideal_ms / measured if measured > 0 else None,
            "of": f"{'bf16_tflops' if cfg['L'] == 1 else 'bf16_tflops_sustained'} and hbm_gbs, {how}",
            "formula": "sum over touched experts of max(n_e x 9,830,400 flop / tensor peak, 1,382,400 B / HBM peak)"}


def expert_load(ids_layers):
    """Tokens per expert of each layer's routing: experts touched (U), the largest and the mean load
    over the touched experts, their ratio (the load imbalance) and, for one layer, the whole sorted
    histogram."""
    counts = [np.bincount(l.reshape(-1), minlength=E) for l in ids_layers]
    U = [int(np.count_nonzero(c)) for c in counts]
    mx = [int(c.max()) for c in counts]
    mean = [float(c[c > 0].mean()) for c in counts]
    rec = {"experts_touched": U[0] if len(U) == 1 else float(np.mean(U)),
           "max_tokens_per_expert": mx[0] if len(mx) == 1 else float(np.mean(mx)),
           "mean_tokens_per_touched_expert": mean[0] if len(mean) == 1 else float(np.mean(mean)),
           "max_over_mean": float(np.mean([a / b for a, b in zip(mx, mean)]))}
    if len(counts) == 1:
        c = counts[0]
        rec["tokens_per_expert_sorted"] = sorted((int(v) for v in c[c > 0]), reverse=True)
    else:
        rec["per_layer"] = "mean over layers"
    return rec


def measure_e2e(qre, cfg, exs, wr, bias, x_host, ws, flush, dev, n, world):
    """The user's call: strata_moe_layer_host / strata_moe_stack_host on page-locked host buffers, on a
    stream of its own.  Each call copies the step's input in, runs it, copies the result out and
    returns after synchronising, so the host wall clock around the call is the whole step."""
    import torch
    T, L = cfg["T"], cfg["L"]
    src = torch.from_numpy(x_host)
    hx = src.clone().pin_memory()
    hout = torch.empty_like(hx).pin_memory()
    s = torch.cuda.Stream(device=dev)
    if L == 1:
        call = qre.prepare_layer_host(exs[0], wr[0], None if bias is None else bias[0], hx, T, 0, hout, None, None,
                                      ws, stream=s)
    else:
        call = qre.prepare_stack_host(exs, wr, bias, L, hx, T, None, None, ws, stream=s)
    tot = 0.0
    for i in range(n + 3):
        if L > 1:
            hx.copy_(src)  # the stack call updates x in place: every step starts from the same input
        if flush is not None:
            flush.fill_(i & 0xFF)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        call()
        if i >= 3:
            tot += time.perf_counter() - t0
    nbytes = T * 2560 * 4
    return {"value": world * T * n / tot, "unit": "tokens/s", "h2d_bytes_per_step": nbytes,
            "d2h_bytes_per_step": nbytes, "steps": n,
            "timing": "host wall clock around strata_moe_layer_host / strata_moe_stack_host through the binding's "
                      "prepared call (page-locked buffers; copy in, compute, copy out, stream sync inside the call)"}


# ------------------------------------------------------------------------------------------------
# CPU oracle (baseline / reference arm)
# ------------------------------------------------------------------------------------------------
def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleSample:
    """A bounded sample of a workload for the oracle: `tokens` tokens drawn like the workload's (its
    router, bias and layer-0 experts; for one-token and verify-window workloads, more tokens of the same
    distribution so that every thread has one), one layer.  A 48-layer workload's per-token time is the
    one-layer time x 48."""

    def __init__(self, cfg_id, seed, tokens):
        import oracle
        self.oracle = oracle
        c = gen.CONFIGS[cfg_id]
        cfg = gen.config_inputs(cfg_id, seed, T=tokens, L=1)
        self.name = c["name"]
        self.layers = c["L"]
        self.x = np.ascontiguousarray(cfg["x"][:tokens])
        self.tokens = self.x.shape[0]
        self.wr, self.bias, self.residual = cfg["wr"][0], cfg["bias"][0], cfg["residual"]
        r = oracle.route(self.x, self.wr, self.bias, residual=self.residual)
        self.blobs = [None] * E
        for e in np.unique(r["ids"]):
            self.blobs[int(e)] = gen.canonical_blob(seed, 0, int(e))

    def run(self, threads):
        t0 = time.perf_counter()
        self.oracle.moe_layer(self.x, self.wr, self.bias, self.blobs, residual=self.residual, n_threads=threads)
        return time.perf_counter() - t0

    def rate(self, seconds):
        """Tokens of the workload per second, from one layer's time over the sample."""
        return self.tokens / seconds / self.layers

    def describe(self, reps, seconds, threads):
        return (f"{self.tokens} token(s) x 1 layer of {self.name} on {threads} thread(s), repeated {reps}x in "
                f"{seconds:.1f} s" + (f", per-token time x{self.layers} layers" if self.layers > 1 else ""))


def oracle_baseline(cfg_id, seed, budget_s, single_thread=False):
    """The oracle timed on every host core (threads = cores, one token per thread at least), repeated
    until budget_s; with single_thread also one token on one thread."""
    cores = host_cores()
    smp = OracleSample(cfg_id, seed, cores)
    reps, el = 0, 0.0
    while el < budget_s or reps == 0:
        el += smp.run(cores)
        reps += 1
    rec = {"value": smp.rate(el / reps), "unit": "tokens/s", "cores": cores, "threads": cores, "host_cores": cores,
           "kind": "oracle", "sample": smp.describe(reps, el, cores)}
    if single_thread:
        one = OracleSample(cfg_id, seed, 1)
        r1, e1 = 0, 0.0
        while e1 < budget_s / 3 or r1 == 0:
            e1 += one.run(1)
            r1 += 1
        rec["single_thread"] = {"value": one.rate(e1 / r1), "unit": "tokens/s", "threads": 1,
                                "sample": one.describe(r1, e1, 1)}
    return rec


def reference_arm(args, rank):
    """--impl reference: the oracle on the host cores, each step one bounded sample of the headline
    workload (one token per core, one layer; x48 for a 48-layer workload)."""
    if rank != 0:
        return None
    cfg_id = args.config
    K = args.steps if args.steps is not None else 5
    W = args.warmup
    cores = host_cores()
    smp = OracleSample(cfg_id, args.seed, cores)
    for _ in range(min(W, 1)):
        smp.run(cores)
    step_s = [smp.run(cores) for _ in range(K)]
    value = smp.rate(float(np.mean(step_s)))
    cfg = gen.CONFIGS[cfg_id]
    conf = workload_config(dict(name=cfg["name"], T=cfg["T"], L=cfg["L"]), args.seed, 1, cfg["L"] == 1 and cfg["T"] <= 8)
    cpu = {"value": value, "unit": "tokens/s", "cores": cores, "threads": cores, "host_cores": cores,
           "kind": "oracle", "sample": smp.describe(K, float(np.sum(step_s)), cores)}
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 0,
            "steps": K, "warmup": W, "ms_per_step": 1e3 * float(np.mean(step_s)), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": conf, "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------------------------------------------------------
def measure_gb300(args, rank, world, local_rank):
    import torch

    import quantized_routed_expert_top10_gb300 as qre
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    head = args.config
    subs = () if args.no_subconfigs else tuple(c for c in SUBCONFIGS if c != head)
    n_layers = max(workload(c, args.seed, args.layers)["L"] for c in (head,) + subs)
    arena = Arena(qre, args.seed, dev, n_layers)
    W = max(3, args.warmup)
    K = args.steps if args.steps is not None else DEFAULT_STEPS[head]
    rec = measure_workload(qre, arena, head, args, K, W, world, dev, local_rank,
                           e2e_calls=max(20, min(K, 500)) if gen.CONFIGS[head]["T"] <= 8 else max(10, min(K, 30)))
    sub = {}
    for c in subs:
        r = measure_workload(qre, arena, c, args, SUB_STEPS[c], W, world, dev, local_rank,
                             e2e_calls=200 if gen.CONFIGS[c]["T"] <= 8 else 30)
        sub[str(c)] = r
    result = {
        "metric": METRIC,
        "value": rec["value"],
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": rec["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": rec["dtype"],
        "data": "synthetic (seeded Philox4x32-10 inputs; random Q2_0 experts; no trained weights)",
        "config": rec["config"],
        "roofline": rec["roofline"],
        "clocks": rec["clocks"],
        "e2e": rec["e2e"],
        "gpu_launches": rec["gpu_launches"],
    }
    for key in ("step_tc", "kernel_ms_per_step", "expert_load", "expert_roofline", "distinct_experts_per_layer"):
        if key in rec:
            result[key] = rec[key]
    if sub:
        result["configs"] = sub
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return result


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        res = reference_arm(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    res = measure_gb300(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = oracle_baseline(args.config, args.seed, budget_s=15.0,
                                                  single_thread=gen.CONFIGS[args.config]["T"] <= 8)
            for c, r in res.get("configs", {}).items():
                r["cpu_baseline"] = oracle_baseline(int(c), args.seed, budget_s=4.0,
                                                    single_thread=int(c) in (0, 1))
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
