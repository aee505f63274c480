"""Benchmark of the GB300 block-scaled fused MoE layer.

Default workload (one "step" = one whole fused_moe_a8w4 call: sort,
activation quantisation, stage-1 GEMM + SiLU/requant, stage-2 GEMM +
weighted reduction, BF16 output): the DeepSeek-V4.1-Flash TP4 backbone MoE
at the largest decode bucket of its sweep, M=768 tokens, H=5120,
I=576 padded to 640, 384 experts, top-6, uniform routing, seeded synthetic
inputs (AITER #5609 "Add DeepSeek V4.1 Flash TP4 gfx950 MoE tuning",
Configuration). The other buckets of that sweep are reported under "sweep",
the gating kernel (router logits -> top-k ids and weights, 384 experts,
top-6) at the bench M and at M=16384 under "router" (µs, GB/s of logits
read and ids/weights written, fraction of measured HBM), and the gated call
(router logits in, gating inside the call) at M=6 and the bench M under
"gated".

The prefill half of the metric is reported under "prefill": the skewed
prefill stress (backbone a8w4, M=16384, Zipf(1.2) routing) and the a16w4
385-expert top-7 geometry with the fused shared expert at M=16384, each as
µs/call, TFLOP/s, the fraction of the block-scaled MMA peak (a8w4: the FP8
rate, taken as twice the measured BF16 GEMM rate; a16w4: the BF16 rate), the
fraction of measured HBM bandwidth, and the fraction of the binding roofline
max(bytes / HBM, flops / MMA peak) / time.

Timing: the call is captured once in a CUDA graph; every timed step flushes
L2 (a 256 MiB write, outside the timed events) and replays the graph between
two CUDA events on the launching stream. W untimed warm-up steps come first;
exactly K steps are timed inside a barrier + synchronize bracket, max over
ranks. A second pass of K eager calls records events around each kernel
(moe_profile_*) for the roofline of the dominant kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--M 768]
  python bench.py --impl reference     # the CPU oracle on the host cores
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import moe_inputs as mi  # noqa: E402

# decode sweep of each workload's geometry (the pages' token buckets)
# the draft sweep follows its tuned decode rows (M=5 is the pages' draft row)
SWEEP = {"backbone": mi.TOKENS["backbone"], "draft": [5, 10, 20, 40, 80, 160, 320, 640],
         "ep": mi.TOKENS["ep"],
         "a16w4_384": mi.TOKENS["a16w4"], "a16w4_385": mi.TOKENS["a16w4"], "zipf": []}
L2_FLUSH_BYTES = 256 << 20


WORKLOADS = {
    # --config name: (geometry, routing, description)
    "backbone": ("backbone", "uniform", "DeepSeek-V4.1-Flash TP4 backbone MoE a8w4: H=5120, "
                 "I=576 padded to 640, 384 experts, top-6, uniform routing"),
    "draft": ("draft", "uniform", "DeepSeek-V4.1-Flash TP4 draft MoE a8w4: H=5120, I=576 "
              "padded to 640, 128 experts, top-3, uniform routing"),
    "ep": ("ep", "uniform", "DeepSeek-V4.1-Flash expert-parallel shard a8w4: H=5120, I=2304, "
           "96 local of 384 experts, top-6, uniform routing"),
    "a16w4_384": ("a16w4_384", "uniform", "DeepSeek-V4.1-Flash a16w4: H=5120, I=768, 384 "
                  "experts, top-6, uniform routing"),
    "a16w4_385": ("a16w4_385", "uniform", "DeepSeek-V4.1-Flash a16w4: H=5120, I=768, 385 "
                  "experts, top-7 with the fused shared expert 384"),
    "zipf": ("backbone", "zipf", "DeepSeek-V4.1-Flash TP4 backbone MoE a8w4: H=5120, I=576 "
             "padded to 640, 384 experts, top-6, Zipf(1.2) routing"),
}


def metric_name(M: int, config: str = "backbone") -> str:
    geo = WORKLOADS[config][0]
    variant = "a16w4" if mi.SHAPES[geo].a16 else "a8w4"
    label = config if config.startswith("a16w4") else f"{config} {variant}"
    return f"fused_moe us/call ({label}, M={M})"


def launches_per_call(M: int, topk: int) -> int:
    """Kernels one fused call launches: up to 256 routes the sort and the
    gather are one launch; up to 8192 routes the sort is one CTA group,
    above it a count and a scatter launch; then stage 1, stage 2, finalise."""
    R = M * topk
    if R == 0:
        return 0
    front = 1 if R <= 256 else (2 if R <= 8192 else 3)
    return front + 3


def recorded_traffic(kernel: str, M: int, config: str = "backbone"):
    """DRAM bytes per launch of `kernel` from the committed ncu capture of the
    bench workload, or None when the capture is for another kernel or
    workload, or the kernel sources changed since it was taken (the record
    holds a SHA-256 of them)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "roofline_traffic.json")
    try:
        rec = json.load(open(path))
    except (OSError, ValueError):
        return None
    if rec.get("kernel") != kernel or M != 768 or config != "backbone":
        return None
    h = hashlib.sha256()
    for f in rec.get("source_files", []):
        try:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        except OSError:
            return None
    if h.hexdigest() != rec.get("source_sha256"):
        return None
    return int(rec["traffic_bytes_per_launch"])


def peaks():
    """(HBM GB/s, BF16 dense TFLOP/s burst, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, device) -> float:
    """The largest of every rank's value; every rank gets it (the job's time
    is its slowest rank's)."""
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def us_per_call(total_ms: float, steps: int, world: int) -> float:
    """Whole-job µs per call: each of `world` replicas ran `steps` calls
    within the slowest rank's total_ms."""
    return total_ms * 1000 / (steps * world)


def work_model(shape, ids, M):
    """Algorithmic bytes and flops of one call (valid routes, touched experts)."""
    E, H, Ip, k = shape.E, shape.H, shape.Ip, ids.shape[1]
    flat = ids.reshape(-1)
    valid = flat[(flat >= 0) & (flat < E)]
    R = int(valid.numel())
    Et = int(torch.unique(valid).numel())
    w1_e = 2 * Ip * (H // 2 + H // 32)
    w2_e = H * (Ip // 2 + Ip // 32)
    act = 2 if shape.a16 else 1 + 1 / 32          # bytes per activation / intermediate element
    # stage 1 reads the weights of the touched experts and each token's
    # (quantised) row once, and writes the intermediate of every route;
    # stage 2 reads the weights and the intermediate and adds into the
    # FP32 accumulator
    s1 = Et * w1_e + M * H * act + R * Ip * act
    s2 = Et * w2_e + R * Ip * act + M * H * 4
    call = Et * (w1_e + w2_e) + M * H * 2 * 2 + 2 * R * Ip * act
    flops = 2.0 * R * (2 * Ip * H + H * Ip)
    return dict(R=R, experts_touched=Et, stage1_bytes=s1, stage2_bytes=s2, call_bytes=call,
                flops=flops)


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [ln.split(",") for ln in open(self.path).read().splitlines() if ln.strip()]
        os.unlink(self.path)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                for n, v in zip(names, r[5:9]):
                    if v.strip() == "Active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _touched(case, shape):
    flat = case.topk_ids.reshape(-1)
    return torch.unique(flat[(flat >= 0) & (flat < shape.E)]).tolist()


def oracle_slice(case, shape, experts):
    """One FP64 oracle run over every route of `experts`; returns seconds."""
    from oracle import moe as om
    t0 = time.perf_counter()
    om.fused_moe(case.x, case.topk_ids, case.topk_weights, case.w1, case.w1_scale,
                 case.w2, case.w2_scale, shape.E, a16=shape.a16, experts=experts)
    return time.perf_counter() - t0


def cpu_baseline(case, shape, budget_s: float = 12.0):
    """Time the FP64 oracle on a bounded slice (whole experts) of the call and
    scale to the full call by the touched-expert count."""
    touched = _touched(case, shape)
    done, t_used = 0, 0.0
    chunk = 4
    while done < len(touched) and t_used < budget_s:
        sel = touched[done:done + chunk]
        t_used += oracle_slice(case, shape, sel)
        done += len(sel)
    est_us = t_used / done * len(touched) * 1e6
    return {"value": round(est_us, 1), "unit": "us/call", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": (f"FP64 numpy oracle on {done} of the {len(touched)} touched experts "
                       f"(all their routes) of the M={case.M} call, {t_used:.1f} s, scaled by "
                       f"{len(touched)}/{done}; BLAS threads = host cores")}


def run_reference(args):
    """The reference arm: the CPU oracle as it stands, on the host cores.
    A whole call of the bench workload takes the oracle tens of seconds, so
    each step runs the oracle on the same fixed slice of the call (the first
    `slice` touched experts, every route of each); ms_per_step is the time a
    step really took, and value is the per-call time extrapolated from the
    slice by the touched-expert count (marked so in the line)."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    geo, routing, _ = WORKLOADS[args.config]
    shape = mi.SHAPES[geo]
    case = mi.make_case(geo, args.M, routing=routing)
    touched = _touched(case, shape)
    # size the slice so that warm-up + timed steps take about args.ref_budget
    # seconds per step at most (the first probe step sets the rate)
    probe = oracle_slice(case, shape, touched[:4]) / 4
    n_slice = int(max(1, min(len(touched), args.ref_budget / max(probe, 1e-6))))
    sl = touched[:n_slice]
    for _ in range(args.warmup):
        oracle_slice(case, shape, sl)
    t_steps = [oracle_slice(case, shape, sl) for _ in range(args.steps)]
    step_s = statistics.mean(t_steps)
    v = step_s * len(touched) / n_slice * 1e6
    cb = {"value": round(v, 1), "unit": "us/call", "cores": os.cpu_count(), "kind": "oracle",
          "sample": (f"FP64 numpy oracle on {n_slice} of the {len(touched)} touched experts "
                     f"(all their routes) of the M={args.M} call per step, "
                     f"{step_s:.2f} s per step, scaled by {len(touched)}/{n_slice}; "
                     "BLAS threads = host cores")}
    line = {"impl": "reference", "metric": metric_name(args.M, args.config),
            "value": round(v, 1),
            "unit": "us/call", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(step_s * 1000, 3), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "config": config_dict(args.M, world, args.config), "cpu_baseline": cb,
            "value_extrapolated": {"from_experts": n_slice, "of_experts": len(touched),
                                   "measured_s_per_step": round(step_s, 3)},
            "e2e": {"value": round(v, 1), "unit": "us/call", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


PREFILL = (
    # (key, geometry, tokens, routing)
    ("zipf_a8w4_M16384", "backbone", 16384, "zipf"),
    ("a16w4_385_M16384", "a16w4_385", 16384, "uniform"),
)


def measure_prefill(m, dev, stream, flush, hbm, bf16, backbone_layer, backbone_weights,
                    steps: int = 10):
    """The prefill buckets of the metric: whole-call graph replays with L2
    flushed before each, µs/call (median), TFLOP/s and the fractions of the
    MMA peak, of HBM and of the binding roofline."""
    res = {}
    e_s = torch.cuda.Event(enable_timing=True)
    e_e = torch.cuda.Event(enable_timing=True)
    for key, name, M, routing in PREFILL:
        shape = mi.SHAPES[name]
        if name == "backbone":
            layer, weights = backbone_layer, backbone_weights
        else:
            weights = mi.make_weights(shape, mi.weight_seed(mi.CONFIG_INDEX[name]))
            layer = m.MoeLayer(weights["w1"], weights["w1_scale"], weights["w2"],
                               weights["w2_scale"], a16=shape.a16, device=dev,
                               block_m_table="gb300")
        case = mi.make_case(name, M, routing=routing, weights=weights)
        x, ids, w = case.x.to(dev), case.topk_ids.to(dev), case.topk_weights.to(dev)
        out = torch.empty(M, shape.H, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(layer.workspace_bytes(M, shape.topk), dtype=torch.uint8, device=dev)
        g = time_graph(layer, x, ids, w, out, ws, steps, 3, flush, stream)
        ts = []
        for _ in range(steps):
            flush.zero_()
            e_s.record(stream)
            g.replay()
            e_e.record(stream)
            e_e.synchronize()
            ts.append(e_s.elapsed_time(e_e))
        us = statistics.median(ts) * 1000
        wm = work_model(shape, case.topk_ids, M)
        peak_tf = bf16 * (1 if shape.a16 else 2)
        t_hbm = wm["call_bytes"] / (hbm * 1e3)          # µs
        t_mma = wm["flops"] / (peak_tf * 1e6)           # µs
        res[key] = {
            "workload": (f"{name} {'a16w4' if shape.a16 else 'a8w4'} M={M}, {routing} routing, "
                         f"E={shape.E}, top-{shape.topk}, H={shape.H}, Ip={shape.Ip}"),
            "us": round(us, 1), "tflops": round(wm["flops"] / us / 1e6, 1),
            "mma_peak_tflops": round(peak_tf, 1),
            "mma_peak": ("FP8 rate = 2 x measured BF16 GEMM (MEASURED_PEAKS.json bf16_tflops)"
                         if not shape.a16 else "measured BF16 GEMM (MEASURED_PEAKS.json)"),
            "mma_frac": round(t_mma / us, 4), "hbm_frac": round(t_hbm / us, 4),
            "binding_frac": round(max(t_hbm, t_mma) / us, 4),
            "binding": "mma" if t_mma >= t_hbm else "hbm",
            "flops": wm["flops"], "bytes": int(wm["call_bytes"]),
            "experts_touched": wm["experts_touched"], "routes": wm["R"],
            "replays": steps}
        del g, ws, out, x, ids, w
        if name != "backbone":
            del layer
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return res


def config_dict(M, world, config: str = "backbone"):
    geo, _, desc = WORKLOADS[config]
    shp = mi.SHAPES[geo]
    return {"workload": f"{desc}; M={M} tokens",
            "tokens": M, "H": shp.H, "I": shp.I, "Ip": shp.Ip, "experts": shp.E,
            "topk": shp.topk,
            "route_block": "shipped GB300 tuning rows of the geometry, else the library rule",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "flushed (256 MiB write) before every timed step"}


def time_graph(layer, x, ids, w, out, ws, steps, warmup, flush, stream):
    for _ in range(warmup):
        layer(x, ids, w, out=out, ws=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        layer(x, ids, w, out=out, ws=ws)
    torch.cuda.synchronize()
    for _ in range(2):
        flush.zero_()
        g.replay()
    torch.cuda.synchronize()
    return g


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--M", type=int, default=768)
    ap.add_argument("--config", default="backbone", choices=sorted(WORKLOADS),
                    help="workload geometry and routing (default: the backbone decode bucket)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-budget", type=float, default=4.0,
                    help="reference arm: seconds of oracle work per step (about)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args)
        return

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    import block_scaled_moe_sort_gb300 as m

    geo, routing, _ = WORKLOADS[args.config]
    shape = mi.SHAPES[geo]
    weights = mi.make_weights(shape, mi.weight_seed(mi.CONFIG_INDEX[geo]))
    layer = m.MoeLayer(weights["w1"], weights["w1_scale"], weights["w2"], weights["w2_scale"],
                       a16=shape.a16, device=dev, block_m_table="gb300")
    case = mi.make_case(geo, args.M, routing=routing, weights=weights)
    x, ids, w = case.x.to(dev), case.topk_ids.to(dev), case.topk_weights.to(dev)
    M, k = args.M, shape.topk
    out = torch.empty(M, shape.H, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(layer.workspace_bytes(M, k), dtype=torch.uint8, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    hbm, bf16, peak_kind = peaks()
    wm = work_model(shape, case.topk_ids, M)

    with torch.cuda.stream(stream):
        g = time_graph(layer, x, ids, w, out, ws, args.steps, args.warmup, flush, stream)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        sampler = ClockSampler(local)
        sampler.start()
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            g.replay()
            ends[i].record(stream)
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        clocks = sampler.stop()
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        total_ms = sum(step_ms)
        if world > 1:
            total_ms = max_over_ranks(total_ms, dev)
        call_us = us_per_call(total_ms, args.steps, world)

        # ---- per-kernel timing pass (eager calls, events around each kernel)
        m.moe_profile_enable(True)
        m.moe_profile_collect()
        for i in range(args.steps):
            flush.zero_()
            layer(x, ids, w, out=out, ws=ws)
        torch.cuda.synchronize()
        kms, ncalls = m.moe_profile_collect()
        m.moe_profile_enable(False)
        kmean = {kk: v / max(ncalls, 1) for kk, v in kms.items()}

        # ---- end to end through the public API with host buffers
        xh = case.x.pin_memory()
        idh = case.topk_ids.pin_memory()
        wh = case.topk_weights.pin_memory()
        oh = torch.empty(M, shape.H, dtype=torch.bfloat16).pin_memory()
        e_s = torch.cuda.Event(enable_timing=True)
        e_e = torch.cuda.Event(enable_timing=True)
        e2e_ms = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            e_s.record(stream)
            x.copy_(xh, non_blocking=True)
            ids.copy_(idh, non_blocking=True)
            w.copy_(wh, non_blocking=True)
            layer(x, ids, w, out=out, ws=ws)
            oh.copy_(out, non_blocking=True)
            e_e.record(stream)
            e_e.synchronize()
            if i >= args.warmup:
                e2e_ms.append(e_s.elapsed_time(e_e))
        e2e_us = statistics.mean(e2e_ms) * 1000

        # ---- decode sweep of the same geometry
        sweep = {}
        if not args.no_sweep:
            for Ms in SWEEP[args.config]:
                c = mi.make_case(geo, Ms, routing=routing, weights=weights)
                xs, ids_s, w_s = c.x.to(dev), c.topk_ids.to(dev), c.topk_weights.to(dev)
                o_s = torch.empty(Ms, shape.H, dtype=torch.bfloat16, device=dev)
                ws_s = torch.empty(layer.workspace_bytes(Ms, k), dtype=torch.uint8, device=dev)
                gs = time_graph(layer, xs, ids_s, w_s, o_s, ws_s, 5, 3, flush, stream)
                ts = []
                for _ in range(10):
                    flush.zero_()
                    e_s.record(stream)
                    gs.replay()
                    e_e.record(stream)
                    e_e.synchronize()
                    ts.append(e_s.elapsed_time(e_e))
                us = statistics.median(ts) * 1000
                wms = work_model(shape, c.topk_ids, Ms)
                sweep[str(Ms)] = {"us": round(us, 2),
                                  "tflops": round(wms["flops"] / us / 1e6, 2),
                                  "hbm_frac": round(wms["call_bytes"] / us / 1e3 / hbm, 3)}
                del gs

        # ---- gating kernel (router logits -> topk ids / weights), bench M and
        # M=16384: event timing of one launch, L2 flushed before each
        router = {}
        if not args.no_sweep:
            for Mr in (M, 16384):
                gr = torch.Generator().manual_seed(5000 + Mr)
                logits = torch.randn(Mr, shape.E, generator=gr, dtype=torch.float32).to(dev)
                for _ in range(3):
                    m.moe_router_topk(logits, k, stream=stream)
                torch.cuda.synchronize()
                ts = []
                for _ in range(20):
                    flush.zero_()
                    e_s.record(stream)
                    m.moe_router_topk(logits, k, stream=stream)
                    e_e.record(stream)
                    e_e.synchronize()
                    ts.append(e_s.elapsed_time(e_e))
                us = statistics.median(ts) * 1000
                nbytes = Mr * shape.E * 4 + Mr * k * 8
                router[str(Mr)] = {"us": round(us, 2), "bytes": nbytes,
                                   "gbs": round(nbytes / us / 1e3, 1),
                                   "hbm_frac": round(nbytes / us / 1e3 / hbm, 3)}

    # ---- gated calls (router logits -> gating + fused call), at decode
    # sizes with the gating inside the call's first kernel and at the bench M
    gated = {}
    if not args.no_sweep and not shape.a16:
        e_s = torch.cuda.Event(enable_timing=True)
        e_e = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for Mg in sorted({6, M}):
                gr = torch.Generator().manual_seed(6000 + Mg)
                lg = torch.randn(Mg, shape.E_route, generator=gr, dtype=torch.float32).to(dev)
                xg = mi.make_case(geo, Mg, routing=routing, weights=weights).x.to(dev)
                og = torch.empty(Mg, shape.H, dtype=torch.bfloat16, device=dev)
                ig = torch.empty(Mg, k, dtype=torch.int32, device=dev)
                wg = torch.empty(Mg, k, dtype=torch.float32, device=dev)
                wsg = torch.empty(layer.workspace_bytes(Mg, k), dtype=torch.uint8, device=dev)

                def gcall():
                    m.fused_moe_gated(xg, lg, k, layer.w1, layer.w1_scale, layer.w2,
                                      layer.w2_scale, layer.E, layer.Ip, out=og, ws=wsg,
                                      topk_ids=ig, topk_weights=wg, stream=stream)
                for _ in range(3):
                    gcall()
                torch.cuda.synchronize()
                gg = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gg, stream=stream):
                    gcall()
                ts = []
                for _ in range(10):
                    flush.zero_()
                    e_s.record(stream)
                    gg.replay()
                    e_e.record(stream)
                    e_e.synchronize()
                    ts.append(e_s.elapsed_time(e_e))
                gated[str(Mg)] = {"us": round(statistics.median(ts) * 1000, 2),
                                  "front": "one launch (gating, sort, gather)" if Mg * k <= 256
                                  else "gating launch + sort + gather"}
                del gg

    prefill = {}
    if not args.no_prefill:
        with torch.cuda.stream(stream):
            prefill = measure_prefill(m, dev, stream, flush, hbm, bf16, layer, weights)

    # ---- roofline of the dominant kernel
    dom = max(("stage1_gemm", "stage2_gemm"), key=lambda kk: kmean[kk])
    dom_bytes = wm["stage1_bytes"] if dom == "stage1_gemm" else wm["stage2_bytes"]
    dom_ms = kmean[dom]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    roof = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
            "unit": "GB/s", "frac": round(achieved / hbm, 4),
            "traffic": recorded_traffic(dom, M, args.config),
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)",
            "algorithmic_bytes": int(dom_bytes), "kernel_us": round(dom_ms * 1000, 2)}

    line = {
        "metric": metric_name(M, args.config), "value": round(call_us, 2), "unit": "us/call", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": ("bf16 x mxfp4 (fp32 accumulate)" if shape.a16
                  else "fp8e4m3 x mxfp4 (fp32 accumulate)"),
        "data": "synthetic (seeded, random-init weights)", "config": config_dict(M, world, args.config),
        "tflops": round(wm["flops"] / call_us / 1e6, 2),
        "call_hbm_frac": round(wm["call_bytes"] / call_us / 1e3 / hbm, 4),
        "kernels_us": {kk: round(v * 1000, 2) for kk, v in kmean.items()},
        "roofline": roof,
        "e2e": {"value": round(e2e_us, 2), "unit": "us/call",
                "h2d_bytes_per_step": int(x.numel() * 2 + ids.numel() * 4 + w.numel() * 4),
                "d2h_bytes_per_step": int(out.numel() * 2)},
        "gpu_launches": launches_per_call(M, k) * args.steps,
        "clocks": clocks,
        "work": wm,
    }
    if sweep:
        line["sweep"] = sweep
    if router:
        line["router"] = router
    if prefill:
        line["prefill"] = prefill
    if gated:
        line["gated"] = gated
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, shape)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
