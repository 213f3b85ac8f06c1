"""Benchmark of the NVFP4 MoE expert layer (libnvfp4moe) on GB300.

One step = one forward of the whole layer (route, quantise, permute, gate/up
GEMM with fused SwiGLU + requantisation, down GEMM, finalize) over one batch
of seeded synthetic tokens whose inputs are resident in HBM.  Prints one
JSON line: the headline is the prefill-sized layer (T=16384, E=64, k=8,
H=7168, I=4096; compute-bound, measured against the FP4 tensor peak), and a
"secondary" object times the decode layer (T=128, E=256, k=8, H=6144,
I=2048; weight-streaming, measured against HBM) in the same run.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on a bounded sample

With N > 1 (torchrun) every rank runs an independent replica of the layer:
the layer has no exchange step, so there is no collective on the data path.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from nvfp4_block_scaled_07_gb300 import workloads as W  # noqa: E402

METRIC = "NVFP4 MoE layer TFLOPS, HBM GB/s, tokens/s, % of GB300 roofline (1 GPU)"
DEFAULT_WORKLOAD = "prefill_t16384"
SECONDARY_WORKLOAD = "decode_t128"
CPU_BUDGET_S = 10.0                  # oracle seconds the cpu_baseline leg samples
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense FP4 / BF16 tensor ratio


def recorded_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` from the ncu record in profiles/, or
    None when there is none for this workload or the kernel sources changed
    since it was taken."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    src = "".join(open(os.path.join(ROOT, n)).read() for n in rec.get("source_files", []))
    if hashlib.sha256(src.encode()).hexdigest() != rec.get("source_sha256"):
        return None
    return rec.get(workload, {}).get(kernel)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only)
# ----------------------------------------------------------------------------
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    """The slowest rank's value: every rank's timed region must end before
    the job's does."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms_per_step):
    """Whole-job rate: the units every replica processed in one step over the
    slowest rank's step time."""
    return units_per_rank * world / (ms_per_step * 1e-3)


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# the CUDA path
# ----------------------------------------------------------------------------
def step_with_kernel_events(B, layer, x, logits, ev):
    """One layer forward with events between its steps (MoELayer.prepare,
    gemm_gate_up, gemm_down, finalize: the calls forward() makes, in the
    same order, on the current stream).  An event between two kernels ends
    their launch overlap, so these per-kernel durations are those of
    isolated launches."""
    ev[0].record()
    layer.prepare(x, logits)
    ev[1].record()
    layer.gemm_gate_up()
    ev[2].record()
    layer.gemm_down()
    ev[3].record()
    layer.finalize()
    ev[4].record()


def kernel_names(fused_prepare):
    return ["prepare", "gemm_gate_up_swiglu", "gemm_down", "finalize"]


def tile_name(t):
    return {-2: "token-major, CTA pairs (256 tokens x 256 weight rows, static schedule)",
            -1: "token-major (128 tokens x 256 weight rows)", 0: "weight rows as M, token tiles up to 128",
            128: "weight rows as M, token tiles up to 128", 256: "weight rows as M, token tiles up to 256"}.get(t, str(t))


def bench_config(w, fmt, k_primary, n_active, world):
    """The `config` object of the JSON line, identical in both arms: the
    workload's shape and generator settings, its format and routing, the
    active experts under seed-0 routing and how L2 is kept out of the
    measurement (the weights streamed per step exceed the 129 MB L2)."""
    k0 = w.k if k_primary is None else k_primary
    w_bytes = n_active * W.fp4_bytes(3 * w.H * w.I, fmt)
    return {"workload": w.name, **w.describe(), "active_experts": int(n_active), "format": fmt,
            "routing": "top-k" if k0 == w.k else f"batch-aware, k_primary={k0}",
            "l2": "inputs larger than L2: %.2f GB of %s weights streamed per step" % (w_bytes / 1e9, fmt.upper()),
            "parallelism": "replicas" if world > 1 else "single GPU"}


def measure_layer(args, w, world, rank, with_e2e=True):
    """Times the layer of workload `w` on this rank's GPU: the device-timed
    steps, per-kernel event times, the end-to-end steps with host buffers
    and the clocks.  Returns (record, layer, inputs)."""
    from nvfp4_block_scaled_07_gb300 import binding as B
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = W.device_inputs(w, seed=args.seed + rank, device=dev)
    layer = B.MoELayer(inp["w_gu"], inp["w_d"], w.k, w.score, w.renormalize, w.h_scale, bias=inp["bias"],
                       T=w.T, tile_n=(args.tile_gate_up, args.tile_down), fused_prepare=not args.separate_prepare,
                       k_primary=args.k_primary, fmt=args.format, dynamic_schedule=not args.static_schedule,
                       tiled_weights=args.weights == "tiled", fused_finalize=args.fused_finalize)
    del inp["w_gu"], inp["w_d"]
    torch.cuda.empty_cache()
    x, logits = inp["x"], inp["logits"]
    for _ in range(args.warmup):
        layer(x, logits)
    B.sync_status()
    counts = layer.perm.counts.cpu().numpy()
    n_active = int((counts > 0).sum())
    stream = torch.cuda.current_stream()

    # ---- device-timed region: inputs resident in HBM, the layer as a user calls it ----
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(torch.cuda.current_device()) as clk:
        start.record(stream)
        for _ in range(args.steps):
            layer(x, logits)
        stop.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    B.sync_status()
    ms_step = max_over_ranks(start.elapsed_time(stop) / args.steps, world)

    # ---- kernel-timing region: the same steps with events between the calls ----
    names = kernel_names(layer.fused_prepare)
    n_ev = len(names) + 1
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for s in range(args.steps):
        step_with_kernel_events(B, layer, x, logits, evs[s])
    torch.cuda.synchronize()
    barrier(world)
    B.sync_status()
    per_kernel = np.array([[evs[s][i].elapsed_time(evs[s][i + 1]) for i in range(n_ev - 1)]
                           for s in range(args.steps)])
    kern_ms = per_kernel.mean(axis=0)
    ms_step_events = float(per_kernel.sum(axis=1).mean())

    # ---- end to end: pinned host inputs in, result out, every step ----
    # Every step copies its inputs in from pinned host memory and its output
    # back.  The copies run on their own streams (the copy engines) and
    # overlap the neighbouring steps' compute: step i + 1's inputs go in
    # while step i computes, step i's output comes back while step i + 1
    # computes (two device buffers of each, reused every other step once the
    # step that used them has finished with them).
    e2e = None
    if with_e2e:
        x_h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True).copy_(x)
        lg_h = torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True).copy_(logits)
        out_h = torch.empty((w.T, w.H), dtype=torch.bfloat16, pin_memory=True)
        xs = [torch.empty_like(x) for _ in range(2)]
        lgs = [torch.empty_like(logits) for _ in range(2)]
        outs = [torch.empty((w.T, w.H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
        h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
        ev = lambda: torch.cuda.Event()
        in_ready = [ev() for _ in range(args.steps)]
        done = [ev() for _ in range(args.steps)]
        back = [ev() for _ in range(args.steps)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        e0.record(h2d_s)
        for i in range(args.steps):
            j = i % 2
            with torch.cuda.stream(h2d_s):
                if i >= 2:
                    h2d_s.wait_event(done[i - 2])  # step i - 2 has read buffers j
                xs[j].copy_(x_h, non_blocking=True)
                lgs[j].copy_(lg_h, non_blocking=True)
                in_ready[i].record(h2d_s)
            with torch.cuda.stream(stream):
                stream.wait_event(in_ready[i])
                if i >= 2:
                    stream.wait_event(back[i - 2])  # step i - 2's output is back on the host
                layer(xs[j], lgs[j], out=outs[j])
                done[i].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(done[i])
                out_h.copy_(outs[j], non_blocking=True)
                back[i].record(d2h_s)
        e1.record(d2h_s)
        torch.cuda.synchronize()
        barrier(world)
        e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
        h2d = x_h.numel() * x_h.element_size() + lg_h.numel() * lg_h.element_size()
        d2h = out_h.numel() * out_h.element_size()
        e2e = {"value": round(job_throughput(w.T, world, e2e_ms), 1), "unit": "tokens/s",
               "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "copies": "pinned host buffers, H2D and D2H on their own streams overlapping the neighbouring "
                         "steps' compute"}
        del x_h, lg_h, out_h, xs, lgs, outs

    # ---- derived numbers ----
    hbm_peak, bf16_peak, peak_kind = measured_peaks()
    fp4_peak = bf16_peak * FP4_OVER_BF16
    R = w.T * w.k
    flops = W.algorithmic_flops(w)
    fb = lambda n: W.fp4_bytes(n, layer.fmt)
    w_bytes_active = n_active * fb(3 * w.H * w.I)
    alg_bytes = w_bytes_active + 2 * w.T * w.H * 2
    tokens_s = job_throughput(w.T, world, ms_step)
    gemms = {}
    for kname, n_rows, k_dim, mult in (("gemm_gate_up_swiglu", 2 * w.I, w.H, 4.0), ("gemm_down", w.H, w.I, 2.0)):
        g_ms = float(kern_ms[names.index(kname)])
        g_bytes = n_active * fb(n_rows * k_dim) + fb(R * k_dim) + (fb(R * w.I) if kname == "gemm_gate_up_swiglu"
                                                                   else 2 * R * w.H)
        g_flops = mult * R * w.H * w.I
        bound = "hbm" if g_bytes / (hbm_peak * 1e9) >= g_flops / (fp4_peak * 1e12) else "tensor"
        if bound == "hbm":
            achieved, peak, unit = g_bytes / (g_ms * 1e-3) / 1e9, hbm_peak, "GB/s"
        else:
            achieved, peak, unit = g_flops / (g_ms * 1e-3) / 1e12, fp4_peak, "TFLOP/s"
        gemms[kname] = {"kernel": kname, "bound": bound, "achieved": round(achieved, 1), "peak": round(peak, 1),
                        "unit": unit, "frac": round(achieved / peak, 4),
                        "algorithmic": g_bytes if bound == "hbm" else g_flops,
                        "algorithmic_unit": "bytes per launch" if bound == "hbm" else "FLOP per launch",
                        "traffic": recorded_traffic(w.name, kname) if layer.fmt == "nvfp4" else None,
                        "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy)" if bound == "hbm" else
                        f"{peak_kind} bf16 burst (MEASURED_PEAKS.json bf16_tflops) x {FP4_OVER_BF16:g} nominal "
                        "fp4/bf16 ratio"}
    layer_frac = max(alg_bytes / (hbm_peak * 1e9), flops / (fp4_peak * 1e12)) / (ms_step * 1e-3)
    rec = {
        "value": round(tokens_s, 1), "unit": "tokens/s", "ms_per_step": round(ms_step, 4),
        "config": bench_config(w, layer.fmt, layer.k_primary, n_active, world),
        "tflops": round(flops * world / (ms_step * 1e-3) / 1e12, 2),
        "hbm_gbs": round(alg_bytes * world / (ms_step * 1e-3) / 1e9, 1),
        "layer_roofline_frac": round(layer_frac, 4),
        "kernels_ms": {n: round(float(v), 4) for n, v in zip(names, kern_ms)},
        "ms_per_step_with_events": round(ms_step_events, 4),
        "roofline": gemms["gemm_gate_up_swiglu"],
        "roofline_down": gemms["gemm_down"],
        "clocks": clk.summary(),
        "gpu_launches": layer.launches_per_forward * args.steps,
    }
    if e2e is not None:
        rec["e2e"] = e2e
    return rec, layer, inp


def run_ours(args, w):
    from nvfp4_block_scaled_07_gb300 import binding as B
    world, rank, local = dist_setup(args.gpus)
    B.device_check()
    rec, layer, inp = measure_layer(args, w, world, rank)
    res = {
        "metric": METRIC, "value": rec["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "data": "synthetic",
        "dtype": "mxfp4 (e2m1 x ue8m0 scales per 32, fp32 accumulate)" if layer.fmt == "mxfp4" else
                 "nvfp4 (e2m1 x ue4m3 scales, fp32 accumulate)",
        "config": rec["config"],
        **{k: rec[k] for k in ("tflops", "hbm_gbs", "layer_roofline_frac", "kernels_ms", "ms_per_step_with_events",
                               "roofline", "roofline_down", "e2e", "clocks")},
        "prepare": "fused (one launch)" if layer.fused_prepare else "separate (route, quantise, permute)",
        "finalize": "fused into the down GEMM (float32 atomics) + conversion" if layer.fused_finalize else
                    "separate gather-reduce in slot order",
        "gemm_plans": {g: [{"tiles": tile_name(B.gemm_tile_choice(w.E, n, w.T * w.k, t)), "expert_rows": list(r)}
                           for t, r in plan]
                       for g, n, plan in (("gate_up", 2 * w.I, layer.plan()[0]), ("down", w.H, layer.plan()[1]))},
        "autotuned": w.T in layer.plans,
        "gemm_schedule": "dynamic" if layer.g_ws is not None else "static",
        "weights": "tiled" if isinstance(layer.w_gu_packed, B.TiledWeights) else "row-major",
    }
    launches = rec["gpu_launches"]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, args, layer_inputs=(inp["x"], inp["logits"], inp["bias"], layer))
    del layer, inp
    torch.cuda.empty_cache()
    if args.secondary and args.secondary not in ("none", w.name):
        w2 = {**W.WORKLOADS, **W.PROFILE_WORKLOADS}[args.secondary]
        rec2, layer2, inp2 = measure_layer(args, w2, world, rank)
        launches += rec2.pop("gpu_launches")
        res["secondary"] = {"workload": w2.name, "unit": "tokens/s", **rec2}
        del layer2, inp2
        torch.cuda.empty_cache()
    res["gpu_launches"] = launches
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ----------------------------------------------------------------------------
# the CPU oracle on a bounded sample (baseline and reference arm)
# ----------------------------------------------------------------------------
def oracle_quantized_weights(w_gu_dev, w_d_dev, experts, fmt="nvfp4"):
    """Oracle quantisation (NVFP4 or MXFP4) of the weights of `experts` (untimed
    setup; the expert matrices are quantised on a thread pool, numpy releases
    the interpreter lock inside its array loops)."""
    from concurrent.futures import ThreadPoolExecutor
    from oracle import nvfp4_moe_oracle as O

    def one(job):
        name, e, src = job
        a = src[int(e)].float().cpu().numpy()
        if fmt == "mxfp4":
            return (name, int(e)), O.quantize_mxfp4(a) + (None,)
        g = O.global_scale(a)
        return (name, int(e)), O.quantize_nvfp4(a, g) + (g,)

    jobs = [(name, e, src) for e in experts for name, src in (("gu", w_gu_dev), ("d", w_d_dev))]
    with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        return dict(ex.map(one, jobs))


def oracle_route(w, lg, b, k_primary=None):
    """The oracle router the layer uses: top-k, or batch-aware with k_primary < k."""
    from oracle import nvfp4_moe_oracle as O
    if k_primary is None or k_primary == w.k:
        return O.route_topk(lg, b, w.k, w.score, w.renormalize)
    return O.route_batch_aware(lg, b, w.k, k_primary, w.score, w.renormalize)


def oracle_sample(w, x32, lg, b, q, experts, islice=None, fmt="nvfp4", k_primary=None, return_out=False):
    """The oracle layer restricted to the routed rows of `experts`.

    Times separately the batch-wide steps (routing of every token, the global
    scale of x, the permutation) and the per-expert steps (quantising the
    expert's token rows, gate/up GEMM, SwiGLU, requantisation, down GEMM and
    the weighted scatter into the output); of the latter, the quantisation
    of the expert's token rows is also reported on its own.  With islice =
    (a, b) only the intermediate columns [a, b) of each expert are computed:
    gate rows [a, b), up rows [I + a, I + b) and the down GEMM over that K
    range (a partial sum of the expert's output); a and b are multiples of
    64.  fmt "mxfp4" runs the MXFP4 layer; k_primary < k routes batch-aware.
    Returns (batch seconds, expert seconds, of which token-row quantisation
    seconds, rows processed, number of active experts), and the float64 sum
    before its bf16 rounding when return_out."""
    from oracle import nvfp4_moe_oracle as O
    mx = fmt == "mxfp4"
    t0 = time.perf_counter()
    idx, wts = oracle_route(w, lg, b, k_primary)
    s_x = None if mx else O.global_scale(x32)
    counts, offsets, p2f, f2p = O.permute(idx, w.E)
    t1 = time.perf_counter()
    out = np.zeros((w.T, w.H))
    rows = 0
    t_xq = 0.0
    for e in experts:
        e = int(e)
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        tok = p2f[r0:r1] // w.k
        gp, gs, gg = q[("gu", e)]
        dp, ds, dg = q[("d", e)]
        a, c = (0, w.I) if islice is None else islice
        blk = 32 if mx else 16
        if (a, c) != (0, w.I):
            sel = np.r_[a:c, w.I + a:w.I + c]
            gp, gs = gp[sel], gs[sel]
            dp, ds = dp[:, a // 2:c // 2], ds[:, a // blk:c // blk]
        sub = np.array([0, r1 - r0])
        tq = time.perf_counter()
        if mx:
            xq, xs = O.quantize_mxfp4(x32[tok])
            t_xq += time.perf_counter() - tq
            h = O.swiglu(O.grouped_gemm_mx(xq, xs, sub, gp[None], gs[None]), c - a).astype(np.float32)
            hq, hs = O.quantize_mxfp4(h)
            y = O.round_to_bf16(O.grouped_gemm_mx(hq, hs, sub, dp[None], ds[None]))
        else:
            xq, xs = O.quantize_nvfp4(x32[tok], s_x)
            t_xq += time.perf_counter() - tq
            gu = O.grouped_gemm(xq, xs, s_x, sub, gp[None], gs[None], np.array([gg]))
            h = O.swiglu(gu, c - a).astype(np.float32)
            hq, hs = O.quantize_nvfp4(h, np.float32(w.h_scale))
            y = O.round_to_bf16(O.grouped_gemm(hq, hs, np.float32(w.h_scale), sub, dp[None], ds[None],
                                               np.array([dg])))
        np.add.at(out, tok, wts.reshape(-1)[p2f[r0:r1]][:, None] * y)
        rows += r1 - r0
    O.round_to_bf16(out)
    t2 = time.perf_counter()
    res = (t1 - t0, t2 - t1, t_xq, rows, int((counts > 0).sum()))
    return res + (out,) if return_out else res


def cpu_baseline(w, args, layer_inputs):
    """The oracle layer, as it stands, on this host's cores: the batch-wide
    steps plus whole active experts (spread over the expert list) one at a
    time until about CPU_BUDGET_S seconds of oracle work, extrapolated by the
    number of active experts."""
    x, logits, bias, layer = layer_inputs
    counts = layer.perm.counts.cpu().numpy()
    active = np.nonzero(counts)[0]
    order = active[np.linspace(0, len(active) - 1, min(len(active), args.cpu_experts)).astype(int)]
    # weights in bf16 for the sampled experts, regenerated from the same seed
    inp = W.device_inputs(w, seed=args.seed, device=x.device)
    fmt, k0 = layer.fmt, (layer.k_primary if layer.k_primary < w.k else None)
    x32 = x.float().cpu().numpy()
    lg = logits.cpu().numpy()
    b = None if bias is None else bias.cpu().numpy()
    t_batch, t_exp, rows, n, n_active = 0.0, 0.0, 0, 0, len(active)
    chunk = max(1, min(len(order), 4))
    for c0 in range(0, len(order), chunk):
        part = order[c0:c0 + chunk]
        q = oracle_quantized_weights(inp["w_gu"], inp["w_d"], part, fmt)      # untimed setup
        for e in part:
            tb, te, _, r, n_active = oracle_sample(w, x32, lg, b, q, [e], fmt=fmt, k_primary=k0)
            t_batch = tb if n == 0 else min(t_batch, tb)
            t_exp += te
            rows += r
            n += 1
            if t_exp >= CPU_BUDGET_S:
                break
        del q
        if t_exp >= CPU_BUDGET_S:
            break
    del inp
    torch.cuda.empty_cache()
    full = t_batch + t_exp * n_active / n
    return {"value": round(w.T / full, 4), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"batch-wide steps ({t_batch:.2f} s) plus {n} of {n_active} active experts ({rows} routed "
                      f"rows, {t_exp:.1f} s) through the float64 oracle; layer time = batch steps + expert time "
                      f"x {n_active / n:.1f} (an extrapolation); elementwise steps on one thread, float64 matmuls "
                      f"on the BLAS pool"}


def run_reference(args, w):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    torch.cuda.set_device(0)
    inp = W.device_inputs(w, seed=args.seed, device=torch.device("cuda", 0))
    print(json.dumps(reference_steps(args, w, inp, world)), flush=True)


def reference_steps(args, w, inp, world=1):
    """The oracle arm: each step one bounded sample of the workload through
    the oracle (format and routing as the layer's), extrapolated to the
    layer.  inp: the workload's tensors on any device.  Returns the JSON
    record."""
    fmt = args.format
    k0 = args.k_primary if args.k_primary is not None and args.k_primary < w.k else None
    x32 = inp["x"].float().cpu().numpy()
    lg = inp["logits"].cpu().numpy()
    b = None if inp["bias"] is None else inp["bias"].cpu().numpy()
    idx, _ = oracle_route(w, lg, b, k0)
    active = np.unique(idx)
    # a small fixed set of experts, quantised once (untimed) and cycled through the steps
    cycle = active[np.linspace(0, len(active) - 1, min(len(active), 4)).astype(int)]
    q = oracle_quantized_weights(inp["w_gu"], inp["w_d"], cycle, fmt)
    del inp
    torch.cuda.empty_cache()
    times = []
    width = min(w.I, 256)
    nsl = -(-w.I // width)                      # the last slice may be narrower
    for s in range(args.warmup + args.steps):
        j = s % (len(cycle) * nsl)
        sl = ((j % nsl) * width, min(w.I, (j % nsl + 1) * width))
        t_batch, t_exp, t_xq, _, n_active = oracle_sample(w, x32, lg, b, q, [cycle[j // nsl]], islice=sl, fmt=fmt,
                                                          k_primary=k0)
        if s >= args.warmup:
            # one slice of one expert per step, extrapolated to the layer: the
            # expert's token rows are quantised once per expert, the rest of
            # the expert's work once per slice
            times.append(t_batch + n_active * (t_xq + nsl * (t_exp - t_xq)))
    ms = float(np.mean(times)) * 1e3
    val = w.T / (ms * 1e-3)
    return {"metric": METRIC, "impl": "reference", "value": round(val, 4), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(w, fmt, k0, len(active), world),
            "cpu_baseline": {"value": round(val, 4), "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": f"per step: the batch-wide steps (routing, global scale, permutation) "
                                       f"plus one {width}-column slice of the intermediate dimension of one active "
                                       f"expert (of a cycled set of 4) for its routed rows through the float64 "
                                       f"oracle; the layer time is extrapolated: the slice's work x {nsl} slices "
                                       f"and the expert's token-row quantisation once, both x the number of active "
                                       f"experts"},
            "e2e": {"value": round(val, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS) + sorted(W.PROFILE_WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--tile-gate-up", type=int, default=0)
    ap.add_argument("--tile-down", type=int, default=0)
    ap.add_argument("--cpu-experts", type=int, default=14,
                    help="most active experts the cpu_baseline leg samples (it stops earlier once its budget is spent)")
    ap.add_argument("--secondary", default=SECONDARY_WORKLOAD,
                    help="workload timed after the headline one, reported under 'secondary' ('none' for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--k-primary", type=int, default=None,
                    help="batch-aware routing: experts each token keeps by its own scores (default k: plain top-k)")
    ap.add_argument("--format", choices=["nvfp4", "mxfp4"], default="nvfp4",
                    help="operand format of the layer (mxfp4: E8M0 scale per 32 elements, no per-tensor scales)")
    ap.add_argument("--weights", choices=["tiled", "rowmajor"], default="tiled",
                    help="expert weight layout of the grouped GEMMs (tiled: each 128 x 128-byte box contiguous)")
    ap.add_argument("--static-schedule", action="store_true",
                    help="grouped GEMMs on static tile stripes instead of the dynamic tile counter")
    ap.add_argument("--fused-finalize", action="store_true",
                    help="finalize fused into the down GEMM (float32 atomics; the sum order is not fixed)")
    ap.add_argument("--separate-prepare", action="store_true",
                    help="route, quantise and permute as separate calls instead of moe_prepare")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = {**W.WORKLOADS, **W.PROFILE_WORKLOADS}[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
