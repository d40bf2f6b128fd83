#!/usr/bin/env python
"""Throughput of the W4A16 MoE expert layer on GB300.

One step = one pass of the whole layer over one synthetic canvas: routing
(top-k + softmax + per-expert pair lists), the grouped gate_up GEMM with the
gated GELU, the grouped down GEMM and the fixed-order combine, all through the
library's C ABI on device-resident inputs.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload canvas256] [--impl ours|reference]
  python bench.py --sampler [--steps K] [--warmup W]

`--sampler` times the per-step sampler instead (entropy, Gumbel-max token and
acceptance over the fp32 logits of a 256-position canvas with a 262,144-token
vocabulary: 268 MB per step) and prints its own JSON line.  `--block` times the
whole MoE block per layer instead (pre-norm and router projection of x, then
the layer, the residual added in the combine) as one moe_w4a16_block call; the
router logits are then formed on the device, not an input.

Under torchrun every rank runs its own canvas on its own GPU (independent
problems, no collective on the data path): weak scaling; value = tokens of all
ranks / max-over-ranks time.  `--impl reference` times the CPU oracle (the
method's plain fp64 definition) on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE expert-layer tokens/s at 256-token canvas; achieved HBM GB/s vs GB300 peak"
FALLBACK_HBM_GBS = 6800.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "expert_gemm_canvas256.txt")
DOMINANT_SRC = [os.path.join(ROOT, "w4a16_moe_expert_router_gb300", "csrc", n) for n in ("gemm_mma.cu", "gemm_common.cuh")]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--workload", default="canvas256")
    p.add_argument("--reduction", type=int, choices=[0, 1], default=0,
                   help="expert GEMM arithmetic: 0 each weight dequantised, 1 group-factorised")
    p.add_argument("--format", type=int, choices=[0, 1, 2], default=0,
                   help="weight format: 0 asymmetric zero-point, 1 affine bias, 2 symmetric")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--e2e-steps", type=int, default=2000)
    p.add_argument("--graph", action="store_true",
                   help="replay each step from a CUDA graph captured once (per weight copy) instead of launching it")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--sampler", action="store_true", help="time the per-step sampler instead of the layer")
    p.add_argument("--noise", type=int, choices=[0, 1], default=0,
                   help="sampler Gumbel noise: 0 one Gumbel per group of four entries, 1 one per token")
    p.add_argument("--block", action="store_true",
                   help="time the whole MoE block per layer (pre-norm, router projection, routing, experts, "
                        "combine with the residual) as one moe_w4a16_block call; logits are not an input")
    return p.parse_args(argv)


# ------------------------------------------------------------ distributed ----

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    group = None
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        group = dist.group.WORLD
    return rank, world, local, group


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- helpers ----

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def source_hash(paths) -> str:
    """First 16 hex digits of the SHA-256 of the files' bytes, concatenated in order."""
    h = hashlib.sha256()
    for path in ([paths] if isinstance(paths, str) else paths):
        with open(path, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    valid only while the kernel source is unchanged since the capture."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    vals = {}
    with open(PROFILE_TRAFFIC) as fh:
        for ln in fh:
            if ":" in ln:
                k, v = ln.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_source_sha256_16") != source_hash(DOMINANT_SRC):
        return None
    try:
        return float(vals["traffic_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": [], "samples": 0}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- our arm ----

def workload_of(args):
    """The named workload with the requested GEMM arithmetic and weight format."""
    import dataclasses
    from w4a16_moe_expert_router_gb300 import synth
    return dataclasses.replace(synth.WORKLOADS[args.workload], reduction=args.reduction, format=args.format)


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    from w4a16_moe_expert_router_gb300 import binding as B
    from w4a16_moe_expert_router_gb300 import build as libbuild
    from w4a16_moe_expert_router_gb300 import runtime, synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py (--impl ours) needs a CUDA GPU")
    libbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wl = workload_of(args)
    layers = wl.layers
    seed = rank  # every rank denoises its own canvas
    x_bits = synth.make_x(wl, seed)
    logits = [synth.make_logits(wl, seed, layer=l) for l in range(layers)]
    # four copies of every layer's weights rotate between steps, so every step reads cold weights
    # (one layer's weights already exceed L2; a 30-layer stack reads 30 distinct layers per step)
    copies = 4 if layers == 1 else 1
    weights, gammas, touched = [], [], []
    for l in range(layers):
        w = synth.make_weights(wl, 0, layer=l)
        gu, dn = runtime.prepare_host(wl, w)
        for _ in range(copies):
            weights.append(runtime.PreparedWeights(torch.from_numpy(gu).to(dev), torch.from_numpy(dn).to(dev)))
        gammas.append(runtime.to_device_f32(synth.make_gamma(wl, 0, layer=l), dev) if wl.rmsnorm else None)
        del w, gu, dn
    if args.block:  # the block's own router weights and pre-norm weight, per layer
        if wl.rmsnorm:
            raise SystemExit("--block takes a workload without the layer-stack RMSNorm (the block is pre-norm)")
        routers = [runtime.to_device_u16(synth.make_router(wl, 0, layer=l), dev) for l in range(layers)]
        gammas_pre = [runtime.to_device_f32(synth.make_gamma_pre(wl, 0, layer=l), dev) for l in range(layers)]
    # a dedicated stream (a CUDA graph cannot capture the legacy default stream)
    stream = torch.cuda.Stream(dev)
    torch.cuda.set_stream(stream)
    sptr = stream.cuda_stream
    buf = runtime.alloc_buffers(wl, device=dev, stream=stream)
    x = runtime.to_device_x(x_bits, dev)
    lg = [runtime.to_device_f32(a, dev) for a in logits]
    outs = [torch.empty((wl.tokens, wl.hidden), dtype=torch.float16, device=dev) for _ in range(2)]

    L = B.lib()
    import ctypes
    sh = buf.shape
    r = buf.routing.c()
    ws_ptr, ws_n = buf.workspace.data_ptr(), buf.workspace.numel()
    wstructs = [B.Weights(w.gate_up.data_ptr(), w.down.data_ptr()) for w in weights]
    shp, rp = ctypes.byref(sh), ctypes.byref(r)

    def layer_calls(l, src, dst, w_i, evs=None):
        """route, experts (gate_up + down in one launch), combine of layer l; events between the calls if given.
        With --block: the one moe_w4a16_block call of layer l (its events all after the call)."""
        if evs is not None:
            evs[0].record(stream)
        if args.block:
            st = L.moe_w4a16_block(shp, src.data_ptr(), gammas_pre[l].data_ptr(), 1e-6, routers[l].data_ptr(), rp,
                                   ctypes.byref(wstructs[w_i]), dst.data_ptr(), ws_ptr, ws_n, sptr)
            if evs is not None:
                for e in evs[1:]:
                    e.record(stream)
            if st:
                raise RuntimeError(f"library call failed with status {st}")
            return
        st = L.moe_w4a16_route(shp, lg[l].data_ptr(), rp, ws_ptr, ws_n, sptr)
        if evs is not None:
            evs[1].record(stream)
        st |= L.moe_w4a16_experts(shp, src.data_ptr(), rp, ctypes.byref(wstructs[w_i]), ws_ptr, ws_n, sptr)
        if evs is not None:
            evs[2].record(stream)
        g = gammas[l]
        st |= L.moe_w4a16_combine(shp, rp, None if g is None else g.data_ptr(), 1e-6, dst.data_ptr(), ws_ptr,
                                  ws_n, sptr)
        if evs is not None:
            evs[3].record(stream)
        if st:
            raise RuntimeError(f"library call failed with status {st}")

    def step(i, evs=None):
        """One step = the whole layer stack over the canvas."""
        src = x
        for l in range(layers):
            dst = outs[l % 2]
            w_i = l * copies + (i % copies)
            layer_calls(l, src, dst, w_i, evs[l] if evs is not None else None)
            src = dst

    # routing statistics for the algorithmic byte count (per layer: experts touched)
    for l in range(layers):
        if args.block:
            layer_calls(l, x, outs[0], l * copies)
        else:
            B.moe_w4a16_route(sh, lg[l], buf.routing, buf.workspace, stream)
        off = buf.routing.expert_offsets.cpu().numpy()
        touched.append(int(np.count_nonzero(np.diff(off))))
    d, f, g1, g2 = wl.hidden, wl.inter, wl.group_gate_up, wl.group_down
    gu_bytes_e = 2 * f * d // 2 + 2 * f * (d // g1) * 4
    dn_bytes_e = d * f // 2 + d * (f // g2) * 4
    layer_bytes = sum(t * (gu_bytes_e + dn_bytes_e) for t in touched)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    graphs = []
    if args.graph:
        # one graph per weight copy: the whole step (every layer's route, experts, combine)
        for c in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step(c)
            graphs.append(g)
        for i in range(args.warmup):
            graphs[i % copies].replay()
        torch.cuda.synchronize(dev)

    K = args.steps
    KA = min(K, 200)  # eager steps with events between the calls, after the timed region
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(layers)] for _ in range(KA)]
    # one event pair per step (nothing between the calls of a step, so the launches of
    # a step keep their programmatic-dependent-launch overlap)
    sev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize(dev)
        t_start.record(stream)
        for i in range(K):
            sev[i][0].record(stream)
            if args.graph:
                graphs[i % copies].replay()
            else:
                step(i)
            sev[i][1].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    elapsed_ms = t_start.elapsed_time(t_end)
    if B.moe_w4a16_read_error(buf.workspace, stream) != B.OK:
        raise RuntimeError("a device-side wait timed out during the timed region")
    max_ms = max_over_ranks(elapsed_ms, world, dev)
    step_ms = np.array([e[0].elapsed_time(e[1]) for e in sev])
    # the per-call attribution comes from eager steps with events between the calls, run after
    # the timed region (those events break the launches' overlap, so the parts sum to more
    # than a timed step)
    for i in range(KA):
        step(i, evs[i])
    torch.cuda.synchronize(dev)

    # per-call averages (route, experts, combine)
    parts = np.zeros((layers, 3))
    for i in range(KA):
        for l in range(layers):
            e = evs[i][l]
            for j in range(3):
                parts[l, j] += e[j].elapsed_time(e[j + 1])
    parts /= KA
    route_us, experts_us, comb_us = (parts.mean(0) * 1e3).tolist()

    tokens_total = wl.tokens * K * world
    value = tokens_total / (max_ms / 1e3)
    ms_per_step = max_ms / K
    peak, peak_src = measured_peak()
    # the expert launch streams every touched expert's weights of both projections once
    achieved = (layer_bytes / layers) / ((route_us if args.block else experts_us) * 1e-6) / 1e9
    layer_gbs = layer_bytes / (ms_per_step * 1e-3) / 1e9

    # end to end through the public API: every step copies its inputs in from pinned host
    # memory and its output back, inside the timed region.  The copies in and the copies out
    # run on two copy streams, double-buffered, so that step i + 1's inputs arrive and step
    # i - 1's output leaves while step i computes (events order each buffer's reuse).  The host loop makes
    # the C calls directly (library, and the CUDA runtime for the copies and events) with
    # argument structures built once, so that it enqueues a step faster than the GPU runs it.
    rt_lib = ctypes.CDLL("libcudart.so.13")
    vp, sz = ctypes.c_void_p, ctypes.c_size_t
    rt_lib.cudaMemcpyAsync.argtypes = [vp, vp, sz, ctypes.c_int, vp]
    rt_lib.cudaEventRecord.argtypes = [vp, vp]
    rt_lib.cudaStreamWaitEvent.argtypes = [vp, vp, ctypes.c_uint]
    rt_lib.cudaEventCreateWithFlags.argtypes = [ctypes.POINTER(vp), ctypes.c_uint]
    H2D, D2H = 1, 2

    def raw_event():
        e = vp()
        if rt_lib.cudaEventCreateWithFlags(ctypes.byref(e), 2) != 0:  # cudaEventDisableTiming
            raise RuntimeError("cudaEventCreateWithFlags failed")
        return e

    in_stream, out_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    cptr, optr = in_stream.cuda_stream, out_stream.cuda_stream
    x_host = torch.from_numpy(x_bits.view(np.float16)).pin_memory()
    lg_host = [torch.from_numpy(a).pin_memory() for a in logits]
    out_host = [torch.empty((wl.tokens, wl.hidden), dtype=torch.float16).pin_memory() for _ in range(2)]
    x_in = [torch.empty_like(x) for _ in range(2)]
    lg_in = [[torch.empty_like(a) for a in lg] for _ in range(2)]
    out_dev = [torch.empty((wl.tokens, wl.hidden), dtype=torch.float16, device=dev) for _ in range(2)]
    ev_in = [raw_event() for _ in range(2)]    # the slot's inputs are on the device
    ev_done = [raw_event() for _ in range(2)]  # the slot's step has finished computing
    ev_out = [raw_event() for _ in range(2)]   # the slot's output has reached the host
    used = [False, False]
    xb, ob = x_host.numel() * 2, wl.tokens * wl.hidden * 2
    lgb = [a.nbytes for a in logits]
    KE = max(1, min(args.e2e_steps, K))

    def e2e_step(i):
        b = i % 2
        st = 0
        if used[b]:
            st |= rt_lib.cudaStreamWaitEvent(cptr, ev_done[b], 0)  # the step before last has read this slot
        st |= rt_lib.cudaMemcpyAsync(x_in[b].data_ptr(), x_host.data_ptr(), xb, H2D, cptr)
        if not args.block:
            for l in range(layers):
                st |= rt_lib.cudaMemcpyAsync(lg_in[b][l].data_ptr(), lg_host[l].data_ptr(), lgb[l], H2D, cptr)
        st |= rt_lib.cudaEventRecord(ev_in[b], cptr)
        st |= rt_lib.cudaStreamWaitEvent(sptr, ev_in[b], 0)
        if used[b]:
            st |= rt_lib.cudaStreamWaitEvent(sptr, ev_out[b], 0)  # the step before last's output is out
        src = x_in[b].data_ptr()
        for l in range(layers):
            dst = out_dev[b].data_ptr() if l == layers - 1 else outs[l % 2].data_ptr()
            w_i = l * copies + (i % copies)
            if args.block:
                st |= L.moe_w4a16_block(shp, src, gammas_pre[l].data_ptr(), 1e-6, routers[l].data_ptr(), rp,
                                        ctypes.byref(wstructs[w_i]), dst, ws_ptr, ws_n, sptr)
            else:
                g = gammas[l]
                st |= L.moe_w4a16_route(shp, lg_in[b][l].data_ptr(), rp, ws_ptr, ws_n, sptr)
                st |= L.moe_w4a16_forward(shp, src, rp, ctypes.byref(wstructs[w_i]),
                                          None if g is None else g.data_ptr(), 1e-6, dst, ws_ptr, ws_n, sptr)
            src = dst
        st |= rt_lib.cudaEventRecord(ev_done[b], sptr)
        st |= rt_lib.cudaStreamWaitEvent(optr, ev_done[b], 0)
        st |= rt_lib.cudaMemcpyAsync(out_host[b].data_ptr(), out_dev[b].data_ptr(), ob, D2H, optr)
        st |= rt_lib.cudaEventRecord(ev_out[b], optr)
        used[b] = True
        if st:
            raise RuntimeError(f"a call of the end-to-end step failed with status {st}")

    for i in range(min(10, KE)):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(KE):
        e2e_step(i)
    for b in range(2):
        rt_lib.cudaStreamWaitEvent(sptr, ev_out[b], 0)  # the last outputs are on the host
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    rt_lib.cudaEventDestroy.argtypes = [vp]
    for e in ev_in + ev_done + ev_out:
        rt_lib.cudaEventDestroy(e)
    h2d = x_bits.nbytes + (0 if args.block else sum(a.nbytes for a in logits))
    d2h = wl.tokens * wl.hidden * 2

    result = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "ms_per_step_median": float(np.median(step_ms)),
        "ms_per_step_min": float(step_ms.min()),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": wl.name + ("_block" if args.block else ""), "tokens": wl.tokens, "hidden": wl.hidden, "inter": wl.inter,
            "experts": wl.experts, "top_k": wl.top_k, "group_gate_up": wl.group_gate_up,
            "group_down": wl.group_down, "layers": layers, "rmsnorm": wl.rmsnorm,
            "reduction": wl.reduction, "weight_format": wl.format,
            "experts_touched_per_layer": touched,
            "l2": f"inputs larger than L2: {layer_bytes / layers / 1e6:.0f} MB of expert weights per layer "
                  f"vs 129 MB L2" + (f"; {copies} weight copies rotate between steps" if copies > 1 else ""),
            "launch": "CUDA graph replay of the whole step" if args.graph else "eager C-ABI calls",
            "parallelism": f"replicas x{world} (one canvas per GPU)",
        },
        "hbm_gbs": layer_gbs,
        "hbm_frac_of_peak": layer_gbs / peak,
        "kernel_us": {"block": route_us} if args.block else {"route": route_us, "experts": experts_us,
                                                              "combine": comb_us},
        "roofline": {
            "kernel": ("the whole moe_w4a16_block call (pre-norm and router projection, routing, row copy, "
                       "expert GEMMs, combine with the residual): the expert weights' bytes over the call's time")
            if args.block else
                      "expert_gemm_mma_kernel (gate_up + down grouped dequant GEMMs in one persistent launch: "
                      "TMA/bulk-copy ring, in-register dequant, m16n8k16 tensor-core MMAs; its timed segment also "
                      "holds the expert-order row copy launched before it)",
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "peak_source": peak_src,
            # the committed counters are of the default instantiation on canvas256
            "traffic": profiled_traffic() if (wl.name, wl.reduction, wl.format, args.block) == ("canvas256", 0, 0, False)
            else None,
            "algorithmic_bytes_per_launch": layer_bytes / layers,
        },
        "e2e": {"value": wl.tokens * KE * world / (e2e_ms / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": KE,
                "copies": "in and out on two copy streams, double-buffered: a step's copies overlap its neighbours' "
                          "computation; "
                          "the host loop calls the library and the CUDA runtime directly"},
        # (pre-norm + router projection,) top-k, grouping (two launches above 512 tokens), row copy,
        # expert GEMMs, combine
        "gpu_launches": K * layers * ((1 if args.block else 0) + (2 if wl.tokens <= 512 else 3) + 3),
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.block:
        result["cpu_baseline"] = cpu_baseline(wl)
        result["cpu_baseline_1core"] = cpu_baseline(wl, nthreads=1)
    return result


# ------------------------------------------------------------ CPU oracle ----

class OracleCase:
    """Seeded inputs of one layer of the workload, generated once, for the CPU oracle."""

    def __init__(self, wl, layer=0):
        from w4a16_moe_expert_router_gb300 import synth
        self.wl = wl
        self.x = synth.make_x(wl, 0)
        self.lg = synth.make_logits(wl, 0, layer=layer)
        self.w = synth.make_weights(wl, 0, layer=layer)
        self.gamma = synth.make_gamma(wl, 0, layer=layer) if wl.rmsnorm else None

    def time_tokens(self, tokens, nthreads):
        """Seconds the oracle takes for routing + experts + combine of the given tokens."""
        import numpy as np

        import oracle
        wl = self.wl
        sel = np.zeros(wl.tokens, np.uint8)
        sel[np.asarray(list(tokens))] = 1
        t0 = time.perf_counter()
        idx, tw = oracle.route(self.lg, wl.top_k)
        oracle.forward(self.x, idx, tw, self.w, group_gate_up=wl.group_gate_up, group_down=wl.group_down,
                       activation=wl.activation, gamma=self.gamma, eps=1e-6, token_sel=sel, nthreads=nthreads,
                       fmt=wl.format)
        return time.perf_counter() - t0


def cpu_baseline(wl, nthreads=None):
    """The oracle on the host cores: all of them on one full layer of the canvas, or one
    core on a sample of its tokens (scaled to the canvas)."""
    nth = nthreads or os.cpu_count() or 1
    per_step = wl.layers  # one canvas through the whole stack
    # the whole canvas either way: the oracle dequantises each touched expert once per call, so a
    # sample of a few tokens would cost far more per token than the canvas does
    secs = OracleCase(wl).time_tokens(range(wl.tokens), nth)
    what = (f"one full {wl.name} layer ({wl.tokens} tokens: routing, fp64 dequantised expert FFNs, combine), "
            f"{nth} thread" + ("s" if nth > 1 else ""))
    return {"value": wl.tokens / (secs * per_step), "unit": "tokens/s", "cores": nth, "kind": "oracle",
            "sample": what + (f"; scaled by {per_step} layers per step" if per_step > 1 else "")}


def run_reference(args, rank, world):
    """The oracle as it stands on the host cores, the unit of cpu_baseline: each step one
    full layer of the canvas (every token routed, its experts dequantised in fp64, the
    combine), scaled by the layers of a stack; at most one warm-up step and a 120 s budget."""
    if rank != 0:
        return None
    wl = workload_of(args)
    nth = os.cpu_count() or 1
    case = OracleCase(wl)
    for i in range(min(args.warmup, 1)):
        case.time_tokens(range(wl.tokens), nth)
    budget_s, t0, done, spent = 120.0, time.perf_counter(), 0, 0.0
    for i in range(args.steps):
        spent += case.time_tokens(range(wl.tokens), nth) * wl.layers
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    value = done * wl.tokens / spent
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": done,
        "warmup": args.warmup, "ms_per_step": 1e3 * spent / done, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "tokens": wl.tokens, "hidden": wl.hidden, "inter": wl.inter,
                   "experts": wl.experts, "top_k": wl.top_k, "layers": wl.layers},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": nth, "kind": "oracle",
                         "sample": f"one full {wl.name} layer of {wl.tokens} tokens per step (routing, fp64 "
                                   f"dequantised expert FFNs, combine), {nth} threads"
                                   + (f"; scaled by {wl.layers} layers per step" if wl.layers > 1 else "")
                                   + (f"; stopped after {done} of {args.steps} steps at the {budget_s:.0f} s budget"
                                      if done < args.steps else "")},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


SAMPLER_METRIC = "sampler steps/s (256 positions x 262,144 vocabulary fp32 logits); achieved HBM GB/s vs GB300 peak"
SAMPLER_PROFILE = os.path.join(ROOT, "profiles", "sampler_pass_p256_v262144.txt")
SAMPLER_SRC = os.path.join(ROOT, "w4a16_moe_expert_router_gb300", "csrc", "sampler.cu")


def run_sampler(args):
    """K sampler calls on device-resident logits (two 268 MB copies alternate, each
    larger than L2), CUDA events on the launching stream; then the same call end to
    end with the logits copied in from pinned host memory and the outputs read back."""
    import torch
    from w4a16_moe_expert_router_gb300 import binding as B
    from w4a16_moe_expert_router_gb300 import build as libbuild
    libbuild.build()
    P, V, seed = 256, 262144, 1234
    steps, warmup = min(args.steps, 2000), max(3, min(args.warmup, 20))
    host = sampler_logits(P, V)
    dev = [torch.from_numpy(h).cuda() for h in host]
    revealed = torch.zeros(P, dtype=torch.uint8, device="cuda")
    tok = torch.empty(P, dtype=torch.int32, device="cuda")
    ent = torch.empty(P, dtype=torch.float32, device="cuda")
    pm = torch.empty(P, dtype=torch.float32, device="cuda")
    acc = torch.empty(P, dtype=torch.uint8, device="cuda")
    cfg = B.make_sampler(P, V, 1.0, 0, 40.0, 0, seed, args.noise)
    ws = torch.empty(B.moe_w4a16_sampler_workspace_bytes(cfg), dtype=torch.uint8, device="cuda")

    def call(i, lg):
        cfg.step = i
        B.moe_w4a16_sample(cfg, lg, revealed, tok, ent, pm, acc, ws)

    for i in range(warmup):
        call(i, dev[i % 2])
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        e0.record()
        for i in range(steps):
            call(i, dev[i % 2])
        e1.record()
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    # end to end: every step copies its logits in from pinned host memory and its four
    # outputs back, inside the timed region.  The logits go in as four chunks on four copy
    # streams (several copy engines at once) into one of two device buffers, so that step
    # i + 1's logits arrive while step i samples; the outputs leave on a stream of their own
    # from one of two output sets.
    pinned = [torch.from_numpy(h).pin_memory() for h in host]
    NC = 4
    in_streams = [torch.cuda.Stream() for _ in range(NC)]
    out_stream = torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    douts = [[torch.empty(P, dtype=t.dtype, device="cuda") for t in (tok, ent, pm, acc)] for _ in range(2)]
    outs_h = [[torch.empty(P, dtype=t.dtype, pin_memory=True) for t in (tok, ent, pm, acc)] for _ in range(2)]
    ev_in = [[torch.cuda.Event() for _ in range(NC)] for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]
    n_el = P * V
    bounds = [n_el * c // NC for c in range(NC + 1)]

    def e2e_call(i):
        b = i % 2
        src, dst = pinned[i % 2].view(-1), dev[b].view(-1)
        for c in range(NC):
            with torch.cuda.stream(in_streams[c]):
                if used[b]:
                    in_streams[c].wait_event(ev_done[b])  # the step before last has read this buffer
                dst[bounds[c]:bounds[c + 1]].copy_(src[bounds[c]:bounds[c + 1]], non_blocking=True)
                ev_in[b][c].record(in_streams[c])
        for c in range(NC):
            cur.wait_event(ev_in[b][c])
        if used[b]:
            cur.wait_event(ev_out[b])  # the step before last's outputs have left this set
        cfg.step = i
        B.moe_w4a16_sample(cfg, dev[b], revealed, *douts[b], ws)
        ev_done[b].record(cur)
        with torch.cuda.stream(out_stream):
            out_stream.wait_event(ev_done[b])
            for o, d in zip(outs_h[b], douts[b]):
                o.copy_(d, non_blocking=True)
            ev_out[b].record(out_stream)
        used[b] = True

    e2e_steps = max(3, min(50, steps))
    for i in range(2):
        e2e_call(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(cur)
    for i in range(e2e_steps):
        e2e_call(i)
    for b in range(2):
        cur.wait_event(ev_out[b])
    t1.record(cur)
    torch.cuda.synchronize()
    e2e_ms = t0.elapsed_time(t1) / e2e_steps
    bytes_step = P * V * 4
    peak, peak_src = measured_peak()
    achieved = bytes_step / (ms * 1e-3) / 1e9
    traffic = None
    if os.path.exists(SAMPLER_PROFILE):
        vals = dict(ln.split(":", 1) for ln in open(SAMPLER_PROFILE) if ":" in ln)
        vals = {k.strip(): v.strip() for k, v in vals.items()}
        if vals.get("kernel_source_sha256_16") == source_hash(SAMPLER_SRC) and vals.get("noise") == str(args.noise):
            try:
                traffic = float(vals["traffic_bytes_per_launch_full_size"])
            except (KeyError, ValueError):
                traffic = None
    res = {
        "metric": SAMPLER_METRIC, "value": 1e3 / ms, "unit": "steps/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": "sampler_p256_v262144", "positions": P, "vocab": V, "logits": "3 * N(0, 1) fp32",
                   "rule": "entropy bound 40", "noise": NOISE_NAMES[args.noise],
                   "l2": "inputs larger than L2: 268 MB of logits per step vs 129 MB L2; two copies alternate"},
        "roofline": {"kernel": "sample_pass_kernel + sample_final_kernel (the whole call: one streaming pass over "
                               "the logits, then one CTA merging the partials and deciding the acceptance)",
                     "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_src, "traffic": traffic, "algorithmic_bytes_per_launch": bytes_step},
        "e2e": {"value": 1e3 / e2e_ms, "unit": "steps/s", "h2d_bytes_per_step": bytes_step,
                "d2h_bytes_per_step": P * (4 + 4 + 4 + 1), "steps": e2e_steps,
                "copies": "logits in as four chunks on four copy streams, double-buffered; outputs out on a "
                          "stream of their own"},
        "gpu_launches": 2 * steps,
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        nth = os.cpu_count() or 1
        sample_p = 32
        t = time.perf_counter()
        oracle.sample(host[0][:sample_p], 1.0, seed, 0, nthreads=nth, noise=args.noise)
        secs = time.perf_counter() - t
        keys = f"Gumbel keys of all {V // 4} groups" if args.noise == 0 else f"Gumbel keys of all {V} tokens"
        res["cpu_baseline"] = {"value": 1.0 / (secs * P / sample_p), "unit": "steps/s", "cores": nth,
                               "kind": "oracle", "sample": f"{sample_p} of the {P} positions (fp64 entropy, "
                                                           f"{keys}), {nth} threads, scaled to a full step"}
    return res


NOISE_NAMES = {0: "one Gumbel per group of four entries", 1: "one Gumbel per token"}


def sampler_logits(P, V, copies=2):
    """The sampler workload's fp32 logits: 3 N(0, 1), one array per alternating copy."""
    import numpy as np
    rng = np.random.default_rng(0)
    return [(rng.standard_normal((P, V), dtype=np.float32) * 3.0) for _ in range(copies)]


def run_sampler_reference(args):
    """The sampler oracle as it stands on the host cores: each step a bounded sample of
    the workload's positions (fp64 entropy and the Gumbel keys of every token),
    scaled to steps/s of the full 256-position step."""
    import oracle
    P, V, seed = 256, 262144, 1234
    nth = os.cpu_count() or 1
    lg = sampler_logits(P, V, copies=1)[0]
    sample_p = max(1, min(P, nth * 2))
    for i in range(min(args.warmup, 1)):
        oracle.sample(lg[:sample_p], 1.0, seed, i, nthreads=nth, noise=args.noise)
    budget_s, t0, done, spent = 120.0, time.perf_counter(), 0, 0.0
    for i in range(args.steps):
        t = time.perf_counter()
        oracle.sample(lg[(i * sample_p) % P:][:sample_p], 1.0, seed, i, nthreads=nth, noise=args.noise)
        spent += (time.perf_counter() - t) * P / sample_p
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    value = done / spent
    return {
        "impl": "reference", "metric": SAMPLER_METRIC, "value": value, "unit": "steps/s", "n_gpus": 1,
        "steps": done, "warmup": args.warmup, "ms_per_step": 1e3 * spent / done, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "sampler_p256_v262144", "positions": P, "vocab": V, "logits": "3 * N(0, 1) fp32",
                   "rule": "entropy bound 40", "noise": NOISE_NAMES[args.noise]},
        "cpu_baseline": {"value": value, "unit": "steps/s", "cores": nth, "kind": "oracle",
                         "sample": f"{sample_p} of the {P} positions per step, {nth} threads, scaled to a full step"},
        "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.sampler:
        if args.impl == "reference":
            if int(os.environ.get("RANK", "0")) == 0:
                print(json.dumps(run_sampler_reference(args)), flush=True)
            return
        print(json.dumps(run_sampler(args)), flush=True)
        return
    if args.impl == "reference":
        # host-only: rank 0 times the oracle, the other ranks exit without work
        rank = int(os.environ.get("RANK", "0"))
        res = run_reference(args, rank, int(os.environ.get("WORLD_SIZE", "1")))
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    rank, world, local, _ = dist_setup()
    res = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
