#!/usr/bin/env python
"""Throughput of the routed NVFP4 MoE expert block on GB300.

One step = the whole hot path over one batch: routing metadata, NVFP4 input
quantization into permuted order, GEMM1 with the fused SwiGLU + requant
epilogue, GEMM2, and the post-expert finalize -- four kernel launches
through the C ABI at decode sizes (routing; the quantizer; both GEMMs in one
persistent launch; the finalize), up to seven at prefill, inputs resident in
HBM. The default workload is the b = 8 decode batch (T = 8, H = 5120,
I = 2048, E = 128, top-8, uniform routing).

Timing: W untimed warm-up steps, then exactly K steps between CUDA events on
the launching stream, bracketed by a barrier and a device synchronize; the
layer's prepared weights rotate over several copies whose total exceeds L2,
so no step reads the previous step's weights from L2. The steps are replayed
from CUDA graphs that each hold one step per weight copy in a row, as
consecutive layers' blocks sit in a captured forward (--no-chain: one graph
per step). For the roofline, the
same steps run once more with the dominant kernel -- the one-launch GEMMs at
decode, GEMM1 at prefill -- bracketed by its own events. `e2e` repeats the
measurement through the public layer call with host (pinned) inputs and
outputs, the copies inside the timed region.

Multi-GPU: replicas only -- each rank runs its own copy of the layer on its
own batch; the value is all ranks' tokens over the slowest rank's time.

`--impl reference` times the CPU oracle (numpy) on a bounded sample of the
same workload instead.
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

METRIC = "MoE-layer tokens/s at 1 GB300 and % of HBM (decode) / FP4 tensor (prefill) roofline"
FALLBACK_HBM_GBS = 6800.0


FALLBACK_BF16_TFLOPS = 1900.0
FP4_PER_BF16 = 13.5 / 2.25  # nominal dense fp4 / bf16 tensor rate

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# the roofline kernel, from one ncu capture of it on this workload's batch,
# and the SHA-256 of the kernel sources it was taken on (gemm.cu,
# gemm_pair.cu, common.cuh, layout.cuh in that order): once those change,
# traffic is null.
NCU_TRAFFIC = {
    "decode_b8": {"kernel": "grouped_gemm_kernel<3, 32>", "bytes": 945_302_272 + 5_205_760,
                  "sources": "8d1187bbfbdb9ebbff0bb9ff741af60e593d16feae5b5d7864421a978982a952"},
    "prefill_t8192_zipf": {"kernel": "gemm1_pair_kernel", "bytes": 1_722_032_896 + 84_068_352,
                           "sources": "8d1187bbfbdb9ebbff0bb9ff741af60e593d16feae5b5d7864421a978982a952"},
}


def _traffic(workload: str, kernel: str):
    """Captured DRAM bytes per launch of `kernel`, or None when there is no
    capture for it or its sources have changed since."""
    import hashlib

    t = NCU_TRAFFIC.get(workload)
    if t is None or not kernel.startswith(t["kernel"]):
        return None
    h = hashlib.sha256()
    for f in ("gemm.cu", "gemm_pair.cu", "common.cuh", "layout.cuh"):
        with open(os.path.join(ROOT, "nvfp4_mixture_experts_route_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return t["bytes"] if h.hexdigest() == t["sources"] else None


def _peaks() -> dict:
    """HBM GB/s and bf16 TFLOP/s (burst, sustained) with their provenance."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            m = json.load(f)
        return {"hbm": float(m["hbm_gbs"]), "bf16": float(m["bf16_tflops"]),
                "bf16_sust": float(m.get("bf16_tflops_sustained", m["bf16_tflops"])), "kind": "measured"}
    except Exception:
        return {"hbm": FALLBACK_HBM_GBS, "bf16": FALLBACK_BF16_TFLOPS, "bf16_sust": 1700.0, "kind": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self) -> dict:
        rows = []
        try:
            with open(self.file.name) as f:
                for ln in f:
                    parts = [p.strip() for p in ln.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.file.name)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def _dist():
    """(world, rank, local rank) from the launcher's environment; for N > 1
    a process group over NCCL (one rank per GPU), or gloo where no GPU is
    visible (the CPU tests of this path)."""
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def _max_over_ranks(world, value: float) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def cpu_oracle_sample(w, raw, batch, a1, a2, tokens: int) -> dict:
    """Time the CPU oracle on the first `tokens` tokens of the batch."""
    from oracle import layer as olayer

    t0 = time.perf_counter()
    olayer.moe_layer(batch["x"][:tokens], batch["topk_ids"][:tokens], batch["topk_weights"][:tokens], raw, a1, a2,
                     raw["gamma"], 1e-6, w.tile_m)
    dt = time.perf_counter() - t0
    return {"value": tokens / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{tokens} of {w.T} tokens of {w.name} ({tokens * w.K} routes), exact fp64/int oracle, "
                      f"numpy BLAS on the host's default thread count, {dt:.2f} s"}


def run_reference(args, w) -> None:
    """The CPU oracle as it stands, one route of the workload per step (the
    GEMM1 + SwiGLU + requant + GEMM2 of that route on its expert, plus its
    share of the finalize), i.e. 1/K token per step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np

    from nvfp4_mixture_experts_route_gb300 import inputs
    from oracle import layer as olayer

    raw = inputs.make_layer(w)
    batch = inputs.make_batch(w)
    a1, a2 = inputs.global_scales(w)
    e2p = np.arange(w.T * w.K, dtype=np.int64).reshape(w.T, w.K)

    def one_route(j: int) -> None:
        t, k = divmod(j % (w.T * w.K), w.K)
        ids = np.full((1, w.K), -1, dtype=np.int32)
        ids[0, k] = batch["topk_ids"][t, k]
        er = olayer.expert_rows(batch["x"][t:t + 1], ids, raw, a1, a2)
        olayer.finalize(er["rows_bf16"], np.where(ids >= 0, e2p[:1], -1), batch["topk_weights"][t:t + 1],
                        raw["gamma"], 1e-6)

    for j in range(args.warmup):
        one_route(j)
    t0 = time.perf_counter()
    for j in range(args.steps):
        one_route(args.warmup + j)
    dt = time.perf_counter() - t0
    value = (args.steps / w.K) / dt
    sample = f"one route (1/{w.K} token) of {w.name} per step, exact oracle, numpy BLAS default threads"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config(w),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(w) -> dict:
    return {"workload": w.name, "T": w.T, "H": w.H, "I": w.I, "E": w.E, "top_k": w.K, "routing": w.routing,
            "tile_m": w.tile_m, "parallelism": "replicas"}


def measure_fp4_peak(B, torch, stream) -> dict:
    """Dense NVFP4 tensor-core rate of this GPU, measured live with the
    library's own probe (moe_fp4_mma_rate: back-to-back tcgen05 kind::mxf4nvf4
    MMAs of 128 x 256 x 64 on shared-memory operands, one CTA per SM, 16 MMAs
    per commit), the best of three launches of about 0.2 s: the burst rate a
    kernel timed on its own between events can reach."""
    status = torch.zeros(1, dtype=torch.int32, device=stream.device)
    B.fp4_mma_rate(256, 0, 16, 1, 64, status=status, stream=stream)
    best = 0.0
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        flops = B.fp4_mma_rate(256, 0, 16, 1, 2000, status=status, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        best = max(best, flops / (e0.elapsed_time(e1) * 1e-3) / 1e12)
    if int(status.item()) != 0:
        raise RuntimeError("fp4 rate probe: device status " + B.STATUS_NAMES.get(int(status.item()), "?"))
    return {"tflops": best, "how": "moe_fp4_mma_rate(n=256, sf_copies=0, mmas_per_commit=16, 1 CTA/SM), "
                                   "best of 3 launches of ~0.2 s, measured in this run"}


class Layer:
    """One prepared layer on this GPU plus rotating copies of its prepared
    weights (together larger than L2), shared by every workload of a run."""

    def __init__(self, args, w, dev):
        from nvfp4_mixture_experts_route_gb300 import binding as B
        from nvfp4_mixture_experts_route_gb300 import inputs
        from nvfp4_mixture_experts_route_gb300.layer import NvFp4MoE

        self.raw = inputs.make_layer(w)
        self.a1, self.a2 = inputs.global_scales(w)
        self.moe = NvFp4MoE(self.raw, self.a1, self.a2, self.raw["gamma"], tile_m=w.tile_m, device=dev)
        self.copies = [self.moe.weights]
        self.keep = [self.moe.prepared]
        self.layer_bytes = sum(t.numel() for t in self.moe.prepared.values())
        for _ in range(max(1, args.copies) - 1):
            p = {k: v.clone() for k, v in self.moe.prepared.items()}
            self.keep.append(p)
            self.copies.append(B.weights_struct(p, self.moe.g1_alphas, self.moe.g1_scale_c, self.moe.g2_alphas))


def measure_workload(args, w, layer: Layer, world, rank, dev, fp4_peak) -> dict:
    """Time one workload's step (graph-replayed, K steps between events) and
    its dominant kernel, and the end-to-end serving call; returns the fields
    of its bench line."""
    import numpy as np
    import torch

    from nvfp4_mixture_experts_route_gb300 import binding as B
    from nvfp4_mixture_experts_route_gb300 import inputs

    batch = inputs.make_batch(w, seed=rank)
    T, K, E, H, I, tile = w.T, w.K, w.E, w.H, w.I, w.tile_m
    moe, copies = layer.moe, layer.copies
    moe.tile_m = tile

    x = torch.from_numpy(batch["x"].view(np.int16)).view(torch.bfloat16).to(dev)
    ids = torch.from_numpy(batch["topk_ids"]).to(dev)
    tw = torch.from_numpy(batch["topk_weights"]).to(dev)
    bufs = moe.buffers(T, K)
    route, ws, rows, out, status = bufs["route"], bufs["ws"], bufs["rows"], bufs["out"], bufs["status"]
    status.zero_()
    stream = torch.cuda.current_stream(dev)

    fused = B.experts_kernels(tile) == 2
    # the whole block in one call at decode sizes (routing, the quantizer,
    # both GEMMs in one launch with the norm's sums of squares in GEMM2's
    # epilogue, then the finalize from them: 4 kernels)
    block = fused

    def step(i, ev=None, split=True):
        wts = copies[i % len(copies)]
        if ev is None and block:
            B.moe_block(wts, ids, tw, route, x=x, a1_gscale=moe.a1_gscale, a2_gscale=moe.a2_gscale,
                        gamma=moe.gamma, eps=moe.eps, weight_before_norm=True, H=H, I=I, E=E, gemm2_rows=rows,
                        row_sumsq=bufs["row_sumsq"], out=out, ws=ws, status=status)
            return
        if ev is None:
            # Routing and the expert body as one call (for few routes the
            # routing runs inside the input quantizer); the GEMMs start as
            # programmatic dependents of the kernel before them.
            B.nvfp4_experts_routed(wts, ids, route, x=x, a1_gscale=moe.a1_gscale, a2_gscale=moe.a2_gscale,
                                   H=H, I=I, E=E, gemm2_rows=rows, ws=ws, status=status)
        else:
            B.route_permute(ids, E, tile, route=route, status=status)
            # The same kernels through the split entry points (plain launches),
            # with events between them for the per-kernel durations.
            B.experts_quantize(route, ws, x=x, a1_gscale=moe.a1_gscale, T=T, H=H, I=I, E=E, K=K,
                               status=status)
            ev[0].record(stream)
            if split:
                B.experts_gemm1(wts, route, ws, a2_gscale=moe.a2_gscale, T=T, H=H, I=I, E=E, K=K,
                                status=status)
                ev[1].record(stream)
                B.experts_gemm2(wts, route, ws, rows, T=T, H=H, I=I, E=E, K=K, status=status)
            else:
                B.experts_gemms(wts, route, ws, rows, a2_gscale=moe.a2_gscale, T=T, H=H, I=I, E=E, K=K,
                                status=status)
                ev[1].record(stream)
            ev[2].record(stream)
            ev[3].record(stream)
        B.post_expert_finalize(rows, route.expanded_to_permuted, tw, moe.gamma, moe.eps, True, out=out,
                               status=status)
        if ev is not None:
            ev[4].record(stream)

    # routing + expert body (routing fused into the quantizer for few
    # routes, else 1 or 3 routing kernels, the quantizer and one or two GEMM
    # launches), then the finalize
    launches_per_step = B.moe_block_kernels(T, K, E, tile) if block else B.routed_experts_kernels(T, K, E, tile) + 1
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES.get(int(status.item()))} during warm-up")

    # CUDA graphs of the step's launches (the ABI calls allocate nothing and
    # never synchronise, so they capture as is): one graph holding len(copies)
    # consecutive steps, one per weight copy, as consecutive layers' blocks
    # sit in a model's captured forward (each step's first kernel is a
    # programmatic dependent of the step before, whose outputs it waits for
    # before touching memory); and one graph per copy holding a single step,
    # for a step count that is not a multiple of len(copies).
    graphs, chain = [], None
    if args.graph:
        for c in range(len(copies)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(c)
            graphs.append(g)
        if getattr(args, "chain", False) and len(copies) > 1:
            chain = torch.cuda.CUDAGraph()
            with torch.cuda.graph(chain):
                for c in range(len(copies)):
                    step(c)
        for i in range(args.warmup):
            graphs[i % len(graphs)].replay()
        if chain is not None:
            chain.replay()
        torch.cuda.synchronize()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index or 0) as clocks:
        start.record(stream)
        i = 0
        if chain is not None:
            while i + len(copies) <= args.steps:
                chain.replay()
                i += len(copies)
        while i < args.steps:
            if graphs:
                graphs[i % len(graphs)].replay()
            else:
                step(i)
            i += 1
        end.record(stream)
        torch.cuda.synchronize()
    total_ms = _max_over_ranks(world, start.elapsed_time(end))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES.get(int(status.item()))} in the timed region")
    del graphs, chain

    # The same steps launched one by one, GEMM launches between events on the
    # launching stream: the per-kernel durations of the roofline.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    for i in range(args.steps):
        step(i, evs[i])
    torch.cuda.synchronize()
    gemm1_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    gemm2_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    finalize_ms = statistics.mean(e[3].elapsed_time(e[4]) for e in evs)
    fused_ms = None
    if fused:
        # the one-launch GEMMs the timed step runs (the launch's time includes
        # the 4-byte-per-route-tile counter memset of the standalone entry point)
        for i in range(args.steps):
            step(i, evs[i], split=False)
        torch.cuda.synchronize()
        fused_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)

    # e2e: the public pipelined serving call from pinned host memory,
    # NvFp4MoE.submit_host on alternating slots (inputs x, topk_ids and
    # topk_weights laid out by input_layout, output in pinned host memory):
    # per step one copy in, the step's graph (routing, expert body, finalize)
    # and one copy out, on three streams ordered by events, so a step's copies
    # overlap its neighbours' kernels; every step's transfers are inside the
    # timed region. (Measured against the zero-copy NvFp4MoE.replay_host,
    # whose kernels read and write the pinned buffers themselves: equal at
    # b=8, 2 % slower at b=64, far slower at prefill sizes, where it copies.)
    # One weight copy: a step streams the touched experts' weights (far
    # larger than L2) from HBM anyway. --no-graph times the eager public call
    # (NvFp4MoE.forward) with two copies around it.
    offs, nbytes = moe.input_layout(T, K)
    moe.weights = copies[0]
    hb = moe.host_buffers(T, K)
    in_h, out_h = hb["host_inputs"], hb["host_out"]
    in_h[offs["x"]:offs["x"] + T * H * 2].copy_(torch.from_numpy(batch["x"].view(np.uint8).reshape(-1)))
    in_h[offs["topk_ids"]:offs["topk_ids"] + T * K * 4].copy_(
        torch.from_numpy(batch["topk_ids"].view(np.uint8).reshape(-1)))
    in_h[offs["topk_weights"]:offs["topk_weights"] + T * K * 4].copy_(
        torch.from_numpy(batch["topk_weights"].view(np.uint8).reshape(-1)))
    gb = moe.graph_buffers(T, K)
    pipelined = args.graph
    if pipelined:
        for slot in moe.host_pipeline(T, K)["slots"]:
            slot["host_inputs"].copy_(in_h)

    def e2e_step(i):
        if pipelined:
            moe.submit_host(T, K, i % 2)
        else:
            gb["inputs"].copy_(in_h, non_blocking=True)
            out_h.copy_(moe.forward(gb["x"], gb["topk_ids"], gb["topk_weights"])[0], non_blocking=True)

    if pipelined:
        moe.pipeline_begin(T, K)
    for i in range(args.warmup):
        e2e_step(i)
    if pipelined:
        moe.pipeline_join(T, K)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    if pipelined:
        moe.pipeline_begin(T, K)
    for i in range(args.steps):
        e2e_step(i)
    if pipelined:
        moe.pipeline_join(T, K)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(world, e0.elapsed_time(e1))
    moe.weights = copies[0]

    touched = np.unique(batch["topk_ids"][batch["topk_ids"] >= 0])
    n_touch = len(touched)
    w13_bytes = 2 * I * (H // 2) + 2 * I * (H // 16)
    w2_bytes = H * (I // 2) + H * (I // 16)
    pk = _peaks()
    peak, peak_kind = pk["hbm"], pk["kind"]
    gemm1_gbs = n_touch * w13_bytes / (gemm1_ms * 1e-3) / 1e9
    fused_gbs = n_touch * (w13_bytes + w2_bytes) / (fused_ms * 1e-3) / 1e9 if fused else None
    live_routes = int(np.sum(batch["topk_ids"] >= 0))
    gemm1_flops = 2.0 * live_routes * (2 * I) * H
    gemm2_flops = 2.0 * live_routes * H * I
    tensor_bound = live_routes >= 8 * w.E * 8  # many routes per expert: the MMA, not HBM, bounds
    tokens_total = T * args.steps * world
    step_ms = total_ms / args.steps
    weight_bytes = n_touch * (w13_bytes + w2_bytes)
    if fused and not tensor_bound:
        roof = {"bound": "hbm",
                "kernel": f"grouped_gemm_kernel<3, {tile}> (GEMM1 + SwiGLU + requant + GEMM2, one launch)",
                "achieved": fused_gbs, "peak": peak, "unit": "GB/s", "frac": fused_gbs / peak,
                "peak_kind": f"{peak_kind} copy bandwidth",
                "traffic": _traffic(w.name, f"grouped_gemm_kernel<3, {tile}>"),
                "algorithmic_bytes": weight_bytes, "launch_ms": fused_ms}
    elif not tensor_bound:
        roof = {"bound": "hbm", "kernel": f"grouped_gemm_kernel<1, {tile}> (GEMM1 + SwiGLU + requant)",
                "achieved": gemm1_gbs, "peak": peak, "unit": "GB/s", "frac": gemm1_gbs / peak,
                "peak_kind": f"{peak_kind} copy bandwidth", "traffic": None,
                "algorithmic_bytes": n_touch * w13_bytes, "launch_ms": gemm1_ms}
    else:
        ach = gemm1_flops / (gemm1_ms * 1e-3) / 1e12
        # 128-row tiles with H and 2I multiples of 256 run GEMM1 in the pair form
        pair = tile == 128 and H % 256 == 0 and (2 * I) % 256 == 0
        g1_kernel = "gemm1_pair_kernel" if pair else f"grouped_gemm_kernel<1, {tile}>"
        roof = {"bound": "tensor", "kernel": g1_kernel + (" (GEMM1 + SwiGLU + requant, tcgen05 cta_group::2 over "
                                                          "two-CTA clusters)" if pair else
                                                          " (GEMM1 + SwiGLU + requant)"),
                "achieved": ach, "peak": fp4_peak["tflops"], "unit": "TFLOP/s", "frac": ach / fp4_peak["tflops"],
                "peak_kind": "measured dense NVFP4 (burst): " + fp4_peak["how"],
                "frac_of_bf16x6": ach / (pk["bf16"] * FP4_PER_BF16),
                "traffic": _traffic(w.name, g1_kernel),
                "algorithmic_flops": gemm1_flops, "launch_ms": gemm1_ms,
                "gemm2": {"achieved": gemm2_flops / (gemm2_ms * 1e-3) / 1e12,
                          "frac": gemm2_flops / (gemm2_ms * 1e-3) / 1e12 / fp4_peak["tflops"],
                          "launch_ms": gemm2_ms}}
    res = {
        "value": tokens_total / (total_ms * 1e-3), "ms_per_step": step_ms,
        "config": {**_config(w), "l2": f"{len(copies)} rotating prepared weight copies "
                                        f"({len(copies) * layer.layer_bytes / 1e9:.2f} GB > L2)",
                   "launch": ((f"CUDA graphs of {len(copies)} consecutive steps ({launches_per_step} kernels "
                               f"per step, chained by programmatic dependent launch)"
                               if getattr(args, "chain", False) and len(copies) > 1
                               else f"CUDA graph per step ({launches_per_step} kernels)") if args.graph
                              else f"eager ({launches_per_step} kernels per step)")},
        "roofline": roof,
        "step_roofline": {"bytes": weight_bytes, "touched_experts": int(n_touch),
                          "achieved_gbs": weight_bytes / (step_ms * 1e-3) / 1e9,
                          "frac_of_measured": weight_bytes / (step_ms * 1e-3) / 1e9 / peak,
                          "frac_of_8tbs": weight_bytes / (step_ms * 1e-3) / 8e12,
                          "gemm1_ms": gemm1_ms, "gemm2_ms": gemm2_ms, "fused_gemms_ms": fused_ms,
                          "finalize_ms": finalize_ms},
        "clocks": clocks.summary(),
        "e2e": {"value": tokens_total / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": in_h.numel(),
                "d2h_bytes_per_step": out_h.numel() * 2,
                "transfer": ("pipelined: per step one copy in and one copy out, on their own streams beside "
                             "the step's graph, two slots" if pipelined else "one copy in, one copy out")},
        "gpu_launches": launches_per_step * args.steps,
    }
    if tensor_bound:
        # the step's HBM bytes as the method moves them: the layer's weights
        # and scales, the bf16 GEMM2 rows written and read back, the
        # intermediate written and read, x and out, the quantized activations
        P, _ = B.route_sizes(T, K, E, tile)
        hbm = (E * (w13_bytes + w2_bytes) + 2 * live_routes * H * 2 + 2 * live_routes * (I // 2 + I // 16)
               + 2 * T * H * 2 + 2 * live_routes * (H // 2 + H // 16))
        res["step_roofline"].update(
            {"bytes": hbm, "achieved_gbs": hbm / (step_ms * 1e-3) / 1e9,
             "frac_of_measured": hbm / (step_ms * 1e-3) / 1e9 / peak, "frac_of_8tbs": hbm / (step_ms * 1e-3) / 8e12,
             "step_tflops": (gemm1_flops + gemm2_flops) / (step_ms * 1e-3) / 1e12,
             "step_frac_of_fp4": (gemm1_flops + gemm2_flops) / (step_ms * 1e-3) / 1e12 / fp4_peak["tflops"]})
    del batch
    return res


def run_ours(args, w) -> None:
    import torch

    from nvfp4_mixture_experts_route_gb300 import binding as B
    from nvfp4_mixture_experts_route_gb300 import inputs

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.load()
    stream = torch.cuda.current_stream(dev)
    fp4_peak = measure_fp4_peak(B, torch, stream)

    layer = Layer(args, w, dev)
    head = measure_workload(args, w, layer, world, rank, dev, fp4_peak)
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e2m1xue4m3 (fp32 accumulate)", "data": "synthetic",
        **{k: head[k] for k in ("config", "roofline", "step_roofline", "clocks", "e2e", "gpu_launches")},
        "fp4_peak": fp4_peak,
    }
    # The other configurations of the same layer (the b = 64 Zipf decode
    # batch and the 8192-token prefill), each timed the same way on the same
    # prepared weights; each reports its own timed region's launches.
    extra = [n for n in args.also.split(",") if n] if args.also is not None else []
    if extra:
        line["workloads"] = {}
        for name in extra:
            wx = inputs.WORKLOADS[name]
            if wx.layer_key != w.layer_key:
                continue
            line["workloads"][name] = measure_workload(args, wx, layer, world, rank, dev, fp4_peak)
    if rank != 0:
        return
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_oracle_sample(w, layer.raw, inputs.make_batch(w, seed=rank), layer.a1, layer.a2,
                                                 tokens=args.cpu_tokens)
    print(json.dumps(line), flush=True)


DENSE_METRIC = "pooler projection tokens/s at 1 GB300 and % of HBM (few tokens) / bf16 tensor (many) roofline"


def run_dense(args, d) -> None:
    """The pooler / unpooler projection alone (moe_dense_bf16), weights
    rotated over copies that together exceed L2."""
    import numpy as np
    import torch

    from nvfp4_mixture_experts_route_gb300 import binding as B
    from nvfp4_mixture_experts_route_gb300 import inputs

    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B.load()
    data = inputs.make_dense(d, seed=rank)
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)  # noqa: E731
    x = bf(data["x"])
    w0 = bf(data["w"])
    w_bytes = w0.numel() * 2
    n_copies = max(args.copies, int(np.ceil(3 * 129e6 / w_bytes)))
    ws_ = [w0] + [w0.clone() for _ in range(n_copies - 1)]
    y = torch.empty((d.T, d.Dout), dtype=torch.bfloat16, device=dev)
    need = B.dense_bf16_workspace_size(d.T, d.Din, d.Dout)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    launches = 1  # one kernel (plus, with a workspace, a small counter memset)

    def step(i):
        B.dense_bf16(x, ws_[i % len(ws_)], out=y, ws=ws, status=status)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    graphs = []
    if args.graph:
        for c in range(len(ws_)):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(c)
            graphs.append(g)
        for i in range(args.warmup):
            graphs[i % len(graphs)].replay()
        torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        start.record(stream)
        for i in range(args.steps):
            if graphs:
                graphs[i % len(graphs)].replay()
            else:
                step(i)
        end.record(stream)
        torch.cuda.synchronize()
    total_ms = _max_over_ranks(world, start.elapsed_time(end))
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES.get(int(status.item()))} in the timed region")

    # e2e: pinned host x in, y out, copies timed
    x_h = torch.from_numpy(data["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    y_h = torch.empty((d.T, d.Dout), dtype=torch.bfloat16).pin_memory()
    x_d = torch.empty_like(x)

    def e2e_step(i):
        x_d.copy_(x_h, non_blocking=True)
        B.dense_bf16(x_d, ws_[i % len(ws_)], out=y, ws=ws, status=status)
        y_h.copy_(y, non_blocking=True)

    for i in range(args.warmup):
        e2e_step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    _barrier(world)
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(args.steps):
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = _max_over_ranks(world, e0.elapsed_time(e1))
    if rank != 0:
        return
    step_ms = total_ms / args.steps
    tokens_total = d.T * args.steps * world
    pk = _peaks()
    alg_bytes = w_bytes + d.T * (d.Din + d.Dout) * 2
    flops = 2.0 * d.T * d.Din * d.Dout
    tensor_bound = d.T >= 256
    kern = "dense_bf16_kernel" + (" (stream-K split, in-kernel ordered fix-up)" if need else "")
    if tensor_bound:
        ach = flops / (step_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "kernel": kern, "achieved": ach, "peak": pk["bf16"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16"], "peak_kind": f"{pk['kind']} burst bf16", "traffic": None,
                "algorithmic_flops": flops, "launch_ms": step_ms}
    else:
        ach = alg_bytes / (step_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": kern, "achieved": ach, "peak": pk["hbm"], "unit": "GB/s",
                "frac": ach / pk["hbm"], "peak_kind": f"{pk['kind']} copy bandwidth", "traffic": None,
                "algorithmic_bytes": alg_bytes, "launch_ms": step_ms}
    line = {
        "metric": DENSE_METRIC, "value": tokens_total / (total_ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (fp32 accumulate)", "data": "synthetic",
        "config": {"workload": d.name, "T": d.T, "Din": d.Din, "Dout": d.Dout, "parallelism": "replicas",
                   "l2": f"{len(ws_)} rotating weight copies ({len(ws_) * w_bytes / 1e9:.2f} GB > L2)",
                   "launch": (f"CUDA graph per step ({launches} kernels)" if graphs
                              else f"eager ({launches} kernels per step)")},
        "roofline": roof,
        "clocks": clocks.summary(),
        "e2e": {"value": tokens_total / (e2e_ms * 1e-3), "unit": "tokens/s",
                "h2d_bytes_per_step": x_h.numel() * 2, "d2h_bytes_per_step": y_h.numel() * 2},
        "gpu_launches": launches * args.steps,
    }
    if world == 1 and not args.no_cpu_baseline:
        from oracle import dense as odense

        tok = min(d.T, 256)
        t0 = time.perf_counter()
        odense.dense_bf16(data["x"][:tok], data["w"])
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": tok / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                                "sample": f"{tok} of {d.T} tokens of {d.name}, fp64 numpy BLAS, {dt:.2f} s"}
    print(json.dumps(line), flush=True)


def run_dense_reference(args, d) -> None:
    """The dense oracle (fp64 numpy BLAS) on min(T, 64) tokens per step."""
    if int(os.environ.get("RANK", "0")) != 0:
        return
    from nvfp4_mixture_experts_route_gb300 import inputs
    from oracle import dense as odense

    data = inputs.make_dense(d)
    tok = min(d.T, 64)
    for _ in range(args.warmup):
        odense.dense_bf16(data["x"][:tok], data["w"])
    t0 = time.perf_counter()
    for _ in range(args.steps):
        odense.dense_bf16(data["x"][:tok], data["w"])
    dt = time.perf_counter() - t0
    value = tok * args.steps / dt
    sample = f"{tok} of {d.T} tokens of {d.name} per step, fp64 numpy BLAS on the host's default threads"
    print(json.dumps({
        "impl": "reference", "metric": DENSE_METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * dt / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": d.name, "T": d.T, "Din": d.Din, "Dout": d.Dout, "parallelism": "replicas"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode_b8")
    ap.add_argument("--copies", type=int, default=4)
    ap.add_argument("--cpu-tokens", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tile-m", type=int, default=0, help="route tile rows (default: the workload's)")
    ap.add_argument("--also", default=None,
                    help="comma-separated further workloads of the same layer, timed in the same run and "
                         "reported under 'workloads' (default with decode_b8: decode_b64_zipf,prefill_t8192_zipf; "
                         "'' for none)")
    ap.add_argument("--no-chain", dest="chain", action="store_false",
                    help="time one graph replay per step instead of graphs of one step per weight copy in a row")
    ap.add_argument("--no-graph", dest="graph", action="store_false",
                    help="launch the timed steps one by one instead of replaying CUDA graphs")
    args = ap.parse_args()
    from nvfp4_mixture_experts_route_gb300 import inputs

    if args.workload in inputs.DENSE_WORKLOADS:
        if args.impl == "reference":
            run_dense_reference(args, inputs.DENSE_WORKLOADS[args.workload])
        else:
            run_dense(args, inputs.DENSE_WORKLOADS[args.workload])
        return
    w = inputs.WORKLOADS[args.workload]
    if args.tile_m:
        import dataclasses

        w = dataclasses.replace(w, tile_m=args.tile_m)
    if args.also is None and args.workload == "decode_b8" and not args.tile_m:
        args.also = "decode_b64_zipf,prefill_t8192_zipf"
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
