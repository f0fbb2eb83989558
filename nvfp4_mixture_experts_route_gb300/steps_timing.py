"""Launch times of the steps around the expert block: the pre-expert RMSNorm +
NVFP4 quant (row-major, and into the permuted workspace), the MuseSpark1x
routing and the expert-TP finalize over 8 partial row buffers. Each entry
point is launched alone between CUDA events (median of 20, launch latency
included) at T = 8 and T = 8192 (H = 5120, E = 128, top-8) on synthetic
inputs.

    python -m nvfp4_mixture_experts_route_gb300.steps_timing
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from . import inputs

H, I, E, K = 5120, 2048, 128, 8


def _median_us(fn, n: int = 20) -> float:
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(n):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) * 1e3)
    return float(np.median(ts))


def measure(T: int, dev: str = "cuda") -> dict:
    """{step: (microseconds per launch, GB/s of the step's algorithmic bytes)}."""
    lib = B.load()
    res = {}
    x = torch.randn((T, H), device=dev).to(torch.bfloat16)
    gamma = (torch.randn(H, device=dev) * 0.1).to(torch.bfloat16)
    g = torch.tensor([500.0], device=dev)
    a = torch.empty((T, H // 2), dtype=torch.uint8, device=dev)
    a_sf = torch.empty((T, H // 16), dtype=torch.uint8, device=dev)

    def norm_quant():
        lib.moe_rmsnorm_nvfp4_quant(x.data_ptr(), gamma.data_ptr(), 1e-6, g.data_ptr(), T, H, a.data_ptr(),
                                    a_sf.data_ptr(), None)

    us = _median_us(norm_quant)
    res["norm_quant"] = (us, (T * H * 2 + T * H // 2 + T * H // 16 + H * 2) / us / 1e3)

    routing = "uniform" if T <= 64 else "zipf"
    tile = 32 if T <= 64 else 128
    ids = torch.from_numpy(inputs.draw_topk(np.random.default_rng(0), T, E, K, routing).astype(np.int32)).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    r = B.route_permute(ids, E, tile, status=st)
    ws = B.alloc_workspace(T, K, E, H, I, tile, dev)

    def norm_quant_permuted():
        B.experts_norm_quantize(r, ws, x=x, gamma=gamma, eps=1e-6, a1_gscale=g, T=T, H=H, I=I, E=E, K=K,
                                status=st)

    us = _median_us(norm_quant_permuted)
    res["norm_quant_permuted"] = (us, (T * H * 2 + T * K * (H // 2 + H // 16) + H * 2) / us / 1e3)

    logits = torch.randn((T, E), device=dev)
    bias = torch.randn(E, device=dev) * 0.1
    tid = torch.empty((T, K), dtype=torch.int32, device=dev)
    tw = torch.empty((T, K), dtype=torch.float32, device=dev)
    us = _median_us(lambda: B.musespark1x_routing(logits, bias, K, topk_ids=tid, topk_weights=tw))
    res["routing"] = (us, (T * E * 4 + E * 4 + T * K * 8) / us / 1e3)

    P, _ = B.route_sizes(T, K, E, tile)
    parts = [torch.randn((P, H), device=dev).to(torch.bfloat16) for _ in range(8)]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    twt = torch.rand((T, K), device=dev)
    us = _median_us(lambda: B.post_expert_finalize_tp(parts, r.expanded_to_permuted, twt, gamma, 1e-6, True, out=out,
                                                      status=st))
    res["finalize_tp8"] = (us, (8 * T * K * H * 2 + T * H * 2) / us / 1e3)
    if int(st.item()) != 0:
        raise RuntimeError(f"device status {B.STATUS_NAMES.get(int(st.item()))}")
    return res


def main() -> None:
    for T in (8, 8192):
        for name, (us, gbs) in measure(T).items():
            print(f"{name:22s} T={T:5d} {us:9.1f} us {gbs:9.1f} GB/s", flush=True)
        torch.cuda.empty_cache()


if __name__ == "__main__":
    main()
