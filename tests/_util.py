"""Helpers shared by the tests: uploads, comparisons, cached oracle runs."""
import functools

import numpy as np
import torch

from nvfp4_mixture_experts_route_gb300 import inputs


def bf16_dev(bits, device="cuda"):
    """bf16 bit patterns (uint16 numpy) -> bf16 device tensor."""
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_host_f64(t):
    """bf16 tensor -> float64 numpy (exact)."""
    return t.detach().float().cpu().numpy().astype(np.float64)


def rel_l2(got, want) -> float:
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.sqrt(np.sum(want * want))
    return float(np.sqrt(np.sum((got - want) ** 2)) / (den if den > 0 else 1.0))


def finite_summary(a) -> str:
    a = np.asarray(a, dtype=np.float64)
    fin = np.isfinite(a)
    big = np.max(np.abs(a[fin])) if fin.any() else float("nan")
    return f"{int(fin.sum())}/{a.size} finite, max |finite| {big:.4g}"


def canon_codes(codes: np.ndarray) -> np.ndarray:
    """e2m1 nibbles with -0 (0x8) mapped to +0 (both decode to zero)."""
    c = np.asarray(codes).astype(np.uint8)
    return np.where((c & 0xF) == 0x8, 0, c & 0xF).astype(np.uint8)


def canon_packed(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed).astype(np.uint8)
    lo, hi = canon_codes(p & 0xF), canon_codes(p >> 4)
    return (lo | (hi << 4)).astype(np.uint8)


@functools.lru_cache(maxsize=4)
def layer_for(name: str):
    return inputs.make_layer(inputs.WORKLOADS[name])
