"""Seeded synthetic inputs for the routed NVFP4 MoE expert block.

This module only draws random data in the shapes and distributions of the
workloads; it holds none of the block's arithmetic. Both the CUDA path (tests,
``bench.py``) and the CPU oracle take their inputs from here, so they see the
same bytes.

Recipe (every workload, base seed 0): ``numpy.random.SeedSequence(seed)``
spawns ten children, used in this order -- x, x_cal, w13, w13_sf, w2, w2_sf,
scalars, gamma, routing, topk weights -- so the layer's weights are the same
for every token count.

* activations x: bf16 N(0, 1), [T, H]
* weights: packed e2m1 bytes uniform over all 256 values (every nibble
  uniform over the 16 codes), w13 [E, 2I, H/2], w2 [E, H, I/2]
* block scales: U[0.5, 2] rounded to the nearest e4m3 (torch's
  ``float8_e4m3fn`` conversion), w13_sf [E, 2I, H/16], w2_sf [E, H, I/16]
* per-expert scalars g1_alphas, g1_scale_c, g2_alphas: fp32 U[0.5, 1.5]
* global scales a1_gscale, a2_gscale: 1.0 for the tiny layer; for the full
  layer the stored calibration (``calibration.json`` beside this module,
  written by ``oracle/calibrate.py`` from a separate x_cal draw)
* post-expert norm gamma: bf16 N(0, 0.1), eps 1e-6
* routing: K distinct experts per token; "uniform" draws them uniformly,
  "zipf" with popularity p(rank) ~ rank^-1.1 over the E experts, ranks mapped
  to experts by a seeded permutation, K distinct experts drawn by successive
  weighted sampling without replacement (done as Gumbel top-K, which has the
  same distribution)
* topk weights: softmax of N(0, 1) over each token's K picks, fp32
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
CALIBRATION_FILE = os.path.join(_HERE, "calibration.json")

CHILDREN = ("x", "x_cal", "w13", "w13_sf", "w2", "w2_sf", "scalars", "gamma", "routing", "weights")
CAL_TOKENS = 8
EPS = 1e-6


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    I: int
    E: int
    K: int
    routing: str  # "uniform" | "zipf"
    tile_m: int
    tp: int = 1
    unit_global_scales: bool = False
    zipf_s: float = 1.1

    @property
    def layer_key(self) -> str:
        return f"E{self.E}_H{self.H}_I{self.I}"


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny_t4", T=4, H=256, I=128, E=8, K=2, routing="uniform", tile_m=32,
                 unit_global_scales=True),
        Workload("decode_b8", T=8, H=5120, I=2048, E=128, K=8, routing="uniform", tile_m=32),
        Workload("decode_b64_zipf", T=64, H=5120, I=2048, E=128, K=8, routing="zipf", tile_m=32),
        Workload("tp8_slice_b32", T=32, H=5120, I=2048, E=128, K=8, routing="uniform", tile_m=32, tp=8),
        Workload("prefill_t8192_zipf", T=8192, H=5120, I=2048, E=128, K=8, routing="zipf", tile_m=128),
    )
}


@dataclass(frozen=True)
class DenseWorkload:
    """The MoE pooler / unpooler projection alone: x bf16 [T, Din] times the
    Linear weight bf16 [Dout, Din]. The pages print neither hidden_size nor
    moe_hidden_size; both are taken as the expert block's H = 5120."""

    name: str
    T: int
    Din: int
    Dout: int


DENSE_WORKLOADS = {
    d.name: d
    for d in (
        DenseWorkload("pooler_b8", T=8, Din=5120, Dout=5120),
        DenseWorkload("pooler_t8192", T=8192, Din=5120, Dout=5120),
    )
}


def make_dense(d: DenseWorkload, seed: int = 0) -> dict[str, np.ndarray]:
    """x ~ N(0, 1) and w ~ N(0, 1/Din) as bf16 bit patterns."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, d.T, d.Din, d.Dout]))
    return {"x": _to_bf16_bits(rng.standard_normal((d.T, d.Din))),
            "w": _to_bf16_bits(rng.standard_normal((d.Dout, d.Din)) / np.sqrt(d.Din))}


def _rngs(seed: int) -> dict[str, np.random.Generator]:
    kids = np.random.SeedSequence(seed).spawn(len(CHILDREN))
    return {name: np.random.default_rng(k) for name, k in zip(CHILDREN, kids)}


def _to_bf16_bits(a: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def _to_e4m3_bits(a: np.ndarray) -> np.ndarray:
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy().copy()


def draw_topk(rng: np.random.Generator, T: int, E: int, K: int, routing: str, zipf_s: float = 1.1,
              perm_rng: np.random.Generator | None = None) -> np.ndarray:
    """K distinct expert ids per token, int32 [T, K]."""
    if routing == "uniform":
        keys = rng.random((T, E))
        return np.argsort(keys, axis=1, kind="stable")[:, :K].astype(np.int32)
    if routing == "zipf":
        perm = (perm_rng or rng).permutation(E)
        popularity = np.empty(E)
        popularity[perm] = np.arange(1, E + 1, dtype=np.float64) ** (-zipf_s)
        gumbel = -np.log(-np.log(rng.random((T, E))))
        keys = np.log(popularity)[None, :] + gumbel
        return np.argsort(-keys, axis=1, kind="stable")[:, :K].astype(np.int32)
    raise ValueError(routing)


def make_layer(w: Workload, seed: int = 0) -> dict[str, np.ndarray]:
    """Raw (unprepared) layer: w13, w13_sf, w2, w2_sf (uint8), g1_alphas,
    g1_scale_c, g2_alphas (fp32 [E]), gamma (bf16 bits [H])."""
    r = _rngs(seed)
    E, H, I = w.E, w.H, w.I
    scalars = r["scalars"].uniform(0.5, 1.5, size=(3, E)).astype(np.float32)
    return {
        "w13": r["w13"].integers(0, 256, size=(E, 2 * I, H // 2), dtype=np.uint8),
        "w13_sf": _to_e4m3_bits(r["w13_sf"].uniform(0.5, 2.0, size=(E, 2 * I, H // 16))),
        "w2": r["w2"].integers(0, 256, size=(E, H, I // 2), dtype=np.uint8),
        "w2_sf": _to_e4m3_bits(r["w2_sf"].uniform(0.5, 2.0, size=(E, H, I // 16))),
        "g1_alphas": scalars[0].copy(),
        "g1_scale_c": scalars[1].copy(),
        "g2_alphas": scalars[2].copy(),
        "gamma": _to_bf16_bits(r["gamma"].normal(0.0, 0.1, size=H)),
    }


def make_batch(w: Workload, seed: int = 0, T: int | None = None) -> dict[str, np.ndarray]:
    """x (bf16 bits [T, H]), topk_ids (int32 [T, K]), topk_weights (fp32 [T, K])."""
    r = _rngs(seed)
    T = w.T if T is None else T
    x = _to_bf16_bits(r["x"].standard_normal((T, w.H)))
    ids = draw_topk(r["routing"], T, w.E, w.K, w.routing, w.zipf_s)
    z = r["weights"].standard_normal((T, w.K))
    z = np.exp(z - z.max(axis=1, keepdims=True))
    weights = (z / z.sum(axis=1, keepdims=True)).astype(np.float32)
    return {"x": x, "topk_ids": ids, "topk_weights": weights}


def calibration_draw(w: Workload, seed: int = 0) -> dict[str, np.ndarray]:
    """The calibration batch: bf16 N(0, 1) x_cal [8, H] and uniform routes."""
    r = _rngs(seed)["x_cal"]
    x = _to_bf16_bits(r.standard_normal((CAL_TOKENS, w.H)))
    ids = draw_topk(r, CAL_TOKENS, w.E, w.K, "uniform")
    return {"x": x, "topk_ids": ids}


def global_scales(w: Workload) -> tuple[float, float]:
    """(a1_gscale, a2_gscale) for the workload's layer."""
    if w.unit_global_scales:
        return 1.0, 1.0
    with open(CALIBRATION_FILE) as f:
        cal = json.load(f)
    entry = cal[w.layer_key]
    return float(np.float32(entry["a1_gscale"])), float(np.float32(entry["a2_gscale"]))
