"""The routed NVFP4 expert block and the post-expert finalize, route by route.

Test infrastructure only (see the package docstring).

The permuted, padded row layout of the kernels is only a device of speed, so
the oracle evaluates each route (t, k) directly (plain definition), then
places its GEMM2 row at the permuted index from :mod:`oracle.routing`.

Steps (argument names from the flashinfer_ops page, ``nvfp4_arguments``, and
the muse_moe_runner page, ``apply_routed`` and
``process_weights_after_loading``):

1. a = NVFP4(x[t]) with a1_gscale                         (:mod:`oracle.quant`)
2. acc1 = a . w13[e]^T over K = H, exact                   (:mod:`oracle.gemm`)
   gate = g1_alphas[e] * acc1[0:I]      ("output1_scale_gate_scalar")
   up   = g1_scale_c[e] * acc1[I:2I]    ("output1_scale_scalar")
   w13 rows [0, I) are the gate (w1) rows, [I, 2I) the up (w3) rows: open
   point 3.
3. h = SiLU(gate) * up, no clamp / alpha / beta (the muse_moe_runner page
   requires W4A4 SwiGLU checkpoints and refuses clamp/alpha/beta).
4. hq = NVFP4(h) with a2_gscale. The pages fold 1/a2 into g1_scale_c; this
   project keeps g1_scale_c free of it and multiplies by a2_gscale in the
   requant instead (open point 2; a caller with the pages' convention passes
   a2_gscale = 1). h is rounded to fp32 before the quantizer, whose decisions
   are taken in fp32 as in the kernel.
5. rows = g2_alphas[e] * (hq . w2[e]^T) over K = I ("output2_scale_scalar"),
   kept in fp64 and rounded once to bf16 (the GEMM2 rows are bf16 on the
   flashinfer_ops page, ``gemm2_rows``).
6. finalize (``MusePostExpertFinalize``): out[t] = sum_k w[t, k] * N(rows[p(t,
   k)]); routes marked -1 add nothing (``_finalize_native`` reads row 0 and
   zeroes it); N is an RMSNorm over all H with zero-centred gamma, the gain
   centre 1 added to the bf16 weight in higher precision
   (``_effective_weight``); the norm's output is fp32 and so is the top-k sum
   (``_finalize_chunk``), copied into the bf16 ``out``.
   Which RMSNorm is open point 1: with g = 1 + gamma,
     weight_before_norm = True  (default):  u = g * r;  N = u / sqrt(mean(u^2) + eps)
     weight_before_norm = False:            N = g * r / sqrt(mean(r^2) + eps)
   The oracle sums in fp64 and also returns bf16(out).

Parity: pinned (finalize against ``torch.nn.functional.rms_norm`` in the K = 1,
w = 1, gamma = 0 special case, invariants (iii)-(vi), the expert-TP identity
in exact arithmetic).
"""
from __future__ import annotations

import numpy as np

from . import gemm as _gemm
from .codecs import bf16_bits_to_f64, round_to_bf16
from .quant import quantize_blocks
from .routing import route_metadata


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """SiLU(gate) * up in fp64."""
    with np.errstate(over="ignore"):
        return gate / (1.0 + np.exp(-gate)) * up


def expert_rows(
    x_bits,
    topk_ids,
    layer: dict,
    a1_gscale: float,
    a2_gscale: float,
    mode: str = "exact",
    return_intermediate: bool = False,
    hq_override: dict | None = None,
):
    """GEMM2 rows of every route, in route order.

    ``x_bits``: bf16 bit patterns [T, H]; ``topk_ids`` int [T, K]; ``layer``
    holds raw (unprepared) NVFP4 weights: w13 codes-packed uint8 [E, 2I, H/2],
    w13_sf [E, 2I, H/16], w2 [E, H, I/2], w2_sf [E, H, I/16], and fp32
    g1_alphas, g1_scale_c, g2_alphas [E].

    ``hq_override`` maps a route index j to (codes [I], sf [I/16]) to run GEMM2
    on a given quantized intermediate.

    Returns dict with ``rows`` fp64 [T*K, H] (zero for unrouted routes),
    ``rows_bf16`` (the same rounded to bf16), ``a_codes``/``a_sf`` per token
    and, if asked, ``h`` fp64 [T*K, I], ``hq_codes`` [T*K, I], ``hq_sf``.
    """
    from .codecs import unpack_nibbles

    gemm = _gemm.gemm_exact if mode == "exact" else _gemm.gemm_exact_int64
    x = bf16_bits_to_f64(x_bits)
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, K = ids.shape
    w13 = layer["w13"]
    E, twoI, half_h = w13.shape
    I = twoI // 2
    H = 2 * half_h

    a_codes, a_sf = quantize_blocks(x.astype(np.float32), a1_gscale)
    rows = np.zeros((T * K, H))
    h_all = np.zeros((T * K, I)) if return_intermediate else None
    hq_codes = np.zeros((T * K, I), dtype=np.uint8) if return_intermediate else None
    hq_sf = np.zeros((T * K, I // 16), dtype=np.uint8) if return_intermediate else None
    flat = ids.reshape(-1)
    for e in np.unique(flat[flat >= 0]):
        js = np.nonzero(flat == e)[0]
        ts = js // K
        w13_codes = unpack_nibbles(w13[e])
        acc1 = gemm(a_codes[ts], a_sf[ts], w13_codes, layer["w13_sf"][e])
        gate = np.float64(np.float32(layer["g1_alphas"][e])) * acc1[:, :I]
        up = np.float64(np.float32(layer["g1_scale_c"][e])) * acc1[:, I:]
        h = swiglu(gate, up)
        qc, qs = quantize_blocks(h.astype(np.float32), a2_gscale)
        if hq_override is not None:
            for n, j in enumerate(js):
                if int(j) in hq_override:
                    qc[n], qs[n] = hq_override[int(j)]
        w2_codes = unpack_nibbles(layer["w2"][e])
        acc2 = gemm(qc, qs, w2_codes, layer["w2_sf"][e])
        rows[js] = np.float64(np.float32(layer["g2_alphas"][e])) * acc2
        if return_intermediate:
            h_all[js] = h
            hq_codes[js] = qc
            hq_sf[js] = qs
    out = {"rows": rows, "rows_bf16": round_to_bf16(rows), "a_codes": a_codes, "a_sf": a_sf}
    if return_intermediate:
        out.update(h=h_all, hq_codes=hq_codes, hq_sf=hq_sf)
    return out


def rms_norm_route(r: np.ndarray, gamma: np.ndarray, eps: float, weight_before_norm: bool) -> np.ndarray:
    """N(r) over the last axis, fp64, with zero-centred gamma (g = 1 + gamma)."""
    g = 1.0 + np.asarray(gamma, dtype=np.float64)
    if weight_before_norm:
        u = g * r
        return u / np.sqrt(np.mean(u * u, axis=-1, keepdims=True) + eps)
    return g * r / np.sqrt(np.mean(r * r, axis=-1, keepdims=True) + eps)


def finalize(
    rows: np.ndarray,
    expanded_to_permuted: np.ndarray,
    topk_weights: np.ndarray,
    gamma_bits: np.ndarray,
    eps: float,
    weight_before_norm: bool = True,
) -> dict[str, np.ndarray]:
    """out[t] = sum_k w[t, k] * N(rows[p(t, k)]), fp64; p = -1 adds nothing.

    ``rows`` are the permuted GEMM2 rows (bf16 values as float64) [P, H];
    ``gamma_bits`` bf16 bit patterns [H]. Returns fp64 ``out`` [T, H] and
    ``out_bf16``."""
    idx = np.asarray(expanded_to_permuted, dtype=np.int64)
    w = np.asarray(topk_weights, dtype=np.float32).astype(np.float64)
    T, K = idx.shape
    H = rows.shape[1] if rows.ndim == 2 and rows.shape[0] else len(gamma_bits)
    gamma = bf16_bits_to_f64(gamma_bits)
    out = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            p = idx[t, k]
            if p < 0:
                continue
            out[t] += w[t, k] * rms_norm_route(rows[p], gamma, eps, weight_before_norm)
    return {"out": out, "out_bf16": round_to_bf16(out)}


def moe_layer(
    x_bits,
    topk_ids,
    topk_weights,
    layer: dict,
    a1_gscale: float,
    a2_gscale: float,
    gamma_bits,
    eps: float,
    tile: int,
    weight_before_norm: bool = True,
    mode: str = "exact",
    return_intermediate: bool = False,
) -> dict:
    """The whole block: metadata, per-route GEMM2 rows placed at their
    permuted indices, and the finalize."""
    ids = np.asarray(topk_ids)
    T, K = ids.shape
    E = layer["w13"].shape[0]
    meta = route_metadata(ids, E, tile)
    er = expert_rows(
        x_bits, ids, layer, a1_gscale, a2_gscale, mode=mode, return_intermediate=return_intermediate
    )
    H = er["rows"].shape[1]
    P = len(meta["permuted_to_token"])
    permuted = np.zeros((P, H))
    e2p = meta["expanded_to_permuted"].reshape(-1)
    live = e2p >= 0
    permuted[e2p[live]] = er["rows_bf16"][live]
    fin = finalize(permuted, meta["expanded_to_permuted"], topk_weights, gamma_bits, eps, weight_before_norm)
    return {"meta": meta, "routes": er, "gemm2_rows": permuted, **fin}
