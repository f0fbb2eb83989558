"""NVFP4 quantization of rows in 16-element blocks.

Test infrastructure only (see the package docstring).

What it computes (flashinfer_ops page, ``FlashInferOps.probe_inputs`` and the
model page, ``MuseSpark1xMoE._prepared_nvfp4_forward``: ``scaled_fp4_quant(x,
global_scale, is_sf_swizzled_layout=False)`` gives e2m1 values ``uint8 [b,
H/2]`` and one e4m3 scale per 16 elements ``[b, H/16]`` in row-major, i.e.
unswizzled, order; the muse_moe_runner page, ``process_weights_after_loading``,
sets the input global scale ``a1_gscale = 1 / a13`` and the intermediate's
``a2_gscale = 1 / a2``):

    amax = max |v_i| over the block
    sf   = e4m3(amax * g / 6)               (6 = largest e2m1 magnitude)
    q_i  = e2m1(v_i * g / sf)  if sf != 0 else +0
    value represented = e2m1(q_i) * e4m3(sf)   (g is not divided back out: it
                                                 is folded into the per-expert
                                                 scalars)

The pages do not print the kernel's arithmetic, so the rounding order is this
project's reading (open point 6): every step is one correctly rounded fp32
operation, in this order --

    s   = fp32(fp32(amax * g) / 6)
    sf  = e4m3_rne_satfinite(s)
    inv = fp32(g / e4m3(sf))
    t_i = fp32(v_i * inv)
    q_i = e2m1_rne_satfinite(t_i)

-- so that the quantized codes, an integer result decided by floating point,
are decided in the same precision on the CPU and in the kernel. Parity:
pinned (brute force over the codec grid, the power-of-two scaling invariant,
the all-zero and saturating special cases).
"""
from __future__ import annotations

import numpy as np

from .codecs import e2m1_encode, e4m3_decode, e4m3_encode, pack_nibbles

BLOCK = 16
E2M1_MAX = 6.0


def quantize_blocks(v, g) -> tuple[np.ndarray, np.ndarray]:
    """Quantize rows ``v`` (float, [..., n], n % 16 == 0; values must be fp32
    representable) with fp32 global scale ``g``.

    Returns (codes uint8 [..., n] one 4-bit code per element, sf uint8
    [..., n/16] e4m3 codes)."""
    v = np.asarray(v, dtype=np.float32)
    g = np.float32(g)
    n = v.shape[-1]
    assert n % BLOCK == 0, "row length must be a multiple of 16"
    blocks = v.reshape(v.shape[:-1] + (n // BLOCK, BLOCK))
    amax = np.max(np.abs(blocks), axis=-1)  # exact
    s = (amax * g).astype(np.float32) / np.float32(E2M1_MAX)
    s = s.astype(np.float32)
    sf = e4m3_encode(s.astype(np.float64))
    sf_val = e4m3_decode(sf).astype(np.float32)  # exact
    nonzero = sf_val > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = np.where(nonzero, g / np.where(nonzero, sf_val, np.float32(1)), 0)
    inv = inv.astype(np.float32)
    t = (blocks * inv[..., None]).astype(np.float32)
    q = e2m1_encode(t.astype(np.float64))
    q = np.where(nonzero[..., None], q, 0).astype(np.uint8)
    return q.reshape(v.shape), sf


def quantize_rows_packed(v, g) -> tuple[np.ndarray, np.ndarray]:
    """As :func:`quantize_blocks`, packed two codes per byte (even element in
    the low nibble): (bytes uint8 [..., n/2], sf uint8 [..., n/16])."""
    q, sf = quantize_blocks(v, g)
    return pack_nibbles(q), sf


def dequantize_blocks(codes, sf) -> np.ndarray:
    """Value represented by codes [..., n] and scales [..., n/16] (float64),
    without the global scale."""
    from .codecs import e2m1_decode

    codes = np.asarray(codes)
    n = codes.shape[-1]
    vals = e2m1_decode(codes).reshape(codes.shape[:-1] + (n // BLOCK, BLOCK))
    return (vals * e4m3_decode(sf)[..., None]).reshape(codes.shape)
