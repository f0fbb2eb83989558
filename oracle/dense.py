"""The MoE pooler / unpooler projection (the model page: ``pooler`` and
``unpooler`` are ``ReplicatedLinear(..., bias=False, quant_config=None)``,
i.e. y = x . w^T on bf16 tensors).

Test infrastructure only (see the package docstring).

    y[t, o] = sum_i x[t, i] * w[o, i]

evaluated in fp64 from the bf16 bit patterns, then rounded once to bf16 (the
layer's output dtype). A bf16 x bf16 product has at most 16 significant bits,
so every product is exact in fp64 and the only rounding before the final one
is the fp64 summation.

Parity: pinned (a brute-force triple loop on tiny inputs, the identity and
permutation weights, which must return x exactly, and linearity in w).
"""
from __future__ import annotations

import numpy as np

from .codecs import bf16_bits_to_f64, round_to_bf16


def dense_f64(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """x bf16 bits [T, Din], w bf16 bits [Dout, Din] -> fp64 [T, Dout]."""
    x = bf16_bits_to_f64(x_bits)
    w = bf16_bits_to_f64(w_bits)
    return x @ w.T


def dense_bf16(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """The projection rounded to bf16 (returned as fp64 values)."""
    return round_to_bf16(dense_f64(x_bits, w_bits))
