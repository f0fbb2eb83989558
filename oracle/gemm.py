"""Block-scaled FP4 products.

Test infrastructure only (see the package docstring).

Both GEMMs of the expert block multiply an NVFP4 activation row by NVFP4
weight rows that share the K axis (K-major weights, ``WeightLayout.MajorK`` on
the flashinfer_ops page; shapes from the expert_tp page, ``StockNvfp4``):

    acc[n] = sum_b  sfA[b] * sfW[n, b] * sum_{i < 16} qA[16b + i] * qW[n, 16b + i]

with q the e2m1 values and sf the e4m3 block scales. The exact mode
evaluates this in int64 after scaling every factor to an integer (e2m1 * 2 in
[-12, 12], e4m3 * 2^9 in [0, 229376]); the result is exact because |acc_int|
<= (K/16) * 229376^2 * 16 * 144 < 2^63 for K <= 5120 * 8. ``acc = acc_int *
2^-20``. The fast mode dequantizes to fp64 and uses a BLAS matmul; it is exact
whenever the sum fits in 53 bits and is otherwise within fp64 rounding.

Parity: pinned (exact mode against a brute-force triple loop on tiny inputs,
fast mode against exact mode).
"""
from __future__ import annotations

import numpy as np

from .codecs import e2m1_decode, e4m3_decode

BLOCK = 16
ACC_SHIFT = 20  # qA * 2, qW * 2, sfA * 2^9, sfW * 2^9


def _q_int(codes) -> np.ndarray:
    """e2m1 codes -> exact integers 2 * value (int8, [-12, 12])."""
    return (e2m1_decode(codes) * 2.0).astype(np.int8)


def _sf_int(sf) -> np.ndarray:
    """e4m3 codes -> exact integers value * 2^9 (int64). Block scales are
    non-negative and finite (the MMA takes them unsigned)."""
    v = e4m3_decode(sf)
    if np.any(~np.isfinite(v)) or np.any(v < 0):
        raise ValueError("block scales must be finite and non-negative")
    return (v * 512.0).astype(np.int64)


def gemm_exact_int64(a_codes, a_sf, w_codes, w_sf) -> np.ndarray:
    """acc [r, n] (float64) for activation rows a [r, K] (codes) with scales
    [r, K/16] against weight rows w [n, K] with scales [n, K/16], summed in
    int64 block by block, exactly as the definition above reads."""
    a_codes = np.atleast_2d(a_codes)
    a_sf = np.atleast_2d(a_sf)
    r, K = a_codes.shape
    n = w_codes.shape[0]
    nb = K // BLOCK
    qa = _q_int(a_codes).reshape(r, nb, BLOCK)
    qw = _q_int(w_codes).reshape(n, nb, BLOCK).astype(np.int64)
    sa = _sf_int(a_sf).reshape(r, nb)
    sw = _sf_int(w_sf).reshape(n, nb)
    out = np.empty((r, n), dtype=np.float64)
    for i in range(r):
        inner = np.einsum("nbk,bk->nb", qw, qa[i].astype(np.int64))
        acc = np.sum(inner * sw * sa[i][None, :], axis=1, dtype=np.int64)
        out[i] = np.ldexp(acc.astype(np.float64), -ACC_SHIFT) if np.all(
            np.abs(acc) < 2**53
        ) else _ldexp_exact(acc)
    return out


def _scaled_int(codes, sf) -> np.ndarray:
    """Rows of codes with their block scale folded in, as exact integers held
    in fp64: (e2m1 * 2) * (e4m3 * 2^9), |value| <= 12 * 229376 < 2^22."""
    codes = np.atleast_2d(codes)
    K = codes.shape[-1]
    q = _q_int(codes).astype(np.float64).reshape(codes.shape[:-1] + (K // BLOCK, BLOCK))
    s = _sf_int(np.atleast_2d(sf)).astype(np.float64)
    return (q * s[..., None]).reshape(codes.shape)


def gemm_exact(a_codes, a_sf, w_codes, w_sf) -> np.ndarray:
    """Same result as :func:`gemm_exact_int64`, through an fp64 BLAS matmul of
    the integer-scaled operands. Every product and every partial sum is an
    integer; when sum_k |a'_k w'_nk| < 2^53 for every output (checked), any
    summation order is exact. Otherwise it falls back to the int64 path."""
    A = _scaled_int(a_codes, a_sf)
    W = _scaled_int(w_codes, w_sf)
    bound = np.abs(A) @ np.abs(W).T
    if np.any(bound >= 2.0**52):
        return gemm_exact_int64(a_codes, a_sf, w_codes, w_sf)
    return np.ldexp(A @ W.T, -ACC_SHIFT)


def _ldexp_exact(acc: np.ndarray) -> np.ndarray:
    # Integers above 2^53 cannot all be held in fp64; the caller only sees
    # them rounded once, here.
    return np.array([float(int(v)) * 2.0**-ACC_SHIFT for v in acc])


def dequantize(codes, sf) -> np.ndarray:
    """Rows [.., K] of codes with scales [.., K/16] -> float64 values."""
    codes = np.asarray(codes)
    K = codes.shape[-1]
    v = e2m1_decode(codes).reshape(codes.shape[:-1] + (K // BLOCK, BLOCK))
    return (v * e4m3_decode(sf)[..., None]).reshape(codes.shape)


def gemm_bruteforce(a_codes, a_sf, w_codes, w_sf) -> np.ndarray:
    """Triple loop over (r, n, k) in Python floats; for tiny pins only."""
    a_codes = np.atleast_2d(a_codes)
    a_sf = np.atleast_2d(a_sf)
    r, K = a_codes.shape
    n = w_codes.shape[0]
    ea = e2m1_decode(a_codes)
    ew = e2m1_decode(w_codes)
    sa = e4m3_decode(a_sf)
    sw = e4m3_decode(w_sf)
    out = np.zeros((r, n))
    for i in range(r):
        for j in range(n):
            s = 0.0
            for k in range(K):
                s += float(ea[i, k] * sa[i, k // BLOCK]) * float(ew[j, k] * sw[j, k // BLOCK])
            out[i, j] = s
    return out
