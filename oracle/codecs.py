"""Exact codecs for the number formats the expert block uses.

Test infrastructure only (see the package docstring).

Formats, from their published definitions (OCP Microscaling Formats spec v1.0,
section 5.3 for E2M1 and the OFP8 spec for E4M3 "fn"):

* E2M1 (the NVFP4 element): 1 sign bit, 2 exponent bits with bias 1, 1
  mantissa bit; exponent field 0 is subnormal (m * 0.5); no inf / NaN. The
  expert_tp page stores two elements per byte (``uint8 [.., H/2]``); the byte's
  low nibble holds the even element (the pages leave the nibble order open;
  this is the plainest reading, stated in the design notes).
* E4M3 "fn" (the NVFP4 block scale, ``torch.float8_e4m3fn`` on the expert_tp
  page, ``StockNvfp4``): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa
  bits; exponent field 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN; the
  largest finite value is 448.
* bfloat16: the top 16 bits of an IEEE fp32.

Encoders round to nearest, ties to the even code, and saturate to the largest
finite magnitude ("satfinite"), the reading of open point 7.
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------
# E2M1
# --------------------------------------------------------------------------


def e2m1_decode(code) -> np.ndarray:
    """Value of 4-bit E2M1 codes (array of ints 0..15) as float64."""
    c = np.asarray(code).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    exp = (c >> 1) & 0x3
    man = c & 0x1
    sub = man * 0.5  # exponent field 0: 0.m x 2^(1-bias), bias 1
    nrm = (1.0 + man * 0.5) * np.exp2(exp.astype(np.float64) - 1.0)
    return sign * np.where(exp == 0, sub, nrm)


def _positive_grid(decode, ncodes: int) -> tuple[np.ndarray, np.ndarray]:
    """Finite non-negative values of a format and their codes, ascending."""
    codes = np.arange(ncodes, dtype=np.int64)
    vals = decode(codes)
    keep = np.isfinite(vals) & (vals >= 0) & ~np.signbit(vals)
    codes, vals = codes[keep], vals[keep]
    order = np.argsort(vals, kind="stable")
    return vals[order], codes[order]


def _round_to_grid(mag: np.ndarray, grid: np.ndarray, gcodes: np.ndarray) -> np.ndarray:
    """Nearest grid point to each non-negative magnitude, ties to the even
    code, clamped to the largest grid value (satfinite)."""
    mag = np.minimum(mag, grid[-1])
    hi = np.clip(np.searchsorted(grid, mag, side="left"), 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_lo = mag - grid[lo]
    d_hi = grid[hi] - mag
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (gcodes[hi] % 2 == 0))
    pick_hi |= hi == lo
    return np.where(pick_hi, gcodes[hi], gcodes[lo])


_E2M1_GRID = _positive_grid(e2m1_decode, 8)


def e2m1_encode(v) -> np.ndarray:
    """E2M1 code (uint8 0..15) of real values, round-to-nearest-even with
    saturation to +-6. The sign bit follows the sign of the input, so a
    negative value that rounds to zero gives the -0 code 0x8."""
    v = np.asarray(v, dtype=np.float64)
    code = _round_to_grid(np.abs(v), *_E2M1_GRID)
    return (code | np.where(np.signbit(v), 0x8, 0)).astype(np.uint8)


# --------------------------------------------------------------------------
# E4M3 (fn)
# --------------------------------------------------------------------------


def e4m3_decode(code) -> np.ndarray:
    """Value of 8-bit E4M3fn codes as float64 (NaN for S.1111.111)."""
    c = np.asarray(code).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    sub = (man / 8.0) * 2.0**-6
    nrm = (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0)
    val = sign * np.where(exp == 0, sub, nrm)
    return np.where((exp == 0xF) & (man == 0x7), np.nan, val)


_E4M3_GRID = _positive_grid(e4m3_decode, 128)


def e4m3_encode(v) -> np.ndarray:
    """E4M3fn code (uint8) of real values, round-to-nearest-even with
    saturation to +-448 (``satfinite``). Inputs must not be NaN."""
    v = np.asarray(v, dtype=np.float64)
    code = _round_to_grid(np.abs(v), *_E4M3_GRID)
    return (code | np.where(np.signbit(v), 0x80, 0)).astype(np.uint8)


# --------------------------------------------------------------------------
# bfloat16
# --------------------------------------------------------------------------


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Value of bf16 bit patterns (uint16) as float64 (exact)."""
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(v) -> np.ndarray:
    """Round real values (float64) to the nearest bf16, ties to even, in one
    rounding step (no detour through fp32). Returns float64 holding bf16
    values. Inputs are finite and inside bf16's normal range or zero; the
    block never produces anything else."""
    v = np.asarray(v, dtype=np.float64)
    m, e = np.frexp(v)  # v = m * 2^e, 0.5 <= |m| < 1
    # bf16 keeps 8 significant bits: |m| * 2^8 in [128, 256).
    return np.ldexp(np.rint(m * 256.0), e - 8)


def bf16_bits(v) -> np.ndarray:
    """bf16 bit patterns (uint16) of values that are already bf16-exact."""
    f = np.asarray(v, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """Pack 4-bit codes [.., 2n] into bytes [.., n], even element in the low
    nibble."""
    c = np.asarray(codes).astype(np.uint8) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    """Inverse of :func:`pack_nibbles`: bytes [.., n] -> codes [.., 2n]."""
    p = np.asarray(packed).astype(np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out
