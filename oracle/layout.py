"""The prepared weight layout, by its documented definition, and the expert-TP
slices.

Test infrastructure only (see the package docstring). Written from the layout
as ``include/moe_nvfp4.h`` documents it for ``moe_prepare_weights``; it shares
no code with the CUDA packer, and the GPU tests compare the two byte for byte.

Raw (the expert_tp page, ``StockNvfp4`` shapes; unswizzled scales):
    w13 uint8 [E, 2I, H/2]   rows [0, I) gate (w1), [I, 2I) up (w3)
    w13_sf e4m3 [E, 2I, H/16]
    w2 uint8 [E, H, I/2]
    w2_sf e4m3 [E, H, I/16]

Prepared:
    p_w13 uint8 [E, 2I, H/2]: prepared row r takes raw row
        16*(r//32) + r%32            if r%32 < 16   (gate)
        I + 16*(r//32) + r%32 - 16   otherwise      (up)
      i.e. gate and up alternate in 16-row granules, so that one 32-row group
      holds the gate and up rows of the same 16 intermediate columns.
    p_w13_sf uint8 [E, 2I/128, H/64, 512]: scale atoms; byte
      (e, mt, kc, 16*m0 + 4*m1 + c) holds the scale of prepared row
      128*mt + 32*m1 + m0 for the 16-element block 4*kc + c
      (m0 < 32, m1 < 4, c < 4).
    p_w2 uint8 [E, H, I/2] = w2 unchanged.
    p_w2_sf uint8 [E, H/128, I/64, 512]: the same atoms over w2_sf's rows
      and blocks.

Needs H % 128 == 0 and I % 64 == 0.

Expert TP (the expert_tp page, module docstring, ``slice_views`` and
``final_shapes``): rank r of tp holds intermediate slice [r I', (r+1) I'),
I' = I / tp, of every expert. The raw slice takes gate rows [r I', (r+1) I')
and up rows [I + r I', I + (r+1) I') of w13 (and w13_sf), and the columns of
that slice of w2 (and w2_sf). The layout identity this layout is built to
keep: for I' % 64 == 0 and H % 128 == 0, the slice view of the prepared
tensors is, byte for byte, the prepared layout of the raw slice.

Parity: pinned (round trip, identity over every slice, refusal cases).
"""
from __future__ import annotations

import numpy as np

ATOM_ROWS = 128
ATOM_KBLOCKS = 4
ATOM_BYTES = 512


def w13_source_row(r: np.ndarray, I: int) -> np.ndarray:
    """Raw w13 row feeding prepared row r."""
    r = np.asarray(r)
    g, j = r // 32, r % 32
    return np.where(j < 16, 16 * g + j, I + 16 * g + (j - 16))


def sf_to_atoms(sf: np.ndarray) -> np.ndarray:
    """[E, R, B] scales -> [E, R/128, B/4, 512] atoms."""
    E, R, B = sf.shape
    assert R % ATOM_ROWS == 0 and B % ATOM_KBLOCKS == 0
    # sf[e, 128*mt + 32*m1 + m0, 4*kc + c] -> atoms[e, mt, kc, 16*m0 + 4*m1 + c]
    v = sf.reshape(E, R // 128, 4, 32, B // 4, 4)  # e, mt, m1, m0, kc, c
    v = v.transpose(0, 1, 4, 3, 2, 5)  # e, mt, kc, m0, m1, c
    return np.ascontiguousarray(v.reshape(E, R // 128, B // 4, ATOM_BYTES))


def atoms_to_sf(atoms: np.ndarray) -> np.ndarray:
    """Inverse of :func:`sf_to_atoms`."""
    E, MT, KC, _ = atoms.shape
    v = atoms.reshape(E, MT, KC, 32, 4, 4)  # e, mt, kc, m0, m1, c
    v = v.transpose(0, 1, 4, 3, 2, 5)  # e, mt, m1, m0, kc, c
    return np.ascontiguousarray(v.reshape(E, MT * 128, KC * 4))


def unsupported(E: int, H: int, I: int) -> str | None:
    """Why the prepared layout cannot hold this shape, or None."""
    if E < 1 or H < 1 or I < 1:
        return "empty layer"
    if H % 128 or I % 64:
        return f"hidden {H} and intermediate {I} must be multiples of 128 and 64"
    return None


def prepare(w13, w13_sf, w2, w2_sf) -> dict[str, np.ndarray]:
    E, twoI, half_h = w13.shape
    I, H = twoI // 2, 2 * half_h
    reason = unsupported(E, H, I)
    if reason:
        raise ValueError(reason)
    src = w13_source_row(np.arange(twoI), I)
    return {
        "w13": np.ascontiguousarray(w13[:, src, :]),
        "w13_sf": sf_to_atoms(np.asarray(w13_sf)[:, src, :]),
        "w2": np.ascontiguousarray(w2),
        "w2_sf": sf_to_atoms(np.asarray(w2_sf)),
    }


def unprepare(p: dict[str, np.ndarray]) -> dict[str, np.ndarray]:
    p_w13 = p["w13"]
    E, twoI, half_h = p_w13.shape
    I = twoI // 2
    src = w13_source_row(np.arange(twoI), I)
    w13 = np.empty_like(p_w13)
    w13[:, src, :] = p_w13
    sf_p = atoms_to_sf(p["w13_sf"])
    w13_sf = np.empty_like(sf_p)
    w13_sf[:, src, :] = sf_p
    return {"w13": w13, "w13_sf": w13_sf, "w2": np.ascontiguousarray(p["w2"]), "w2_sf": atoms_to_sf(p["w2_sf"])}


def raw_slice(raw: dict[str, np.ndarray], r: int, tp: int) -> dict[str, np.ndarray]:
    """Rank r's raw intermediate slice (scalars unchanged)."""
    E, twoI, _ = raw["w13"].shape
    I = twoI // 2
    s = I // tp
    rows = np.concatenate([np.arange(r * s, (r + 1) * s), I + np.arange(r * s, (r + 1) * s)])
    out = dict(raw)
    out["w13"] = np.ascontiguousarray(raw["w13"][:, rows])
    out["w13_sf"] = np.ascontiguousarray(raw["w13_sf"][:, rows])
    out["w2"] = np.ascontiguousarray(raw["w2"][:, :, r * s // 2 : (r + 1) * s // 2])
    out["w2_sf"] = np.ascontiguousarray(raw["w2_sf"][:, :, r * s // 16 : (r + 1) * s // 16])
    return out


def prepared_slice_view(p: dict[str, np.ndarray], r: int, tp: int) -> dict[str, np.ndarray]:
    """Rank r's slice taken from the prepared tensors (copied contiguous)."""
    E, twoI, _ = p["w13"].shape
    I = twoI // 2
    s = I // tp
    return {
        "w13": np.ascontiguousarray(p["w13"][:, 2 * r * s : 2 * (r + 1) * s]),
        "w13_sf": np.ascontiguousarray(p["w13_sf"][:, 2 * r * s // 128 : 2 * (r + 1) * s // 128]),
        "w2": np.ascontiguousarray(p["w2"][:, :, r * s // 2 : (r + 1) * s // 2]),
        "w2_sf": np.ascontiguousarray(p["w2_sf"][:, :, r * s // 64 : (r + 1) * s // 64]),
    }
