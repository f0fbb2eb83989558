"""GPU parity of the tcgen05 grouped GEMMs and of the whole expert block
against the CPU oracle, through the C ABI.

Bars: GEMM2 rows on identical quantized operands within rel-L2 2e-3; final
output within rel-L2 1e-2 (the intermediate requant may flip FP4 codes at
rounding boundaries because h is fp32 on the GPU and fp64 in the oracle);
routing metadata bit-exact (test_gpu_kernels)."""
import time

import numpy as np
import pytest
import torch

from oracle import codecs, layer as olayer, layout as olayout
from nvfp4_mixture_experts_route_gb300 import binding as B
from nvfp4_mixture_experts_route_gb300 import inputs

from _util import bf16_dev, bf16_host_f64, canon_codes, finite_summary, layer_for, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"

GEMM2_BAR = 2e-3
OUT_BAR = 1e-2


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.to(DEV) if dtype is None else t.to(DEV, dtype)


class Prepared:
    """A layer uploaded and prepared once."""

    def __init__(self, raw):
        t = {k: _dev(raw[k]) for k in ("w13", "w13_sf", "w2", "w2_sf")}
        self.E, twoI, hh = raw["w13"].shape
        self.I, self.H = twoI // 2, 2 * hh
        self.p = B.prepare_weights(t["w13"], t["w13_sf"], t["w2"], t["w2_sf"])
        del t
        self.g1a = _dev(raw["g1_alphas"])
        self.g1c = _dev(raw["g1_scale_c"])
        self.g2a = _dev(raw["g2_alphas"])
        self.gamma = bf16_dev(raw["gamma"])
        self.w = B.weights_struct(self.p, self.g1a, self.g1c, self.g2a)


def run_gpu(prep: Prepared, batch, tile, a1, a2, *, hq_override=None, wbn=True, export=True):
    """Routing, quantize, GEMM1, [import hq], GEMM2, finalize. Returns numpy
    views of what the tests compare."""
    E, H, I = prep.E, prep.H, prep.I
    ids = _dev(batch["topk_ids"].astype(np.int32))
    T, K = ids.shape
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    r = B.route_permute(ids, E, tile, status=status)
    ws = B.alloc_workspace(T, K, E, H, I, tile, DEV)
    g1 = torch.tensor([a1], dtype=torch.float32, device=DEV)
    g2 = torch.tensor([a2], dtype=torch.float32, device=DEV)
    B.experts_quantize(r, ws, x=bf16_dev(batch["x"]), a1_gscale=g1, T=T, H=H, I=I, E=E, K=K, status=status)
    B.experts_gemm1(prep.w, r, ws, a2_gscale=g2, T=T, H=H, I=I, E=E, K=K, status=status)
    out = {}
    if export:
        hc, hs = B.experts_export(1, ws, T=T, H=H, I=I, E=E, K=K, tile_m=tile)
        out["hq_codes"], out["hq_sf"] = hc.cpu().numpy(), hs.cpu().numpy()
    if hq_override is not None:
        B.experts_import(1, _dev(hq_override[0]), _dev(hq_override[1]), ws, T=T, H=H, I=I, E=E, K=K, tile_m=tile)
    P, _ = B.route_sizes(T, K, E, tile)
    rows = torch.zeros((max(P, 1), H), dtype=torch.bfloat16, device=DEV)
    B.experts_gemm2(prep.w, r, ws, rows, T=T, H=H, I=I, E=E, K=K, status=status)
    fin = B.post_expert_finalize(rows, r.expanded_to_permuted, _dev(batch["topk_weights"]), prep.gamma, 1e-6, wbn)
    torch.cuda.synchronize()
    out.update(
        status=int(status.item()),
        e2p=r.expanded_to_permuted.cpu().numpy(),
        p2t=r.permuted_to_token.cpu().numpy(),
        rows=bf16_host_f64(rows),
        out=bf16_host_f64(fin),
    )
    return out


def oracle_hq_permuted(er, e2p, P, I):
    """The oracle's quantized intermediate placed at the permuted rows."""
    codes = np.zeros((P, I // 2), np.uint8)
    sf = np.zeros((P, I // 16), np.uint8)
    flat = e2p.reshape(-1)
    live = flat >= 0
    codes[flat[live]] = codecs.pack_nibbles(er["hq_codes"][live])
    sf[flat[live]] = er["hq_sf"][live]
    return codes, sf


def _workload(T, H, I, E, K, routing="uniform", tile=32):
    return inputs.Workload(f"t{T}h{H}i{I}e{E}k{K}", T=T, H=H, I=I, E=E, K=K, routing=routing, tile_m=tile)


SMALL = [
    # (T, H, I, E, K, routing, tile, a1, a2)
    (4, 256, 128, 8, 2, "uniform", 32, 1.0, 1.0),           # the tiny workload
    (37, 512, 256, 8, 4, "uniform", 32, 4.0, 1e-3),        # several tiles, ragged tail
    (29, 640, 384, 4, 3, "zipf", 64, 4.0, 1e-3),           # ragged K (2.5 and 1.5 stages)
    (70, 512, 256, 4, 4, "zipf", 128, 4.0, 1e-3),          # tile 128
    (150, 256, 256, 4, 4, "uniform", 256, 4.0, 1e-3),      # tile 256: two scale atoms per tile
    # I % 128 == 64 (expert-TP slices the prepared layout admits): a GEMM2 K
    # stage of one or three K = 64 steps reads past the row end (zero fill)
    (19, 256, 192, 4, 2, "uniform", 32, 4.0, 1e-3),
    (40, 256, 320, 4, 3, "zipf", 128, 4.0, 1e-3),
    (9, 512, 64, 4, 2, "uniform", 64, 4.0, 1e-3),
    # 128-row tiles with a last K stage of two steps: GEMM2 (K = 384) here,
    # GEMM1 (K = 640) below
    (150, 768, 384, 4, 4, "zipf", 128, 4.0, 1e-3),
    (90, 640, 384, 3, 3, "uniform", 128, 4.0, 1e-3),
]


@pytest.fixture(scope="module")
def small_cases():
    out = []
    for T, H, I, E, K, routing, tile, a1, a2 in SMALL:
        w = _workload(T, H, I, E, K, routing, tile)
        raw = inputs.make_layer(w)
        batch = inputs.make_batch(w)
        out.append((w, raw, batch, tile, a1, a2))
    return out


def _fused_rows(prep, batch, tile, a1, a2, calls=2):
    """quantize, then moe_experts_gemms `calls` times on the same workspace."""
    E, H, I = prep.E, prep.H, prep.I
    ids = _dev(batch["topk_ids"].astype(np.int32))
    T, K = ids.shape
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    r = B.route_permute(ids, E, tile, status=status)
    ws = B.alloc_workspace(T, K, E, H, I, tile, DEV)
    g1 = torch.tensor([a1], dtype=torch.float32, device=DEV)
    g2 = torch.tensor([a2], dtype=torch.float32, device=DEV)
    B.experts_quantize(r, ws, x=bf16_dev(batch["x"]), a1_gscale=g1, T=T, H=H, I=I, E=E, K=K, status=status)
    P, _ = B.route_sizes(T, K, E, tile)
    outs = []
    for _ in range(calls):
        rows = torch.zeros((max(P, 1), H), dtype=torch.bfloat16, device=DEV)
        B.experts_gemms(prep.w, r, ws, rows, a2_gscale=g2, T=T, H=H, I=I, E=E, K=K, status=status)
        outs.append(rows)
    torch.cuda.synchronize()
    return int(status.item()), [bf16_host_f64(o) for o in outs]


FUSED_EXTRA = [
    (1, 256, 128, 8, 1, "uniform", 32, 4.0, 1e-3),      # one route tile: GEMM2 units wait on GEMM1 units
    (3, 512, 384, 2, 2, "uniform", 64, 4.0, 1e-3),      # one expert, few units, ragged K
]


@pytest.mark.parametrize("idx", range(len(SMALL) + len(FUSED_EXTRA)))
def test_fused_gemms_match_split_gemms(small_cases, idx):
    """The one-launch GEMM1+GEMM2 (per-route-tile completion counters) gives
    the split launches' GEMM2 rows bit for bit, at every tile size, and again
    when called a second time on the same workspace."""
    if idx < len(SMALL):
        w, raw, batch, tile, a1, a2 = small_cases[idx]
    else:
        T, H, I, E, K, routing, tile, a1, a2 = FUSED_EXTRA[idx - len(SMALL)]
        w = _workload(T, H, I, E, K, routing, tile)
        raw, batch = inputs.make_layer(w), inputs.make_batch(w)
    prep = Prepared(raw)
    split = run_gpu(prep, batch, tile, a1, a2, export=False)
    assert split["status"] == 0
    status, fused = _fused_rows(prep, batch, tile, a1, a2)
    assert status == 0
    for rows in fused:
        assert np.array_equal(rows, split["rows"])


ROUTED_EXTRA = [
    # (T, H, I, E, K, routing, tile, a1, a2)
    (256, 256, 128, 16, 8, "uniform", 32, 4.0, 1e-3),   # T*K = 2048: most routes routed in the quantizer
    (257, 256, 128, 16, 8, "uniform", 32, 4.0, 1e-3),   # T*K = 2056: the routing kernels, then the body
    (5, 256, 128, 200, 4, "zipf", 64, 4.0, 1e-3),       # E = 200: 8 warps x E histogram, few routes
    (3, 256, 128, 300, 2, "uniform", 32, 4.0, 1e-3),    # E > 256: the routing kernels, then the body
]

_ROUTE_FIELDS = ("expert_counts", "expert_offsets", "expanded_to_permuted", "permuted_to_token", "tile_expert",
                 "tile_row_limit", "totals")


def _routed_vs_split(prep, ids_np, x_bits, tile, a1, a2):
    """(status, route, rows) of route_permute + nvfp4_experts and of
    nvfp4_experts_routed (called twice on the same buffers)."""
    E, H, I = prep.E, prep.H, prep.I
    ids = _dev(ids_np.astype(np.int32))
    T, K = ids.shape
    x = bf16_dev(x_bits)
    g1 = torch.tensor([a1], dtype=torch.float32, device=DEV)
    g2 = torch.tensor([a2], dtype=torch.float32, device=DEV)
    st_a = torch.zeros(1, dtype=torch.int32, device=DEV)
    r_a = B.route_permute(ids, E, tile, status=st_a)
    rows_a, _ = B.nvfp4_experts(prep.w, r_a, x=x, a1_gscale=g1, a2_gscale=g2, T=T, H=H, I=I, E=E, K=K, status=st_a)
    st_b = torch.zeros(1, dtype=torch.int32, device=DEV)
    r_b = B.alloc_route(T, K, E, tile, DEV)
    for f in _ROUTE_FIELDS:  # what the call must overwrite
        getattr(r_b, f).fill_(12345)
    ws = B.alloc_workspace(T, K, E, H, I, tile, DEV)
    outs = []
    for _ in range(2):
        rows_b = torch.zeros_like(rows_a)
        B.nvfp4_experts_routed(prep.w, ids, r_b, x=x, a1_gscale=g1, a2_gscale=g2, H=H, I=I, E=E, gemm2_rows=rows_b,
                               ws=ws, status=st_b)
        outs.append(rows_b)
    torch.cuda.synchronize()
    return (int(st_a.item()), r_a, rows_a), (int(st_b.item()), r_b, outs)


@pytest.mark.parametrize("idx", range(len(SMALL) + len(ROUTED_EXTRA)))
def test_routed_entry_matches_route_then_experts(small_cases, idx):
    """moe_nvfp4_experts_routed writes moe_route_permute's metadata bit for
    bit and moe_nvfp4_experts's GEMM2 rows (every row that carries a route)
    on that route, whether the routing ran inside the input quantizer (few
    routes, tile_m <= 64: 2 kernels) or as its own kernels before the body,
    and again on a second call over the same buffers."""
    if idx < len(SMALL):
        w, raw, batch, tile, a1, a2 = small_cases[idx]
    else:
        T, H, I, E, K, routing, tile, a1, a2 = ROUTED_EXTRA[idx - len(SMALL)]
        w = _workload(T, H, I, E, K, routing, tile)
        raw, batch = inputs.make_layer(w), inputs.make_batch(w)
    prep = Prepared(raw)
    fused = w.T * w.K <= 2048 and w.E <= 256 and tile <= 64
    want_kernels = 2 if fused else B.route_kernels(w.T, w.K, w.E) + B.experts_kernels(tile)
    assert B.routed_experts_kernels(w.T, w.K, w.E, tile) == want_kernels
    (st_a, r_a, rows_a), (st_b, r_b, outs) = _routed_vs_split(prep, batch["topk_ids"], batch["x"], tile, a1, a2)
    assert st_a == 0 and st_b == 0
    for f in _ROUTE_FIELDS:
        assert torch.equal(getattr(r_a, f), getattr(r_b, f)), f
    live = r_a.expanded_to_permuted.reshape(-1)
    live = live[live >= 0]
    for rows_b in outs:
        assert torch.equal(rows_b[live], rows_a[live])


def test_routed_entry_unrouted_and_bad_ids(small_cases):
    """Routes marked -1 are skipped and an id out of range is skipped and
    reported (MOE_ERR_INVALID_ROUTE), by the routing inside the quantizer as
    by moe_route_permute; the rows of the other routes agree bit for bit."""
    w, raw, batch, tile, a1, a2 = small_cases[1]
    assert w.T * w.K <= 2048 and tile <= 64
    ids = batch["topk_ids"].copy()
    ids[::3, 0] = -1
    ids[1, 1] = w.E
    prep = Prepared(raw)
    (st_a, r_a, rows_a), (st_b, r_b, outs) = _routed_vs_split(prep, ids, batch["x"], tile, a1, a2)
    assert st_a == -6 and st_b == -6
    for f in _ROUTE_FIELDS:
        assert torch.equal(getattr(r_a, f), getattr(r_b, f)), f
    live = r_a.expanded_to_permuted.reshape(-1)
    live = live[live >= 0]
    assert len(live) == w.T * w.K - len(ids[::3]) - 1
    for rows_b in outs:
        assert torch.equal(rows_b[live], rows_a[live])


BLOCK_EXTRA = ROUTED_EXTRA + [
    (7, 256, 128, 16, 12, "uniform", 32, 4.0, 1e-3),    # K = 12 > 8: the finalize kernel after the body
    (1, 640, 384, 8, 8, "uniform", 64, 4.0, 1e-3),      # one token, H = 640: a partial column slice
]


def _block_vs_parts(prep, ids_np, batch, tile, a1, a2, wbn, calls=2):
    """(status, route, rows, row_sumsq, out) of route_permute +
    nvfp4_experts_sumsq + post_expert_finalize_sumsq, and of moe_block called
    `calls` times on the same buffers (its outputs of each call)."""
    E, H, I = prep.E, prep.H, prep.I
    ids = _dev(ids_np.astype(np.int32))
    T, K = ids.shape
    x = bf16_dev(batch["x"])
    tw = _dev(batch["topk_weights"])
    g1 = torch.tensor([a1], dtype=torch.float32, device=DEV)
    g2 = torch.tensor([a2], dtype=torch.float32, device=DEV)
    st_a = torch.zeros(1, dtype=torch.int32, device=DEV)
    r_a = B.route_permute(ids, E, tile, status=st_a)
    rows_a, ss_a, _ = B.nvfp4_experts_sumsq(prep.w, r_a, x=x, a1_gscale=g1, a2_gscale=g2, T=T, H=H, I=I, E=E, K=K,
                                            gamma=prep.gamma, weight_before_norm=wbn, status=st_a)
    out_a = B.post_expert_finalize_sumsq(rows_a, ss_a, r_a.expanded_to_permuted, tw, prep.gamma, 1e-6, status=st_a)
    st_b = torch.zeros(1, dtype=torch.int32, device=DEV)
    r_b = B.alloc_route(T, K, E, tile, DEV)
    for f in _ROUTE_FIELDS:
        getattr(r_b, f).fill_(12345)
    ws = B.alloc_workspace(T, K, E, H, I, tile, DEV)
    got = []
    for _ in range(calls):
        rows_b = torch.zeros_like(rows_a)
        ss_b = torch.zeros_like(ss_a)
        out_b = torch.full_like(out_a, 7.0)
        B.moe_block(prep.w, ids, tw, r_b, x=x, a1_gscale=g1, a2_gscale=g2, gamma=prep.gamma, eps=1e-6,
                    weight_before_norm=wbn, H=H, I=I, E=E, gemm2_rows=rows_b, row_sumsq=ss_b, out=out_b, ws=ws,
                    status=st_b)
        got.append((rows_b, ss_b, out_b))
    torch.cuda.synchronize()
    return (int(st_a.item()), r_a, rows_a, ss_a, out_a), (int(st_b.item()), r_b, got)


def _check_block(parts, block):
    (st_a, r_a, rows_a, ss_a, out_a), (st_b, r_b, got) = parts, block
    assert st_a == st_b
    for f in _ROUTE_FIELDS:
        assert torch.equal(getattr(r_a, f), getattr(r_b, f)), f
    live = r_a.expanded_to_permuted.reshape(-1)
    live = live[live >= 0]
    for rows_b, ss_b, out_b in got:
        assert torch.equal(rows_b[live], rows_a[live])
        assert torch.equal(ss_b[live], ss_a[live])
        assert torch.equal(out_b, out_a)


@pytest.mark.parametrize("wbn", [True, False])
@pytest.mark.parametrize("idx", range(len(SMALL) + len(BLOCK_EXTRA)))
def test_block_entry_matches_its_parts(small_cases, idx, wbn):
    """moe_nvfp4_moe_block equals moe_route_permute, moe_nvfp4_experts_sumsq
    and moe_post_expert_finalize_sumsq bit for bit (metadata, live rows,
    their sums of squares, the output), with the finalize by units (K <= 8)
    or per token (K = 12), in both norm readings (gamma ~ N(0, 1)), and again
    on a second call over the same buffers."""
    if idx < len(SMALL):
        w, raw, batch, tile, a1, a2 = small_cases[idx]
    else:
        T, H, I, E, K, routing, tile, a1, a2 = BLOCK_EXTRA[idx - len(SMALL)]
        w = _workload(T, H, I, E, K, routing, tile)
        raw, batch = inputs.make_layer(w), inputs.make_batch(w)
    raw = dict(raw)
    raw["gamma"] = inputs._to_bf16_bits(np.random.default_rng(5).standard_normal(w.H))
    prep = Prepared(raw)
    n = B.moe_block_kernels(w.T, w.K, w.E, tile)
    assert n == B.route_kernels(w.T, w.K, w.E) + B.experts_kernels(tile) + 1
    _check_block(*_block_vs_parts(prep, batch["topk_ids"], batch, tile, a1, a2, wbn))


def test_block_entry_against_the_oracle(small_cases, record_property):
    """The whole block (sums of squares in GEMM2, the finalize from them)
    against the oracle's layer: output within the end-to-end bar, and the
    oracle's finalize of the block's own rows within 2e-3."""
    w, raw, batch, tile, a1, a2 = small_cases[1]
    raw = dict(raw)
    raw["gamma"] = inputs._to_bf16_bits(np.random.default_rng(6).standard_normal(w.H))
    prep = Prepared(raw)
    for wbn in (True, False):
        (_, r_a, _, _, _), (st, r_b, got) = _block_vs_parts(prep, batch["topk_ids"], batch, tile, a1, a2, wbn,
                                                            calls=1)
        assert st == 0
        rows_b, _, out_b = got[0]
        ref = olayer.moe_layer(batch["x"], batch["topk_ids"], batch["topk_weights"], raw, a1, a2, raw["gamma"],
                               1e-6, tile, weight_before_norm=wbn)
        err = rel_l2(bf16_host_f64(out_b), ref["out"])
        e2p = r_b.expanded_to_permuted.cpu().numpy()
        fin = olayer.finalize(bf16_host_f64(rows_b), e2p, batch["topk_weights"], raw["gamma"], 1e-6, wbn)
        err_fin = rel_l2(bf16_host_f64(out_b), fin["out"])
        record_property(f"out_rel_l2_wbn{int(wbn)}", err)
        record_property(f"finalize_rel_l2_wbn{int(wbn)}", err_fin)
        assert err < OUT_BAR and err_fin < 2e-3, (err, err_fin)


def test_block_entry_unrouted_and_bad_ids(small_cases):
    """Routes marked -1 contribute nothing and an id out of range is skipped
    and reported, inside the fused block as in its parts; a token with no
    routes at all gets a zero output row."""
    w, raw, batch, tile, a1, a2 = small_cases[1]
    ids = batch["topk_ids"].copy()
    ids[::3, 0] = -1
    ids[1, 1] = w.E
    ids[2, :] = -1
    prep = Prepared(raw)
    parts, block = _block_vs_parts(prep, ids, batch, tile, a1, a2, True)
    assert parts[0] == -6 and block[0] == -6
    _check_block(parts, block)
    assert not block[2][0][2][2].any()


def test_fused_gemms_finish_while_other_work_holds_most_sms():
    """The one-launch GEMMs hand their units out by ticket to running CTAs
    only, so a GEMM2 unit never waits for a GEMM1 unit that no running CTA
    holds: with another stream's kernel holding all but 16 SMs for 1.5 s
    (longer than every bounded wait), the launch still completes on the SMs
    left, with a clean status and the split launches' rows bit for bit."""
    T, H, I, E, K, tile = 256, 1024, 512, 8, 8, 32
    w = _workload(T, H, I, E, K, "uniform", tile)
    raw, batch = inputs.make_layer(w), inputs.make_batch(w)
    prep = Prepared(raw)
    split = run_gpu(prep, batch, tile, 4.0, 1e-3, export=False)
    assert split["status"] == 0
    ids = _dev(batch["topk_ids"].astype(np.int32))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    r = B.route_permute(ids, E, tile, status=status)
    ws = B.alloc_workspace(T, K, E, H, I, tile, DEV)
    g1 = torch.tensor([4.0], dtype=torch.float32, device=DEV)
    g2 = torch.tensor([1e-3], dtype=torch.float32, device=DEV)
    B.experts_quantize(r, ws, x=bf16_dev(batch["x"]), a1_gscale=g1, T=T, H=H, I=I, E=E, K=K, status=status)
    P, _ = B.route_sizes(T, K, E, tile)
    rows = torch.zeros((P, H), dtype=torch.bfloat16, device=DEV)
    torch.cuda.synchronize()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    other = torch.cuda.Stream()
    B.selftest_occupy(sms - 16, 200 * 1024, 1_500_000_000, stream=other)
    time.sleep(0.1)  # the holding CTAs are resident before the GEMMs launch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    B.experts_gemms(prep.w, r, ws, rows, a2_gscale=g2, T=T, H=H, I=I, E=E, K=K, status=status)
    e1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert np.array_equal(bf16_host_f64(rows), split["rows"])
    # it finished on the 16 free SMs, before the other kernel let go of the rest
    assert e0.elapsed_time(e1) < 1300.0


def test_gemm2_rows_only_16_byte_aligned():
    """GEMM2's 128-row-tile epilogue writes whole 32-byte sectors when the rows
    buffer allows it and 16-byte pieces when it is only 16-byte aligned (the
    header's requirement): both give the same rows."""
    T, H, I, E, K = 70, 512, 256, 4, 4
    w = _workload(T, H, I, E, K, "zipf", 128)
    raw, batch = inputs.make_layer(w), inputs.make_batch(w)
    prep = Prepared(raw)
    ids = _dev(batch["topk_ids"].astype(np.int32))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    r = B.route_permute(ids, E, 128, status=status)
    ws = B.alloc_workspace(T, K, E, H, I, 128, DEV)
    g1 = torch.tensor([4.0], dtype=torch.float32, device=DEV)
    g2 = torch.tensor([1e-3], dtype=torch.float32, device=DEV)
    B.experts_quantize(r, ws, x=bf16_dev(batch["x"]), a1_gscale=g1, T=T, H=H, I=I, E=E, K=K, status=status)
    B.experts_gemm1(prep.w, r, ws, a2_gscale=g2, T=T, H=H, I=I, E=E, K=K, status=status)
    P, _ = B.route_sizes(T, K, E, 128)
    aligned = torch.zeros((P, H), dtype=torch.bfloat16, device=DEV)
    flat = torch.zeros(P * H + 64, dtype=torch.bfloat16, device=DEV)
    base = flat.data_ptr() % 32 // 2  # elements to the next 32-byte boundary
    off = flat[base + 8 : base + 8 + P * H].view(P, H)  # 16 bytes past it
    assert off.data_ptr() % 32 == 16
    B.experts_gemm2(prep.w, r, ws, aligned, T=T, H=H, I=I, E=E, K=K, status=status)
    B.experts_gemm2(prep.w, r, ws, off, T=T, H=H, I=I, E=E, K=K, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(aligned, off)


@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_gemm2_on_identical_operands(small_cases, idx, record_property):
    w, raw, batch, tile, a1, a2 = small_cases[idx]
    er = olayer.expert_rows(batch["x"], batch["topk_ids"], raw, a1, a2, return_intermediate=True)
    prep = Prepared(raw)
    P, _ = B.route_sizes(w.T, w.K, w.E, tile)
    first = run_gpu(prep, batch, tile, a1, a2, export=False)
    hq = oracle_hq_permuted(er, first["e2p"], P, w.I)
    got = run_gpu(prep, batch, tile, a1, a2, hq_override=hq, export=False)
    assert got["status"] == 0
    e2p = got["e2p"].reshape(-1)
    live = e2p >= 0
    rows = got["rows"][e2p[live]]
    want = er["rows_bf16"][live]
    err = rel_l2(rows, want)
    record_property("gemm2_rel_l2", err)
    assert err < GEMM2_BAR, f"rel-L2 {err:.3g}; gpu {finite_summary(rows)}"


@pytest.mark.parametrize("idx", range(len(SMALL)))
def test_gemm1_intermediate_and_end_to_end(small_cases, idx, record_property):
    w, raw, batch, tile, a1, a2 = small_cases[idx]
    ref = olayer.moe_layer(batch["x"], batch["topk_ids"], batch["topk_weights"], raw, a1, a2, raw["gamma"],
                           1e-6, tile, return_intermediate=True)
    prep = Prepared(raw)
    got = run_gpu(prep, batch, tile, a1, a2)
    assert got["status"] == 0
    assert np.array_equal(got["e2p"], ref["meta"]["expanded_to_permuted"])
    e2p = got["e2p"].reshape(-1)
    live = e2p >= 0
    # the requantized intermediate: scales and codes agree except at rare
    # rounding-boundary flips
    g_sf = got["hq_sf"][e2p[live]]
    g_codes = canon_codes(codecs.unpack_nibbles(got["hq_codes"][e2p[live]]))
    w_codes = canon_codes(ref["routes"]["hq_codes"][live])
    sf_match = np.mean(g_sf == ref["routes"]["hq_sf"][live])
    code_match = np.mean(g_codes == w_codes)
    assert sf_match > 0.99 and code_match > 0.99, (sf_match, code_match)
    err_rows = rel_l2(got["rows"][e2p[live]], ref["routes"]["rows_bf16"][live])
    assert err_rows < OUT_BAR, err_rows
    err = rel_l2(got["out"], ref["out"])
    for k, v in (("sf_match", sf_match), ("code_match", code_match), ("rows_rel_l2", err_rows), ("out_rel_l2", err)):
        record_property(k, float(v))
    assert err < OUT_BAR, f"out rel-L2 {err:.3g}; gpu {finite_summary(got['out'])}"


def _pairing_ids(T, layout):
    """topk_ids [T, 2] from (expert, first token, last token + 1) runs of each
    route slot: every token routes slot 0 and slot 1 to distinct experts."""
    ids = np.full((T, 2), -1, np.int32)
    for slot, runs in enumerate(layout):
        for e, t0, t1 in runs:
            ids[t0:t1, slot] = e
    return ids


@pytest.mark.parametrize("case", ["odd_and_even_tiles", "lone_tiles_only"])
def test_pair_gemm1_tile_pairing(case, record_property):
    """GEMM1 at 128-row tiles with H and 2I multiples of 256 runs as 256-row
    MMAs over a pair of consecutive route tiles of one expert. Expert tile
    counts 3 (a pair and a lone last tile), 2 (one pair, the second tile full
    or one row), 1 (a lone partial tile) and 0, against the oracle."""
    T, H, I, E = 300, 512, 256, 6
    w = _workload(T, H, I, E, 2, "uniform", 128)
    raw = inputs.make_layer(w)
    batch = inputs.make_batch(w)
    if case == "odd_and_even_tiles":
        # expert 0: 300 routes (3 tiles), expert 1: 256 (2 full tiles),
        # expert 2: 43 (1 tile), expert 5: 1; experts 3 and 4: none
        batch["topk_ids"] = _pairing_ids(T, [[(0, 0, 300)], [(1, 0, 256), (2, 256, 299), (5, 299, 300)]])
    else:
        # every expert has at most one tile: each pair's second tile is absent
        batch["topk_ids"] = _pairing_ids(T, [[(0, 0, 100), (1, 100, 200), (2, 200, 300)],
                                             [(3, 0, 120), (4, 120, 250), (5, 250, 300)]])
    a1, a2 = 4.0, 1e-3
    ref = olayer.moe_layer(batch["x"], batch["topk_ids"], batch["topk_weights"], raw, a1, a2, raw["gamma"],
                           1e-6, 128, return_intermediate=True)
    got = run_gpu(Prepared(raw), batch, 128, a1, a2)
    assert got["status"] == 0
    assert np.array_equal(got["e2p"], ref["meta"]["expanded_to_permuted"])
    e2p = got["e2p"].reshape(-1)
    live = e2p >= 0
    sf_match = np.mean(got["hq_sf"][e2p[live]] == ref["routes"]["hq_sf"][live])
    code_match = np.mean(canon_codes(codecs.unpack_nibbles(got["hq_codes"][e2p[live]])) ==
                         canon_codes(ref["routes"]["hq_codes"][live]))
    assert sf_match > 0.99 and code_match > 0.99, (sf_match, code_match)
    err_rows = rel_l2(got["rows"][e2p[live]], ref["routes"]["rows_bf16"][live])
    err = rel_l2(got["out"], ref["out"])
    for k, v in (("sf_match", sf_match), ("code_match", code_match), ("rows_rel_l2", err_rows), ("out_rel_l2", err)):
        record_property(k, float(v))
    assert err_rows < OUT_BAR and err < OUT_BAR, (err_rows, err)


def test_pair_gemm1_deterministic_and_capacity_fallback(record_property):
    """The pair-form GEMM1 gives the same bits on every run; a routing with
    more route tiles than its pair list holds (1024) takes the single-CTA
    GEMM1, and the two forms agree on the routes both compute (per route,
    through expanded_to_permuted), both against the oracle on sampled tokens."""
    H, I, E, K = 512, 256, 8, 8
    big = _workload(16384, H, I, E, K, "uniform", 128)  # 131,072 routes: 1024 + tiles
    raw = inputs.make_layer(big)
    batch = inputs.make_batch(big)
    P_big, tiles_big = B.route_sizes(big.T, K, E, 128)
    assert tiles_big > 1024
    small = {k: v[:4096] for k, v in batch.items()}  # 32,768 routes: pair form
    prep = Prepared(raw)
    a1, a2 = 4.0, 1e-3
    one = run_gpu(prep, small, 128, a1, a2)
    two = run_gpu(prep, small, 128, a1, a2)
    assert one["status"] == 0
    assert np.array_equal(one["hq_codes"], two["hq_codes"]) and np.array_equal(one["out"], two["out"])
    fall = run_gpu(prep, batch, 128, a1, a2)
    assert fall["status"] == 0
    # the same routes' intermediate rows in both layouts
    e_s = one["e2p"].reshape(-1)
    e_b = fall["e2p"].reshape(-1)[: e_s.size]
    live = e_s >= 0
    same_codes = np.mean(np.all(one["hq_codes"][e_s[live]] == fall["hq_codes"][e_b[live]], axis=1))
    record_property("pair_vs_single_identical_rows", float(same_codes))
    assert same_codes > 0.999
    # sampled tokens of each run against the oracle
    rng = np.random.default_rng(3)
    for got, bt in ((one, small), (fall, batch)):
        toks = np.sort(rng.choice(bt["topk_ids"].shape[0], 24, replace=False))
        sub = {k: v[toks] for k, v in bt.items()}
        ref = olayer.moe_layer(sub["x"], sub["topk_ids"], sub["topk_weights"], raw, a1, a2, raw["gamma"], 1e-6, 128)
        assert rel_l2(got["out"][toks], ref["out"]) < OUT_BAR


def test_pair_gemm1_without_routes():
    """No route at all (every id -1) at the pair form's shapes: no tile, no
    unit; the launch completes with a clean status and a zero output."""
    T, H, I, E = 40, 512, 256, 4
    w = _workload(T, H, I, E, 2, "uniform", 128)
    raw = inputs.make_layer(w)
    batch = inputs.make_batch(w)
    batch["topk_ids"] = np.full((T, 2), -1, np.int32)
    got = run_gpu(Prepared(raw), batch, 128, 4.0, 1e-3, export=False)
    assert got["status"] == 0
    assert not got["out"].any()


@pytest.mark.parametrize("idx", range(len(SMALL)))
@pytest.mark.parametrize("wbn", [True, False])
def test_fused_sums_of_squares_and_streaming_finalize(small_cases, idx, wbn, record_property):
    """moe_nvfp4_experts_sumsq: the rows equal moe_nvfp4_experts's bit for bit;
    every written row's 32-column sums of squares equal, to fp32 rounding,
    the fp64 sums of the stored bf16 values (gain-weighted in the weight-
    before-norm reading); the split GEMM2 / one-launch entry points write the
    same partials; moe_post_expert_finalize_sumsq equals the oracle's
    finalize of those rows (gamma ~ N(0, 1) so that the two readings differ)."""
    w, raw, batch, tile, a1, a2 = small_cases[idx]
    raw = dict(raw)
    raw["gamma"] = inputs._to_bf16_bits(np.random.default_rng(3).standard_normal(w.H))
    prep = Prepared(raw)
    T, K, E, H, I = w.T, w.K, w.E, w.H, w.I
    ids = _dev(batch["topk_ids"].astype(np.int32))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    r = B.route_permute(ids, E, tile, status=status)
    g1 = torch.tensor([a1], dtype=torch.float32, device=DEV)
    g2 = torch.tensor([a2], dtype=torch.float32, device=DEV)
    x = bf16_dev(batch["x"])
    plain, _ = B.nvfp4_experts(prep.w, r, x=x, a1_gscale=g1, a2_gscale=g2, T=T, H=H, I=I, E=E, K=K, status=status)
    rows, ss, ws = B.nvfp4_experts_sumsq(prep.w, r, x=x, a1_gscale=g1, a2_gscale=g2, T=T, H=H, I=I, E=E, K=K,
                                         gamma=prep.gamma, weight_before_norm=wbn, status=status)
    # the split entry points' partials
    rows2 = torch.zeros_like(rows)
    ss2 = torch.zeros_like(ss)
    B.experts_gemm2_sumsq(prep.w, r, ws, rows2, ss2, gamma=prep.gamma, weight_before_norm=wbn, T=T, H=H, I=I, E=E,
                          K=K, status=status)
    ss3 = torch.zeros_like(ss)
    B.experts_gemms_sumsq(prep.w, r, ws, torch.zeros_like(rows), ss3, a2_gscale=g2, gamma=prep.gamma,
                          weight_before_norm=wbn, T=T, H=H, I=I, E=E, K=K, status=status)
    tw = _dev(batch["topk_weights"])
    out = B.post_expert_finalize_sumsq(rows, ss, r.expanded_to_permuted, tw, prep.gamma, 1e-6, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    e2p = r.expanded_to_permuted.cpu().numpy()
    live = e2p.reshape(-1)
    live = live[live >= 0]
    assert torch.equal(rows[live], plain[live])
    got_rows = bf16_host_f64(rows)[live]
    gain = 1.0 + codecs.bf16_bits_to_f64(raw["gamma"]) if wbn else np.ones(H)
    want_ss = ((got_rows * gain[None, :]) ** 2).reshape(len(live), H // 32, 32).sum(axis=-1)
    got_ss = ss.cpu().numpy().astype(np.float64)[live]
    assert np.allclose(got_ss, want_ss, rtol=1e-5, atol=0), np.max(np.abs(got_ss / want_ss - 1))
    assert np.array_equal(ss2.cpu().numpy()[live], ss.cpu().numpy()[live])
    assert np.array_equal(ss3.cpu().numpy()[live], ss.cpu().numpy()[live])
    want = olayer.finalize(bf16_host_f64(rows), e2p, batch["topk_weights"], raw["gamma"], 1e-6, wbn)
    got = bf16_host_f64(out)
    err = rel_l2(got, want["out"])
    record_property("finalize_rel_l2", err)
    assert err < 2e-3
    rms = np.sqrt(np.mean(want["out"] ** 2))
    assert (np.abs(got - want["out_bf16"]) <= np.abs(want["out_bf16"]) * 2.0**-7 + 1e-4 * rms).all()


def test_weight_before_norm_reading_end_to_end(small_cases):
    w, raw, batch, tile, a1, a2 = small_cases[1]
    raw = dict(raw)
    raw["gamma"] = inputs._to_bf16_bits(np.random.default_rng(0).standard_normal(w.H))
    prep = Prepared(raw)
    for wbn in (True, False):
        ref = olayer.moe_layer(batch["x"], batch["topk_ids"], batch["topk_weights"], raw, a1, a2, raw["gamma"],
                               1e-6, tile, weight_before_norm=wbn)
        got = run_gpu(prep, batch, tile, a1, a2, wbn=wbn, export=False)
        assert rel_l2(got["out"], ref["out"]) < OUT_BAR


def test_determinism(small_cases):
    w, raw, batch, tile, a1, a2 = small_cases[2]
    prep = Prepared(raw)
    a = run_gpu(prep, batch, tile, a1, a2)
    b = run_gpu(prep, batch, tile, a1, a2)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["hq_codes"], b["hq_codes"])


def test_unrouted_routes_contribute_nothing(small_cases):
    w, raw, batch, tile, a1, a2 = small_cases[1]
    batch = dict(batch)
    ids = batch["topk_ids"].copy()
    ids[::2, 0] = -1
    batch["topk_ids"] = ids
    ref = olayer.moe_layer(batch["x"], ids, batch["topk_weights"], raw, a1, a2, raw["gamma"], 1e-6, tile)
    got = run_gpu(Prepared(raw), batch, tile, a1, a2, export=False)
    assert rel_l2(got["out"], ref["out"]) < OUT_BAR


# ---------------------------------------------------------------------------
# Full-size layer (H = 5120, I = 2048, E = 128): decode, TP slices, prefill
# ---------------------------------------------------------------------------
@pytest.fixture(scope="module")
def full():
    raw = layer_for("decode_b8")
    return raw, Prepared(raw)


def test_decode_b8_full_size(full, record_property):
    raw, prep = full
    w = inputs.WORKLOADS["decode_b8"]
    a1, a2 = inputs.global_scales(w)
    batch = inputs.make_batch(w)
    ref = olayer.moe_layer(batch["x"], batch["topk_ids"], batch["topk_weights"], raw, a1, a2, raw["gamma"],
                           1e-6, w.tile_m, return_intermediate=True)
    got = run_gpu(prep, batch, w.tile_m, a1, a2)
    assert got["status"] == 0
    e2p = got["e2p"].reshape(-1)
    err_rows = rel_l2(got["rows"][e2p], ref["routes"]["rows_bf16"])
    err = rel_l2(got["out"], ref["out"])
    record_property("out_rel_l2", err)
    record_property("rows_rel_l2", err_rows)
    assert err < OUT_BAR and err_rows < OUT_BAR, (err, err_rows)
    # GEMM2 alone on the oracle's intermediate
    P, _ = B.route_sizes(w.T, w.K, w.E, w.tile_m)
    hq = oracle_hq_permuted(ref["routes"], got["e2p"], P, w.I)
    same = run_gpu(prep, batch, w.tile_m, a1, a2, hq_override=hq, export=False)
    err2 = rel_l2(same["rows"][e2p], ref["routes"]["rows_bf16"])
    record_property("gemm2_rel_l2", err2)
    assert err2 < GEMM2_BAR


@pytest.mark.parametrize("name", ["decode_b8", "decode_b64_zipf"])
def test_routed_entry_full_size(full, name):
    """At full size (H = 5120, I = 2048, E = 128, K = 8) the routing inside
    the input quantizer gives moe_route_permute's metadata and the split
    path's GEMM2 rows bit for bit."""
    raw, prep = full
    w = inputs.WORKLOADS[name]
    a1, a2 = inputs.global_scales(w)
    batch = inputs.make_batch(w)
    assert B.routed_experts_kernels(w.T, w.K, w.E, w.tile_m) == 2
    (st_a, r_a, rows_a), (st_b, r_b, outs) = _routed_vs_split(prep, batch["topk_ids"], batch["x"], w.tile_m, a1, a2)
    assert st_a == 0 and st_b == 0
    for f in _ROUTE_FIELDS:
        assert torch.equal(getattr(r_a, f), getattr(r_b, f)), f
    live = r_a.expanded_to_permuted.reshape(-1)
    for rows_b in outs:
        assert torch.equal(rows_b[live], rows_a[live])


@pytest.mark.parametrize("name", ["decode_b8", "decode_b64_zipf"])
def test_block_entry_full_size(full, name):
    """At full size the whole block in 4 kernels (routing, the quantizer,
    both GEMMs with the sums of squares in one launch, the finalize) equals
    its parts bit for bit."""
    raw, prep = full
    w = inputs.WORKLOADS[name]
    a1, a2 = inputs.global_scales(w)
    batch = inputs.make_batch(w)
    assert B.moe_block_kernels(w.T, w.K, w.E, w.tile_m) == 4
    parts, block = _block_vs_parts(prep, batch["topk_ids"], batch, w.tile_m, a1, a2, True)
    assert parts[0] == 0
    _check_block(parts, block)


def test_expert_tp_identity(full, record_property):
    """The expert_tp page: the GEMM2 rows of the tp = 8 intermediate slices
    (I' = 256) are K-partials whose sum is the full-width row.

    Exact part: with I' % 16 == 0 every requant block lies inside a slice, so
    each slice's quantized intermediate (GEMM1 + SwiGLU + requant on the
    slice's own prepared weights) equals, bit for bit, the same columns of
    the full-width run's.

    Rows part: the slices run one after another on this GPU and their bf16
    partial rows are summed in fp32 with one bf16 rounding (the page's
    probe_rel_l2). Each partial and the full-width row were rounded to bf16
    once, so the difference is a sum of independent roundings of relative
    size at most 2^-9 (RMS 2^-9/sqrt(3)); the bar is three times the RMS this
    predicts from the rows themselves, and never above 1e-2."""
    raw, prep = full
    w = inputs.WORKLOADS["tp8_slice_b32"]
    a1, a2 = inputs.global_scales(w)
    batch = inputs.make_batch(w)
    full_run = run_gpu(prep, batch, w.tile_m, a1, a2)
    e2p = full_run["e2p"].reshape(-1)
    s = w.I // w.tp
    acc = np.zeros((len(e2p), w.H), dtype=np.float32)
    sq_parts = 0.0
    for r in range(w.tp):
        sl = olayout.raw_slice(raw, r, w.tp)
        part = run_gpu(Prepared(sl), batch, w.tile_m, a1, a2)
        assert np.array_equal(part["e2p"], full_run["e2p"])
        assert np.array_equal(part["hq_codes"][e2p], full_run["hq_codes"][e2p][:, r * s // 2:(r + 1) * s // 2])
        assert np.array_equal(part["hq_sf"][e2p], full_run["hq_sf"][e2p][:, r * s // 16:(r + 1) * s // 16])
        rows_r = part["rows"][e2p]
        acc += rows_r.astype(np.float32)
        sq_parts += float(np.sum(rows_r ** 2))
        torch.cuda.empty_cache()
    summed = codecs.round_to_bf16(acc.astype(np.float64))
    want = full_run["rows"][e2p]
    sq_full = float(np.sum(want ** 2))
    predicted = np.sqrt((sq_parts + 2.0 * sq_full) * 2.0**-18 / 3.0 / sq_full)
    err = rel_l2(summed, want)
    record_property("tp_sum_rel_l2", err)
    record_property("tp_predicted_rms", float(predicted))
    assert err < min(3.0 * predicted, OUT_BAR), (err, predicted)
    pick = np.array([0, 31])
    ref = olayer.expert_rows(batch["x"][pick], batch["topk_ids"][pick], raw, a1, a2)
    mask = np.isin(np.arange(w.T * w.K) // w.K, pick)
    assert rel_l2(summed[mask], ref["rows_bf16"]) < OUT_BAR


def _oracle_out_for_tokens(er, e2p_routes, batch, tokens, gamma_bits):
    """The oracle's finalize of the given tokens from route-indexed rows
    (er from expert_rows over a batch whose routes are the tokens' routes)."""
    K = batch["topk_ids"].shape[1]
    idx = np.where(e2p_routes >= 0, np.arange(e2p_routes.size).reshape(e2p_routes.shape), -1)
    return olayer.finalize(er["rows_bf16"], idx, batch["topk_weights"][tokens], gamma_bits, 1e-6)["out"]


def _gemm2_on_oracle_hq(prep, batch, tile, a1, a2, gpu_run, er, routes):
    """GEMM2 rows after importing the oracle's quantized intermediate for the
    given routes (route index j -> er row n) into the GPU's own intermediate."""
    e2p = gpu_run["e2p"].reshape(-1)
    codes, sf = gpu_run["hq_codes"].copy(), gpu_run["hq_sf"].copy()
    rows_p = e2p[routes]
    codes[rows_p] = codecs.pack_nibbles(er["hq_codes"])
    sf[rows_p] = er["hq_sf"]
    return run_gpu(prep, batch, tile, a1, a2, hq_override=(codes, sf), export=False)


def test_decode_b64_zipf_full_size(full, record_property):
    """decode b = 64 with Zipf routing at full size, every token: the
    metadata bit-exact, the GEMM2 rows of all 512 routes on the oracle's
    quantized intermediate within 2e-3, the rows end to end and the output
    of all 64 tokens within 1e-2."""
    raw, prep = full
    w = inputs.WORKLOADS["decode_b64_zipf"]
    a1, a2 = inputs.global_scales(w)
    batch = inputs.make_batch(w)
    ref = olayer.moe_layer(batch["x"], batch["topk_ids"], batch["topk_weights"], raw, a1, a2, raw["gamma"],
                           1e-6, w.tile_m, return_intermediate=True)
    got = run_gpu(prep, batch, w.tile_m, a1, a2)
    assert got["status"] == 0
    assert np.array_equal(got["e2p"], ref["meta"]["expanded_to_permuted"])
    assert np.array_equal(got["p2t"], ref["meta"]["permuted_to_token"])
    e2p = got["e2p"].reshape(-1)
    err_rows = rel_l2(got["rows"][e2p], ref["routes"]["rows_bf16"])
    err = rel_l2(got["out"], ref["out"])
    same = _gemm2_on_oracle_hq(prep, batch, w.tile_m, a1, a2, got,
                               {"hq_codes": ref["routes"]["hq_codes"], "hq_sf": ref["routes"]["hq_sf"]},
                               np.arange(w.T * w.K))
    err2 = rel_l2(same["rows"][e2p], ref["routes"]["rows_bf16"])
    for k, v in (("out_rel_l2", err), ("rows_rel_l2", err_rows), ("gemm2_rel_l2", err2)):
        record_property(k, v)
    assert err < OUT_BAR and err_rows < OUT_BAR and err2 < GEMM2_BAR, (err, err_rows, err2)


def _pick_prefill_experts(ids, E):
    """Whole experts to hold to the oracle at prefill: the hottest (most route
    tiles), one of median size, the highest-index expert with routes, and one
    whose routes fill a single partial tile (fewest routes otherwise)."""
    counts = np.bincount(ids[ids >= 0].ravel(), minlength=E)
    nz = np.nonzero(counts)[0]
    hot = int(np.argmax(counts))
    med = int(nz[np.argsort(counts[nz], kind="stable")[len(nz) // 2]])
    top = int(nz.max())
    single = [int(e) for e in nz if counts[e] < 128 and e not in (hot, med, top)]
    part = single[0] if single else int(nz[np.argmin(counts[nz])])
    return [hot, med, top, part], counts


def test_prefill_t8192_whole_experts_and_256_tokens(full, record_property):
    """Prefill T = 8192 with Zipf routing and 128-row route tiles (about 570
    live tiles, the persistent grids' rings wrapping over thousands of
    units): every route of four whole experts -- the hottest (58 tiles), a
    median one, the highest-index one and one whose routes fill a single
    partial tile -- and the output of 256 tokens spread over the batch,
    against the oracle.

    GEMM2 rows of those experts on the oracle's quantized intermediate within
    2e-3 (the flashinfer_ops page's identical-operand comparison), their
    requantized intermediate code for code and scale for scale (> 0.99; flips
    only at rounding boundaries), their rows end to end and the 256 tokens'
    output within 1e-2 (rel-L2 with fp64 norms, as the expert_tp page's
    probe_rel_l2); the routing metadata bit-exact."""
    from oracle import routing as orouting

    raw, prep = full
    w = inputs.WORKLOADS["prefill_t8192_zipf"]
    a1, a2 = inputs.global_scales(w)
    batch = inputs.make_batch(w)
    ids = batch["topk_ids"]
    experts, counts = _pick_prefill_experts(ids, w.E)
    got = run_gpu(prep, batch, w.tile_m, a1, a2)
    assert got["status"] == 0
    meta = orouting.route_metadata(ids, w.E, w.tile_m)
    assert np.array_equal(got["e2p"], meta["expanded_to_permuted"])
    assert np.array_equal(got["p2t"], meta["permuted_to_token"])
    e2p = got["e2p"].reshape(-1)

    # every route of the chosen experts
    routes = np.nonzero(np.isin(ids.reshape(-1), experts))[0]
    tok = np.unique(routes // w.K)
    sub_ids = np.where(np.isin(ids[tok], experts), ids[tok], -1).astype(np.int32)
    er = olayer.expert_rows(batch["x"][tok], sub_ids, raw, a1, a2, return_intermediate=True)
    # the live routes of the sub-batch, in order, are `routes` (both
    # token-major, then k, over ascending tokens)
    live = sub_ids.reshape(-1) >= 0
    er_live = {k: er[k][live] for k in ("rows_bf16", "hq_codes", "hq_sf")}
    gpu_rows = got["rows"][e2p[routes]]
    g_sf = got["hq_sf"][e2p[routes]]
    g_codes = canon_codes(codecs.unpack_nibbles(got["hq_codes"][e2p[routes]]))
    sf_match = float(np.mean(g_sf == er_live["hq_sf"]))
    code_match = float(np.mean(g_codes == canon_codes(er_live["hq_codes"])))
    err_rows = rel_l2(gpu_rows, er_live["rows_bf16"])
    same = _gemm2_on_oracle_hq(prep, batch, w.tile_m, a1, a2, got, er_live, routes)
    assert same["status"] == 0
    ids_flat = ids.reshape(-1)[routes]
    per_expert = {}
    for e in experts:
        m = ids_flat == e
        per_expert[e] = rel_l2(same["rows"][e2p[routes[m]]], er_live["rows_bf16"][m])
        record_property(f"gemm2_rel_l2_e{e}_n{int(counts[e])}", per_expert[e])
    err2 = rel_l2(same["rows"][e2p[routes]], er_live["rows_bf16"])

    # 256 tokens spread over the batch, all of their routes
    pick = np.linspace(0, w.T - 1, 256).astype(np.int64)
    er_t = olayer.expert_rows(batch["x"][pick], ids[pick], raw, a1, a2)
    want_out = _oracle_out_for_tokens(er_t, ids[pick], batch, pick, raw["gamma"])
    err_out = rel_l2(got["out"][pick], want_out)
    err_rows_t = rel_l2(got["rows"][e2p.reshape(w.T, w.K)[pick].reshape(-1)], er_t["rows_bf16"])
    for k, v in (("sf_match", sf_match), ("code_match", code_match), ("rows_rel_l2", err_rows),
                 ("gemm2_rel_l2", err2), ("out_rel_l2_256", err_out), ("rows_rel_l2_256", err_rows_t)):
        record_property(k, v)
    assert sf_match > 0.99 and code_match > 0.99, (sf_match, code_match)
    assert max(per_expert.values()) < GEMM2_BAR and err2 < GEMM2_BAR, per_expert
    assert err_rows < OUT_BAR and err_rows_t < OUT_BAR and err_out < OUT_BAR, (err_rows, err_rows_t, err_out)


def test_graphed_serving_path_matches_eager():
    """NvFp4MoE.replay (the step captured once as a CUDA graph on static
    buffers) gives the eager forward's output bit for bit, for two batches
    written into the same static inputs."""
    from nvfp4_mixture_experts_route_gb300.layer import NvFp4MoE

    w = inputs.WORKLOADS["tiny_t4"]
    raw = inputs.make_layer(w)
    moe = NvFp4MoE(raw, 1.0, 1.0, raw["gamma"], tile_m=w.tile_m)
    gb = moe.graph_buffers(w.T, w.K)
    for seed in (0, 1):
        batch = inputs.make_batch(w, seed=seed)
        x = bf16_dev(batch["x"])
        ids = torch.from_numpy(batch["topk_ids"]).to("cuda")
        tw = torch.from_numpy(batch["topk_weights"]).to("cuda")
        eager = moe.forward(x, ids, tw)[0].clone()
        gb["x"].copy_(x)
        gb["topk_ids"].copy_(ids)
        gb["topk_weights"].copy_(tw)
        got = moe.replay(w.T, w.K)
        torch.cuda.synchronize()
        assert torch.equal(got, eager)


def test_zero_copy_serving_step_matches_device_step():
    """The zero-copy serving step (its kernels read x, topk_ids and
    topk_weights from pinned host memory and the finalize writes the output
    there) gives the device-buffer step's output bit for bit, for two batches
    written into the same pinned inputs between replays of one graph."""
    from nvfp4_mixture_experts_route_gb300.layer import NvFp4MoE

    w = inputs.WORKLOADS["tiny_t4"]
    raw = inputs.make_layer(w)
    moe = NvFp4MoE(raw, 1.0, 1.0, raw["gamma"], tile_m=w.tile_m)
    hb = moe.host_buffers(w.T, w.K)
    assert B.device_reads_host(hb["host_inputs"]) and B.device_reads_host(hb["host_out"])
    assert not B.device_reads_host(torch.zeros(16, dtype=torch.uint8))  # pageable: not registered
    assert moe.zero_copy(w.T, w.K)
    offs, _ = moe.input_layout(w.T, w.K)
    for seed in (0, 1):
        batch = inputs.make_batch(w, seed=seed)
        x = bf16_dev(batch["x"])
        ids = torch.from_numpy(batch["topk_ids"]).to("cuda")
        tw = torch.from_numpy(batch["topk_weights"]).to("cuda")
        want = moe.forward(x, ids, tw)[0].cpu()
        hi = hb["host_inputs"]
        hi[offs["x"]:offs["x"] + x.numel() * 2].copy_(torch.from_numpy(batch["x"].view(np.uint8).reshape(-1)))
        hi[offs["topk_ids"]:offs["topk_ids"] + ids.numel() * 4].copy_(
            torch.from_numpy(batch["topk_ids"].view(np.uint8).reshape(-1)))
        hi[offs["topk_weights"]:offs["topk_weights"] + tw.numel() * 4].copy_(
            torch.from_numpy(batch["topk_weights"].view(np.uint8).reshape(-1)))
        got = moe.replay_host(w.T, w.K)
        torch.cuda.synchronize()
        assert torch.equal(got, want)


@pytest.mark.parametrize("T,tile", [(300, 128), (4, 32)])
def test_pipelined_serving_call_matches_eager(T, tile):
    """NvFp4MoE.submit_host on alternating slots (copy in, step graph and
    copy out on three streams) gives each step the eager forward's output of
    that step's batch bit for bit, with six different batches in flight two
    at a time and every slot refilled only after its previous step's event."""
    import dataclasses

    from nvfp4_mixture_experts_route_gb300.layer import NvFp4MoE

    w = dataclasses.replace(inputs.WORKLOADS["tiny_t4"], T=T, tile_m=tile)
    raw = inputs.make_layer(w)
    moe = NvFp4MoE(raw, 1.0, 1.0, raw["gamma"], tile_m=w.tile_m)
    offs, _ = moe.input_layout(w.T, w.K)
    slots = moe.host_pipeline(w.T, w.K)["slots"]
    batches = [inputs.make_batch(w, seed=seed) for seed in range(6)]
    want = []
    for batch in batches:
        x = bf16_dev(batch["x"])
        ids = torch.from_numpy(batch["topk_ids"]).to("cuda")
        tw = torch.from_numpy(batch["topk_weights"]).to("cuda")
        want.append(moe.forward(x, ids, tw)[0].cpu())
    got, events = [None] * len(batches), []
    moe.pipeline_begin(w.T, w.K)
    for i, batch in enumerate(batches):
        slot = slots[i % 2]
        if i >= 2:
            events[i - 2].synchronize()
            got[i - 2] = slot["host_out"].clone()
        hi = slot["host_inputs"]
        hi[offs["x"]:offs["x"] + w.T * w.H * 2].copy_(torch.from_numpy(batch["x"].view(np.uint8).reshape(-1)))
        hi[offs["topk_ids"]:offs["topk_ids"] + w.T * w.K * 4].copy_(
            torch.from_numpy(batch["topk_ids"].view(np.uint8).reshape(-1)))
        hi[offs["topk_weights"]:offs["topk_weights"] + w.T * w.K * 4].copy_(
            torch.from_numpy(batch["topk_weights"].view(np.uint8).reshape(-1)))
        events.append(moe.submit_host(w.T, w.K, i % 2))
    moe.pipeline_join(w.T, w.K)
    torch.cuda.synchronize()
    for i in (len(batches) - 2, len(batches) - 1):
        got[i] = slots[i % 2]["host_out"].clone()
    for i in range(len(batches)):
        assert torch.equal(got[i], want[i]), i


@pytest.mark.parametrize("name", ["decode_b8", "decode_b64_zipf", "prefill_t8192_zipf"])
def test_timed_launch_path_matches_split_path(full, name):
    """The routed body then the plain finalize (for decode tiles the routing
    inside the quantizer and one persistent launch of both GEMMs, for
    prefill tiles the routing kernels, the quantizer and two GEMM launches,
    each a programmatic dependent that prefetches weights; eager and as a
    graph replay) gives exactly the split entry points' output at full size;
    those are held to the oracle above; so does the host-staged serving call
    (its copies inside the graph). moe_experts_gemms at that size gives the
    split GEMM2 rows too. The whole-block call (bench.py's step at decode
    sizes) gives the same rows and the output up to the order of fp32
    sums."""
    from nvfp4_mixture_experts_route_gb300.layer import NvFp4MoE

    raw, prep = full
    w = inputs.WORKLOADS[name]
    a1, a2 = inputs.global_scales(w)
    batch = inputs.make_batch(w)
    split = run_gpu(prep, batch, w.tile_m, a1, a2, export=False)
    assert split["status"] == 0
    moe = NvFp4MoE(raw, a1, a2, raw["gamma"], tile_m=w.tile_m, fused_norm=False)
    x = bf16_dev(batch["x"])
    ids = torch.from_numpy(batch["topk_ids"]).to(DEV)
    tw = torch.from_numpy(batch["topk_weights"]).to(DEV)
    eager = bf16_host_f64(moe.forward(x, ids, tw)[0])
    assert np.array_equal(eager, split["out"])
    gb = moe.graph_buffers(w.T, w.K)
    gb["x"].copy_(x)
    gb["topk_ids"].copy_(ids)
    gb["topk_weights"].copy_(tw)
    graphed = bf16_host_f64(moe.replay(w.T, w.K))
    assert np.array_equal(graphed, split["out"])
    # the serving call with its host copies inside the graph
    hb = moe.host_buffers(w.T, w.K)
    hb["host_inputs"].copy_(gb["inputs"].cpu())
    host = moe.replay_host(w.T, w.K)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host_f64(host), split["out"])
    # the pipelined serving call (bench.py's e2e form for larger steps)
    for slot in moe.host_pipeline(w.T, w.K)["slots"]:
        slot["host_inputs"].copy_(hb["host_inputs"])
    moe.pipeline_begin(w.T, w.K)
    for i in range(3):
        moe.submit_host(w.T, w.K, i % 2)
    moe.pipeline_join(w.T, w.K)
    torch.cuda.synchronize()
    for slot in moe.host_pipeline(w.T, w.K)["slots"]:
        assert np.array_equal(bf16_host_f64(slot["host_out"]), split["out"])
    status, fused = _fused_rows(prep, batch, w.tile_m, a1, a2, calls=1)
    assert status == 0 and np.array_equal(fused[0], split["rows"])
    # The layer through the whole-block call (the norm's sums of squares
    # fused into GEMM2, the finalize from them: what bench.py times at decode
    # sizes): the same rows bit for bit; the output equal up to the order of
    # the fp32 sums; its graph replays equal its eager call; the layer's
    # default picks it exactly for route tiles of at most 64 rows.
    del moe
    torch.cuda.empty_cache()
    fn = NvFp4MoE(raw, a1, a2, raw["gamma"], tile_m=w.tile_m, fused_norm=True)
    got, bufs = fn.forward(x, ids, tw)
    got = bf16_host_f64(got)
    torch.cuda.synchronize()
    assert int(bufs["status"].item()) == 0
    P, _ = B.route_sizes(w.T, w.K, w.E, w.tile_m)
    live = split["e2p"].reshape(-1)
    live = live[live >= 0]
    assert np.array_equal(bf16_host_f64(bufs["rows"])[live], split["rows"][live])
    assert rel_l2(got, split["out"]) < 1e-3
    assert (np.abs(got - split["out"]) <= np.abs(split["out"]) * 2.0**-7 + 1e-3 * np.sqrt(np.mean(split["out"] ** 2))).all()
    gb = fn.graph_buffers(w.T, w.K)
    gb["x"].copy_(x)
    gb["topk_ids"].copy_(ids)
    gb["topk_weights"].copy_(tw)
    assert np.array_equal(bf16_host_f64(fn.replay(w.T, w.K)), got)
    hb = fn.host_buffers(w.T, w.K)
    hb["host_inputs"].copy_(gb["inputs"].cpu())
    assert fn.zero_copy(w.T, w.K) == (B.experts_kernels(w.tile_m) == 2)
    host = fn.replay_host(w.T, w.K)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host_f64(host), got)
    fn.fused_norm = None
    auto = bf16_host_f64(fn.forward(x, ids, tw)[0])
    assert np.array_equal(auto, got if B.experts_kernels(w.tile_m) == 2 else split["out"])
