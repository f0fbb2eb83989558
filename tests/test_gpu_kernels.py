"""GPU parity of the routing, input-quantization, weight-preparation and
finalize kernels against the CPU oracle, through the C ABI."""
import dataclasses

import numpy as np
import pytest
import torch

from oracle import codecs, layer as olayer, layout as olayout, quant as oquant, routing as orouting
from nvfp4_mixture_experts_route_gb300 import binding as B
from nvfp4_mixture_experts_route_gb300 import inputs

from _util import bf16_dev, bf16_host_f64, canon_packed, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _route_gpu(ids_np, E, tile, status=None):
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).to(DEV)
    r = B.route_permute(ids, E, tile, status=status)
    torch.cuda.synchronize()
    return r


def _route_np(r):
    return {
        "expert_counts": r.expert_counts.cpu().numpy(),
        "expert_offsets": r.expert_offsets.cpu().numpy(),
        "expanded_to_permuted": r.expanded_to_permuted.cpu().numpy(),
        "permuted_to_token": r.permuted_to_token.cpu().numpy(),
        "tile_expert": r.tile_expert.cpu().numpy(),
        "tile_row_limit": r.tile_row_limit.cpu().numpy(),
        "totals": r.totals.cpu().numpy(),
    }


def _assert_route_equal(got, want):
    P = len(want["permuted_to_token"])
    MT = len(want["tile_expert"])
    for k in ("expert_counts", "expert_offsets", "expanded_to_permuted", "totals"):
        assert np.array_equal(got[k], want[k]), k
    assert np.array_equal(got["permuted_to_token"][:P], want["permuted_to_token"])
    assert np.array_equal(got["tile_expert"][:MT], want["tile_expert"])
    assert np.array_equal(got["tile_row_limit"][:MT], want["tile_row_limit"])


ROUTE_CASES = [
    ("tiny_t4", 0), ("decode_b8", 0), ("decode_b64_zipf", 0), ("tp8_slice_b32", 0),
    ("prefill_t8192_zipf", 0), ("decode_b8", 1),
]


@pytest.mark.parametrize("name,seed", ROUTE_CASES)
@pytest.mark.parametrize("tile", [32, 128])
def test_route_permute_bit_exact(name, seed, tile):
    w = inputs.WORKLOADS[name]
    ids = inputs.make_batch(w, seed=seed)["topk_ids"]
    want = orouting.route_metadata(ids, w.E, tile)
    got = _route_np(_route_gpu(ids, w.E, tile))
    _assert_route_equal(got, want)


@pytest.mark.parametrize("tile", [32, 64, 256])
def test_route_permute_edge_cases(tile):
    rng = np.random.default_rng(3)
    cases = [
        np.full((40, 1), 5, np.int32),                 # all routes on one expert
        np.array([[3, 0]], np.int32),                  # one token
        -np.ones((7, 3), np.int32),                    # nothing routed
        inputs.draw_topk(rng, 1000, 1024, 8, "zipf"),  # E = 1024, many tiles
        inputs.draw_topk(rng, 77, 16, 8, "uniform"),   # ragged
    ]
    mixed = inputs.draw_topk(rng, 50, 32, 4, "uniform")
    mixed[::3, 1] = -1
    cases.append(mixed)
    for ids in cases:
        E = max(8, int(ids.max()) + 1)
        E = 1024 if ids.shape == (1000, 8) else E
        want = orouting.route_metadata(ids, E, tile)
        _assert_route_equal(_route_np(_route_gpu(ids, E, tile)), want)


@pytest.mark.parametrize("tile", [32, 128])
def test_route_permute_many_routes_edge_cases(tile):
    """Route counts that take the segmented (count / scan / scatter) path:
    exactly two segments, a short last segment, everything on one expert,
    nothing routed, E = 1024 with ragged segments, and -1 holes."""
    rng = np.random.default_rng(11)
    cases = [
        (inputs.draw_topk(rng, 512, 64, 8, "uniform"), 64),     # R = 4096: two segments
        (inputs.draw_topk(rng, 1531, 128, 8, "zipf"), 128),     # R = 12248: short tail
        (np.full((6000, 1), 7, np.int32), 8),                   # one expert takes all
        (-np.ones((4100, 2), np.int32), 16),                    # nothing routed
        (inputs.draw_topk(rng, 2047, 1024, 3, "zipf"), 1024),   # E = 1024, ragged
    ]
    holes = inputs.draw_topk(rng, 3000, 32, 4, "uniform")
    holes[::5, 2] = -1
    cases.append((holes, 32))
    for ids, E in cases:
        want = orouting.route_metadata(ids, E, tile)
        _assert_route_equal(_route_np(_route_gpu(ids, E, tile)), want)


def test_route_permute_many_routes_refuses_bad_ids():
    ids = inputs.draw_topk(np.random.default_rng(12), 2048, 64, 4, "uniform")
    ids[1500, 3] = 64
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    _route_gpu(ids, 64, 32, status=status)
    assert int(status.item()) == -6


def test_route_permute_refuses_bad_ids():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    _route_gpu(np.array([[0, 8], [1, 2]], np.int32), 8, 32, status=status)
    assert int(status.item()) == -6
    status.zero_()
    _route_gpu(np.array([[-3, 1]], np.int32), 8, 32, status=status)
    assert int(status.item()) == -6


def test_route_permute_empty():
    r = B.route_permute(torch.empty((0, 8), dtype=torch.int32, device=DEV), 128, 32)
    torch.cuda.synchronize()
    assert r.totals.cpu().tolist() == [0, 0]
    assert not r.expert_counts.cpu().numpy().any()


def test_route_permute_deterministic():
    w = inputs.WORKLOADS["prefill_t8192_zipf"]
    ids = inputs.make_batch(w)["topk_ids"]
    a = _route_np(_route_gpu(ids, w.E, 128))
    b = _route_np(_route_gpu(ids, w.E, 128))
    for k in a:
        assert np.array_equal(a[k], b[k])


# ---------------------------------------------------------------------------
# Step a1: quantization into permuted order
# ---------------------------------------------------------------------------
def _quant_case(T, H, E, K, tile, g, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    x = inputs._to_bf16_bits(rng.standard_normal((T, H)) * scale)
    ids = inputs.draw_topk(rng, T, E, K, "uniform")
    r = _route_gpu(ids, E, tile)
    I = 128
    ws = B.alloc_workspace(T, K, E, H, I, tile, DEV)
    g_dev = torch.tensor([g], dtype=torch.float32, device=DEV)
    B.experts_quantize(r, ws, x=bf16_dev(x), a1_gscale=g_dev, T=T, H=H, I=I, E=E, K=K)
    codes, scales = B.experts_export(0, ws, T=T, H=H, I=I, E=E, K=K, tile_m=tile)
    torch.cuda.synchronize()
    return x, r, codes.cpu().numpy(), scales.cpu().numpy(), ws


@pytest.mark.parametrize("T,H,E,K,tile,g,scale", [
    (4, 256, 8, 2, 32, 1.0, 1.0),
    (8, 5120, 128, 8, 32, 618.8201293945312, 1.0),
    (37, 1024, 16, 4, 64, 3.0, 100.0),        # ragged, several tiles, saturation
    (300, 512, 8, 8, 256, 2.0, 1.0),          # two scale atoms per tile
    (256, 5120, 16, 8, 128, 3.0, 1.0),        # full row width: ten 32-block chunks per token
    (16, 256, 4, 2, 128, 1e-3, 1e-5),         # scales in the e4m3 subnormals / zero
    # prefill-sized batches: many tokens per route tile, a ragged last chunk,
    # K < 8, the decode tile size, subnormal scales
    (1100, 5120, 128, 8, 128, 618.8201293945312, 1.0),
    (1030, 1152, 16, 3, 32, 3.0, 100.0),
    (2048, 256, 8, 8, 256, 1e-3, 1e-5),
])
def test_quantize_permute_bit_exact(T, H, E, K, tile, g, scale):
    x, r, codes, scales, _ = _quant_case(T, H, E, K, tile, g, scale=scale)
    want_q, want_sf = oquant.quantize_blocks(codecs.bf16_bits_to_f64(x).astype(np.float32), g)
    want_packed = codecs.pack_nibbles(want_q)
    p2t = r.permuted_to_token.cpu().numpy()
    total = int(r.totals[1].item())
    live = np.nonzero(p2t[:total] >= 0)[0]
    pad = np.nonzero(p2t[:total] < 0)[0]
    assert np.array_equal(scales[live], want_sf[p2t[live]])
    assert np.array_equal(canon_packed(codes[live]), canon_packed(want_packed[p2t[live]]))
    assert not scales[pad].any()  # padding rows: zero scales (their codes are not written)


@pytest.mark.parametrize("T", [300, 1100])  # warps per token chunk; staged rows (1024 tokens and more)
def test_quantize_skips_route_rows_out_of_range(T):
    H, E, K, tile, g = 1024, 16, 4, 64, 3.0
    x, r, codes0, scales0, ws = _quant_case(T, H, E, K, tile, g)
    P, _ = B.route_sizes(T, K, E, tile)
    e2p = r.expanded_to_permuted.clone()
    bad = [(5, 1, P), (T - 1, 3, P + 1000), (T // 2, 0, -7)]
    victims = [int(e2p[t, k].item()) for t, k, _ in bad]
    for t, k, v in bad:
        e2p[t, k] = v
    ws.fill_(0x5A)  # rows that are never written keep this byte
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    B.experts_quantize(dataclasses.replace(r, expanded_to_permuted=e2p), ws, x=bf16_dev(x),
                       a1_gscale=torch.tensor([g], dtype=torch.float32, device=DEV), T=T, H=H, I=128, E=E, K=K,
                       status=status)
    codes, scales = B.experts_export(0, ws, T=T, H=H, I=128, E=E, K=K, tile_m=tile)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    codes, scales = codes.cpu().numpy(), scales.cpu().numpy()
    p2t = r.permuted_to_token.cpu().numpy()
    total = int(r.totals[1].item())
    live = np.setdiff1d(np.nonzero(p2t[:total] >= 0)[0], victims)
    assert np.array_equal(codes[live], codes0[live]) and np.array_equal(scales[live], scales0[live])
    assert (codes[victims] == 0x5A).all() and (scales[victims] == 0x5A).all()
    pad = np.nonzero(p2t[:total] < 0)[0]
    assert not scales[pad].any()


@pytest.mark.parametrize("T", [12, 260])
def test_quantize_prequantized_input_is_a_gather(T):
    H, E, K, tile = 512, 8, 4, 32
    rng = np.random.default_rng(1)
    a = rng.integers(0, 256, (T, H // 2), dtype=np.uint8)
    a_sf = rng.integers(0, 0x7F, (T, H // 16), dtype=np.uint8)
    ids = inputs.draw_topk(rng, T, E, K, "uniform")
    r = _route_gpu(ids, E, tile)
    ws = B.alloc_workspace(T, K, E, H, 128, tile, DEV)
    B.experts_quantize(r, ws, a=torch.from_numpy(a).to(DEV), a_sf=torch.from_numpy(a_sf).to(DEV),
                       T=T, H=H, I=128, E=E, K=K)
    codes, scales = B.experts_export(0, ws, T=T, H=H, I=128, E=E, K=K, tile_m=tile)
    p2t = r.permuted_to_token.cpu().numpy()
    live = np.nonzero(p2t >= 0)[0]
    assert np.array_equal(codes.cpu().numpy()[live], a[p2t[live]])
    assert np.array_equal(scales.cpu().numpy()[live], a_sf[p2t[live]])


def test_workspace_import_export_round_trip():
    T, H, I, E, K, tile = 20, 256, 256, 8, 4, 64
    P, _ = B.route_sizes(T, K, E, tile)
    ws = B.alloc_workspace(T, K, E, H, I, tile, DEV)
    rng = np.random.default_rng(2)
    codes = torch.from_numpy(rng.integers(0, 256, (P, I // 2), dtype=np.uint8)).to(DEV)
    scales = torch.from_numpy(rng.integers(0, 256, (P, I // 16), dtype=np.uint8)).to(DEV)
    B.experts_import(1, codes, scales, ws, T=T, H=H, I=I, E=E, K=K, tile_m=tile)
    c2, s2 = B.experts_export(1, ws, T=T, H=H, I=I, E=E, K=K, tile_m=tile)
    assert torch.equal(c2, codes) and torch.equal(s2, scales)


# ---------------------------------------------------------------------------
# moe_prepare_weights against the oracle's packer; the TP layout identity
# ---------------------------------------------------------------------------
def _prepare_gpu(raw):
    t = {k: torch.from_numpy(np.ascontiguousarray(raw[k])).to(DEV) for k in ("w13", "w13_sf", "w2", "w2_sf")}
    p = B.prepare_weights(t["w13"], t["w13_sf"], t["w2"], t["w2_sf"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in p.items()}


@pytest.mark.parametrize("E,H,I", [(8, 256, 128), (3, 512, 192), (2, 1024, 512)])
def test_prepare_weights_bytes(E, H, I):
    rng = np.random.default_rng(E * H + I)
    raw = {
        "w13": rng.integers(0, 256, (E, 2 * I, H // 2), dtype=np.uint8),
        "w13_sf": rng.integers(0, 256, (E, 2 * I, H // 16), dtype=np.uint8),
        "w2": rng.integers(0, 256, (E, H, I // 2), dtype=np.uint8),
        "w2_sf": rng.integers(0, 256, (E, H, I // 16), dtype=np.uint8),
    }
    got = _prepare_gpu(raw)
    want = olayout.prepare(raw["w13"], raw["w13_sf"], raw["w2"], raw["w2_sf"])
    for k in want:
        assert np.array_equal(got[k], want[k]), k


def test_tp_slice_layout_identity_on_gpu():
    """A TP slice of the GPU-prepared tensors is, byte for byte, the GPU
    preparation of the raw slice (tp = 8, I' = 256)."""
    E, H, I, tp = 4, 512, 2048, 8
    rng = np.random.default_rng(7)
    raw = {
        "w13": rng.integers(0, 256, (E, 2 * I, H // 2), dtype=np.uint8),
        "w13_sf": rng.integers(0, 256, (E, 2 * I, H // 16), dtype=np.uint8),
        "w2": rng.integers(0, 256, (E, H, I // 2), dtype=np.uint8),
        "w2_sf": rng.integers(0, 256, (E, H, I // 16), dtype=np.uint8),
    }
    full = _prepare_gpu(raw)
    for r in range(tp):
        sl = olayout.raw_slice(raw, r, tp)
        got = olayout.prepared_slice_view(full, r, tp)
        want = _prepare_gpu(sl)
        for k in want:
            assert np.array_equal(got[k], want[k]), (k, r)


# ---------------------------------------------------------------------------
# Step a7: the post-expert finalize on given bf16 rows
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T,K,H,gamma_sd,scale", [
    (4, 2, 256, 1.0, 1.0),
    (8, 8, 5120, 1.0, 3e4),
    (33, 8, 4096, 0.1, 1e-3),
    (5, 3, 16384, 1.0, 1.0),
    (3, 1, 8, 0.5, 1.0),
    # the two-CTA register kernel (K <= 8, H % 16 == 0, H <= 8192): many
    # waves, the widest row, a row of three vectors per CTA; and K > 8
    (600, 8, 5120, 1.0, 1.0),
    (5, 8, 8192, 0.5, 1.0),
    (9, 4, 48, 1.0, 1.0),
    (7, 12, 1024, 1.0, 1.0),
    # many tokens: the persistent kernel whose rows stream through a ring of
    # shared-memory slots (several tokens per CTA, fewer slots than K for
    # the widest row)
    (1024, 8, 5120, 1.0, 1.0),
    (1500, 6, 2048, 0.5, 1e2),
    (1030, 8, 4096, 1.0, 1.0),
    (1024, 40, 512, 1.0, 1.0),  # more than 32 routes per token
])
@pytest.mark.parametrize("wbn", [True, False])
def test_finalize_parity(T, K, H, gamma_sd, scale, wbn):
    rng = np.random.default_rng(T * K + H)
    P = T * K + 5
    rows_bits = inputs._to_bf16_bits(rng.standard_normal((P, H)) * scale)
    gamma = inputs._to_bf16_bits(rng.standard_normal(H) * gamma_sd)
    e2p = rng.permutation(P)[: T * K].reshape(T, K).astype(np.int32)
    e2p[0, -1] = -1  # an unrouted route
    w = rng.random((T, K)).astype(np.float32)
    want = olayer.finalize(codecs.bf16_bits_to_f64(rows_bits), e2p, w, gamma, 1e-6, wbn)
    out = B.post_expert_finalize(bf16_dev(rows_bits), torch.from_numpy(e2p).to(DEV), torch.from_numpy(w).to(DEV),
                                 bf16_dev(gamma), 1e-6, wbn)
    got = bf16_host_f64(out)
    assert rel_l2(got, want["out"]) < 2e-3
    # per element: at most one bf16 step from the correctly rounded value
    rms = np.sqrt(np.mean(want["out"] ** 2))
    bound = np.abs(want["out_bf16"]) * 2.0**-7 + 1e-4 * rms
    assert (np.abs(got - want["out_bf16"]) <= bound).all()


@pytest.mark.parametrize("K,H,T", [(8, 5120, 6), (3, 1024, 6), (4, 16384, 6), (8, 5120, 1024)])
def test_finalize_skips_out_of_range_rows(K, H, T):
    """Entries of expanded_to_permuted past the rows buffer (num_rows and
    beyond) or below -1 are never read: the route adds nothing, as a -1 route
    does (the muse_moe_runner page, _finalize_native: unrouted routes read as
    zero rows), and the status word holds MOE_ERR_INVALID_ROUTE. The staged
    (K * H * 2 bytes in shared memory) and the register kernels are both
    covered, and the persistent ring kernel of many tokens."""
    rng = np.random.default_rng(K * H)
    P = T * K
    rows_bits = inputs._to_bf16_bits(rng.standard_normal((P, H)))
    gamma = inputs._to_bf16_bits(rng.standard_normal(H) * 0.1)
    e2p = rng.permutation(P).reshape(T, K).astype(np.int32)
    bad = e2p.copy()
    bad[0, 0] = P          # one past the buffer
    bad[2, K - 1] = 1 << 30
    bad[4, 0] = -7
    w = rng.random((T, K)).astype(np.float32)
    want = olayer.finalize(codecs.bf16_bits_to_f64(rows_bits), np.where((bad >= 0) & (bad < P), bad, -1), w, gamma,
                           1e-6, True)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = B.post_expert_finalize(bf16_dev(rows_bits), torch.from_numpy(bad).to(DEV), torch.from_numpy(w).to(DEV),
                                 bf16_dev(gamma), 1e-6, True, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    assert rel_l2(bf16_host_f64(out), want["out"]) < 2e-3
    # the streaming finalize from sums of squares skips the same entries
    rows64 = codecs.bf16_bits_to_f64(rows_bits)
    g = 1.0 + codecs.bf16_bits_to_f64(gamma)
    ss = ((rows64 * g[None, :]) ** 2).reshape(P, H // 32, 32).sum(axis=-1).astype(np.float32)
    status.zero_()
    out2 = B.post_expert_finalize_sumsq(bf16_dev(rows_bits), torch.from_numpy(ss).to(DEV),
                                        torch.from_numpy(bad).to(DEV), torch.from_numpy(w).to(DEV), bf16_dev(gamma),
                                        1e-6, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    assert rel_l2(bf16_host_f64(out2), want["out"]) < 2e-3
    # the same rows with the valid map: status stays 0
    status.zero_()
    B.post_expert_finalize(bf16_dev(rows_bits), torch.from_numpy(e2p).to(DEV), torch.from_numpy(w).to(DEV),
                           bf16_dev(gamma), 1e-6, True, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.parametrize("wbn", [True, False])
def test_finalize_ring_kernel_against_staged_kernel(wbn):
    """The persistent ring kernel (1024 tokens and more) and the one-CTA-per-
    token staged kernel (fewer) compute the same values in different
    reduction orders: on the same tokens they agree to within one bf16 step
    per element, and a token with no route gives a zero row in both."""
    rng = np.random.default_rng(77)
    T, K, H = 1024, 8, 5120
    P = T * K + 64
    rows = bf16_dev(inputs._to_bf16_bits(rng.standard_normal((P, H))))
    gamma = bf16_dev(inputs._to_bf16_bits(rng.standard_normal(H) * 0.3))
    e2p_np = rng.permutation(P)[: T * K].reshape(T, K).astype(np.int32)
    e2p_np[5, 2] = -1
    e2p_np[900, :] = -1  # a token with no route at all
    e2p = torch.from_numpy(e2p_np).to(DEV)
    w = torch.from_numpy(rng.random((T, K)).astype(np.float32)).to(DEV)
    many = B.post_expert_finalize(rows, e2p, w, gamma, 1e-6, wbn)
    few = B.post_expert_finalize(rows, e2p[: T - 1].contiguous(), w[: T - 1].contiguous(), gamma, 1e-6, wbn)
    torch.cuda.synchronize()
    a, b = many[: T - 1].double(), few.double()
    assert ((a - b).abs() <= b.abs() * 2.0**-7 + 1e-6).all()
    assert rel_l2(a.cpu().numpy(), b.cpu().numpy()) < 1e-3
    assert not many[900].float().abs().any() and not few[900].float().abs().any()


def test_finalize_readings_are_distinguished():
    """With gamma ~ N(0, 1) the two norm readings differ by far more than
    the bar, so the parity test above pins which one the kernel computes."""
    rng = np.random.default_rng(5)
    T, K, H = 4, 4, 1024
    rows_bits = inputs._to_bf16_bits(rng.standard_normal((T * K, H)))
    gamma = inputs._to_bf16_bits(rng.standard_normal(H))
    e2p = np.arange(T * K, dtype=np.int32).reshape(T, K)
    w = np.full((T, K), 0.25, np.float32)
    r = codecs.bf16_bits_to_f64(rows_bits)
    a = olayer.finalize(r, e2p, w, gamma, 1e-6, False)["out"]
    b = olayer.finalize(r, e2p, w, gamma, 1e-6, True)["out"]
    assert rel_l2(a, b) > 0.1


def test_bounded_wait_times_out_and_context_survives():
    """The failure path of every pipelined kernel: a wait on an mbarrier that
    nothing completes gives up at a forced 2 ms limit with MOE_ERR_TIMEOUT in
    the status word, a second waiter leaves through the abort flag well
    before its own 1 s limit, and the context then runs kernels normally."""
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    result = torch.zeros(3, dtype=torch.int32, device=DEV)
    B.selftest_wait_timeout(2_000_000, status, result)
    torch.cuda.synchronize()
    r = result.cpu().tolist()
    assert int(status.item()) == -5
    assert r[0] == 1 and r[1] == 1
    assert r[2] < 500_000  # microseconds: the abort flag, not the 1 s limit
    ids = np.array([[0, 3], [3, 1]], np.int32)
    got = _route_np(_route_gpu(ids, 8, 32))
    _assert_route_equal(got, orouting.route_metadata(ids, 8, 32))


def test_counter_wait_times_out_and_context_survives():
    """The one-launch expert GEMMs' wait of a GEMM2 unit for its route
    tile's GEMM1 units (a GPU-scope acquire poll of a completion counter):
    on a counter that stays 0 it gives up at a forced 2 ms limit with
    MOE_ERR_TIMEOUT, a second waiter leaves through the abort flag, the
    counter is left untouched and the context then runs kernels normally."""
    counter = torch.zeros(1, dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    result = torch.zeros(3, dtype=torch.int32, device=DEV)
    B.selftest_counter_timeout(2_000_000, counter, status, result)
    torch.cuda.synchronize()
    r = result.cpu().tolist()
    assert int(status.item()) == -5
    assert r[0] == 1 and r[1] == 1
    assert r[2] < 500_000  # microseconds: the abort flag, not the 1 s limit
    assert int(counter.item()) == 0
    ids = np.array([[0, 3], [3, 1]], np.int32)
    got = _route_np(_route_gpu(ids, 8, 32))
    _assert_route_equal(got, orouting.route_metadata(ids, 8, 32))
