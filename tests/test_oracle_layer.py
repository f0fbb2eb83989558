"""Pins of the oracle's expert block and post-expert finalize (no GPU)."""
import numpy as np
import torch

from oracle import codecs, layer, layout, routing
from nvfp4_mixture_experts_route_gb300 import inputs

TINY = inputs.WORKLOADS["tiny_t4"]


def test_finalize_k1_unit_weight_is_plain_rmsnorm():
    rng = np.random.default_rng(0)
    H = 256
    rows = codecs.round_to_bf16(rng.standard_normal((3, H)) * 50)
    gamma = np.zeros(H, np.uint16)  # bf16 +0
    e2p = np.array([[2], [0], [1]])
    w = np.ones((3, 1), np.float32)
    for wbn in (True, False):
        out = layer.finalize(rows, e2p, w, gamma, 1e-6, wbn)["out"]
        ref = torch.nn.functional.rms_norm(torch.from_numpy(rows[[2, 0, 1]]), (H,), eps=1e-6).numpy()
        assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_finalize_readings_against_torch_rms_norm_with_weight():
    rng = np.random.default_rng(1)
    H = 128
    r = codecs.round_to_bf16(rng.standard_normal((1, H)) * 3)
    gamma_bits = codecs.bf16_bits(codecs.round_to_bf16(rng.standard_normal(H)))
    g = 1.0 + codecs.bf16_bits_to_f64(gamma_bits)
    e2p, w = np.array([[0]]), np.ones((1, 1), np.float32)
    rt = torch.from_numpy(r)
    gt = torch.from_numpy(g)
    # reading (A): the weight multiplies the normalised row
    a = layer.finalize(r, e2p, w, gamma_bits, 1e-6, weight_before_norm=False)["out"]
    assert np.allclose(a, torch.nn.functional.rms_norm(rt, (H,), weight=gt, eps=1e-6).numpy(), rtol=1e-12)
    # reading (B): the weight scales the row before it is normalised
    b = layer.finalize(r, e2p, w, gamma_bits, 1e-6, weight_before_norm=True)["out"]
    assert np.allclose(b, torch.nn.functional.rms_norm(rt * gt, (H,), eps=1e-6).numpy(), rtol=1e-12)
    assert not np.allclose(a, b, rtol=1e-3)


def test_finalize_unrouted_and_weights():
    H = 64
    rows = codecs.round_to_bf16(np.random.default_rng(2).standard_normal((4, H)))
    gamma = np.zeros(H, np.uint16)
    e2p = np.array([[0, -1, 3], [-1, -1, -1]])
    w = np.array([[0.5, 100.0, 0.25], [1, 1, 1]], np.float32)
    out = layer.finalize(rows, e2p, w, gamma, 1e-6)["out"]
    n = lambda v: v / np.sqrt(np.mean(v * v) + 1e-6)  # noqa: E731
    assert np.allclose(out[0], 0.5 * n(rows[0]) + 0.25 * n(rows[3]), rtol=1e-13)
    assert not out[1].any()


def test_swiglu_matches_torch_silu():
    rng = np.random.default_rng(3)
    gate, up = rng.standard_normal(1000) * 20, rng.standard_normal(1000)
    ref = (torch.nn.functional.silu(torch.from_numpy(gate)) * torch.from_numpy(up)).numpy()
    assert np.allclose(layer.swiglu(gate, up), ref, rtol=1e-14, atol=0)
    assert layer.swiglu(np.array([-1e5]), np.array([3.0]))[0] == 0.0


def _constant_layer(E=2, H=256, I=128, gate_code=2, up_code=1):
    """All-ones activations against gate rows of one value and up rows of
    another: acc1, h and acc2 have closed forms."""
    sf1 = 0x38  # 1.0
    w13 = np.zeros((E, 2 * I, H // 2), np.uint8)
    w13[:, :I] = gate_code | (gate_code << 4)
    w13[:, I:] = up_code | (up_code << 4)
    return {
        "w13": w13,
        "w13_sf": np.full((E, 2 * I, H // 16), sf1, np.uint8),
        "w2": np.full((E, H, I // 2), 0x22, np.uint8),  # 1.0
        "w2_sf": np.full((E, H, I // 16), sf1, np.uint8),
        "g1_alphas": np.array([0.5, 1.0], np.float32)[:E],
        "g1_scale_c": np.array([2.0, 0.25], np.float32)[:E],
        "g2_alphas": np.array([3.0, 1.0], np.float32)[:E],
    }


def test_gate_up_order_and_scalars_closed_form():
    H, I = 256, 128
    L = _constant_layer()
    # x = 6.0 everywhere quantizes to code 7 with scale 1.0 at g = 1.
    x = codecs.bf16_bits(np.full((1, H), 6.0))
    er = layer.expert_rows(x, np.array([[0]]), L, 1.0, 1.0, return_intermediate=True)
    acc_gate, acc_up = 6.0 * 1.0 * H, 6.0 * 0.5 * H  # gate rows 1.0, up rows 0.5
    gate, up = 0.5 * acc_gate, 2.0 * acc_up
    h = gate / (1 + np.exp(-gate)) * up
    assert np.allclose(er["h"][0], h, rtol=1e-15)
    # h = 768 * 1536 everywhere: sf = e4m3(h / 6) saturates at 448, codes at 6
    assert (er["hq_sf"][0] == 0x7E).all() and (er["hq_codes"][0] == 7).all()
    assert np.allclose(er["rows"][0], 3.0 * (6.0 * 448.0) * 1.0 * I)


def test_tp_identity_exact_in_oracle():
    """The expert_tp page: the GEMM2 rows of the tp intermediate slices are
    K-partials whose sum is the full row. In exact arithmetic the oracle's
    partial rows sum to its full rows bit for bit (I' % 16 == 0 keeps every
    requant block inside a slice)."""
    w = inputs.Workload("t", T=6, H=256, I=256, E=8, K=2, routing="uniform", tile_m=32)
    L = inputs.make_layer(w)
    L["g2_alphas"] = np.ones_like(L["g2_alphas"])  # keep the fp64 scaling exact
    b = inputs.make_batch(w)
    full = layer.expert_rows(b["x"], b["topk_ids"], L, 2.0, 1e-3)
    tp = 4
    acc = np.zeros_like(full["rows"])
    for r in range(tp):
        part = layer.expert_rows(b["x"], b["topk_ids"], layout.raw_slice(L, r, tp), 2.0, 1e-3)
        acc += part["rows"]
    assert np.array_equal(acc, full["rows"])


def _tiny_run(**kw):
    L = inputs.make_layer(TINY)
    b = inputs.make_batch(TINY)
    return L, b, layer.moe_layer(b["x"], b["topk_ids"], b["topk_weights"], L, 1.0, 1.0, L["gamma"], 1e-6, 32, **kw)


def test_token_permutation_equivariance():
    L, b, ref = _tiny_run()
    perm = np.array([2, 0, 3, 1])
    got = layer.moe_layer(b["x"][perm], b["topk_ids"][perm], b["topk_weights"][perm], L, 1.0, 1.0, L["gamma"], 1e-6, 32)
    assert np.allclose(got["out"], ref["out"][perm], rtol=1e-12, atol=1e-12)


def test_k_order_invariance():
    L, b, ref = _tiny_run()
    got = layer.moe_layer(b["x"], b["topk_ids"][:, ::-1], b["topk_weights"][:, ::-1], L, 1.0, 1.0, L["gamma"], 1e-6, 32)
    assert np.allclose(got["out"], ref["out"], rtol=1e-12, atol=1e-12)


def test_scale_invariance_of_the_norm():
    """Scaling g2_alphas[e] by c > 0 scales expert e's rows; the per-route
    norm removes it (up to eps and the bf16 rounding of the rows, exact for a
    power of two)."""
    L, b, ref = _tiny_run()
    L2 = dict(L)
    L2["g2_alphas"] = L["g2_alphas"] * np.float32(4.0)
    got = layer.moe_layer(b["x"], b["topk_ids"], b["topk_weights"], L2, 1.0, 1.0, L["gamma"], 1e-6, 32)
    assert np.allclose(got["out"], ref["out"], rtol=1e-9, atol=1e-9)


def test_linearity_in_weights():
    L, b, ref = _tiny_run()
    e2p = ref["meta"]["expanded_to_permuted"]
    w = b["topk_weights"]
    one = layer.finalize(ref["gemm2_rows"], e2p, w, L["gamma"], 1e-6)["out"]
    two = layer.finalize(ref["gemm2_rows"], e2p, 2 * w, L["gamma"], 1e-6)["out"]
    assert np.allclose(two, 2 * one, rtol=1e-14)
    assert np.array_equal(one, ref["out"])


def test_tiny_metadata_and_rows_placement():
    L, b, ref = _tiny_run()
    meta = routing.route_metadata(b["topk_ids"], TINY.E, 32)
    for key in meta:
        assert np.array_equal(meta[key], ref["meta"][key])
    e2p = meta["expanded_to_permuted"].reshape(-1)
    assert np.array_equal(ref["gemm2_rows"][e2p], ref["routes"]["rows_bf16"])
