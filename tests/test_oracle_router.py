"""Pins of the oracle's MuseSpark1x routing and fused pre-expert norm + quant
(no GPU)."""
import numpy as np
import pytest
import scipy.special
import torch

from oracle import codecs, quant, router
from nvfp4_mixture_experts_route_gb300 import inputs


def test_sigmoid_matches_scipy():
    x = np.linspace(-30, 30, 2001).astype(np.float32)
    assert np.allclose(router.sigmoid_f32(x), scipy.special.expit(x.astype(np.float64)), rtol=1e-6, atol=1e-30)


def test_topk_brute_force():
    rng = np.random.default_rng(0)
    T, E, K = 20, 64, 8
    logits = rng.standard_normal((T, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.1).astype(np.float32)
    ids, w = router.musespark1x_routing(logits, bias, K)
    s = scipy.special.expit(logits.astype(np.float64))
    for t in range(T):
        want = np.argsort(-(s[t] + bias), kind="stable")[:K]
        assert list(ids[t]) == list(want)
        sel = s[t, want]
        assert np.allclose(w[t], sel / sel.sum(), rtol=1e-6)
        assert abs(w[t].sum() - 1.0) < 1e-12


def test_bias_steers_choice_not_weights():
    logits = np.array([[3.0, 2.0, -4.0, 1.0]], np.float32)
    bias = np.array([0.0, 0.0, 5.0, 0.0], np.float32)
    ids, w = router.musespark1x_routing(logits, bias, 2)
    assert list(ids[0]) == [2, 0]  # expert 2 only chosen through its bias
    s = scipy.special.expit(np.array([-4.0, 3.0]))
    assert np.allclose(w[0], s / s.sum())


def test_ties_padding_scale_and_eps():
    logits = np.zeros((3, 6), np.float32)
    ids, w = router.musespark1x_routing(logits, np.zeros(6, np.float32), 3, route_scale=2.5,
                                        is_padding=np.array([0, 1, 0], bool))
    assert list(ids[0]) == [0, 1, 2] and list(ids[1]) == [-1, -1, -1]
    assert np.allclose(w[0], 2.5 / 3) and not w[1].any()
    # very negative logits: scores ~0, the eps keeps the division finite
    ids, w = router.musespark1x_routing(np.full((1, 4), -200.0, np.float32), np.zeros(4, np.float32), 2)
    assert np.isfinite(w).all() and (w >= 0).all()


def test_rmsnorm_matches_torch_rms_norm_then_quant():
    rng = np.random.default_rng(1)
    T, H = 5, 512
    x = inputs._to_bf16_bits(rng.standard_normal((T, H)) * 3)
    gamma = inputs._to_bf16_bits(rng.standard_normal(H) * 0.3)
    y, codes, sf = router.rmsnorm_nvfp4(x, gamma, 1e-6, 40.0)
    g = torch.from_numpy(1.0 + codecs.bf16_bits_to_f64(gamma))
    ref = torch.nn.functional.rms_norm(torch.from_numpy(codecs.bf16_bits_to_f64(x)), (H,), weight=g, eps=1e-6)
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    q2, s2 = quant.quantize_blocks(ref.numpy().astype(np.float32), 40.0)
    assert np.array_equal(codes, q2) and np.array_equal(sf, s2)


@pytest.mark.parametrize("gs", [1.0, 448.0 * 6 / 4])
def test_rmsnorm_unit_rms_rows(gs):
    """Rows already of unit RMS with gamma = 0 pass through the norm
    unchanged (up to eps), so their codes equal the plain quantizer's."""
    rng = np.random.default_rng(2)
    H = 256
    v = rng.standard_normal((3, H))
    v /= np.sqrt(np.mean(v * v, axis=1, keepdims=True))
    x = inputs._to_bf16_bits(v)
    y, codes, sf = router.rmsnorm_nvfp4(x, np.zeros(H, np.uint16), 0.0, gs)
    xv = codecs.bf16_bits_to_f64(x)
    assert np.allclose(y, xv / np.sqrt(np.mean(xv * xv, axis=1, keepdims=True)), rtol=1e-15)
