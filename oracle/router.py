"""MuseSpark1x expert routing from router logits, and the fused pre-expert
RMSNorm + NVFP4 input quantization.

Test infrastructure only (see the package docstring).

Routing (the model page, ``MuseSpark1xMoE.__init__``: ``MuseSpark1xRouter(top_k,
num_experts, expert_bias, route_scale, router_score_normalization="sigmoid",
router_score_division_eps=1e-15)`` and the experts' ``scoring_func="sigmoid",
e_score_correction_bias=expert_bias, renormalize=True,
routed_scaling_factor=route_scale``; the muse_moe_runner page,
``validate_deployment``: "sigmoid + expert bias + sum-renormalize, no expert
groups, route_scale == 1.0"):

    s      = sigmoid(logits)                      per token, over the E experts
    chosen = the K experts with the largest s + expert_bias
    w      = s[chosen] / (sum(s[chosen]) + eps) * route_scale

The bias only steers the choice; the weights use the unbiased scores. The
pages do not print the kernel, so two details are this project's reading:
equal choice values rank the lower expert index first, and a token flagged
as padding gets ids -1 (routes the experts skip, as the model page notes for
padding rows) and weights 0.

The choice is an integer decided by floating point, so it is taken in the
kernel's precision: s in fp32 as 1 / (1 + exp(-x)) and s + bias in fp32; the
weights are then computed in fp64 from those fp32 scores.

Pre-expert norm (the model page: ``pre_expert_norm = MuseSpark1xRMSNorm(
has_weight=True, zero_centered_gamma=True, post_norm_gain_center_type="one")``;
``norm_fuses_into_nvfp4_quant`` requires ``not norm.applies_weight_before_norm``;
``norm_quant_trtllm_nvfp4(pooled, ..., norm.weight, eps, gain_center,
global_scale)``):

    y = x / sqrt(mean(x^2) + eps) * (1 + gamma)      (weight after the norm)
    (a, a_sf) = NVFP4(y) with the input global scale

computed in fp64 and rounded to fp32 before the fp32 quantizer (the kernel
keeps y in fp32; the codes may differ from the oracle's where y lies within
rounding of a code boundary).

Parity: pinned (sigmoid against scipy's expit, brute-force top-K, the bias
steering only the choice, renormalisation, padding; the norm against
torch.nn.functional.rms_norm).
"""
from __future__ import annotations

import numpy as np

from .codecs import bf16_bits_to_f64
from .quant import quantize_blocks


def sigmoid_f32(logits) -> np.ndarray:
    x = np.asarray(logits, dtype=np.float32)
    with np.errstate(over="ignore"):
        return (np.float32(1.0) / (np.float32(1.0) + np.exp(-x))).astype(np.float32)


def musespark1x_routing(logits, expert_bias, top_k: int, route_scale: float = 1.0, eps: float = 1e-15,
                        is_padding=None) -> tuple[np.ndarray, np.ndarray]:
    """(topk_ids int32 [T, K], topk_weights float64 [T, K])."""
    s = sigmoid_f32(logits)
    choice = (s + np.asarray(expert_bias, dtype=np.float32)[None, :]).astype(np.float32)
    T, E = s.shape
    ids = np.full((T, top_k), -1, dtype=np.int32)
    w = np.zeros((T, top_k), dtype=np.float64)
    for t in range(T):
        if is_padding is not None and is_padding[t]:
            continue
        order = sorted(range(E), key=lambda e: (-float(choice[t, e]), e))[:top_k]
        ids[t] = order
        sc = s[t, order].astype(np.float64)
        w[t] = sc / (sc.sum() + eps) * route_scale
    return ids, w


def rmsnorm_nvfp4(x_bits, gamma_bits, eps: float, gscale: float):
    """Pre-expert RMSNorm (weight 1 + gamma after the norm) and NVFP4 quant.
    Returns (y float64 [T, H], codes uint8 [T, H] one code per element,
    sf uint8 [T, H/16])."""
    x = bf16_bits_to_f64(x_bits)
    g = 1.0 + bf16_bits_to_f64(gamma_bits)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g
    codes, sf = quantize_blocks(y.astype(np.float32), gscale)
    return y, codes, sf
