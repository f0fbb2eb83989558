"""GPU parity of the pooler / unpooler projection (tcgen05 kind::f16 GEMM)
against the oracle, through the C ABI."""
import numpy as np
import pytest
import torch

from oracle import codecs, dense as odense
from nvfp4_mixture_experts_route_gb300 import binding as B
from nvfp4_mixture_experts_route_gb300 import inputs

from _util import bf16_dev, bf16_host_f64, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ulp_bf16(v):
    """Spacing of bf16 numbers at |v| (normal range)."""
    a = np.maximum(np.abs(v), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("T,Din,Dout", [
    (1, 64, 128),        # one stage, one tile
    (8, 5120, 5120),     # decode-sized: stream-K split, partial tiles summed in CTA order
    (64, 2048, 1280),    # 10 tiles on every CTA: each range spans tile boundaries
    (8, 64, 5120),       # one K step per tile: every CTA owns whole tiles
    (37, 320, 384),      # ragged tokens, odd stage count
    (300, 1024, 256),    # 256-token tiles with a ragged tail
])
def test_dense_bf16_parity(T, Din, Dout):
    rng = np.random.default_rng(T * 7 + Din)
    x = inputs._to_bf16_bits(rng.standard_normal((T, Din)))
    w = inputs._to_bf16_bits(rng.standard_normal((Dout, Din)) / np.sqrt(Din))
    y = B.dense_bf16(bf16_dev(x), bf16_dev(w))
    torch.cuda.synchronize()
    got = bf16_host_f64(y)
    ref = odense.dense_f64(x, w)
    # one bf16 rounding of an fp32 sum: within 1 ulp of the exact sum plus the
    # fp32 accumulation error (|x|.|w| * Din * 2^-24, generous)
    bound = _ulp_bf16(ref) + np.abs(codecs.bf16_bits_to_f64(x)) @ np.abs(codecs.bf16_bits_to_f64(w)).T * Din * 2.0 ** -24
    assert np.all(np.abs(got - ref) <= bound)
    assert rel_l2(got, ref) < 3e-3


def test_dense_bf16_identity_is_exact():
    rng = np.random.default_rng(5)
    T, D = 50, 256
    x = inputs._to_bf16_bits(rng.standard_normal((T, D)))
    y = B.dense_bf16(bf16_dev(x), bf16_dev(inputs._to_bf16_bits(np.eye(D))))
    torch.cuda.synchronize()
    assert np.array_equal(bf16_host_f64(y), codecs.bf16_bits_to_f64(x))


def test_dense_bf16_deterministic_and_empty():
    rng = np.random.default_rng(6)
    x = bf16_dev(inputs._to_bf16_bits(rng.standard_normal((8, 2048))))
    w = bf16_dev(inputs._to_bf16_bits(rng.standard_normal((1024, 2048)) / 45))
    assert B.dense_bf16_workspace_size(8, 2048, 1024) > 0  # the sliced path
    a = B.dense_bf16(x, w)
    b = B.dense_bf16(x, w)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    e = B.dense_bf16(torch.empty((0, 2048), dtype=torch.bfloat16, device=DEV), w)
    torch.cuda.synchronize()
    assert e.shape == (0, 1024)


def test_dense_bf16_prefill_sampled():
    """T = 8192 tokens through 5120 x 5120 (256-token tiles, whole tiles per CTA),
    checked on 64 sampled tokens."""
    rng = np.random.default_rng(7)
    T, D = 8192, 5120
    x = inputs._to_bf16_bits(rng.standard_normal((T, D)))
    w = inputs._to_bf16_bits(rng.standard_normal((D, D)) / np.sqrt(D))
    y = B.dense_bf16(bf16_dev(x), bf16_dev(w))
    torch.cuda.synchronize()
    rows = np.sort(rng.choice(T, 64, replace=False))
    got = bf16_host_f64(y[torch.from_numpy(rows).to(DEV)])
    ref = odense.dense_f64(x[rows], w)
    assert rel_l2(got, ref) < 3e-3
