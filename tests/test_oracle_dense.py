"""Pins of the oracle's pooler / unpooler projection (no GPU)."""
import numpy as np

from oracle import codecs, dense
from nvfp4_mixture_experts_route_gb300 import inputs


def test_brute_force_triple_loop():
    """Small-integer bf16 values keep every product and sum exact, so the
    BLAS result must equal a plain triple loop bit for bit."""
    rng = np.random.default_rng(0)
    T, Din, Dout = 3, 7, 5
    x = inputs._to_bf16_bits(rng.integers(-8, 9, (T, Din)).astype(np.float64) / 2)
    w = inputs._to_bf16_bits(rng.integers(-8, 9, (Dout, Din)).astype(np.float64) / 4)
    xv, wv = codecs.bf16_bits_to_f64(x), codecs.bf16_bits_to_f64(w)
    want = np.zeros((T, Dout))
    for t in range(T):
        for o in range(Dout):
            acc = 0.0
            for i in range(Din):
                acc += xv[t, i] * wv[o, i]
            want[t, o] = acc
    assert np.array_equal(dense.dense_f64(x, w), want)


def test_identity_and_permutation_return_x():
    rng = np.random.default_rng(1)
    T, D = 9, 64
    x = inputs._to_bf16_bits(rng.standard_normal((T, D)))
    eye = inputs._to_bf16_bits(np.eye(D))
    assert np.array_equal(dense.dense_bf16(x, eye), codecs.bf16_bits_to_f64(x))
    perm = rng.permutation(D)
    pw = inputs._to_bf16_bits(np.eye(D)[perm])
    assert np.array_equal(dense.dense_bf16(x, pw), codecs.bf16_bits_to_f64(x)[:, perm])


def test_linear_in_the_weight():
    """Two weights with disjoint supports: the products of their sum are the
    sums of their products (all exact in fp64)."""
    rng = np.random.default_rng(2)
    T, Din, Dout = 4, 32, 8
    x = inputs._to_bf16_bits(rng.standard_normal((T, Din)))
    w = rng.standard_normal((Dout, Din))
    mask = rng.random((Dout, Din)) < 0.5
    w1 = inputs._to_bf16_bits(np.where(mask, w, 0.0))
    w2 = inputs._to_bf16_bits(np.where(mask, 0.0, w))
    both = inputs._to_bf16_bits(codecs.bf16_bits_to_f64(w1) + codecs.bf16_bits_to_f64(w2))
    lhs = dense.dense_f64(x, both)
    rhs = dense.dense_f64(x, w1) + dense.dense_f64(x, w2)
    assert np.allclose(lhs, rhs, rtol=1e-14, atol=1e-14)
