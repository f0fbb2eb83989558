"""Pins of the oracle's block-scaled FP4 products (no GPU)."""
import numpy as np
import pytest

from oracle import codecs, gemm


def _rand(rng, r, K, sf_hi=0x7E):
    return rng.integers(0, 16, (r, K)).astype(np.uint8), rng.integers(0, sf_hi + 1, (r, K // 16)).astype(np.uint8)


@pytest.mark.parametrize("r,n,K", [(1, 3, 16), (2, 5, 64), (3, 4, 96)])
def test_exact_against_brute_force(r, n, K):
    rng = np.random.default_rng(r * 100 + K)
    a, sa = _rand(rng, r, K)
    w, sw = _rand(rng, n, K)
    ref = gemm.gemm_bruteforce(a, sa, w, sw)
    assert np.array_equal(gemm.gemm_exact(a, sa, w, sw), ref)
    assert np.array_equal(gemm.gemm_exact_int64(a, sa, w, sw), ref)


def test_blas_and_int64_agree_full_width():
    rng = np.random.default_rng(9)
    a, sa = _rand(rng, 4, 5120)
    w, sw = _rand(rng, 64, 5120, sf_hi=0x50)
    assert np.array_equal(gemm.gemm_exact(a, sa, w, sw), gemm.gemm_exact_int64(a, sa, w, sw))


def test_closed_forms():
    K = 5120
    one, one_sf = np.full((1, K), 2, np.uint8), np.full((1, K // 16), 0x38, np.uint8)  # 1.0, scale 1.0
    assert gemm.gemm_exact(one, one_sf, one, one_sf)[0, 0] == K
    # alternating signs cancel
    w = np.tile(np.array([2, 10], np.uint8), K // 2)[None, :]
    assert gemm.gemm_exact(one, one_sf, w, one_sf)[0, 0] == 0
    # largest magnitudes: 6 * 448 on both sides -> needs the int64 fallback
    big, big_sf = np.full((1, K), 7, np.uint8), np.full((1, K // 16), 0x7E, np.uint8)
    want = K * (6.0 * 448.0) ** 2
    assert gemm.gemm_exact(big, big_sf, big, big_sf)[0, 0] == want
    # a transposed operand would mix rows: row j of w only meets itself
    w2 = np.zeros((3, K), np.uint8)
    w2[1] = 2
    assert list(gemm.gemm_exact(one, one_sf, w2, np.repeat(one_sf, 3, 0))[0]) == [0, K, 0]


def test_scale_applies_per_block():
    K = 64
    a = np.full((1, K), 2, np.uint8)
    sa = np.array([[0x38, 0x40, 0x30, 0x48]], np.uint8)  # 1, 2, 0.5, 4
    w = np.full((1, K), 2, np.uint8)
    sw = np.array([[0x38, 0x38, 0x40, 0x38]], np.uint8)  # 1, 1, 2, 1
    assert gemm.gemm_exact(a, sa, w, sw)[0, 0] == 16 * (1 * 1 + 2 * 1 + 0.5 * 2 + 4 * 1)
    assert float(codecs.e4m3_decode(0x48)) == 4.0


def test_refuses_nan_scales():
    a = np.full((1, 16), 2, np.uint8)
    with pytest.raises(ValueError):
        gemm.gemm_exact(a, np.array([[0x7F]], np.uint8), a, np.array([[0x38]], np.uint8))
