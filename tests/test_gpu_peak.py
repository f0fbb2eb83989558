"""The dense NVFP4 tensor-core rate probe (moe_fp4_mma_rate) runs every
supported variant to completion with a clean status word, and refuses the
variants that do not fit tensor memory on the host."""
import pytest
import torch

from nvfp4_mixture_experts_route_gb300 import binding as B

VARIANTS = [
    # (n, sf_copies, mmas_per_commit, ctas_per_sm, ring)
    (128, 0, 4, 1, 3), (128, 0, 4, 2, 3), (128, 1, 4, 2, 3), (128, 0, 16, 2, 3), (128, 2, 4, 2, 3),
    (128, 3, 4, 2, 3), (128, 4, 4, 2, 3), (128, 5, 4, 2, 3), (128, 2, 4, 1, 5), (128, 3, 4, 1, 5),
    (256, 0, 4, 1, 3), (256, 1, 4, 1, 3), (256, 0, 16, 1, 3), (256, 2, 4, 1, 3), (256, 3, 4, 1, 3),
    (256, 1, 4, 1, 5), (256, 2, 4, 1, 5), (256, 3, 4, 1, 5), (256, 4, 4, 1, 5), (256, 5, 4, 1, 5),
]


def test_unfitting_variants_refused_on_host():
    import ctypes as C

    lib = B.load()
    f = C.c_double()
    for n, sf, mpc, ctas, ring, want in ((256, 0, 4, 2, 3, -2), (128, 1, 16, 1, 3, -2), (128, 3, 16, 1, 3, -2),
                                         (128, 1, 4, 2, 5, -2), (64, 0, 4, 1, 3, -1), (128, 0, 4, 3, 3, -1),
                                         (128, 6, 4, 1, 3, -1), (128, 1, 4, 1, 4, -1)):
        assert lib.moe_fp4_mma_rate(n, sf, mpc, ctas, ring, 0, 8, C.byref(f), None, None) == want
        assert b"fp4 rate" in lib.moe_last_error()
    assert lib.moe_fp4_mma_rate(128, 0, 4, 1, 3, 2, 8, C.byref(f), None, None) == -1  # warp_issue 0 or 1
    for n, sf, stages in ((64, 0, 8), (128, 2, 8), (256, 1, 0)):
        assert lib.moe_fp4_mma_rate_pair(n, sf, stages, C.byref(f), None, None) == -1
        assert b"fp4 rate pair" in lib.moe_last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("warp_issue", [False, True])
@pytest.mark.parametrize("variant", VARIANTS)
def test_rate_probe_runs(variant, warp_issue, record_property):
    n, sf, mpc, ctas, ring = variant
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.fp4_mma_rate(n, sf, mpc, ctas, 64, status=status, ring=ring, warp_issue=warp_issue)  # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    flops = B.fp4_mma_rate(n, sf, mpc, ctas, 2048 // mpc * 4, status=status, ring=ring, warp_issue=warp_issue)
    e1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert flops == 2.0 * 128 * n * 64 * mpc * (2048 // mpc * 4) * sms * ctas
    tflops = flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
    record_property("tflops", tflops)
    # a rate above the part's nominal dense FP4 figure would mean the MMAs
    # did not run
    assert 0 < tflops < 20000


@pytest.mark.gpu
def test_same_kernel_with_more_shared_memory_later():
    # n = 128, one stage of copies once, 4 MMAs per commit: the same kernel
    # runs with 96 KB of shared memory at two CTAs per SM and 160 KB at one;
    # the larger request after the smaller one raises the kernel's limit again
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for warp_issue in (False, True):
        for ctas in (2, 1):
            B.fp4_mma_rate(128, 0, 4, ctas, 64, status=status, warp_issue=warp_issue)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.gpu
@pytest.mark.parametrize("n,sf", [(128, 0), (128, 1), (256, 0), (256, 1)])
def test_pair_rate_probe_runs(n, sf, record_property):
    """The cta_group::2 form: clusters of two CTAs allocate tensor memory
    together and rank 0 issues M = 256 MMAs over both; every variant ends
    with a clean status word."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.fp4_mma_rate_pair(n, sf, 16, status=status)  # warm-up
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    flops = B.fp4_mma_rate_pair(n, sf, 2048, status=status)
    e1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    sms = torch.cuda.get_device_properties(0).multi_processor_count & ~1
    assert flops == 2.0 * 256 * n * 64 * 4 * 2048 * (sms // 2)
    tflops = flops / (e0.elapsed_time(e1) * 1e-3) / 1e12
    record_property("tflops", tflops)
    assert 0 < tflops < 20000
