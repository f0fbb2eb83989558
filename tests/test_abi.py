"""The C-ABI library loads, exports every declared entry point, and checks
its arguments on the host (no GPU calls)."""
import ctypes as C
import os

import pytest

from nvfp4_mixture_experts_route_gb300 import binding as B
from nvfp4_mixture_experts_route_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

@pytest.fixture(scope="module")
def lib():
    build.build()
    return B.load()


def test_every_declared_symbol_is_exported(lib):
    names = B.declared_symbols()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(B._SIGNATURES) == set(names)


def test_version_and_sizes(lib):
    assert lib.moe_abi_version() == 5
    assert B.prepared_sizes(128, 5120, 2048) == [
        128 * 4096 * 2560, 128 * 4096 * 320, 128 * 5120 * 1024, 128 * 5120 * 128]
    assert B.route_sizes(8, 8, 128, 32) == (2048, 64)
    assert B.route_sizes(8192, 8, 128, 128) == (128 * (128 + (65536 - 128) // 128), 128 + (65536 - 128) // 128)
    assert B.route_sizes(0, 8, 128, 32) == (0, 0)


def test_workspace_size_formula(lib):
    T, K, E, H, I, tm = 8, 8, 128, 5120, 2048, 32
    P, MT = B.route_sizes(T, K, E, tm)

    def up(v):
        return (v + 1023) // 1024 * 1024

    # codes row-major; scales as one 512-byte atom per K=64 step per 128 rows of a tile;
    # then one int32 completion counter per route tile and the unit ticket
    want = (up(P * H // 2) + up(MT * (H // 64) * 512) + up(P * I // 2) + up(MT * (I // 64) * 512)
            + up((MT + 1) * 4))
    assert B.experts_workspace_size(T, K, E, H, I, tm) == want


@pytest.mark.parametrize("call,code", [
    (lambda: B.prepared_sizes(8, 192, 128), "MOE_ERR_UNSUPPORTED"),
    (lambda: B.prepared_sizes(8, 256, 96), "MOE_ERR_UNSUPPORTED"),
    (lambda: B.route_sizes(4, 2, 8, 48), "MOE_ERR_UNSUPPORTED"),
    (lambda: B.route_sizes(4, 2, 0, 32), "MOE_ERR_INVALID_ARG"),
    (lambda: B.experts_workspace_size(4, 2, 8, 256, 96, 32), "MOE_ERR_UNSUPPORTED"),
    (lambda: B.experts_workspace_size(4, 2, 8, 192, 128, 32), "MOE_ERR_UNSUPPORTED"),
])
def test_host_refusals(lib, call, code):
    with pytest.raises(B.MoeError) as ei:
        call()
    assert code in str(ei.value)
    assert lib.moe_last_error()


def test_null_pointers_refused_before_any_launch(lib):
    rc = lib.moe_route_permute(None, 4, 2, 8, 32, None, None, None, None, None, None, None, None, None)
    assert rc == -1 and b"null" in lib.moe_last_error()
    rc = lib.moe_post_expert_finalize(None, 8, None, None, None, 1e-6, 1, 4, 2, 256, None, None, None)
    assert rc == -1
    rc = lib.moe_post_expert_finalize(None, 8, None, None, None, 1e-6, 1, 4, 2, 250, None, None, None)
    assert rc == -1 and b"shape" in lib.moe_last_error()
    rc = lib.moe_post_expert_finalize(None, -1, None, None, None, 1e-6, 1, 4, 2, 256, None, None, None)
    assert rc == -1 and b"shape" in lib.moe_last_error()
    w = B.MoeWeights()
    r = B.MoeRoute()
    rc = lib.moe_nvfp4_experts(C.byref(w), None, None, None, None, None, C.byref(r), 4, 256, 128, 8, 2, 32,
                               None, None, 0, None, None)
    assert rc == -1
    # misaligned workspace
    w = B.MoeWeights(*([16] * 7))
    r = B.MoeRoute(16, 16, 16, 16)
    rc = lib.moe_experts_gemm2(C.byref(w), C.byref(r), 4, 256, 128, 8, 2, 32, 16, 1040, 1 << 20, None, None)
    assert rc == -1 and b"aligned" in lib.moe_last_error()
    # undersized workspace
    rc = lib.moe_experts_gemm2(C.byref(w), C.byref(r), 4, 256, 128, 8, 2, 32, 16, 1024, 16, None, None)
    assert rc == -3
    # the routed entry (routing inside the quantizer at these sizes): null
    # routing buffers, then an undersized workspace
    rc = lib.moe_nvfp4_experts_routed(C.byref(w), 16, 16, None, None, 16, 16, 4, 256, 128, 8, 2, 32, None, 16, 16,
                                      16, 16, 16, 16, 16, 1024, 1 << 20, None, None)
    assert rc == -1 and b"null" in lib.moe_last_error()
    rc = lib.moe_nvfp4_experts_routed(C.byref(w), 16, 16, None, None, 16, 16, 4, 256, 128, 8, 2, 32, 16, 16, 16,
                                      16, 16, 16, 16, 16, 1024, 16, None, None)
    assert rc == -3
    rc = lib.moe_nvfp4_experts_routed(C.byref(B.MoeWeights()), 16, 16, None, None, 16, 16, 4, 256, 128, 8, 2, 32,
                                      16, 16, 16, 16, 16, 16, 16, 16, 1024, 1 << 20, None, None)
    assert rc == -1
    # the whole block: no output, then no row sums of squares
    rc = lib.moe_nvfp4_moe_block(C.byref(w), 16, 16, 16, None, None, 16, 16, 16, 1e-6, 1, 4, 256, 128, 8, 2, 32,
                                 16, 16, 16, 16, 16, 16, 16, 16, 16, None, 1024, 1 << 20, None, None)
    assert rc == -1 and b"out" in lib.moe_last_error()
    rc = lib.moe_nvfp4_moe_block(C.byref(w), 16, 16, 16, None, None, 16, 16, 16, 1e-6, 1, 4, 256, 128, 8, 2, 32,
                                 16, 16, 16, 16, 16, 16, 16, 16, None, 16, 1024, 1 << 20, None, None)
    assert rc == -1 and b"row_sumsq" in lib.moe_last_error()


def test_experts_kernel_count():
    assert B.experts_kernels(32) == 2 and B.experts_kernels(64) == 2
    assert B.experts_kernels(128) == 3 and B.experts_kernels(256) == 3
    with pytest.raises(B.MoeError):
        B.experts_kernels(48)


def test_route_kernel_count():
    """One CTA for few routes, count / scan / scatter from 2 full segments
    of 2048 routes whose last segment holds E slots."""
    assert B.route_kernels(8, 8, 128) == 1
    assert B.route_kernels(511, 8, 64) == 1      # 4088 routes: one segment
    assert B.route_kernels(512, 8, 64) == 3      # 4096 routes: two segments
    assert B.route_kernels(8192, 8, 128) == 3
    assert B.route_kernels(0, 8, 128) == 1
    assert B.route_kernels(2047, 2, 1024) == 1   # 4094 routes: one segment


def test_routed_experts_kernel_count():
    """Routing runs inside the input quantizer (2 kernels in all) for at most
    2048 routes, at most 256 experts and tile_m <= 64; otherwise the routing
    kernels come first, then the body's kernels (none when nothing routes)."""
    assert B.routed_experts_kernels(8, 8, 128, 32) == 2
    assert B.routed_experts_kernels(64, 8, 128, 32) == 2
    assert B.routed_experts_kernels(256, 8, 128, 64) == 2    # 2048 routes
    assert B.routed_experts_kernels(257, 8, 128, 32) == 1 + 2
    assert B.routed_experts_kernels(8, 8, 300, 32) == 1 + 2  # E > 256
    assert B.routed_experts_kernels(8, 8, 128, 128) == 1 + 3
    assert B.routed_experts_kernels(8192, 8, 128, 128) == 3 + 3
    assert B.routed_experts_kernels(0, 8, 128, 32) == 1
    with pytest.raises(B.MoeError):
        B.routed_experts_kernels(8, 8, 128, 48)


def test_moe_block_kernel_count():
    """The whole block is the routing kernels (1 or 3), the body's (2 for
    tiles of at most 64 rows, else 3) and the finalize; nothing but the
    routing kernel when there are no routes."""
    assert B.moe_block_kernels(8, 8, 128, 32) == 1 + 2 + 1
    assert B.moe_block_kernels(64, 8, 128, 32) == 1 + 2 + 1
    assert B.moe_block_kernels(8, 12, 128, 32) == 1 + 2 + 1
    assert B.moe_block_kernels(8192, 8, 128, 128) == 3 + 3 + 1
    assert B.moe_block_kernels(0, 8, 128, 32) == 1
    with pytest.raises(B.MoeError):
        B.moe_block_kernels(8, 8, 128, 48)


def test_selftest_arguments_refused_before_launch(lib):
    assert lib.moe_selftest_wait_timeout(2_000_000, None, None, None) == -1
    assert lib.moe_selftest_wait_timeout(10, 16, 16, None) == -1          # below 1 us
    assert lib.moe_selftest_wait_timeout(5_000_000_000, 16, 16, None) == -1  # above 1 s
    assert lib.moe_selftest_counter_timeout(2_000_000, None, 16, 16, None) == -1
    assert lib.moe_selftest_counter_timeout(2_000_000, 18, 16, 16, None) == -1  # misaligned counter
    assert lib.moe_selftest_counter_timeout(10, 16, 16, 16, None) == -1       # below 1 us


def test_header_compiles_as_c_and_cpp():
    """include/moe_nvfp4.h is a plain C header: no C++ types leak into the
    boundary, and it also compiles as C++."""
    import shutil
    import subprocess

    hdr = os.path.join(ROOT, "include", "moe_nvfp4.h")
    for cc, std, lang in (("gcc", "-std=c99", "c"), ("g++", "-std=c++17", "c++")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} not installed")
        r = subprocess.run([cc, "-fsyntax-only", std, "-Wall", "-Wextra", "-Werror", "-x", lang, hdr],
                           capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
