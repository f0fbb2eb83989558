"""ctypes binding of libmoe_nvfp4.so (declared in include/moe_nvfp4.h).

Argument marshalling only: every step of the expert block runs in the
library's CUDA kernels. PyTorch supplies device memory (``torch.empty``) and
the current CUDA stream. There is no fallback: if the library is missing, or
a call fails, this module raises.

The functions carry the C entry points' names without the ``moe_`` prefix.
"""
from __future__ import annotations

import ctypes as C
import os
from dataclasses import dataclass

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_nvfp4.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "moe_nvfp4.h")

MOE_OK = 0
STATUS_NAMES = {
    0: "MOE_OK",
    -1: "MOE_ERR_INVALID_ARG",
    -2: "MOE_ERR_UNSUPPORTED",
    -3: "MOE_ERR_WORKSPACE",
    -4: "MOE_ERR_CUDA",
    -5: "MOE_ERR_TIMEOUT",
    -6: "MOE_ERR_INVALID_ROUTE",
}


class MoeError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class MoeWeights(C.Structure):
    _fields_ = [
        ("w13", C.c_void_p),
        ("w13_sf", C.c_void_p),
        ("w2", C.c_void_p),
        ("w2_sf", C.c_void_p),
        ("g1_alphas", C.c_void_p),
        ("g1_scale_c", C.c_void_p),
        ("g2_alphas", C.c_void_p),
    ]


class MoeRoute(C.Structure):
    _fields_ = [
        ("permuted_to_token", C.c_void_p),
        ("tile_expert", C.c_void_p),
        ("tile_row_limit", C.c_void_p),
        ("totals", C.c_void_p),
        ("expanded_to_permuted", C.c_void_p),
    ]


_P = C.c_void_p
_I = C.c_int
_SIGNATURES = {
    "moe_last_error": ([], C.c_char_p),
    "moe_abi_version": ([], _I),
    "moe_device_reads_host": ([_P], _I),
    "moe_route_kernels": ([_I, _I, _I], _I),
    "moe_experts_kernels": ([_I], _I),
    "moe_prepared_sizes": ([_I, _I, _I, C.POINTER(C.c_size_t)], _I),
    "moe_prepare_weights": ([_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_route_sizes": ([_I, _I, _I, _I, C.POINTER(_I), C.POINTER(_I)], _I),
    "moe_route_permute": ([_P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_experts_workspace_size": ([_I, _I, _I, _I, _I, _I, C.POINTER(C.c_size_t)], _I),
    "moe_nvfp4_experts": (
        [C.POINTER(MoeWeights), _P, _P, _P, _P, _P, C.POINTER(MoeRoute), _I, _I, _I, _I, _I, _I, _P, _P,
         C.c_size_t, _P, _P],
        _I,
    ),
    "moe_nvfp4_experts_routed": (
        [C.POINTER(MoeWeights), _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P,
         _P, C.c_size_t, _P, _P],
        _I,
    ),
    "moe_routed_experts_kernels": ([_I, _I, _I, _I], _I),
    "moe_nvfp4_moe_block": (
        [C.POINTER(MoeWeights), _P, _P, _P, _P, _P, _P, _P, _P, C.c_float, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P,
         _P, _P, _P, _P, _P, _P, _P, _P, C.c_size_t, _P, _P],
        _I,
    ),
    "moe_moe_block_kernels": ([_I, _I, _I, _I], _I),
    "moe_nvfp4_experts_sumsq": (
        [C.POINTER(MoeWeights), _P, _P, _P, _P, _P, C.POINTER(MoeRoute), _I, _I, _I, _I, _I, _I, _P, _P, _I, _P,
         _P, C.c_size_t, _P, _P],
        _I,
    ),
    "moe_experts_gemm2_sumsq": (
        [C.POINTER(MoeWeights), C.POINTER(MoeRoute), _I, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, C.c_size_t, _P,
         _P], _I),
    "moe_experts_gemms_sumsq": (
        [C.POINTER(MoeWeights), _P, C.POINTER(MoeRoute), _I, _I, _I, _I, _I, _I, _P, _P, _I, _P, _P, C.c_size_t,
         _P, _P], _I),
    "moe_post_expert_finalize_sumsq": ([_P, _P, _I, _P, _P, _P, C.c_float, _I, _I, _I, _P, _P, _P], _I),
    "moe_experts_quantize": (
        [_P, _P, _P, _P, C.POINTER(MoeRoute), _I, _I, _I, _I, _I, _I, _P, C.c_size_t, _P, _P],
        _I,
    ),
    "moe_experts_gemm1": (
        [C.POINTER(MoeWeights), _P, C.POINTER(MoeRoute), _I, _I, _I, _I, _I, _I, _P, C.c_size_t, _P, _P],
        _I,
    ),
    "moe_experts_gemms": (
        [C.POINTER(MoeWeights), _P, C.POINTER(MoeRoute), _I, _I, _I, _I, _I, _I, _P, _P, C.c_size_t, _P, _P],
        _I,
    ),
    "moe_experts_gemm2": (
        [C.POINTER(MoeWeights), C.POINTER(MoeRoute), _I, _I, _I, _I, _I, _I, _P, _P, C.c_size_t, _P, _P],
        _I,
    ),
    "moe_experts_export": ([_I, _P, C.c_size_t, _I, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_experts_import": ([_I, _P, _P, _I, _I, _I, _I, _I, _I, _P, C.c_size_t, _P], _I),
    "moe_post_expert_finalize": ([_P, _I, _P, _P, _P, C.c_float, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_nvfp4_experts_noalloc": (
        [C.POINTER(MoeWeights), _P, _P, _P, _P, _P, C.POINTER(MoeRoute), _I, _I, _I, _I, _I, _I, _P, _P, _P],
        _I,
    ),
    "moe_noalloc_scratch_bytes": ([], C.c_size_t),
    "moe_post_expert_finalize_tp": (
        [C.POINTER(C.c_void_p), _I, _I, _P, _P, _P, C.c_float, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_musespark1x_routing": ([_P, _P, _P, _I, _I, _I, C.c_float, C.c_float, _P, _P, _P], _I),
    "moe_rmsnorm_nvfp4_quant": ([_P, _P, C.c_float, _P, _I, _I, _P, _P, _P], _I),
    "moe_dense_bf16_workspace_size": ([_I, _I, _I, C.POINTER(C.c_size_t)], _I),
    "moe_dense_bf16": ([_P, _P, _I, _I, _I, _P, _P, C.c_size_t, _P, _P], _I),
    "moe_fp4_mma_rate": ([_I, _I, _I, _I, _I, _I, _I, C.POINTER(C.c_double), _P, _P], _I),
    "moe_fp4_mma_rate_pair": ([_I, _I, _I, C.POINTER(C.c_double), _P, _P], _I),
    "moe_selftest_wait_timeout": ([C.c_uint64, _P, _P, _P], _I),
    "moe_selftest_occupy": ([_I, _I, C.c_uint64, _P], _I),
    "moe_selftest_counter_timeout": ([C.c_uint64, _P, _P, _P, _P], _I),
    "moe_experts_norm_quantize": (
        [_P, _P, C.c_float, _P, C.POINTER(MoeRoute), _I, _I, _I, _I, _I, _I, _P, C.c_size_t, _P, _P], _I),
}

_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load the library (once). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise FileNotFoundError(
                f"{path} is missing: build it with `python -m nvfp4_mixture_experts_route_gb300.build`"
            )
        lib = C.CDLL(path)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


def declared_symbols() -> list[str]:
    """Entry points declared in include/moe_nvfp4.h."""
    import re

    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(moe_\w+)\s*\(", text, re.M)))


def _check(rc: int) -> None:
    if rc != MOE_OK:
        raise MoeError(rc, load().moe_last_error().decode())


# ---------------------------------------------------------------------------
# Torch-facing helpers: pointers, streams, allocation.
# ---------------------------------------------------------------------------
def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream=None) -> int:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def prepared_sizes(E: int, H: int, I: int) -> list[int]:
    out = (C.c_size_t * 4)()
    _check(load().moe_prepared_sizes(E, H, I, out))
    return list(out)


def prepare_weights(w13, w13_sf, w2, w2_sf, stream=None) -> dict:
    """Raw uint8 weight tensors on the device -> prepared tensors."""
    import torch

    E, twoI, half_h = w13.shape
    H, I = 2 * half_h, twoI // 2
    sizes = prepared_sizes(E, H, I)
    dev = w13.device
    out = {
        "w13": torch.empty((E, 2 * I, H // 2), dtype=torch.uint8, device=dev),
        "w13_sf": torch.empty((E, 2 * I // 128, H // 64, 512), dtype=torch.uint8, device=dev),
        "w2": torch.empty((E, H, I // 2), dtype=torch.uint8, device=dev),
        "w2_sf": torch.empty((E, H // 128, I // 64, 512), dtype=torch.uint8, device=dev),
    }
    assert [t.numel() for t in out.values()] == sizes
    for t in (w13, w13_sf, w2, w2_sf):
        assert t.is_contiguous() and t.dtype == torch.uint8
    _check(load().moe_prepare_weights(
        _ptr(w13), _ptr(w13_sf), _ptr(w2), _ptr(w2_sf), E, H, I,
        _ptr(out["w13"]), _ptr(out["w13_sf"]), _ptr(out["w2"]), _ptr(out["w2_sf"]), _stream(stream)))
    return out


def route_kernels(T: int, K: int, E: int) -> int:
    """Kernels route_permute launches for this shape (1 or 3)."""
    n = load().moe_route_kernels(T, K, E)
    if n < 0:
        _check(n)
    return n


def experts_kernels(tile_m: int) -> int:
    """Kernels nvfp4_experts launches for this route-tile size (2 or 3)."""
    n = load().moe_experts_kernels(tile_m)
    if n < 0:
        _check(n)
    return n


def routed_experts_kernels(T: int, K: int, E: int, tile_m: int) -> int:
    """Kernels nvfp4_experts_routed launches for these sizes (2 when the
    routing runs inside the input quantizer)."""
    n = load().moe_routed_experts_kernels(T, K, E, tile_m)
    if n < 0:
        _check(n)
    return n


def device_reads_host(t) -> bool:
    """Whether the library's kernels may read / write the host tensor `t`
    through its own address (page-locked, mapped at the same address)."""
    return bool(load().moe_device_reads_host(_ptr(t)))


def moe_block_kernels(T: int, K: int, E: int, tile_m: int) -> int:
    """Kernels moe_block launches for these sizes (3 when routing runs inside
    the input quantizer)."""
    n = load().moe_moe_block_kernels(T, K, E, tile_m)
    if n < 0:
        _check(n)
    return n


def route_sizes(T: int, K: int, E: int, tile_m: int) -> tuple[int, int]:
    P, MT = C.c_int(), C.c_int()
    _check(load().moe_route_sizes(T, K, E, tile_m, C.byref(P), C.byref(MT)))
    return P.value, MT.value


@dataclass
class Route:
    expert_counts: object
    expert_offsets: object
    expanded_to_permuted: object
    permuted_to_token: object
    tile_expert: object
    tile_row_limit: object
    totals: object
    tile_m: int

    def struct(self) -> MoeRoute:
        return MoeRoute(_ptr(self.permuted_to_token), _ptr(self.tile_expert), _ptr(self.tile_row_limit),
                        _ptr(self.totals), _ptr(self.expanded_to_permuted))


def alloc_route(T: int, K: int, E: int, tile_m: int, device) -> Route:
    import torch

    P, MT = route_sizes(T, K, E, tile_m)
    i32 = dict(dtype=torch.int32, device=device)
    return Route(
        torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty((T, K), **i32),
        torch.empty(max(P, 1), **i32), torch.empty(max(MT, 1), **i32), torch.empty(max(MT, 1), **i32),
        torch.empty(2, **i32), tile_m,
    )


def route_permute(topk_ids, E: int, tile_m: int, route: Route | None = None, status=None, stream=None) -> Route:
    T, K = topk_ids.shape
    r = route or alloc_route(T, K, E, tile_m, topk_ids.device)
    _check(load().moe_route_permute(
        _ptr(topk_ids), T, K, E, tile_m, _ptr(r.expert_counts), _ptr(r.expert_offsets),
        _ptr(r.expanded_to_permuted), _ptr(r.permuted_to_token), _ptr(r.tile_expert),
        _ptr(r.tile_row_limit), _ptr(r.totals), _ptr(status), _stream(stream)))
    return r


def weights_struct(p: dict, g1_alphas, g1_scale_c, g2_alphas) -> MoeWeights:
    return MoeWeights(_ptr(p["w13"]), _ptr(p["w13_sf"]), _ptr(p["w2"]), _ptr(p["w2_sf"]),
                      _ptr(g1_alphas), _ptr(g1_scale_c), _ptr(g2_alphas))


def experts_workspace_size(T, K, E, H, I, tile_m) -> int:
    n = C.c_size_t()
    _check(load().moe_experts_workspace_size(T, K, E, H, I, tile_m, C.byref(n)))
    return n.value


def alloc_workspace(T, K, E, H, I, tile_m, device):
    """A 1024-byte aligned uint8 workspace tensor (the caching allocator
    aligns to 512; one extra KiB is sliced to alignment)."""
    import torch

    n = experts_workspace_size(T, K, E, H, I, tile_m)
    raw = torch.empty(n + 1024, dtype=torch.uint8, device=device)
    off = (-raw.data_ptr()) % 1024
    return raw[off: off + n]


def nvfp4_experts_routed(w: MoeWeights, topk_ids, route: Route, *, x=None, a=None, a_sf=None, a1_gscale,
                         a2_gscale, H, I, E, gemm2_rows=None, ws=None, status=None, stream=None):
    """moe_nvfp4_experts_routed: routing into `route` (allocated with
    alloc_route) and the expert body, in one call."""
    import torch

    T, K = topk_ids.shape
    tile_m = route.tile_m
    P, _ = route_sizes(T, K, E, tile_m)
    dev = route.totals.device
    if gemm2_rows is None:
        gemm2_rows = torch.empty((max(P, 1), H), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = alloc_workspace(T, K, E, H, I, tile_m, dev)
    _check(load().moe_nvfp4_experts_routed(
        C.byref(w), _ptr(topk_ids), _ptr(x), _ptr(a), _ptr(a_sf), _ptr(a1_gscale), _ptr(a2_gscale), T, H, I, E,
        K, tile_m, _ptr(route.expert_counts), _ptr(route.expert_offsets), _ptr(route.expanded_to_permuted),
        _ptr(route.permuted_to_token), _ptr(route.tile_expert), _ptr(route.tile_row_limit), _ptr(route.totals),
        _ptr(gemm2_rows), _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))
    return gemm2_rows, ws


def moe_block(w: MoeWeights, topk_ids, topk_weights, route: Route, *, x=None, a=None, a_sf=None, a1_gscale,
              a2_gscale, gamma, eps: float, weight_before_norm: bool = True, H, I, E, gemm2_rows=None,
              row_sumsq=None, out=None, ws=None, status=None, stream=None):
    """moe_nvfp4_moe_block: routing into `route`, the expert body with the
    sums of squares fused into GEMM2 and the finalize, in one call. Returns
    (out, gemm2_rows, row_sumsq, ws)."""
    import torch

    T, K = topk_ids.shape
    tile_m = route.tile_m
    P, _ = route_sizes(T, K, E, tile_m)
    dev = route.totals.device
    if gemm2_rows is None:
        gemm2_rows = torch.empty((max(P, 1), H), dtype=torch.bfloat16, device=dev)
    if row_sumsq is None:
        row_sumsq = torch.empty((max(P, 1), H // 32), dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = alloc_workspace(T, K, E, H, I, tile_m, dev)
    _check(load().moe_nvfp4_moe_block(
        C.byref(w), _ptr(topk_ids), _ptr(topk_weights), _ptr(x), _ptr(a), _ptr(a_sf), _ptr(a1_gscale),
        _ptr(a2_gscale), _ptr(gamma), float(eps), 1 if weight_before_norm else 0, T, H, I, E, K, tile_m,
        _ptr(route.expert_counts), _ptr(route.expert_offsets), _ptr(route.expanded_to_permuted),
        _ptr(route.permuted_to_token), _ptr(route.tile_expert), _ptr(route.tile_row_limit), _ptr(route.totals),
        _ptr(gemm2_rows), _ptr(row_sumsq), _ptr(out), _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))
    return out, gemm2_rows, row_sumsq, ws


def nvfp4_experts(w: MoeWeights, route: Route, *, x=None, a=None, a_sf=None, a1_gscale, a2_gscale,
                  T, H, I, E, K, gemm2_rows=None, ws=None, status=None, stream=None):
    import torch

    tile_m = route.tile_m
    P, _ = route_sizes(T, K, E, tile_m)
    dev = route.totals.device
    if gemm2_rows is None:
        gemm2_rows = torch.empty((max(P, 1), H), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = alloc_workspace(T, K, E, H, I, tile_m, dev)
    rs = route.struct()
    _check(load().moe_nvfp4_experts(
        C.byref(w), _ptr(x), _ptr(a), _ptr(a_sf), _ptr(a1_gscale), _ptr(a2_gscale), C.byref(rs),
        T, H, I, E, K, tile_m, _ptr(gemm2_rows), _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))
    return gemm2_rows, ws


def nvfp4_experts_sumsq(w: MoeWeights, route: Route, *, x=None, a=None, a_sf=None, a1_gscale, a2_gscale,
                        T, H, I, E, K, gamma, weight_before_norm: bool = True, gemm2_rows=None, row_sumsq=None,
                        ws=None, status=None, stream=None):
    """The expert body with the post-expert norm's sums of squares fused into
    GEMM2 (see moe_nvfp4_experts_sumsq); returns (rows, row_sumsq, ws)."""
    import torch

    tile_m = route.tile_m
    P, _ = route_sizes(T, K, E, tile_m)
    dev = route.totals.device
    if gemm2_rows is None:
        gemm2_rows = torch.empty((max(P, 1), H), dtype=torch.bfloat16, device=dev)
    if row_sumsq is None:
        row_sumsq = torch.empty((max(P, 1), H // 32), dtype=torch.float32, device=dev)
    if ws is None:
        ws = alloc_workspace(T, K, E, H, I, tile_m, dev)
    rs = route.struct()
    _check(load().moe_nvfp4_experts_sumsq(
        C.byref(w), _ptr(x), _ptr(a), _ptr(a_sf), _ptr(a1_gscale), _ptr(a2_gscale), C.byref(rs),
        T, H, I, E, K, tile_m, _ptr(gemm2_rows), _ptr(gamma), 1 if weight_before_norm else 0, _ptr(row_sumsq),
        _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))
    return gemm2_rows, row_sumsq, ws


def experts_quantize(route: Route, ws, *, x=None, a=None, a_sf=None, a1_gscale=None, T, H, I, E, K,
                     status=None, stream=None):
    rs = route.struct()
    _check(load().moe_experts_quantize(_ptr(x), _ptr(a), _ptr(a_sf), _ptr(a1_gscale), C.byref(rs), T, H, I, E,
                                       K, route.tile_m, _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))


def experts_gemm1(w: MoeWeights, route: Route, ws, *, a2_gscale, T, H, I, E, K, status=None, stream=None):
    rs = route.struct()
    _check(load().moe_experts_gemm1(C.byref(w), _ptr(a2_gscale), C.byref(rs), T, H, I, E, K, route.tile_m,
                                    _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))


def experts_gemm2(w: MoeWeights, route: Route, ws, gemm2_rows, *, T, H, I, E, K, status=None, stream=None):
    rs = route.struct()
    _check(load().moe_experts_gemm2(C.byref(w), C.byref(rs), T, H, I, E, K, route.tile_m, _ptr(gemm2_rows),
                                    _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))


def experts_gemms(w: MoeWeights, route: Route, ws, gemm2_rows, *, a2_gscale, T, H, I, E, K, status=None,
                  stream=None):
    """GEMM1 and GEMM2 in one persistent launch (equal to experts_gemm1 then experts_gemm2)."""
    rs = route.struct()
    _check(load().moe_experts_gemms(C.byref(w), _ptr(a2_gscale), C.byref(rs), T, H, I, E, K, route.tile_m,
                                    _ptr(gemm2_rows), _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))


def experts_gemm2_sumsq(w: MoeWeights, route: Route, ws, gemm2_rows, row_sumsq, *, gamma,
                        weight_before_norm: bool = True, T, H, I, E, K, status=None, stream=None):
    rs = route.struct()
    _check(load().moe_experts_gemm2_sumsq(C.byref(w), C.byref(rs), T, H, I, E, K, route.tile_m, _ptr(gemm2_rows),
                                          _ptr(gamma), 1 if weight_before_norm else 0, _ptr(row_sumsq), _ptr(ws),
                                          ws.numel(), _ptr(status), _stream(stream)))


def experts_gemms_sumsq(w: MoeWeights, route: Route, ws, gemm2_rows, row_sumsq, *, a2_gscale, gamma,
                        weight_before_norm: bool = True, T, H, I, E, K, status=None, stream=None):
    rs = route.struct()
    _check(load().moe_experts_gemms_sumsq(C.byref(w), _ptr(a2_gscale), C.byref(rs), T, H, I, E, K, route.tile_m,
                                          _ptr(gemm2_rows), _ptr(gamma), 1 if weight_before_norm else 0,
                                          _ptr(row_sumsq), _ptr(ws), ws.numel(), _ptr(status), _stream(stream)))


def experts_export(which: int, ws, *, T, H, I, E, K, tile_m, stream=None):
    import torch

    P, _ = route_sizes(T, K, E, tile_m)
    Kc = I if which else H
    codes = torch.empty((P, Kc // 2), dtype=torch.uint8, device=ws.device)
    scales = torch.empty((P, Kc // 16), dtype=torch.uint8, device=ws.device)
    _check(load().moe_experts_export(which, _ptr(ws), ws.numel(), T, H, I, E, K, tile_m, _ptr(codes),
                                     _ptr(scales), _stream(stream)))
    return codes, scales


def experts_import(which: int, codes, scales, ws, *, T, H, I, E, K, tile_m, stream=None):
    _check(load().moe_experts_import(which, _ptr(codes), _ptr(scales), T, H, I, E, K, tile_m, _ptr(ws),
                                     ws.numel(), _stream(stream)))


def noalloc_scratch_bytes() -> int:
    return int(load().moe_noalloc_scratch_bytes())


def nvfp4_experts_noalloc(w: MoeWeights, route: Route, *, x=None, a=None, a_sf=None, a1_gscale, a2_gscale,
                          T, H, I, E, K, gemm2_rows=None, status=None, stream=None):
    """moe_nvfp4_experts on the library's own fixed device scratch array (no
    workspace argument, nothing allocated by the call itself)."""
    import torch

    P, _ = route_sizes(T, K, E, route.tile_m)
    if gemm2_rows is None:
        gemm2_rows = torch.empty((max(P, 1), H), dtype=torch.bfloat16, device=route.totals.device)
    rs = route.struct()
    _check(load().moe_nvfp4_experts_noalloc(
        C.byref(w), _ptr(x), _ptr(a), _ptr(a_sf), _ptr(a1_gscale), _ptr(a2_gscale), C.byref(rs),
        T, H, I, E, K, route.tile_m, _ptr(gemm2_rows), _ptr(status), _stream(stream)))
    return gemm2_rows


def post_expert_finalize(rows, expanded_to_permuted, topk_weights, gamma, eps: float,
                         weight_before_norm: bool = True, out=None, status=None, stream=None):
    """rows: bf16 [num_rows, H]; entries of expanded_to_permuted outside
    [-1, num_rows) are skipped and recorded in status (MOE_ERR_INVALID_ROUTE)."""
    import torch

    T, K = expanded_to_permuted.shape
    H = gamma.numel()
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=gamma.device)
    _check(load().moe_post_expert_finalize(
        _ptr(rows), rows.shape[0], _ptr(expanded_to_permuted), _ptr(topk_weights), _ptr(gamma), float(eps),
        1 if weight_before_norm else 0, T, K, H, _ptr(out), _ptr(status), _stream(stream)))
    return out


def post_expert_finalize_sumsq(rows, row_sumsq, expanded_to_permuted, topk_weights, gamma, eps: float, out=None,
                               status=None, stream=None):
    """Finalize from GEMM2's fused sums of squares (see the header)."""
    import torch

    T, K = expanded_to_permuted.shape
    H = gamma.numel()
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=gamma.device)
    _check(load().moe_post_expert_finalize_sumsq(
        _ptr(rows), _ptr(row_sumsq), min(rows.shape[0], row_sumsq.shape[0]), _ptr(expanded_to_permuted),
        _ptr(topk_weights), _ptr(gamma), float(eps), T, K, H, _ptr(out), _ptr(status), _stream(stream)))
    return out


def post_expert_finalize_tp(row_parts, expanded_to_permuted, topk_weights, gamma, eps: float,
                            weight_before_norm: bool = True, out=None, status=None, stream=None):
    """Finalize from tp K-partial row buffers (summed in fp32, one bf16
    rounding, before the norm)."""
    import torch

    T, K = expanded_to_permuted.shape
    H = gamma.numel()
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=gamma.device)
    arr = (C.c_void_p * len(row_parts))(*[r.data_ptr() for r in row_parts])
    num_rows = min(r.shape[0] for r in row_parts)
    _check(load().moe_post_expert_finalize_tp(
        arr, len(row_parts), num_rows, _ptr(expanded_to_permuted), _ptr(topk_weights), _ptr(gamma), float(eps),
        1 if weight_before_norm else 0, T, K, H, _ptr(out), _ptr(status), _stream(stream)))
    return out


def musespark1x_routing(logits, expert_bias, top_k: int, route_scale: float = 1.0, eps: float = 1e-15,
                        is_padding=None, topk_ids=None, topk_weights=None, stream=None):
    import torch

    T, E = logits.shape
    if topk_ids is None:
        topk_ids = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    if topk_weights is None:
        topk_weights = torch.empty((T, top_k), dtype=torch.float32, device=logits.device)
    _check(load().moe_musespark1x_routing(_ptr(logits), _ptr(expert_bias), _ptr(is_padding), T, E, top_k,
                                          float(route_scale), float(eps), _ptr(topk_ids), _ptr(topk_weights),
                                          _stream(stream)))
    return topk_ids, topk_weights


def rmsnorm_nvfp4_quant(x, gamma, eps: float, gscale, stream=None):
    import torch

    T, H = x.shape
    a = torch.empty((T, H // 2), dtype=torch.uint8, device=x.device)
    a_sf = torch.empty((T, H // 16), dtype=torch.uint8, device=x.device)
    _check(load().moe_rmsnorm_nvfp4_quant(_ptr(x), _ptr(gamma), float(eps), _ptr(gscale), T, H, _ptr(a),
                                          _ptr(a_sf), _stream(stream)))
    return a, a_sf


def experts_norm_quantize(route: Route, ws, *, x, gamma, eps: float, a1_gscale, T, H, I, E, K, status=None,
                          stream=None):
    rs = route.struct()
    _check(load().moe_experts_norm_quantize(_ptr(x), _ptr(gamma), float(eps), _ptr(a1_gscale), C.byref(rs), T,
                                            H, I, E, K, route.tile_m, _ptr(ws), ws.numel(), _ptr(status),
                                            _stream(stream)))


def dense_bf16_workspace_size(T: int, Din: int, Dout: int) -> int:
    n = C.c_size_t()
    _check(load().moe_dense_bf16_workspace_size(T, Din, Dout, C.byref(n)))
    return n.value


def dense_bf16(x, w, *, out=None, ws=None, status=None, stream=None):
    """Pooler / unpooler projection: bf16 y [T, Dout] = x [T, Din] . w[Dout, Din]^T."""
    import torch

    T, Din = x.shape
    Dout = w.shape[0]
    y = out if out is not None else torch.empty((T, Dout), dtype=torch.bfloat16, device=x.device)
    need = dense_bf16_workspace_size(T, Din, Dout)
    if need and ws is None:
        ws = torch.empty(need, dtype=torch.uint8, device=x.device)
    _check(load().moe_dense_bf16(_ptr(x), _ptr(w), T, Din, Dout, _ptr(y), _ptr(ws), ws.numel() if ws is not None else 0,
                                 _ptr(status), _stream(stream)))
    return y


def fp4_mma_rate(n: int, sf_copies: int, mmas_per_commit: int, ctas_per_sm: int, stages: int, status=None,
                 stream=None, ring: int = 3, warp_issue: bool = False) -> float:
    """Launch the dense NVFP4 tensor-core rate probe (see the header);
    returns the launch's FLOPs. Time it with events on the same stream."""
    f = C.c_double()
    _check(load().moe_fp4_mma_rate(n, int(sf_copies), mmas_per_commit, ctas_per_sm, ring, int(warp_issue), stages,
                                   C.byref(f), _ptr(status), _stream(stream)))
    return f.value


def fp4_mma_rate_pair(n: int, sf_copies: int, stages: int, status=None, stream=None) -> float:
    """Launch the pair-form (cta_group::2) rate probe (see the header);
    returns the launch's FLOPs. Time it with events on the same stream."""
    f = C.c_double()
    _check(load().moe_fp4_mma_rate_pair(n, int(sf_copies), stages, C.byref(f), _ptr(status), _stream(stream)))
    return f.value


def selftest_wait_timeout(limit_ns: int, status, result, stream=None) -> None:
    """Run the bounded-wait failure path (see the header); status int32 [1]
    and result int32 [3] on the device."""
    _check(load().moe_selftest_wait_timeout(int(limit_ns), _ptr(status), _ptr(result), _stream(stream)))


def selftest_counter_timeout(limit_ns: int, counter, status, result, stream=None) -> None:
    """The completion-counter wait's failure path on a counter that stays 0
    (see moe_selftest_counter_timeout)."""
    _check(load().moe_selftest_counter_timeout(int(limit_ns), _ptr(counter), _ptr(status), _ptr(result),
                                               _stream(stream)))



def selftest_occupy(ctas: int, smem_bytes: int, ns: int, stream=None) -> None:
    """Hold SMs for ns nanoseconds from another stream (see the header)."""
    _check(load().moe_selftest_occupy(int(ctas), int(smem_bytes), int(ns), _stream(stream)))
