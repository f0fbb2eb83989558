"""moe_nvfp4_experts_noalloc: the expert body on the library's own fixed
device scratch array, for callers that cannot allocate device memory (graph
capture, allocator-free serving loops, plug-ins given no memory).

Collected last on purpose (file name), so that a run stopping at the first
failure has already run every other test. Passes alone in a fresh process
(the first call sets up the scratch address) and after the other tests.
"""
import numpy as np
import pytest
import torch

from nvfp4_mixture_experts_route_gb300 import binding as B
from nvfp4_mixture_experts_route_gb300 import inputs

from _util import bf16_dev, rel_l2


def test_oversized_workspace_refused_before_any_work():
    """A shape whose workspace exceeds the fixed array is refused on the host
    with MOE_ERR_WORKSPACE; nothing is dereferenced or launched."""
    B.load()
    T, K, E, H, I, tile = 8192, 8, 128, 5120, 2048, 128
    assert B.experts_workspace_size(T, K, E, H, I, tile) > B.noalloc_scratch_bytes()
    w = B.MoeWeights(*([16] * 7))
    r = B.MoeRoute(16, 16, 16, 16)
    import ctypes as C

    rc = B.load().moe_nvfp4_experts_noalloc(C.byref(w), 16, None, None, 16, 16, C.byref(r), T, H, I, E, K,
                                           tile, 16, None, None)
    assert rc == -3 and b"workspace" in B.load().moe_last_error()


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_point_on_two_calls():
    dev = "cuda"
    w = inputs.Workload("noalloc_t37", T=37, H=512, I=256, E=8, K=4, routing="uniform", tile_m=32)
    raw = inputs.make_layer(w)
    batch = inputs.make_batch(w)
    a1, a2 = 4.0, 1e-3
    t = {k: torch.from_numpy(raw[k]).to(dev) for k in ("w13", "w13_sf", "w2", "w2_sf")}
    prep = B.prepare_weights(t["w13"], t["w13_sf"], t["w2"], t["w2_sf"])
    f32 = dict(dtype=torch.float32, device=dev)
    g1a, g1c, g2a = (torch.from_numpy(raw[k]).to(**f32) for k in ("g1_alphas", "g1_scale_c", "g2_alphas"))
    weights = B.weights_struct(prep, g1a, g1c, g2a)
    ids = torch.from_numpy(batch["topk_ids"]).to(dev)
    x = bf16_dev(batch["x"])
    s1, s2 = torch.tensor([a1], **f32), torch.tensor([a2], **f32)
    route = B.route_permute(ids, w.E, w.tile_m)
    dims = dict(T=w.T, H=w.H, I=w.I, E=w.E, K=w.K)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    want, _ = B.nvfp4_experts(weights, route, x=x, a1_gscale=s1, a2_gscale=s2, status=status, **dims)
    got1 = B.nvfp4_experts_noalloc(weights, route, x=x, a1_gscale=s1, a2_gscale=s2, status=status, **dims)
    got2 = B.nvfp4_experts_noalloc(weights, route, x=x, a1_gscale=s1, a2_gscale=s2, status=status, **dims)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    e2p = route.expanded_to_permuted.cpu().numpy().reshape(-1)
    live = torch.from_numpy(e2p[e2p >= 0]).to(dev)
    # The same deterministic kernels on the same operands, only the workspace
    # placed elsewhere: the live rows must be equal bit for bit (rel-L2 is
    # reported only to describe a mismatch).
    ref = want[live]
    for got in (got1, got2):
        assert torch.equal(got[live], ref), rel_l2(got[live].float().cpu().numpy(), ref.float().cpu().numpy())
