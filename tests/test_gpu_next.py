"""GPU parity of the steps around the expert block: MuseSpark1x routing, the
fused pre-expert RMSNorm + NVFP4 quant, and the expert-TP tail finalize."""
import numpy as np
import pytest
import torch

from oracle import codecs, layer as olayer, router as orouter
from nvfp4_mixture_experts_route_gb300 import binding as B
from nvfp4_mixture_experts_route_gb300 import inputs

from _util import bf16_dev, bf16_host_f64, canon_codes, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("T,E,K,bias_sd", [(64, 128, 8, 0.05), (8, 1024, 32, 0.2), (33, 72, 6, 0.0), (5, 8, 8, 1.0)])
def test_musespark1x_routing_parity(T, E, K, bias_sd):
    rng = np.random.default_rng(T + E)
    logits = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    bias = (rng.standard_normal(E) * bias_sd).astype(np.float32)
    pad = np.zeros(T, np.uint8)
    pad[1::5] = 1
    ids, w = B.musespark1x_routing(torch.from_numpy(logits).to(DEV), torch.from_numpy(bias).to(DEV), K,
                                   is_padding=torch.from_numpy(pad).to(DEV))
    torch.cuda.synchronize()
    want_ids, want_w = orouter.musespark1x_routing(logits, bias, K, is_padding=pad.astype(bool))
    got_ids = ids.cpu().numpy()
    # the choice is unique unless two choice values tie within fp32 rounding
    s = orouter.sigmoid_f32(logits)
    c = np.sort(s + bias, axis=1)[:, ::-1]
    clear = (c[:, K - 1] - c[:, K] > 1e-6) if K < E else np.ones(T, bool)
    rows = clear | pad.astype(bool)
    assert np.array_equal(got_ids[rows], want_ids[rows])
    assert np.allclose(w.cpu().numpy()[rows], want_w[rows], rtol=2e-6, atol=1e-7)
    # whatever the order, every chosen set is valid: K distinct in-range experts
    live = ~pad.astype(bool)
    assert all(len(set(r)) == K and r.min() >= 0 and r.max() < E for r in got_ids[live])


def test_routing_feeds_the_block_end_to_end():
    w = inputs.WORKLOADS["tiny_t4"]
    raw = inputs.make_layer(w)
    batch = inputs.make_batch(w)
    rng = np.random.default_rng(9)
    logits = rng.standard_normal((w.T, w.E)).astype(np.float32)
    bias = np.zeros(w.E, np.float32)
    ids, tw = B.musespark1x_routing(torch.from_numpy(logits).to(DEV), torch.from_numpy(bias).to(DEV), w.K)
    from nvfp4_mixture_experts_route_gb300.layer import NvFp4MoE

    moe = NvFp4MoE(raw, 1.0, 1.0, raw["gamma"], tile_m=w.tile_m)
    out, _ = moe.forward(bf16_dev(batch["x"]), ids, tw)
    torch.cuda.synchronize()
    want_ids, want_w = orouter.musespark1x_routing(logits, bias, w.K)
    assert np.array_equal(ids.cpu().numpy(), want_ids)
    ref = olayer.moe_layer(batch["x"], want_ids, want_w.astype(np.float32), raw, 1.0, 1.0, raw["gamma"], 1e-6,
                           w.tile_m)
    assert rel_l2(bf16_host_f64(out), ref["out"]) < 1e-2


@pytest.mark.parametrize("T,H,gs,scale", [(4, 256, 1.0, 1.0), (37, 5120, 618.8201293945312, 3.0), (9, 1024, 2.0, 1e3),
                                          (5, 6144, 4.0, 1.0)])  # H > 5120: one CTA per row
def test_rmsnorm_nvfp4_quant_parity(T, H, gs, scale):
    rng = np.random.default_rng(T * H)
    x = inputs._to_bf16_bits(rng.standard_normal((T, H)) * scale)
    gamma = inputs._to_bf16_bits(rng.standard_normal(H) * 0.1)
    g = torch.tensor([gs], dtype=torch.float32, device=DEV)
    a, a_sf = B.rmsnorm_nvfp4_quant(bf16_dev(x), bf16_dev(gamma), 1e-6, g)
    torch.cuda.synchronize()
    y, codes, sf = orouter.rmsnorm_nvfp4(x, gamma, 1e-6, gs)
    got_codes = canon_codes(codecs.unpack_nibbles(a.cpu().numpy()))
    got_sf = a_sf.cpu().numpy()
    # y is fp32 on the GPU and fp64 here: codes agree except at rare rounding boundaries
    assert np.mean(got_sf == sf) > 0.999
    assert np.mean(got_codes == canon_codes(codes)) > 0.999
    deq = codecs.e2m1_decode(got_codes).reshape(T, H // 16, 16) * codecs.e4m3_decode(got_sf)[..., None]
    want = codecs.e2m1_decode(codes).reshape(T, H // 16, 16) * codecs.e4m3_decode(sf)[..., None]
    assert rel_l2(deq, want) < 1e-3


@pytest.mark.parametrize("T,H,I,E,K,tile,routing", [
    (21, 512, 128, 8, 4, 32, "uniform"),
    (300, 5120, 256, 16, 8, 128, "zipf"),     # a CTA per permuted row, 128-row tiles
    (600, 5120, 256, 16, 8, 128, "zipf"),     # one warp per token
    (9, 6144, 128, 8, 2, 64, "uniform"),      # H > 5120: one CTA per permuted row
])
def test_norm_quantize_into_permuted_workspace_equals_gathered_linear(T, H, I, E, K, tile, routing):
    """moe_experts_norm_quantize writes exactly the row-major kernel's codes
    and scales of each route's token into its permuted row, and zero scales
    into every padding row of the tiles in use."""
    rng = np.random.default_rng(4)
    x = bf16_dev(inputs._to_bf16_bits(rng.standard_normal((T, H))))
    gamma = bf16_dev(inputs._to_bf16_bits(rng.standard_normal(H) * 0.1))
    g = torch.tensor([3.0], dtype=torch.float32, device=DEV)
    ids = torch.from_numpy(inputs.draw_topk(rng, T, E, K, routing)).to(DEV)
    r = B.route_permute(ids, E, tile)
    ws = B.alloc_workspace(T, K, E, H, I, tile, DEV)
    B.experts_norm_quantize(r, ws, x=x, gamma=gamma, eps=1e-6, a1_gscale=g, T=T, H=H, I=I, E=E, K=K)
    codes, scales = B.experts_export(0, ws, T=T, H=H, I=I, E=E, K=K, tile_m=tile)
    a, a_sf = B.rmsnorm_nvfp4_quant(x, gamma, 1e-6, g)
    torch.cuda.synchronize()
    p2t = r.permuted_to_token.cpu().numpy()
    total = int(r.totals[1].item())
    live = np.nonzero(p2t[:total] >= 0)[0]
    pad = np.nonzero(p2t[:total] < 0)[0]
    assert np.array_equal(codes.cpu().numpy()[live], a.cpu().numpy()[p2t[live]])
    assert np.array_equal(scales.cpu().numpy()[live], a_sf.cpu().numpy()[p2t[live]])
    assert not scales.cpu().numpy()[pad].any()


@pytest.mark.parametrize("nparts,H,T,K", [(8, 5120, 6, 4), (4, 256, 6, 4), (1, 1024, 6, 4),
                                          # many tokens: the persistent kernel that streams every
                                          # route's part rows through a shared-memory ring
                                          (8, 5120, 1024, 4), (3, 2048, 1100, 4), (2, 4096, 1030, 4),
                                          # more than 32 routes per token
                                          (2, 512, 1024, 36)])
def test_expert_tp_tail_finalize(nparts, H, T, K):
    rng = np.random.default_rng(nparts * H + T)
    P = T * K + 3
    parts = [inputs._to_bf16_bits(rng.standard_normal((P, H)) / np.sqrt(nparts)) for _ in range(nparts)]
    gamma = inputs._to_bf16_bits(rng.standard_normal(H) * 0.5)
    e2p = rng.permutation(P)[: T * K].reshape(T, K).astype(np.int32)
    e2p[2, 1] = -1
    e2p[5, :] = -1  # a token with no route: a zero row
    w = rng.random((T, K)).astype(np.float32)
    summed = sum(codecs.bf16_bits_to_f64(p).astype(np.float32) for p in parts)
    rows = codecs.round_to_bf16(summed.astype(np.float64))
    want = olayer.finalize(rows, e2p, w, gamma, 1e-6)
    dev_parts = [bf16_dev(p) for p in parts]
    got = B.post_expert_finalize_tp(dev_parts, torch.from_numpy(e2p).to(DEV), torch.from_numpy(w).to(DEV),
                                    bf16_dev(gamma), 1e-6)
    torch.cuda.synchronize()
    assert rel_l2(bf16_host_f64(got), want["out"]) < 2e-3
    # per element: at most one bf16 step from the correctly rounded value
    rms = np.sqrt(np.mean(want["out"] ** 2))
    assert (np.abs(bf16_host_f64(got) - want["out_bf16"]) <= np.abs(want["out_bf16"]) * 2.0**-7 + 1e-4 * rms).all()
    if nparts == 1:
        one = B.post_expert_finalize(dev_parts[0], torch.from_numpy(e2p).to(DEV), torch.from_numpy(w).to(DEV),
                                     bf16_dev(gamma), 1e-6)
        assert torch.equal(one, got)
