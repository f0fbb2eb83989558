// The single-CTA routing of few routes (step a2), shared by the routing
// kernel (route.cu) and the fused routing + quantization kernel (quant.cu).
// Warp w of the CTA owns a contiguous segment of the routes; pass 1 builds a
// warp-private histogram (__match_any_sync groups equal experts in a chunk of
// 32 routes, the group leader adds the group size); a scan over the warps and
// one over the experts give each warp its first row per expert; pass 2 hands
// out rows in ascending expanded index j = t*K + k.
#pragma once
#include "common.cuh"

namespace moe {

// The single-CTA routing, NT threads (E <= NT): 1024 in general, 256 for few
// routes and experts, where the per-expert scans over the warps and the
// block barriers are the latency. hist: shared memory [NT/32][E]. With
// write_global the metadata go to the caller's buffers (counts, offsets,
// expanded_to_permuted, permuted_to_token, the tile tables, totals); the
// fused routing + quantization kernel (quant.cu) also asks for a copy in its
// own shared memory (e2p_s [R], limit_s [MT], totals_s [2]; null if not).
template <int NT>
__device__ __forceinline__ void route_small(const int32_t* __restrict__ topk_ids, int T, int K, int E, int tile_m,
                                            int P, int MT, int32_t* hist, bool write_global,
                                            int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_offsets,
                                            int32_t* __restrict__ expanded_to_permuted,
                                            int32_t* __restrict__ permuted_to_token, int32_t* __restrict__ tile_expert,
                                            int32_t* __restrict__ tile_row_limit, int32_t* __restrict__ totals,
                                            int32_t* e2p_s, int32_t* limit_s, int32_t* totals_s, int32_t* status) {
  constexpr int NW = NT / 32;
  __shared__ int32_t warp_sums[NW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = T * K;
  const int seg = (R + NW - 1) / NW;
  const int beg = min(R, warp * seg), end = min(R, beg + seg);

  for (int i = tid; i < NW * E; i += NT) hist[i] = 0;
  if (write_global) {
    for (int i = tid; i < P; i += NT) permuted_to_token[i] = -1;
    for (int i = tid; i < MT; i += NT) {
      tile_expert[i] = -1;
      tile_row_limit[i] = -1;
    }
  }
  if (limit_s != nullptr)
    for (int i = tid; i < MT; i += NT) limit_s[i] = -1;
  __syncthreads();

  // Pass 1: warp-private histogram.
  int32_t* my = hist + warp * E;
  bool bad = false;
  for (int base = beg; base < end; base += 32) {
    const int j = base + lane;
    int e = (j < end) ? topk_ids[j] : -1;
    if (e < -1 || e >= E) {
      bad = true;
      e = -1;
    }
    // Lanes without a route get a key no expert uses, unique per lane.
    const int key = (e >= 0) ? e : -2 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
  }
  if (bad && write_global) record_status(status, MOE_ERR_INVALID_ROUTE);
  __syncthreads();

  // Per expert: scan over warps (warp-relative starts) and the padded count.
  int padded = 0, count = 0;
  if (tid < E) {
    for (int w = 0; w < NW; ++w) {
      const int c = hist[w * E + tid];
      hist[w * E + tid] = count;
      count += c;
    }
    padded = (count + tile_m - 1) / tile_m * tile_m;
  }
  // Block-wide exclusive scan of padded over the experts (E <= NT).
  int incl = padded;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int sw = lane < NW ? warp_sums[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, sw, d);
      if (lane >= d) sw += v;
    }
    if (lane < NW) warp_sums[lane] = sw;  // inclusive over warps
  }
  __syncthreads();
  const int offset = incl - padded + (warp > 0 ? warp_sums[warp - 1] : 0);
  const int total = warp_sums[NW - 1];
  if (tid < E) {
    for (int w = 0; w < NW; ++w) hist[w * E + tid] += offset;
    // Tiles of this expert: [offset/tile_m, (offset+padded)/tile_m).
    const int t0 = offset / tile_m, nt = padded / tile_m;
    if (write_global) {
      expert_counts[tid] = count;
      expert_offsets[tid] = offset;
      for (int i = 0; i < nt; ++i) {
        tile_expert[t0 + i] = tid;
        tile_row_limit[t0 + i] = offset + count;
      }
    }
    if (limit_s != nullptr)
      for (int i = 0; i < nt; ++i) limit_s[t0 + i] = offset + count;
  }
  if (tid == 0) {
    if (write_global) {
      expert_offsets[E] = total;
      totals[0] = total / tile_m;
      totals[1] = total;
    }
    if (totals_s != nullptr) {
      totals_s[0] = total / tile_m;
      totals_s[1] = total;
    }
  }
  __syncthreads();

  // Pass 2: hand out rows in ascending j.
  for (int base = beg; base < end; base += 32) {
    const int j = base + lane;
    int e = (j < end) ? topk_ids[j] : -1;
    if (e < -1 || e >= E) e = -1;
    const int key = (e >= 0) ? e : -2 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (e >= 0) {
      const int rank = __popc(peers & ((1u << lane) - 1u));
      const int p = my[e] + rank;
      if (write_global) {
        expanded_to_permuted[j] = p;
        permuted_to_token[p] = j / K;
      }
      if (e2p_s != nullptr) e2p_s[j] = p;
    } else if (j < end) {
      if (write_global) expanded_to_permuted[j] = -1;
      if (e2p_s != nullptr) e2p_s[j] = -1;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
}

}  // namespace moe
