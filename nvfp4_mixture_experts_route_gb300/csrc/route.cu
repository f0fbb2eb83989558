// Routing metadata (step a2): per-expert histogram, padded offsets, the
// stable expanded->permuted map, permuted->token, and the tile tables.
//
// What is computed follows the flashinfer_ops page (FlashInferOps.slot names
// the tensors; gemm2_rows bounds the padded rows): counts[e], offsets as the
// exclusive prefix of ceil(counts/tile)*tile, routes of one expert in
// ascending expanded index j = t*K + k, tiles enumerated by (expert, index).
//
// For few routes one CTA of 1024 threads does it all, deterministically and
// without global atomics (many routes take the three-kernel path below): warp w owns a contiguous segment of the routes, so the order of
// its routes is the order of j. Pass 1 builds a warp-private histogram
// hist[w][e] (warp __match_any_sync groups equal experts in a 32-route chunk;
// the group leader adds the group size). A per-expert scan over the warps and
// a block scan over the experts turn it into each warp's first row per
// expert. Pass 2 walks the segment again and hands out rows in order (rank
// inside the chunk = peers below the lane).
#include "common.cuh"
#include "route_small.cuh"

namespace moe {

constexpr int kRouteThreads = 1024;
constexpr int kRouteWarps = kRouteThreads / 32;

template <int NT>
__global__ void __launch_bounds__(NT, 1)
    route_permute_kernel(const int32_t* __restrict__ topk_ids, int T, int K, int E, int tile_m,
                         int P, int MT, int32_t* __restrict__ expert_counts,
                         int32_t* __restrict__ expert_offsets,
                         int32_t* __restrict__ expanded_to_permuted,
                         int32_t* __restrict__ permuted_to_token, int32_t* __restrict__ tile_expert,
                         int32_t* __restrict__ tile_row_limit, int32_t* __restrict__ totals,
                         int32_t* status) {
  extern __shared__ int32_t hist[];  // [NT/32][E]
  // Launched in plain stream order; the kernels after it wait for it to
  // complete before they read what it writes.
  pdl_trigger();
  route_small<NT>(topk_ids, T, K, E, tile_m, P, MT, hist, true, expert_counts, expert_offsets,
                  expanded_to_permuted, permuted_to_token, tile_expert, tile_row_limit, totals, nullptr, nullptr,
                  nullptr, status);
}

// ---------------------------------------------------------------------------
// Many routes (prefill): three kernels over G segments of `seg` routes each,
// with the same result. Segment g's per-expert counts travel through
// expanded_to_permuted[g*seg .. g*seg+E) (a segment holds at least E routes),
// which is its own output region, so no scratch memory is needed:
//   count:   per-segment histogram (shared-memory atomics) into those slots;
//            also fills permuted_to_token and the tile tables with -1.
//   scan:    one CTA: per expert, the exclusive prefix over segments, the
//            counts, padded offsets, tile tables and totals; each slot becomes
//            the first row of its (segment, expert).
//   scatter: per segment, the single-CTA kernel's two passes (warp-private
//            histogram, rows handed out in ascending j) from those bases.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kRouteThreads) route_count_kernel(
    const int32_t* __restrict__ topk_ids, int R, int E, int seg, int P, int MT,
    int32_t* __restrict__ e2p, int32_t* __restrict__ permuted_to_token,
    int32_t* __restrict__ tile_expert, int32_t* __restrict__ tile_row_limit, int32_t* status) {
  extern __shared__ int32_t h[];  // [E]
  pdl_trigger();
  const int tid = threadIdx.x;
  const int beg = blockIdx.x * seg, end = min(R, beg + seg);
  for (int e = tid; e < E; e += kRouteThreads) h[e] = 0;
  const int nthreads = gridDim.x * kRouteThreads, gtid = blockIdx.x * kRouteThreads + tid;
  for (int i = gtid; i < P; i += nthreads) permuted_to_token[i] = -1;
  for (int i = gtid; i < MT; i += nthreads) {
    tile_expert[i] = -1;
    tile_row_limit[i] = -1;
  }
  __syncthreads();
  bool bad = false;
  for (int j = beg + tid; j < end; j += kRouteThreads) {
    const int e = topk_ids[j];
    if (e < -1 || e >= E)
      bad = true;
    else if (e >= 0)
      atomicAdd(&h[e], 1);
  }
  if (bad) record_status(status, MOE_ERR_INVALID_ROUTE);
  __syncthreads();
  for (int e = tid; e < E; e += kRouteThreads) e2p[beg + e] = h[e];
}

__global__ void __launch_bounds__(kRouteThreads, 1) route_scan_kernel(
    int E, int tile_m, int G, int seg, int32_t* __restrict__ e2p,
    int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_offsets,
    int32_t* __restrict__ tile_expert, int32_t* __restrict__ tile_row_limit,
    int32_t* __restrict__ totals) {
  __shared__ int32_t warp_sums[kRouteWarps];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Segments are read and written in batches of 8 so that the loads of a
  // batch are in flight together.
  constexpr int kBatch = 8;
  int count = 0, padded = 0;
  if (tid < E) {
    for (int g0 = 0; g0 < G; g0 += kBatch) {
      int c[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) c[u] = g0 + u < G ? e2p[(size_t)(g0 + u) * seg + tid] : 0;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (g0 + u < G) e2p[(size_t)(g0 + u) * seg + tid] = count;  // exclusive prefix
        count += c[u];
      }
    }
    padded = (count + tile_m - 1) / tile_m * tile_m;
  }
  int incl = padded;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += v;
  }
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int sw = warp_sums[lane];
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, sw, d);
      if (lane >= d) sw += v;
    }
    warp_sums[lane] = sw;
  }
  __syncthreads();
  const int offset = incl - padded + (warp > 0 ? warp_sums[warp - 1] : 0);
  const int total = warp_sums[kRouteWarps - 1];
  if (tid < E) {
    expert_counts[tid] = count;
    expert_offsets[tid] = offset;
    for (int g0 = 0; g0 < G; g0 += kBatch) {
      int c[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) c[u] = g0 + u < G ? e2p[(size_t)(g0 + u) * seg + tid] : 0;
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        if (g0 + u < G) e2p[(size_t)(g0 + u) * seg + tid] = c[u] + offset;
    }
    const int t0 = offset / tile_m, nt = padded / tile_m;
    for (int i = 0; i < nt; ++i) {
      tile_expert[t0 + i] = tid;
      tile_row_limit[t0 + i] = offset + count;
    }
  }
  if (tid == 0) {
    expert_offsets[E] = total;
    totals[0] = total / tile_m;
    totals[1] = total;
  }
}

__global__ void __launch_bounds__(kRouteThreads, 1) route_scatter_kernel(
    const int32_t* __restrict__ topk_ids, int R, int K, int E, int seg, int32_t* __restrict__ e2p,
    int32_t* __restrict__ permuted_to_token) {
  extern __shared__ int32_t hist[];  // [kRouteWarps][E]
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cbeg = blockIdx.x * seg, cend = min(R, cbeg + seg);
  const int wseg = (cend - cbeg + kRouteWarps - 1) / kRouteWarps;
  const int beg = min(cend, cbeg + warp * wseg), end = min(cend, beg + wseg);
  for (int i = tid; i < kRouteWarps * E; i += kRouteThreads) hist[i] = 0;
  __syncthreads();
  // Pass 1: warp-private histogram of this segment.
  int32_t* my = hist + warp * E;
  for (int base = beg; base < end; base += 32) {
    const int j = base + lane;
    int e = (j < end) ? topk_ids[j] : -1;
    if (e < -1 || e >= E) e = -1;
    const int key = (e >= 0) ? e : -2 - lane;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
  }
  __syncthreads();
  // Each warp's first row per expert: the segment's base plus the warps before.
  if (tid < E) {
    int run = e2p[cbeg + tid];
    for (int w = 0; w < kRouteWarps; ++w) {
      const int c = hist[w * E + tid];
      hist[w * E + tid] = run;
      run += c;
    }
  }
  __syncthreads();  // every base slot is read before pass 2 overwrites them
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
      e2p[j] = p;
      permuted_to_token[p] = j / K;
    } else if (j < end) {
      e2p[j] = -1;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) my[e] += __popc(peers);
    __syncwarp();
  }
}

// Segments for the many-route path: G = R / kSegRoutes of ceil(R / G) routes,
// taken only when there are at least two and the last holds E slots.
constexpr int kSegRoutes = 2048;
static bool multi_segments(int R, int E, int* G, int* seg) {
  const int g = R / kSegRoutes;
  if (g < 2) return false;
  const int s = (R + g - 1) / g;
  if (R - (g - 1) * s < E) return false;
  *G = g;
  *seg = s;
  return true;
}

size_t route_smem_bytes(int E) { return sizeof(int32_t) * kRouteWarps * (size_t)E; }

int route_kernel_count(int T, int K, int E) {
  int G = 0, seg = 0;
  return multi_segments(T * K, E, &G, &seg) ? 3 : 1;
}

cudaError_t launch_route_permute(const int32_t* topk_ids, int T, int K, int E, int tile_m, int P,
                                 int MT, int32_t* counts, int32_t* offsets, int32_t* e2p,
                                 int32_t* p2t, int32_t* tile_expert, int32_t* tile_row_limit,
                                 int32_t* totals, int32_t* status, cudaStream_t stream) {
  const size_t smem = route_smem_bytes(E);
  int G = 0, seg = 0;
  if (multi_segments(T * K, E, &G, &seg)) {
    cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(route_scatter_kernel),
                                        (int)route_smem_bytes(1024));
    if (err != cudaSuccess) return err;
    route_count_kernel<<<G, kRouteThreads, sizeof(int32_t) * (size_t)E, stream>>>(
        topk_ids, T * K, E, seg, P, MT, e2p, p2t, tile_expert, tile_row_limit, status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    err = launch_kernel(route_scan_kernel, dim3(1), dim3(kRouteThreads), 0, stream, true, E, tile_m, G,
                        seg, e2p, counts, offsets, tile_expert, tile_row_limit, totals);
    if (err != cudaSuccess) return err;
    return launch_kernel(route_scatter_kernel, dim3(G), dim3(kRouteThreads), smem, stream, true,
                         topk_ids, T * K, K, E, seg, e2p, p2t);
  }
  if (T * K <= 2048 && E <= 256) {
    route_permute_kernel<256><<<1, 256, sizeof(int32_t) * 8 * (size_t)E, stream>>>(
        topk_ids, T, K, E, tile_m, P, MT, counts, offsets, e2p, p2t, tile_expert, tile_row_limit,
        totals, status);
    return cudaGetLastError();
  }
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(route_permute_kernel<kRouteThreads>),
                                      (int)route_smem_bytes(1024));
  if (err != cudaSuccess) return err;
  route_permute_kernel<kRouteThreads><<<1, kRouteThreads, smem, stream>>>(
      topk_ids, T, K, E, tile_m, P, MT, counts, offsets, e2p, p2t, tile_expert, tile_row_limit,
      totals, status);
  return cudaGetLastError();
}

}  // namespace moe
