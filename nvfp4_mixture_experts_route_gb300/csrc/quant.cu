// Step a1: NVFP4 quantization of the activations, written straight into the
// permuted, padded row order the grouped GEMMs read (the "model" page's
// scaled_fp4_quant(x, a1_gscale, is_sf_swizzled_layout=False), then the
// routing's permutation, in one pass).
//
// Per 16-element block, every step one correctly rounded fp32 operation:
//   s = (amax * g) / 6;  sf = e4m3_rn_satfinite(s);  inv = g / float(sf);
//   q_i = e2m1_rn_satfinite(v_i * inv)   (all codes 0 when sf decodes to 0)
//
// Workspace layout of a quantized operand with K columns, P permuted rows in
// tiles of tile_m rows (S = ceil(tile_m / 128) scale atoms per tile column):
//   codes  uint8 [P, K/2], row-major
//   scales uint8 [P/tile_m, K/64, S, 512]: for row i of tile tau, block b:
//          byte ((tau*K/64 + b/4)*S + i/128)*512 + 16*(i%32) + 4*((i%128)/32) + b%4
// i.e. the tcgen05 scale atom of each K=64 step of each 128-row group of a
// tile, so one bulk copy per pipeline stage brings every scale of the tile.
#include "common.cuh"
#include "layout.cuh"
#include "route_small.cuh"

namespace moe {

// Routes up to which routing runs inside the input quantizer: every CTA
// redoes it, so it must stay a few microseconds of one CTA's work.
constexpr int kFusedMaxRoutes = 2048;

__device__ __forceinline__ void quantize_block16(const float (&v)[16], float g, uint32_t& lo,
                                                 uint32_t& hi, uint32_t& sf_code) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const float s = (amax * g) / 6.0f;
  sf_code = f32_to_e4m3(s);
  const float sfv = e4m3_to_f32(sf_code);
  lo = hi = 0;
  if (sfv > 0.f) {
    const float inv = g / sfv;
#pragma unroll
    for (int i = 0; i < 8; i += 2) lo |= f32x2_to_e2m1x2(v[i] * inv, v[i + 1] * inv) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; i += 2)
      hi |= f32x2_to_e2m1x2(v[8 + i] * inv, v[9 + i] * inv) << (4 * i);
  }
}

// Token work item (a warp, token t, chunk j): lane l quantizes the BPL
// adjacent blocks from b = 32 BPL j + BPL l of the token once and writes
// their 8 BPL code bytes to the row of each of the token's routes with one
// store; the first lane of each 4-block group writes the group's 4 scale
// bytes (contiguous in the scale atom). Two blocks per lane (the standalone
// kernel) halve the per-route lookups, address arithmetic and store
// instructions per byte, which bound it at one block per lane. Lanes k and
// k + 32 of the item first look up route k's permuted row (expanded_to_
// permuted) and the offset of that row's scale bytes for block 0, so the
// per-block work is a shuffle and the stores. Padding work item (a warp,
// tile tau, group c): lane i zeroes the 4 scale bytes of rows 32j + i
// (j < tile_m / 32) of the tile that lie past its row limit; with a zero
// block scale the codes, always finite e2m1 values, contribute exactly 0 to
// every product, so padding-row codes are never written. The padding items
// come first, then the token items. Reads x once; writes each route row once.
//
// A route row outside [-1, P) is skipped and recorded in *status as
// MOE_ERR_INVALID_ROUTE (by the token's first chunk item).
// e2p and tile_row_limit may point to global or shared memory (the fused
// routing + quantization kernel keeps its own copy of the routing there);
// n_tiles is the number of route tiles in use.
template <int BPL>
__device__ __forceinline__ void quantize_permute_items(
    const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ a_in,
    const uint8_t* __restrict__ a_sf_in, const float* __restrict__ gscale, const int32_t* e2p,
    const int32_t* tile_row_limit, int n_tiles, int T, int K, int H, int tile_m, int P, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, int32_t* __restrict__ done, int n_done, int32_t* status) {
  // the per-tile GEMM1 completion counters and the unit ticket of the
  // one-launch expert GEMMs that follow
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n_done; i += gridDim.x * blockDim.x) done[i] = 0;
  const int ng = H / 64;  // four-block groups per row
  const int nb = H / 16;
  const float g = (x != nullptr) ? *gscale : 0.f;
  const int S = sf_atoms_per_tile(tile_m);
  const int lane = threadIdx.x & 31;
  const int warp0 = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * (blockDim.x / 32);
  // Padding: one warp per (tile, group).
  {
    const int n_pad = n_tiles * ng;
    for (int w = warp0; w < n_pad; w += nwarps) {
      const int tau = w / ng, c = w - (w / ng) * ng;
      const int limit = tile_row_limit[tau];
      for (int j = 0; j < tile_m; j += 32) {
        const int p = tau * tile_m + j + lane;
        if (p >= limit)
          *reinterpret_cast<uint32_t*>(scales + act_sf_offset(p, 4 * c, tile_m, ng, S)) = 0u;
      }
    }
  }
  // Tokens: one warp per (token, chunk of 32 BPL blocks), lane l taking the
  // BPL adjacent blocks b0 = 32 BPL j + BPL l, ... . nb is a multiple of 8,
  // so a lane's blocks, and a quad's lanes, are all in range or all out of it.
  const int nchunks = (nb + 32 * BPL - 1) / (32 * BPL);
  constexpr unsigned kFull = 0xFFFFFFFFu;
  constexpr int kQuadLanes = 4 / BPL;  // lanes holding one 4-block group
  const size_t group_step = (size_t)S * kAtomBytes;  // scale bytes between consecutive 4-block groups
  for (int w = warp0; w < T * nchunks; w += nwarps) {
    const int t = w / nchunks, j = w - t * nchunks;
    // routes k = lane and lane + 32: permuted row and its block-0 scale offset
    int p_lo = -1, p_hi = -1;
    size_t s_lo = 0, s_hi = 0;
    if (lane < K) {
      p_lo = e2p[(size_t)t * K + lane];
      if (p_lo < -1 || p_lo >= P) {
        if (j == 0) record_status(status, MOE_ERR_INVALID_ROUTE);
        p_lo = -1;
      }
      if (p_lo >= 0) s_lo = act_sf_offset(p_lo, 0, tile_m, ng, S);
    }
    if (lane + 32 < K) {
      p_hi = e2p[(size_t)t * K + lane + 32];
      if (p_hi < -1 || p_hi >= P) {
        if (j == 0) record_status(status, MOE_ERR_INVALID_ROUTE);
        p_hi = -1;
      }
      if (p_hi >= 0) s_hi = act_sf_offset(p_hi, 0, tile_m, ng, S);
    }
    const int b0 = 32 * BPL * j + BPL * lane;
    const bool on = b0 < nb;  // every lane stays for the warp-wide shuffles
    uint32_t q[2 * BPL];      // the lane's code words, block i in q[2i], q[2i+1]
    uint32_t sf_mine = 0;     // its scale bytes, block i in byte i
#pragma unroll
    for (int i = 0; i < 2 * BPL; ++i) q[i] = 0u;
    if (on && x != nullptr) {
      const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H + 16 * b0);
      uint4 u[2 * BPL];
#pragma unroll
      for (int i = 0; i < 2 * BPL; ++i) u[i] = src[i];
#pragma unroll
      for (int i = 0; i < BPL; ++i) {
        const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&u[2 * i]);
        const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&u[2 * i + 1]);
        float v[16];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f0 = __bfloat1622float2(h0[e]);
          const float2 f1 = __bfloat1622float2(h1[e]);
          v[2 * e] = f0.x;
          v[2 * e + 1] = f0.y;
          v[8 + 2 * e] = f1.x;
          v[8 + 2 * e + 1] = f1.y;
        }
        uint32_t sfc;
        quantize_block16(v, g, q[2 * i], q[2 * i + 1], sfc);
        sf_mine |= sfc << (8 * i);
      }
    } else if (on) {
#pragma unroll
      for (int i = 0; i < BPL; ++i) {
        const uint2 c = *reinterpret_cast<const uint2*>(a_in + (size_t)t * (H / 2) + 8 * (b0 + i));
        q[2 * i] = c.x;
        q[2 * i + 1] = c.y;
        sf_mine |= (uint32_t)a_sf_in[(size_t)t * nb + b0 + i] << (8 * i);
      }
    }
    // the quad's four scale bytes, block 4 * (b0 / 4) in the low byte
    const int base = lane & ~(kQuadLanes - 1);
    uint32_t sf4 = 0;
#pragma unroll
    for (int r = 0; r < kQuadLanes; ++r) sf4 |= __shfl_sync(kFull, sf_mine, base + r) << (8 * BPL * r);
    const size_t sf_b = (size_t)(b0 >> 2) * group_step;
    const bool quad_first = (lane & (kQuadLanes - 1)) == 0;
    for (int k = 0; k < K; ++k) {
      const int p = __shfl_sync(kFull, k < 32 ? p_lo : p_hi, k & 31);
      if (p < 0) continue;  // the same p in every lane
      const size_t so = __shfl_sync(kFull, k < 32 ? s_lo : s_hi, k & 31);
      if (on) {
        uint8_t* dst = codes + (size_t)p * (H / 2) + 8 * b0;
        if constexpr (BPL == 2)
          *reinterpret_cast<uint4*>(dst) = make_uint4(q[0], q[1], q[2], q[3]);
        else
          *reinterpret_cast<uint2*>(dst) = make_uint2(q[0], q[1]);
        if (quad_first) *reinterpret_cast<uint32_t*>(scales + so + sf_b) = sf4;
      }
    }
  }
}

__global__ void __launch_bounds__(256) quantize_permute_kernel(
    const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ a_in,
    const uint8_t* __restrict__ a_sf_in, const float* __restrict__ gscale,
    const int32_t* __restrict__ e2p, const int32_t* __restrict__ tile_row_limit,
    const int32_t* __restrict__ totals, int T, int K, int H, int tile_m, int P, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales, int32_t* __restrict__ done, int n_done, int32_t* status) {
  pdl_wait();
  pdl_trigger();
  quantize_permute_items<2>(x, a_in, a_sf_in, gscale, e2p, tile_row_limit, totals[0], T, K, H, tile_m, P, codes,
                            scales, done, n_done, status);
}

// Steps a2 and a1 in one kernel, for few routes (T*K <= kFusedMaxRoutes,
// E <= 256): every CTA runs the single-CTA routing into its own shared
// memory (a few microseconds of work, far less than a kernel boundary on
// the step's critical path), CTA 0 also writes the routing metadata out,
// and each CTA then quantizes its share of the items from its shared copy.
// The results equal the routing kernel's followed by quantize_permute_kernel.
// Shared memory: hist [8][E], e2p_s [T*K], limit_s [MT], totals_s [2].
__global__ void __launch_bounds__(256) route_quantize_kernel(
    const int32_t* __restrict__ topk_ids, int T, int K, int E, int tile_m, int P, int MT,
    int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_offsets,
    int32_t* __restrict__ expanded_to_permuted, int32_t* __restrict__ permuted_to_token,
    int32_t* __restrict__ tile_expert, int32_t* __restrict__ tile_row_limit, int32_t* __restrict__ totals,
    const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ a_in, const uint8_t* __restrict__ a_sf_in,
    const float* __restrict__ gscale, int H, uint8_t* __restrict__ codes, uint8_t* __restrict__ scales,
    int32_t* __restrict__ done, int32_t* status) {
  extern __shared__ int32_t rq_smem[];
  int32_t* hist = rq_smem;
  int32_t* e2p_s = hist + 8 * E;
  int32_t* limit_s = e2p_s + T * K;
  int32_t* totals_s = limit_s + MT;
  // the previous kernel in the stream may still read what CTA 0 writes
  pdl_wait();
  const bool writer = blockIdx.x == 0;
  route_small<256>(topk_ids, T, K, E, tile_m, P, MT, hist, writer, expert_counts, expert_offsets,
                   expanded_to_permuted, permuted_to_token, tile_expert, tile_row_limit, totals, e2p_s, limit_s,
                   totals_s, status);
  // The GEMMs that follow read the route totals and tile table as a prefetch
  // hint before they wait for this grid (and again, for their work, after):
  // push CTA 0's copy out before this grid lets them launch.
  if (writer) __threadfence();
  pdl_trigger();
  quantize_permute_items<1>(x, a_in, a_sf_in, gscale, e2p_s, limit_s, totals_s[0], T, K, H, tile_m, P, codes,
                            scales, done, MT + 1, status);
}

// Scale atoms <-> row-major scales [rows, K/16].
__global__ void act_scales_io_kernel(int to_linear, uint8_t* __restrict__ atoms,
                                     uint8_t* __restrict__ linear, int rows, int K, int tile_m) {
  const int nb = K / 16;
  const int S = sf_atoms_per_tile(tile_m);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
       idx < (long long)rows * nb; idx += (long long)gridDim.x * blockDim.x) {
    const int p = (int)(idx / nb), b = (int)(idx % nb);
    const size_t o = act_sf_offset(p, b, tile_m, K / 64, S);
    if (to_linear)
      linear[idx] = atoms[o];
    else
      atoms[o] = linear[idx];
  }
}

static int grid_for(long long work, int threads) {
  long long g = (work + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > 152 * 16) g = 152 * 16;
  return (int)g;
}

cudaError_t launch_quantize_permute(const void* x, const void* a, const void* a_sf,
                                    const float* a1_gscale, const int32_t* e2p,
                                    const int32_t* tile_row_limit, const int32_t* totals, int T,
                                    int K, int H, int tile_m, int P, int n_done, uint8_t* codes,
                                    uint8_t* scales, int32_t* done, int32_t* status, cudaStream_t stream) {
  // per route tile a GEMM1 counter, then the unit ticket
  const int MT = n_done - 1;
  // enough warps for one padding item each (one global read then one store
  // per lane), and one warp per token item
  const long long pad_threads = (long long)MT * (H / 64) * 32,
                  tok_threads = (long long)T * ((H / 16 + 63) / 64) * 32;
  const int grid = grid_for(pad_threads > tok_threads ? pad_threads : tok_threads, 256);
  return launch_kernel(quantize_permute_kernel, dim3(grid), dim3(256), 0, stream, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), reinterpret_cast<const uint8_t*>(a),
                       reinterpret_cast<const uint8_t*>(a_sf), a1_gscale, e2p, tile_row_limit, totals,
                       T, K, H, tile_m, P, codes, scales, done, n_done, status);
}

size_t route_quantize_smem(int T, int K, int E, int MT) {
  return sizeof(int32_t) * ((size_t)8 * E + (size_t)T * K + (size_t)MT + 2);
}

bool route_quantize_fits(int T, int K, int E) { return T * K <= kFusedMaxRoutes && E <= 256; }

cudaError_t launch_route_quantize(const int32_t* topk_ids, int T, int K, int E, int tile_m, int P, int MT,
                                  int32_t* counts, int32_t* offsets, int32_t* e2p, int32_t* p2t,
                                  int32_t* tile_expert, int32_t* tile_row_limit, int32_t* totals, const void* x,
                                  const void* a, const void* a_sf, const float* a1_gscale, int H, uint8_t* codes,
                                  uint8_t* scales, int32_t* done, int32_t* status, cudaStream_t stream) {
  // One CTA per SM at most: the routing is redone in every CTA, and fewer
  // CTAs leave room beside them for the GEMM CTAs that launch early.
  static int sms = 0;
  if (sms == 0) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 148;
    sms = n;
  }
  const long long pad_threads = (long long)MT * (H / 64) * 32,
                  tok_threads = (long long)T * ((H / 16 + 31) / 32) * 32;
  int grid = grid_for(pad_threads > tok_threads ? pad_threads : tok_threads, 256);
  if (grid > sms) grid = sms;
  const size_t smem = route_quantize_smem(T, K, E, MT);
  return launch_kernel(route_quantize_kernel, dim3(grid), dim3(256), smem, stream, true, topk_ids, T, K, E,
                       tile_m, P, MT, counts, offsets, e2p, p2t, tile_expert, tile_row_limit, totals,
                       reinterpret_cast<const __nv_bfloat16*>(x), reinterpret_cast<const uint8_t*>(a),
                       reinterpret_cast<const uint8_t*>(a_sf), a1_gscale, H, codes, scales, done, status);
}

cudaError_t launch_act_scales_io(int to_linear, uint8_t* atoms, uint8_t* linear, int K,
                                 int tile_m, int P, cudaStream_t stream) {
  const int grid = grid_for((long long)P * (K / 16), 256);
  act_scales_io_kernel<<<grid, 256, 0, stream>>>(to_linear, atoms, linear, P, K, tile_m);
  return cudaGetLastError();
}

}  // namespace moe
