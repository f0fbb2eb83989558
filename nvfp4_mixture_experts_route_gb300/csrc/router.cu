// Two steps that feed the expert block:
//
//  * MuseSpark1x routing from router logits (the model page's
//    fused_musespark1x_routing; MuseSpark1xRouter with sigmoid scores, an
//    expert bias that only steers the choice, sum-renormalised weights with a
//    division eps, route_scale; no expert groups):
//        s = sigmoid(logits); chosen = top-K of s + bias (lower index first
//        on equal values); w = s[chosen] / (sum + eps) * route_scale;
//        padding tokens get ids -1 and weights 0.
//    One warp per token; each lane owns experts lane, lane+32, ...; K rounds
//    of a warp arg-max pick the experts in order. (E <= 1024.)
//
//  * The pre-expert RMSNorm fused into the NVFP4 input quantization (the
//    model page's norm_quant_trtllm_nvfp4; the norm's zero-centred weight is
//    applied after the normalisation, the only kind the page fuses):
//        y = x / sqrt(mean(x^2) + eps) * (1 + gamma);  (a, a_sf) = NVFP4(y)
//    One CTA per output row: a first pass over the row for the sum of
//    squares, a second that normalises and quantizes 16-element blocks. It
//    writes either the row-major layout of scaled_fp4_quant or straight into
//    the permuted workspace of the expert body (like the plain quantizer).
#include <float.h>

#include "common.cuh"
#include "layout.cuh"

namespace moe {

// EPL experts per lane (E <= 32 * EPL): the per-lane arrays and the arg-max
// scans are sized at compile time, so a 128-expert router scans 4 slots per
// lane, not 32.
template <int EPL>
__global__ void __launch_bounds__(256)
    musespark1x_routing_kernel(const float* __restrict__ logits, const float* __restrict__ bias,
                               const uint8_t* __restrict__ is_padding, int T, int E, int K,
                               float route_scale, float eps, int32_t* __restrict__ ids,
                               float* __restrict__ weights) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (t >= T) return;
  if (is_padding != nullptr && is_padding[t]) {
    for (int k = lane; k < K; k += 32) {
      ids[(size_t)t * K + k] = -1;
      weights[(size_t)t * K + k] = 0.f;
    }
    return;
  }
  float s[EPL], c[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int j = lane + 32 * i;
    if (j < E) {
      const float x = logits[(size_t)t * E + j];
      s[i] = 1.0f / (1.0f + expf(-x));
      c[i] = s[i] + bias[j];
    } else {
      s[i] = 0.f;
      c[i] = -FLT_MAX;
    }
  }
  uint32_t taken = 0;
  int my_id = -1;
  float my_s = 0.f;
  for (int k = 0; k < K; ++k) {
    float best = -FLT_MAX;
    int best_j = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int j = lane + 32 * i;
      if (j < E && !((taken >> i) & 1u) && (c[i] > best || (c[i] == best && j < best_j))) {
        best = c[i];
        best_j = j;
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, d);
      const int oj = __shfl_xor_sync(0xffffffffu, best_j, d);
      if (ob > best || (ob == best && oj < best_j)) {
        best = ob;
        best_j = oj;
      }
    }
    // the owner lane marks the expert and hands its unbiased score on
    float sw = 0.f;
    if ((best_j & 31) == lane) {
      const int slot = best_j >> 5;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == slot) sw = s[i];
      taken |= 1u << slot;
    }
    sw = __shfl_sync(0xffffffffu, sw, best_j & 31);
    if (lane == k) {
      my_id = best_j;
      my_s = sw;
    }
  }
  float sum = (lane < K) ? my_s : 0.f;
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, d);
  if (lane < K) {
    ids[(size_t)t * K + lane] = my_id;
    weights[(size_t)t * K + lane] = my_s / (sum + eps) * route_scale;
  }
}

cudaError_t launch_musespark1x_routing(const float* logits, const float* bias, const uint8_t* pad, int T,
                                       int E, int K, float route_scale, float eps, int32_t* ids,
                                       float* weights, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int warps = 8;
  const dim3 grid((T + warps - 1) / warps), block(32 * warps);
  const int epl = (E + 31) / 32;
  if (epl <= 1)
    musespark1x_routing_kernel<1><<<grid, block, 0, stream>>>(logits, bias, pad, T, E, K, route_scale, eps, ids, weights);
  else if (epl <= 2)
    musespark1x_routing_kernel<2><<<grid, block, 0, stream>>>(logits, bias, pad, T, E, K, route_scale, eps, ids, weights);
  else if (epl <= 4)
    musespark1x_routing_kernel<4><<<grid, block, 0, stream>>>(logits, bias, pad, T, E, K, route_scale, eps, ids, weights);
  else if (epl <= 8)
    musespark1x_routing_kernel<8><<<grid, block, 0, stream>>>(logits, bias, pad, T, E, K, route_scale, eps, ids, weights);
  else if (epl <= 16)
    musespark1x_routing_kernel<16><<<grid, block, 0, stream>>>(logits, bias, pad, T, E, K, route_scale, eps, ids, weights);
  else
    musespark1x_routing_kernel<32><<<grid, block, 0, stream>>>(logits, bias, pad, T, E, K, route_scale, eps, ids, weights);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Pre-expert RMSNorm + NVFP4 quant
// ---------------------------------------------------------------------------
constexpr int kNqThreads = 256;

__device__ __forceinline__ void load16(const __nv_bfloat16* p, float (&v)[16]) {
  const uint4* q = reinterpret_cast<const uint4*>(p);
  const uint4 u0 = q[0], u1 = q[1];
  const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&u0);
  const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&u1);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f0 = __bfloat1622float2(h0[i]);
    const float2 f1 = __bfloat1622float2(h1[i]);
    v[2 * i] = f0.x;
    v[2 * i + 1] = f0.y;
    v[8 + 2 * i] = f1.x;
    v[8 + 2 * i + 1] = f1.y;
  }
}

__device__ __forceinline__ void nvfp4_block(const float (&v)[16], float g, uint32_t& lo, uint32_t& hi,
                                            uint32_t& sfc) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  sfc = f32_to_e4m3((amax * g) / 6.0f);
  const float sfv = e4m3_to_f32(sfc);
  lo = hi = 0;
  if (sfv > 0.f) {
    const float inv = g / sfv;
#pragma unroll
    for (int i = 0; i < 8; i += 2) lo |= f32x2_to_e2m1x2(v[i] * inv, v[i + 1] * inv) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; i += 2) hi |= f32x2_to_e2m1x2(v[8 + i] * inv, v[9 + i] * inv) << (4 * i);
  }
}

// PERMUTED: rows are permuted rows < totals[1] (token from permuted_to_token,
// padding rows get zero scales, scales in the workspace atom layout);
// otherwise rows are tokens and the output is row-major codes / scales.
template <bool PERMUTED>
__global__ void __launch_bounds__(kNqThreads)
    rmsnorm_nvfp4_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
                         float eps, const float* __restrict__ gscale,
                         const int32_t* __restrict__ permuted_to_token,
                         const int32_t* __restrict__ totals, int T, int H, int tile_m,
                         uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  __shared__ float red[kNqThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int nb = H / 16;
  const int rows = PERMUTED ? totals[1] : T;
  const float g = *gscale;
  const int S = sf_atoms_per_tile(tile_m);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const int t = PERMUTED ? permuted_to_token[row] : row;
    if (t < 0) {  // padding row: zero scales (uniform across the CTA)
      for (int b = threadIdx.x; b < nb; b += kNqThreads)
        scales[act_sf_offset(row, b, tile_m, H / 64, S)] = 0;
      continue;
    }
    const __nv_bfloat16* xr = x + (size_t)t * H;
    float ss = 0.f;
    for (int b = threadIdx.x; b < nb; b += kNqThreads) {
      float v[16];
      load16(xr + 16 * b, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
    __syncthreads();  // red[] free from the previous row
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    float total = 0.f;
#pragma unroll
    for (int w = 0; w < kNqThreads / 32; ++w) total += red[w];
    const float inv = 1.0f / sqrtf(total / (float)H + eps);
    for (int b = threadIdx.x; b < nb; b += kNqThreads) {
      float v[16], gm[16];
      load16(xr + 16 * b, v);
      load16(gamma + 16 * b, gm);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = (v[i] * inv) * (1.0f + gm[i]);
      uint32_t lo, hi, sfc;
      nvfp4_block(v, g, lo, hi, sfc);
      *reinterpret_cast<uint2*>(codes + (size_t)row * (H / 2) + 8 * b) = make_uint2(lo, hi);
      if (PERMUTED)
        scales[act_sf_offset(row, b, tile_m, H / 64, S)] = static_cast<uint8_t>(sfc);
      else
        scales[(size_t)row * nb + b] = static_cast<uint8_t>(sfc);
    }
  }
}

// The same norm and quantization with one warp per token, for H <= 5120
// (NCH <= 10 chunks of 32 blocks of 16): lane l holds blocks 32 j + l of the
// token in registers, so the row is read once, the sum of squares is one
// warp reduction (lanes in order over their blocks, then an xor butterfly)
// and no block barrier is needed. Row-major output as scaled_fp4_quant, or
// (PERMUTED) each token quantized once and written to the rows of its routes
// (lanes k and k + 32 look up route k's row and its block-0 scale offset; the
// first lane of a quad writes the quad's four scale bytes), then one warp per
// (route tile, four-block group) zeroes the scales of the tile's padding rows.
template <int NCH, bool PERMUTED>
__global__ void __launch_bounds__(kNqThreads)
    rmsnorm_nvfp4_warp_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
                              float eps, const float* __restrict__ gscale, const int32_t* __restrict__ e2p,
                              const int32_t* __restrict__ tile_row_limit, const int32_t* __restrict__ totals,
                              int T, int K, int H, int tile_m, uint8_t* __restrict__ codes,
                              uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  constexpr unsigned kFull = 0xFFFFFFFFu;
  const int nb = H / 16, ng = H / 64;
  const float g = *gscale;
  const int S = sf_atoms_per_tile(tile_m);
  const int lane = threadIdx.x & 31;
  const int warp0 = blockIdx.x * (kNqThreads / 32) + (threadIdx.x >> 5);
  const int nwarps = gridDim.x * (kNqThreads / 32);
  const size_t group_step = (size_t)S * kAtomBytes;
  for (int t = warp0; t < T; t += nwarps) {
    // routes k = lane and lane + 32: permuted row and its block-0 scale offset
    int p_lo = -1, p_hi = -1;
    if (PERMUTED) {
      if (lane < K) p_lo = e2p[(size_t)t * K + lane];
      if (lane + 32 < K) p_hi = e2p[(size_t)t * K + lane + 32];
    }
    uint4 u[NCH][2];
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int b = 32 * j + lane;
      if (b < nb) {
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H + 16 * b);
        u[j][0] = src[0];
        u[j][1] = src[1];
      } else {
        u[j][0] = u[j][1] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u[j][0]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        ss = fmaf(f.x, f.x, ss);
        ss = fmaf(f.y, f.y, ss);
      }
    }
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(kFull, ss, d);
    const float inv = 1.0f / sqrtf(ss / (float)H + eps);
    const size_t s_lo = (PERMUTED && p_lo >= 0) ? act_sf_offset(p_lo, 0, tile_m, ng, S) : 0;
    const size_t s_hi = (PERMUTED && p_hi >= 0) ? act_sf_offset(p_hi, 0, tile_m, ng, S) : 0;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int b = 32 * j + lane;
      const bool on = b < nb;  // every lane stays for the warp-wide shuffles
      uint32_t lo = 0, hi = 0, sfc = 0;
      if (on) {
        float v[16], gm[16];
        const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&u[j][0]);
        const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&u[j][1]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f0 = __bfloat1622float2(h0[i]);
          const float2 f1 = __bfloat1622float2(h1[i]);
          v[2 * i] = f0.x;
          v[2 * i + 1] = f0.y;
          v[8 + 2 * i] = f1.x;
          v[8 + 2 * i + 1] = f1.y;
        }
        load16(gamma + 16 * b, gm);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = (v[i] * inv) * (1.0f + gm[i]);
        nvfp4_block(v, g, lo, hi, sfc);
      }
      if (!PERMUTED) {
        if (on) {
          *reinterpret_cast<uint2*>(codes + (size_t)t * (H / 2) + 8 * b) = make_uint2(lo, hi);
          scales[(size_t)t * nb + b] = static_cast<uint8_t>(sfc);
        }
        continue;
      }
      // the quad's four scale bytes, block 4 * (b / 4) in the low byte
      const int base = lane & ~3;
      const uint32_t sf4 = __shfl_sync(kFull, sfc, base) | (__shfl_sync(kFull, sfc, base + 1) << 8) |
                           (__shfl_sync(kFull, sfc, base + 2) << 16) | (__shfl_sync(kFull, sfc, base + 3) << 24);
      const size_t sf_b = (size_t)(b >> 2) * group_step;
      for (int k = 0; k < K; ++k) {
        const int p = __shfl_sync(kFull, k < 32 ? p_lo : p_hi, k & 31);
        if (p < 0) continue;  // the same p in every lane
        const size_t so = __shfl_sync(kFull, k < 32 ? s_lo : s_hi, k & 31);
        if (on) {
          *reinterpret_cast<uint2*>(codes + (size_t)p * (H / 2) + 8 * b) = make_uint2(lo, hi);
          if ((b & 3) == 0) *reinterpret_cast<uint32_t*>(scales + so + sf_b) = sf4;
        }
      }
    }
  }
  if (PERMUTED) {
    // padding rows of the route tiles in use: zero block scales
    const int n_pad = totals[0] * ng;
    for (int w = warp0; w < n_pad; w += nwarps) {
      const int tau = w / ng, c = w - (w / ng) * ng;
      const int limit = tile_row_limit[tau];
      for (int j = 0; j < tile_m; j += 32) {
        const int p = tau * tile_m + j + lane;
        if (p >= limit) *reinterpret_cast<uint32_t*>(scales + act_sf_offset(p, 4 * c, tile_m, ng, S)) = 0u;
      }
    }
  }
}

static int nq_grid(int rows) {
  int g = rows < 1 ? 1 : rows;
  return g > 152 * 8 ? 152 * 8 : g;
}

// Warp-per-token kernels for H <= 5120 (NCH chunks).
template <bool PERMUTED>
static cudaError_t launch_nq_warp(int nch, dim3 grid, cudaStream_t stream, const __nv_bfloat16* x,
                                  const __nv_bfloat16* gamma, float eps, const float* gscale, const int32_t* e2p,
                                  const int32_t* limit, const int32_t* totals, int T, int K, int H, int tile_m,
                                  uint8_t* codes, uint8_t* scales) {
#define MOE_NQ_CASE(n)                                                                                    \
  case n:                                                                                                 \
    return launch_kernel(rmsnorm_nvfp4_warp_kernel<n, PERMUTED>, grid, dim3(kNqThreads), 0, stream, true, x, \
                         gamma, eps, gscale, e2p, limit, totals, T, K, H, tile_m, codes, scales);
  switch (nch) {
    MOE_NQ_CASE(1)
    MOE_NQ_CASE(2)
    MOE_NQ_CASE(3)
    MOE_NQ_CASE(4)
    MOE_NQ_CASE(5)
    MOE_NQ_CASE(6)
    MOE_NQ_CASE(7)
    MOE_NQ_CASE(8)
    MOE_NQ_CASE(9)
    MOE_NQ_CASE(10)
  }
#undef MOE_NQ_CASE
  return cudaErrorInvalidValue;
}

// At most two CTAs per SM (one is resident at a time at H = 5120: 254
// registers): the warps loop over tokens and padding items, so a grid past
// that would only add waves.
static int nq_warp_grid(long long warps) {
  long long g = (warps + kNqThreads / 32 - 1) / (kNqThreads / 32);
  if (g < 1) g = 1;
  return (int)(g > 152 * 2 ? 152 * 2 : g);
}

cudaError_t launch_rmsnorm_nvfp4(const void* x, const void* gamma, float eps, const float* gscale, int T,
                                 int H, void* a, void* a_sf, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const auto xp = reinterpret_cast<const __nv_bfloat16*>(x);
  const auto gp = reinterpret_cast<const __nv_bfloat16*>(gamma);
  // one CTA per row: faster here than a warp per token (measured 41 against
  // 49 us at T = 8192, 11.5 against 14.1 us at T = 8)
  return launch_kernel(rmsnorm_nvfp4_kernel<false>, dim3(nq_grid(T)), dim3(kNqThreads), 0, stream, true, xp, gp,
                       eps, gscale, (const int32_t*)nullptr, (const int32_t*)nullptr, T, H, 32,
                       reinterpret_cast<uint8_t*>(a), reinterpret_cast<uint8_t*>(a_sf));
}

cudaError_t launch_rmsnorm_nvfp4_permuted(const void* x, const void* gamma, float eps, const float* gscale,
                                          const int32_t* p2t, const int32_t* e2p, const int32_t* tile_row_limit,
                                          const int32_t* totals, int T, int K, int H, int tile_m, int P, int MT,
                                          uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  const auto xp = reinterpret_cast<const __nv_bfloat16*>(x);
  const auto gp = reinterpret_cast<const __nv_bfloat16*>(gamma);
  const int nch = (H / 16 + 31) / 32;
  // many tokens: a warp per token reads x once and writes every route row
  // (131 against 292 us at T = 8192, top-8); few tokens: a CTA per permuted
  // row spreads the work wider (17 against 28 us at T = 8)
  if (nch <= 10 && T >= 512) {
    const long long pad = (long long)MT * (H / 64);
    return launch_nq_warp<true>(nch, dim3(nq_warp_grid(pad > T ? pad : T)), stream, xp, gp, eps, gscale, e2p,
                                tile_row_limit, totals, T, K, H, tile_m, codes, scales);
  }
  return launch_kernel(rmsnorm_nvfp4_kernel<true>, dim3(nq_grid(P)), dim3(kNqThreads), 0, stream, true, xp, gp,
                       eps, gscale, p2t, totals, 0, H, tile_m, codes, scales);
}

}  // namespace moe
