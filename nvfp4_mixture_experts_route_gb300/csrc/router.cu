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
//    of a warp arg-max pick the experts in order.
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

constexpr int kRouteMaxPerLane = 32;  // E <= 1024

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
  float s[kRouteMaxPerLane], c[kRouteMaxPerLane];
#pragma unroll
  for (int i = 0; i < kRouteMaxPerLane; ++i) {
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
    for (int i = 0; i < kRouteMaxPerLane; ++i) {
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
      for (int i = 0; i < kRouteMaxPerLane; ++i)
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
  musespark1x_routing_kernel<<<(T + warps - 1) / warps, 32 * warps, 0, stream>>>(
      logits, bias, pad, T, E, K, route_scale, eps, ids, weights);
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

static int nq_grid(int rows) {
  int g = rows < 1 ? 1 : rows;
  return g > 152 * 8 ? 152 * 8 : g;
}

cudaError_t launch_rmsnorm_nvfp4(const void* x, const void* gamma, float eps, const float* gscale, int T,
                                 int H, void* a, void* a_sf, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  return launch_kernel(rmsnorm_nvfp4_kernel<false>, dim3(nq_grid(T)), dim3(kNqThreads), 0, stream, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), reinterpret_cast<const __nv_bfloat16*>(gamma),
                       eps, gscale, (const int32_t*)nullptr, (const int32_t*)nullptr, T, H, 32,
                       reinterpret_cast<uint8_t*>(a), reinterpret_cast<uint8_t*>(a_sf));
}

cudaError_t launch_rmsnorm_nvfp4_permuted(const void* x, const void* gamma, float eps, const float* gscale,
                                          const int32_t* p2t, const int32_t* totals, int H, int tile_m, int P,
                                          uint8_t* codes, uint8_t* scales, cudaStream_t stream) {
  return launch_kernel(rmsnorm_nvfp4_kernel<true>, dim3(nq_grid(P)), dim3(kNqThreads), 0, stream, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), reinterpret_cast<const __nv_bfloat16*>(gamma),
                       eps, gscale, p2t, totals, 0, H, tile_m, codes, scales);
}

}  // namespace moe
