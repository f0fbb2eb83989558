// Step a7: the MuseSpark1x post-expert finalize (the muse_moe_runner page,
// MusePostExpertFinalize: per-route RMSNorm with zero-centred gamma, fp32
// norm output, fp32 top-k weighted sum, copied into the bf16 output; routes
// marked -1 add nothing).
//
// One CTA per token. Each thread owns 8-element (16-byte) vectors of the
// hidden dimension; for every route k the CTA loads the GEMM2 row, reduces
// the sum of squares across the block, and adds w * u / rms into fp32
// registers. HBM traffic: K rows of H bf16 in, one row out.
#include "common.cuh"

namespace moe {

constexpr int kFinThreads = 256;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();  // red[] free from the previous use
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kFinThreads / 32; ++w) s += red[w];  // fixed order
  return s;
}

// VPT: 8-element vectors per thread (ceil(H / 8 / 256)), a template so that
// the per-thread arrays stay in registers.
template <int VPT>
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(
    const __nv_bfloat16* __restrict__ rows, const int32_t* __restrict__ e2p,
    const float* __restrict__ topk_w, const __nv_bfloat16* __restrict__ gamma, float eps,
    int weight_before_norm, int K, int H, __nv_bfloat16* __restrict__ out) {
  __shared__ float red[kFinThreads / 32];
  const int t = blockIdx.x;
  const int nvec = H / 8;
  float g[VPT][8];
  float acc[VPT][8];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * kFinThreads;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      acc[i][q] = 0.f;
      g[i][q] = 1.f;
    }
    if (v < nvec) {
      const uint4 u = *reinterpret_cast<const uint4*>(gamma + 8 * v);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]);
        g[i][2 * q] = 1.f + f.x;  // gain centre added in fp32
        g[i][2 * q + 1] = 1.f + f.y;
      }
    }
  }
  const float inv_h = 1.0f / (float)H;
  for (int k = 0; k < K; ++k) {
    const int p = e2p[(size_t)t * K + k];
    if (p < 0) continue;  // uniform across the block
    const float wk = topk_w[(size_t)t * K + k];
    float u[VPT][8];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = threadIdx.x + i * kFinThreads;
#pragma unroll
      for (int q = 0; q < 8; ++q) u[i][q] = 0.f;
      if (v < nvec) {
        const uint4 raw = *reinterpret_cast<const uint4*>(rows + (size_t)p * H + 8 * v);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(h[q]);
          u[i][2 * q] = f.x;
          u[i][2 * q + 1] = f.y;
        }
        if (weight_before_norm) {
#pragma unroll
          for (int q = 0; q < 8; ++q) u[i][q] *= g[i][q];
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) ss = fmaf(u[i][q], u[i][q], ss);
      }
    }
    const float total = block_sum(ss, red);
    const float c = wk / sqrtf(total * inv_h + eps);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float n = weight_before_norm ? u[i][q] * c : (u[i][q] * c) * g[i][q];
        acc[i][q] += n;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * kFinThreads;
    if (v < nvec) {
      uint4 o;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(acc[i][2 * q], acc[i][2 * q + 1]);
      *reinterpret_cast<uint4*>(out + (size_t)t * H + 8 * v) = o;
    }
  }
}

cudaError_t launch_finalize(const void* rows, const int32_t* e2p, const float* w,
                            const void* gamma, float eps, int weight_before_norm, int T, int K,
                            int H, void* out, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const int vpt = ceil_div(H / 8, kFinThreads);
  auto rp = reinterpret_cast<const __nv_bfloat16*>(rows);
  auto gp = reinterpret_cast<const __nv_bfloat16*>(gamma);
  auto op = reinterpret_cast<__nv_bfloat16*>(out);
#define MOE_FIN_CASE(n)                                                                     \
  case n:                                                                                   \
    finalize_kernel<n><<<T, kFinThreads, 0, stream>>>(rp, e2p, w, gp, eps, weight_before_norm, \
                                                      K, H, op);                              \
    break;
  switch (vpt) {
    MOE_FIN_CASE(1)
    MOE_FIN_CASE(2)
    MOE_FIN_CASE(3)
    MOE_FIN_CASE(4)
    MOE_FIN_CASE(5)
    MOE_FIN_CASE(6)
    MOE_FIN_CASE(7)
    MOE_FIN_CASE(8)
    default:
      return cudaErrorInvalidValue;
  }
#undef MOE_FIN_CASE
  return cudaGetLastError();
}

}  // namespace moe
