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

namespace moe {

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

// Work item (token t, group c of four 16-element blocks): the group is
// quantized once and its 32 code bytes and 4 scale bytes (contiguous in the
// scale atom) are written to the row of each of the token's routes, found
// through expanded_to_permuted. The first items (they loop over rows, so
// they start first) zero the scales of the padding rows of each live tile
// (rows tile_row_limit .. the tile's end):
// with a zero block scale the codes, always finite e2m1 values, contribute
// exactly 0 to every product, so padding-row codes are never written.
// Reads x once; writes each route row once.
__global__ void __launch_bounds__(256, 6) quantize_permute_kernel(
    const __nv_bfloat16* __restrict__ x, const uint8_t* __restrict__ a_in,
    const uint8_t* __restrict__ a_sf_in, const float* __restrict__ gscale,
    const int32_t* __restrict__ e2p, const int32_t* __restrict__ tile_row_limit,
    const int32_t* __restrict__ totals, int T, int K, int H, int tile_m, uint8_t* __restrict__ codes,
    uint8_t* __restrict__ scales) {
  pdl_wait();
  pdl_trigger();
  const int ng = H / 64;  // four-block groups per row
  const int nb = H / 16;
  const long long n_pad = (long long)totals[0] * ng;
  const long long n_all = n_pad + (long long)T * ng;
  const float g = (x != nullptr) ? *gscale : 0.f;
  const int S = sf_atoms_per_tile(tile_m);
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < n_all;
       idx += (long long)gridDim.x * blockDim.x) {
    if (idx >= n_pad) {
      const long long i2 = idx - n_pad;
      const int t = (int)(i2 / ng), c = (int)(i2 % ng);
      uint4 q0, q1;  // 32 code bytes: blocks 4c .. 4c+3
      uint32_t sf4;  // their 4 scale bytes, block 4c in the low byte
      if (x != nullptr) {
        const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)t * H + 64 * c);
        uint32_t lo[4], hi[4], sfc[4];
#pragma unroll
        for (int bq = 0; bq < 4; ++bq) {
          const uint4 u0 = src[2 * bq], u1 = src[2 * bq + 1];
          const __nv_bfloat162* h0 = reinterpret_cast<const __nv_bfloat162*>(&u0);
          const __nv_bfloat162* h1 = reinterpret_cast<const __nv_bfloat162*>(&u1);
          float v[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f0 = __bfloat1622float2(h0[i]);
            const float2 f1 = __bfloat1622float2(h1[i]);
            v[2 * i] = f0.x;
            v[2 * i + 1] = f0.y;
            v[8 + 2 * i] = f1.x;
            v[8 + 2 * i + 1] = f1.y;
          }
          quantize_block16(v, g, lo[bq], hi[bq], sfc[bq]);
        }
        q0 = make_uint4(lo[0], hi[0], lo[1], hi[1]);
        q1 = make_uint4(lo[2], hi[2], lo[3], hi[3]);
        sf4 = sfc[0] | (sfc[1] << 8) | (sfc[2] << 16) | (sfc[3] << 24);
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(a_in + (size_t)t * (H / 2) + 32 * c);
        q0 = src[0];
        q1 = src[1];
        sf4 = *reinterpret_cast<const uint32_t*>(a_sf_in + (size_t)t * nb + 4 * c);
      }
      for (int k = 0; k < K; ++k) {
        const int p = e2p[(size_t)t * K + k];
        if (p < 0) continue;
        uint4* dst = reinterpret_cast<uint4*>(codes + (size_t)p * (H / 2) + 32 * c);
        dst[0] = q0;
        dst[1] = q1;
        *reinterpret_cast<uint32_t*>(scales + act_sf_offset(p, 4 * c, tile_m, H / 64, S)) = sf4;
      }
    } else {
      const int tau = (int)(idx / ng), c = (int)(idx % ng);
      const int end = (tau + 1) * tile_m;
      for (int p = tile_row_limit[tau]; p < end; ++p)
        *reinterpret_cast<uint32_t*>(scales + act_sf_offset(p, 4 * c, tile_m, H / 64, S)) = 0u;
    }
  }
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
                                    int K, int H, int tile_m, int P, int MT, uint8_t* codes,
                                    uint8_t* scales, cudaStream_t stream) {
  (void)P;
  const int grid = grid_for((long long)(T + MT) * (H / 64), 256);
  return launch_kernel(quantize_permute_kernel, dim3(grid), dim3(256), 0, stream, true,
                       reinterpret_cast<const __nv_bfloat16*>(x), reinterpret_cast<const uint8_t*>(a),
                       reinterpret_cast<const uint8_t*>(a_sf), a1_gscale, e2p, tile_row_limit, totals,
                       T, K, H, tile_m, codes, scales);
}

cudaError_t launch_act_scales_io(int to_linear, uint8_t* atoms, uint8_t* linear, int K,
                                 int tile_m, int P, cudaStream_t stream) {
  const int grid = grid_for((long long)P * (K / 16), 256);
  act_scales_io_kernel<<<grid, 256, 0, stream>>>(to_linear, atoms, linear, P, K, tile_m);
  return cudaGetLastError();
}

}  // namespace moe
