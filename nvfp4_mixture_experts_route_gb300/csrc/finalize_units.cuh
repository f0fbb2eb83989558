// The post-expert finalize from GEMM2's sums of squares, in units of
// (token, 256 columns per warp) done by four warps together
// (finalize_sumsq_units_kernel).
//
// Per token t and route k (row p = expanded_to_permuted[t, k]):
//   coef_k = w[t, k] / sqrt(sum_c row_ss[p][c] / H + eps)
//   out[t] = bf16((1 + gamma) * sum_k coef_k * rows[p]),  fp32, route order.
// The H/32 partials of route k are summed by 16 lanes of one warp as float4s
// (lane j takes float4s j, j + 16, ..., adding .x, .y, .z, .w in turn; then
// an xor butterfly over the 16 lanes); warp wi sums routes 2 wi and 2 wi + 1
// and the coefficients go through shared memory to the other warps (a named
// barrier, id 1, over the unit's warps).
#pragma once
#include "common.cuh"

namespace moe {

constexpr int kFinUnitMaxK = 8;    // routes per token the units take
constexpr int kFinUnitWarps = 4;   // warps of a unit (each sums 2 routes' partials)

struct FinArgs {
  const __nv_bfloat16* rows;  // [num_rows, H]
  const float* row_ss;        // [num_rows, H / 32]
  const int32_t* e2p;         // [T, K]
  const float* w;             // [T, K]
  const __nv_bfloat16* gamma; // [H]
  __nv_bfloat16* out;         // [T, H]
  int32_t* status;
  float eps;
  int K, H, num_rows;
};

static __device__ __forceinline__ void fin_bar_sync(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// What of a unit does not depend on the rows: lane k < K holds route k's
// row and weight; every lane its gain vector (8 columns from v).
struct FinPre {
  int t, v, pk;
  float wk;
  uint4 gain;
};

static __device__ __forceinline__ FinPre fin_prepare(const FinArgs& a, int t, int v, int lane) {
  FinPre f;
  f.t = t;
  f.v = v;
  f.pk = -1;
  f.wk = 0.f;
  if (lane < a.K) {
    f.pk = __ldcg(a.e2p + (size_t)t * a.K + lane);
    if (f.pk < -1 || f.pk >= a.num_rows) {
      record_status(a.status, MOE_ERR_INVALID_ROUTE);
      f.pk = -1;
    }
    f.wk = __ldcg(a.w + (size_t)t * a.K + lane);
  }
  f.gain = f.v < a.H / 8 ? __ldg(reinterpret_cast<const uint4*>(a.gamma + 8 * f.v)) : make_uint4(0, 0, 0, 0);
  return f;
}

}  // namespace moe

namespace moe {

// The rest of a unit: warp wi of its kFinUnitWarps, all reaching the named
// barrier once (nthreads = 32 * kFinUnitWarps). The loads of the rows and of
// the warp's share of the partial sums are in flight together.
static __device__ __forceinline__ void fin_finish_inl(const FinArgs& a, const FinPre& f, int lane, int wi,
                                                     float* coef_s, int nthreads) {
  const int K = a.K, H = a.H, G4 = H / 128;
  const bool on = f.v < H / 8;
  uint4 raw[kFinUnitMaxK];
#pragma unroll
  for (int k = 0; k < kFinUnitMaxK; ++k) {
    const int rp = __shfl_sync(0xFFFFFFFFu, f.pk, k);
    raw[k] = (on && k < K && rp >= 0) ? __ldcg(reinterpret_cast<const uint4*>(a.rows + (size_t)rp * H) + f.v)
                                      : make_uint4(0, 0, 0, 0);
  }
  // this half-warp's route and its share of the partial sums
  const int k = 2 * wi + (lane >> 4), j = lane & 15;
  const int my = __shfl_sync(0xFFFFFFFFu, f.pk, k & 31);
  const float wk = __shfl_sync(0xFFFFFFFFu, f.wk, k & 31);
  const bool mine = k < K && my >= 0;
  const float4* src = reinterpret_cast<const float4*>(a.row_ss + (size_t)(mine ? my : 0) * (H / 32));
  float ss = 0.f;
  for (int m0 = j; m0 < G4; m0 += 64) {
    float4 x[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      x[i] = (mine && m0 + 16 * i < G4) ? __ldcg(src + m0 + 16 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (m0 + 16 * i < G4) {
        ss += x[i].x;
        ss += x[i].y;
        ss += x[i].z;
        ss += x[i].w;
      }
    }
  }
#pragma unroll
  for (int d = 1; d < 16; d <<= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, d);
  if (j == 0 && k < K) coef_s[k] = mine ? wk / sqrtf(ss / (float)H + a.eps) : 0.f;
  fin_bar_sync(nthreads);
  float2 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.f, 0.f);
#pragma unroll
  for (int kk = 0; kk < kFinUnitMaxK; ++kk) {
    if (kk >= K) break;
    const float c = coef_s[kk];
    const float2 ck = make_float2(c, c);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[kk]);
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = ffma2(__bfloat1622float2(h[q]), ck, acc[q]);
  }
  if (!on) return;
  const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&f.gain);
  uint4 o;
  __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 gf = __bfloat1622float2(gh[q]);
    const float2 r = fmul2(acc[q], make_float2(1.f + gf.x, 1.f + gf.y));  // gain centre added in fp32
    oh[q] = __floats2bfloat162_rn(r.x, r.y);
  }
  *reinterpret_cast<uint4*>(a.out + (size_t)f.t * H + 8 * f.v) = o;
}

}  // namespace moe
