// Step a7: the MuseSpark1x post-expert finalize (the muse_moe_runner page,
// MusePostExpertFinalize: per-route RMSNorm with zero-centred gamma, fp32
// norm output, fp32 top-k weighted sum, copied into the bf16 output; routes
// marked -1 add nothing).
//
// One CTA per token. Each thread owns 8-element (16-byte) vectors of the
// hidden dimension. Routes are taken in chunks of up to kFinChunk: the CTA
// first issues the loads of every row of the chunk (so their latencies
// overlap), then reduces all of the chunk's sums of squares in one block
// reduction, then adds w * u / rms into fp32 registers. HBM traffic: K rows
// of H bf16 in, one row out.
#include <algorithm>

#include "common.cuh"
#include "finalize_units.cuh"

namespace moe {

constexpr int kFinThreads = 256;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kFinChunk = 8;  // most routes per chunk (fewer for wide rows)
constexpr int kMaxParts = 16;  // K-partial row buffers the expert-TP tail sums

// The GEMM2 rows, or the expert-TP tail's tp K-partial row buffers: a row is
// bf16(sum over parts, in fp32) -- the expert_tp page's "FP32 sum, one BF16
// rounding" -- before the norm; with one part it is read as is.
struct RowParts {
  const __nv_bfloat16* p[kMaxParts];
  int n;
};

// A route's row index as read from expanded_to_permuted: -1 (not routed) and
// [0, num_rows) are valid; anything else records MOE_ERR_INVALID_ROUTE and
// is treated as -1, so that no row outside the buffer is ever read (each
// thread of the CTA takes the same decision; only thread 0 records it).
__device__ __forceinline__ int checked_row(int p, int num_rows, int32_t* status) {
  if (p < -1 || p >= num_rows) {
    if (threadIdx.x == 0) record_status(status, MOE_ERR_INVALID_ROUTE);
    return -1;
  }
  return p;
}

__device__ __forceinline__ uint4 load_row_vec(const RowParts& parts, size_t off) {
  if (parts.n == 1) return *reinterpret_cast<const uint4*>(parts.p[0] + off);
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  for (int r = 0; r < parts.n; ++r) {
    const uint4 u = *reinterpret_cast<const uint4*>(parts.p[r] + off);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(h[q]);
      acc[2 * q] += f.x;
      acc[2 * q + 1] += f.y;
    }
  }
  uint4 o;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
  return o;
}

// VPT: 8-element vectors per thread (ceil(H / 8 / 256)) and CH: routes per
// chunk, templates so that the per-thread arrays stay in registers.
template <int VPT, int CH>
__global__ void __launch_bounds__(kFinThreads) finalize_kernel(
    const RowParts rows, const int32_t* __restrict__ e2p,
    const float* __restrict__ topk_w, const __nv_bfloat16* __restrict__ gamma, float eps,
    int weight_before_norm, int K, int H, int num_rows, __nv_bfloat16* __restrict__ out, int32_t* status) {
  __shared__ float red[kFinWarps][CH];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
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
  for (int k0 = 0; k0 < K; k0 += CH) {
    const int kc = min(CH, K - k0);
    int pr[CH];
    uint4 raw[CH][VPT];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      pr[c] = c < kc ? checked_row(e2p[(size_t)t * K + k0 + c], num_rows, status) : -1;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = threadIdx.x + i * kFinThreads;
        raw[c][i] = (pr[c] >= 0 && v < nvec) ? load_row_vec(rows, (size_t)pr[c] * H + 8 * v)
                                              : make_uint4(0, 0, 0, 0);
      }
    }
    float ss[CH];
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      ss[c] = 0.f;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[c][i]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(h[q]);
          const float a = weight_before_norm ? f.x * g[i][2 * q] : f.x;
          const float b = weight_before_norm ? f.y * g[i][2 * q + 1] : f.y;
          ss[c] = fmaf(a, a, ss[c]);
          ss[c] = fmaf(b, b, ss[c]);
        }
      }
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) ss[c] += __shfl_xor_sync(0xffffffffu, ss[c], d);
    }
    __syncthreads();  // red[] is free from the previous chunk
    if (lane == 0) {
#pragma unroll
      for (int c = 0; c < CH; ++c) red[warp][c] = ss[c];
    }
    __syncthreads();
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      if (pr[c] < 0) continue;  // uniform across the block
      float total = 0.f;
#pragma unroll
      for (int w = 0; w < kFinWarps; ++w) total += red[w][c];  // fixed order
      const float coef = topk_w[(size_t)t * K + k0 + c] / sqrtf(total * inv_h + eps);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[c][i]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(h[q]);
          // (r * g) * coef in both readings; the reading only moves g inside
          // or outside the mean of squares above.
          acc[i][2 * q] += (f.x * g[i][2 * q]) * coef;
          acc[i][2 * q + 1] += (f.y * g[i][2 * q + 1]) * coef;
        }
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

// The same finalize with the token's K rows staged in shared memory by bulk
// copies, one mbarrier per route: one thread issues them all up front, and
// the CTA normalises route k as soon as its row has landed while the later
// rows are still in flight (a route's coefficient needs only its own sum of
// squares). Two CTAs per SM keep two tokens' rows in flight without holding
// registers. One CTA per token; each thread owns VPT 8-element vectors of
// the hidden dimension, converts each of its row elements once, and applies
// the gain to the weighted sum at the end (both readings apply g to the
// normalised row: out = g * sum_k coef_k r_k). Used when K * H * 2 bytes fit
// kFinStagedMaxBytes.
constexpr int kFinStagedMaxBytes = 100 * 1024;
constexpr int kFinMaxK = 64;

template <int VPT>
__global__ void __launch_bounds__(kFinThreads, 2) finalize_staged_kernel(
    const __nv_bfloat16* __restrict__ rows, const int32_t* __restrict__ e2p,
    const float* __restrict__ topk_w, const __nv_bfloat16* __restrict__ gamma, float eps,
    int weight_before_norm, int K, int H, int num_rows, __nv_bfloat16* __restrict__ out, int32_t* status) {
  extern __shared__ __align__(16) uint8_t staged[];  // K rows of H bf16
  __shared__ __align__(8) uint64_t bar[kFinMaxK];
  __shared__ float red[2][kFinWarps];
  __shared__ int32_t rowp[kFinMaxK];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = H / 8;
  const uint32_t row_bytes = (uint32_t)H * 2;
  if (threadIdx.x == 0) {
    for (int k = 0; k < K; ++k) mbar_init(smem_u32(&bar[k]), 1);
    fence_barrier_init();
    for (int k = 0; k < K; ++k) {
      const int p = checked_row(e2p[(size_t)t * K + k], num_rows, status);
      rowp[k] = p;
      if (p >= 0) {
        mbar_arrive_expect_tx(smem_u32(&bar[k]), row_bytes);
        bulk_load(smem_u32(staged) + k * row_bytes, rows + (size_t)p * H, row_bytes,
                  smem_u32(&bar[k]));
      }
    }
  }
  // gain g = 1 + gamma (fp32) while the rows arrive
  // Pairs of hidden-dimension elements in packed fp32x2 arithmetic.
  float2 g[VPT][4], acc[VPT][4];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * kFinThreads;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      g[i][q] = make_float2(1.f, 1.f);
      acc[i][q] = make_float2(0.f, 0.f);
    }
    if (v < nvec) {
      const uint4 u = *reinterpret_cast<const uint4*>(gamma + 8 * v);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]);
        g[i][q] = make_float2(1.f + f.x, 1.f + f.y);  // gain centre added in fp32
      }
    }
  }
  __syncthreads();  // rowp[] and the barriers' initialisation are visible
  const __nv_bfloat16* srow = reinterpret_cast<const __nv_bfloat16*>(staged);
  const float inv_h = 1.0f / (float)H;
  for (int k = 0; k < K; ++k) {
    if (rowp[k] < 0) continue;  // uniform across the block
    // Bounded wait for route k's row (a bulk copy of a valid row always
    // lands; the limit only keeps a broken launch from spinning forever).
    // A CTA that gives up waits, bounded, for its other copies and exits
    // without writing output.
    {
      const uint64_t t0 = global_timer_ns();
      bool ok = true;
      while (!mbar_try_wait(smem_u32(&bar[k]), 0)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
          ok = false;
          break;
        }
      }
      if (!ok) {
        for (int j = k; j < K; ++j)
          if (rowp[j] >= 0) mbar_wait_cleanup(smem_u32(&bar[j]), 0);
        return;
      }
    }
    float2 f[VPT][4];  // route k's row, converted once
    float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = threadIdx.x + i * kFinThreads;
      const uint4 u = v < nvec ? *reinterpret_cast<const uint4*>(srow + (size_t)k * H + 8 * v)
                               : make_uint4(0, 0, 0, 0);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        f[i][q] = __bfloat1622float2(h[q]);
        const float2 a = weight_before_norm ? fmul2(f[i][q], g[i][q]) : f[i][q];
        ss2 = ffma2(a, a, ss2);
      }
    }
    float ss = ss2.x + ss2.y;
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
    if (lane == 0) red[k & 1][warp] = ss;  // two buffers: one barrier per route
    __syncthreads();
    float total = 0.f;
#pragma unroll
    for (int w = 0; w < kFinWarps; ++w) total += red[k & 1][w];  // fixed order
    const float ck = topk_w[(size_t)t * K + k] / sqrtf(total * inv_h + eps);
    const float2 ck2 = make_float2(ck, ck);
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][q] = ffma2(f[i][q], ck2, acc[i][q]);
  }
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * kFinThreads;
    if (v < nvec) {
      uint4 o;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 r = fmul2(acc[i][q], g[i][q]);
        h[q] = __floats2bfloat162_rn(r.x, r.y);
      }
      *reinterpret_cast<uint4*>(out + (size_t)t * H + 8 * v) = o;
    }
  }
}

// The finalize made persistent for many tokens: a CTA takes tokens
// blockIdx.x, + gridDim.x, ... and streams their route rows through a ring
// of row buffers in shared memory (as many as kFinRingBytes hold, at most
// kFinRingMaxSlots). A producer warp's lane 0 issues the bulk copy of each
// valid route row into the next free slot (one full and one empty mbarrier
// per slot), running up to a ring ahead across token boundaries, so the rows
// of the next token are in flight while this one is reduced. The
// kFinRingThreads consumer threads take the rows in the same order: each
// loads its VPT 8-element vectors of the row into registers (kept as bf16,
// converted where used), hands the slot back (one arrival per consumer
// warp), reduces the row's sum of squares (one barrier of the consumer warps
// per route) and adds coef_k r_k; after a
// token's last route it applies the gain and stores the output row. A route's
// reduction is a chain of dependent steps; the SM's kFinRingCtas CTAs run as
// many such chains at once.
// Both sides read expanded_to_permuted and skip the same entries (-1, and
// out-of-range ones, which the producer records as MOE_ERR_INVALID_ROUTE).
// Every wait is bounded. A producer that gives up stops issuing and lets its
// copies in flight land; the consumers then run through their remaining
// routes without waiting (every wait returns at once once the CTA's abort
// flag is up), so that each of them passes the same per-route barriers, and
// a thread whose wait gave up stores nothing.
constexpr int kFinRingThreads = 128;
constexpr int kFinRingWarps = kFinRingThreads / 32;
// Three CTAs per SM with the gain held in registers: 149.9 us at T = 8192,
// H = 5120, top-8 (the copies alone, timed without the arithmetic, 110 us);
// two CTAs of eight consumer warps 203 us; four CTAs of four warps re-reading
// the gain per row 201 us, holding it in registers (spills) 396 us.
constexpr int kFinRingCtas = 3;  // per SM
constexpr int kFinRingMaxSlots = 16;
constexpr int kFinRingBytes = 60 * 1024;
constexpr int kFinRingMinTokens = 1024;

template <int VPT>
__global__ void __launch_bounds__(kFinRingThreads + 32, kFinRingCtas) finalize_ring_kernel(
    const __nv_bfloat16* __restrict__ rows, const int32_t* __restrict__ e2p,
    const float* __restrict__ topk_w, const __nv_bfloat16* __restrict__ gamma, float eps,
    int weight_before_norm, int T, int K, int H, int num_rows, int R, __nv_bfloat16* __restrict__ out,
    int32_t* status) {
  extern __shared__ __align__(16) uint8_t ring[];  // R rows of H bf16
  __shared__ __align__(8) uint64_t full[kFinRingMaxSlots];
  __shared__ __align__(8) uint64_t empty[kFinRingMaxSlots];
  __shared__ float red[2][kFinRingWarps];
  __shared__ int abort_flag;
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = H / 8;
  const uint32_t row_bytes = (uint32_t)H * 2;
  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kFinRingWarps);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == kFinRingWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      int n = 0;  // rows issued
      bool stop = false;
      for (int t = blockIdx.x; t < T && !stop; t += gridDim.x) {
        for (int k = 0; k < K; ++k) {
          int p = e2p[(size_t)t * K + k];
          if (p < -1 || p >= num_rows) {
            record_status(status, MOE_ERR_INVALID_ROUTE);
            p = -1;
          }
          if (p < 0) continue;
          const int slot = n % R, use = n / R;
          if (use > 0 && !mbar_wait(smem_u32(&empty[slot]), (use - 1) & 1, &abort_flag, status)) {
            stop = true;
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&full[slot]), row_bytes);
          bulk_load(smem_u32(ring) + slot * row_bytes, rows + (size_t)p * H, row_bytes, smem_u32(&full[slot]));
          ++n;
        }
      }
      // every copy issued has landed before the CTA's shared memory goes
      for (int j = max(0, n - R); j < n; ++j) mbar_wait_cleanup(smem_u32(&full[j % R]), (j / R) & 1);
    }
    return;
  }
  // ------------------------------ consumers ------------------------------
  // gain g = 1 + gamma (fp32), pairs of hidden-dimension elements
  float2 g[VPT][4];
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * kFinRingThreads;
    const uint4 u = v < nvec ? __ldg(reinterpret_cast<const uint4*>(gamma + 8 * v)) : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(h[q]);
      g[i][q] = make_float2(1.f + f.x, 1.f + f.y);  // gain centre added in fp32
    }
  }
  const float inv_h = 1.0f / (float)H;
  int n = 0;       // rows consumed
  bool ok = true;  // every wait of this thread ended with its row landed
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    float2 acc[VPT][4];
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][q] = make_float2(0.f, 0.f);
    for (int k = 0; k < K; ++k) {
      const int p = e2p[(size_t)t * K + k];
      if (p < 0 || p >= num_rows) continue;  // the producer's decision, uniform across the CTA
      const float wk = topk_w[(size_t)t * K + k];
      const int slot = n % R;
      ok = mbar_wait(smem_u32(&full[slot]), (n / R) & 1, &abort_flag, status) && ok;
      const __nv_bfloat16* srow = reinterpret_cast<const __nv_bfloat16*>(ring + slot * row_bytes);
      uint4 raw[VPT];  // route k's row, kept as bf16 (converted again when added)
      float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = threadIdx.x + i * kFinRingThreads;
        raw[i] = v < nvec ? *reinterpret_cast<const uint4*>(srow + 8 * v) : make_uint4(0, 0, 0, 0);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[i]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __bfloat1622float2(h[q]);
          const float2 a = weight_before_norm ? fmul2(f, g[i][q]) : f;
          ss2 = ffma2(a, a, ss2);
        }
      }
      // the slot's bytes are in registers: hand it back to the producer
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
      float ss = ss2.x + ss2.y;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
      if (lane == 0) red[n & 1][warp] = ss;  // two buffers: one barrier per route
      fin_bar_sync(kFinRingThreads);
      float total = 0.f;
#pragma unroll
      for (int w = 0; w < kFinRingWarps; ++w) total += red[n & 1][w];  // fixed order
      // w / sqrt(ms + eps) as w * rsqrt(ms + eps): within 2 ulp in fp32, far
      // below the bf16 output's step, and fewer instructions on the route's
      // chain (142.7 against 149.9 us at T = 8192)
      const float ck = wk * rsqrtf(total * inv_h + eps);
      const float2 ck2 = make_float2(ck, ck);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[i]);
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = ffma2(__bfloat1622float2(h[q]), ck2, acc[i][q]);
      }
      ++n;
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = threadIdx.x + i * kFinRingThreads;
      if (v < nvec && ok) {
        uint4 o;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 r = fmul2(acc[i][q], g[i][q]);
          h[q] = __floats2bfloat162_rn(r.x, r.y);
        }
        *reinterpret_cast<uint4*>(out + (size_t)t * H + 8 * v) = o;
      }
    }
  }
}

// The expert-TP tail's form of the ring kernel: a route's row is the sum of
// nparts partial row buffers (fp32 sum in part order, one bf16 rounding:
// load_row_vec's arithmetic), so the producer copies each route's nparts
// part rows into consecutive slots, and the consumers add them up (the slot
// goes back as soon as its part is in registers) before the route's norm.
// Two CTAs per SM: the fp32 sums of a route's vectors take registers that
// three CTAs would not have.
constexpr int kFinRingPartsCtas = 2;
constexpr int kFinRingPartsBytes = 96 * 1024;

template <int VPT>
__global__ void __launch_bounds__(kFinRingThreads + 32, kFinRingPartsCtas) finalize_ring_parts_kernel(
    const RowParts parts, const int32_t* __restrict__ e2p, const float* __restrict__ topk_w,
    const __nv_bfloat16* __restrict__ gamma, float eps, int weight_before_norm, int T, int K, int H, int num_rows,
    int R, __nv_bfloat16* __restrict__ out, int32_t* status) {
  extern __shared__ __align__(16) uint8_t ring[];  // R part rows of H bf16
  __shared__ __align__(8) uint64_t full[kFinRingMaxSlots];
  __shared__ __align__(8) uint64_t empty[kFinRingMaxSlots];
  __shared__ float red[2][kFinRingWarps];
  __shared__ int abort_flag;
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nvec = H / 8, np = parts.n;
  const uint32_t row_bytes = (uint32_t)H * 2;
  if (threadIdx.x == 0) {
    for (int i = 0; i < R; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kFinRingWarps);
    }
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (warp == kFinRingWarps) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      int n = 0;  // part rows issued
      bool stop = false;
      for (int t = blockIdx.x; t < T && !stop; t += gridDim.x) {
        for (int k = 0; k < K && !stop; ++k) {
          int p = e2p[(size_t)t * K + k];
          if (p < -1 || p >= num_rows) {
            record_status(status, MOE_ERR_INVALID_ROUTE);
            p = -1;
          }
          if (p < 0) continue;
          for (int j = 0; j < np; ++j) {
            const int slot = n % R, use = n / R;
            if (use > 0 && !mbar_wait(smem_u32(&empty[slot]), (use - 1) & 1, &abort_flag, status)) {
              stop = true;
              break;
            }
            mbar_arrive_expect_tx(smem_u32(&full[slot]), row_bytes);
            bulk_load(smem_u32(ring) + slot * row_bytes, parts.p[j] + (size_t)p * H, row_bytes,
                      smem_u32(&full[slot]));
            ++n;
          }
        }
      }
      // every copy issued has landed before the CTA's shared memory goes
      for (int j = max(0, n - R); j < n; ++j) mbar_wait_cleanup(smem_u32(&full[j % R]), (j / R) & 1);
    }
    return;
  }
  // ------------------------------ consumers ------------------------------
  float2 g[VPT][4];  // gain g = 1 + gamma (fp32)
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int v = threadIdx.x + i * kFinRingThreads;
    const uint4 u = v < nvec ? __ldg(reinterpret_cast<const uint4*>(gamma + 8 * v)) : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(h[q]);
      g[i][q] = make_float2(1.f + f.x, 1.f + f.y);
    }
  }
  const float inv_h = 1.0f / (float)H;
  int n = 0;       // part rows consumed
  int nr = 0;      // routes reduced
  bool ok = true;  // every wait of this thread ended with its row landed
  for (int t = blockIdx.x; t < T; t += gridDim.x) {
    float2 acc[VPT][4];
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[i][q] = make_float2(0.f, 0.f);
    for (int k = 0; k < K; ++k) {
      const int p = e2p[(size_t)t * K + k];
      if (p < 0 || p >= num_rows) continue;  // the producer's decision, uniform across the CTA
      const float wk = topk_w[(size_t)t * K + k];
      // the route's row: fp32 sum of its parts in part order, one bf16 rounding
      float2 sum[VPT][4];
#pragma unroll
      for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int q = 0; q < 4; ++q) sum[i][q] = make_float2(0.f, 0.f);
      for (int j = 0; j < np; ++j) {
        const int slot = n % R;
        ok = mbar_wait(smem_u32(&full[slot]), (n / R) & 1, &abort_flag, status) && ok;
        const __nv_bfloat16* srow = reinterpret_cast<const __nv_bfloat16*>(ring + slot * row_bytes);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
          const int v = threadIdx.x + i * kFinRingThreads;
          const uint4 u = v < nvec ? *reinterpret_cast<const uint4*>(srow + 8 * v) : make_uint4(0, 0, 0, 0);
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(h[q]);
            sum[i][q].x += f.x;
            sum[i][q].y += f.y;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
        ++n;
      }
      uint4 raw[VPT];  // the route's row, bf16
      float2 ss2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw[i]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          h[q] = __floats2bfloat162_rn(sum[i][q].x, sum[i][q].y);
          const float2 f = __bfloat1622float2(h[q]);
          const float2 a = weight_before_norm ? fmul2(f, g[i][q]) : f;
          ss2 = ffma2(a, a, ss2);
        }
      }
      float ss = ss2.x + ss2.y;
#pragma unroll
      for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, d);
      if (lane == 0) red[nr & 1][warp] = ss;  // two buffers: one barrier per route
      fin_bar_sync(kFinRingThreads);
      float total = 0.f;
#pragma unroll
      for (int w = 0; w < kFinRingWarps; ++w) total += red[nr & 1][w];  // fixed order
      const float ck = wk * rsqrtf(total * inv_h + eps);
      const float2 ck2 = make_float2(ck, ck);
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[i]);
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[i][q] = ffma2(__bfloat1622float2(h[q]), ck2, acc[i][q]);
      }
      ++nr;
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = threadIdx.x + i * kFinRingThreads;
      if (v < nvec && ok) {
        uint4 o;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 r = fmul2(acc[i][q], g[i][q]);
          h[q] = __floats2bfloat162_rn(r.x, r.y);
        }
        *reinterpret_cast<uint4*>(out + (size_t)t * H + 8 * v) = o;
      }
    }
  }
}

// The finalize for few tokens (decode batches), where its latency counts:
// one CTA per token and one thread per 8-element vector of the hidden
// dimension (H / 8 threads, H up to 5120), each loading its vector of all K
// (<= 8) route rows at once (the rows were just written, mostly still in
// L2). Every thread's share of each route's sum of squares goes to shared
// memory, one warp per route sums them in a fixed order, and after a
// single block barrier every thread adds coef_k * r_k from its registers and
// applies the gain: out = bf16(g * sum_k coef_k r_k). One reduction round
// for all routes, where the staged kernel waits on one per route.
constexpr int kFinFewMaxK = 8;
constexpr int kFinFewMaxThreads = 640;
constexpr int kFinFewMaxTokens = 128;

__global__ void __launch_bounds__(kFinFewMaxThreads, 1) finalize_few_kernel(
    const __nv_bfloat16* __restrict__ rows, int num_rows, const int32_t* __restrict__ e2p,
    const float* __restrict__ topk_w, const __nv_bfloat16* __restrict__ gamma, float eps,
    int weight_before_norm, int K, int H, __nv_bfloat16* __restrict__ out, int32_t* status) {
  __shared__ __align__(16) float part[kFinFewMaxThreads][kFinFewMaxK];
  __shared__ float coef[kFinFewMaxK];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int v = threadIdx.x, lane = v & 31, warp = v >> 5, nwarps = blockDim.x >> 5;
  const bool on = v < H / 8;
  uint4 raw[kFinFewMaxK];
#pragma unroll
  for (int k = 0; k < kFinFewMaxK; ++k) {
    const int p = k < K ? checked_row(e2p[(size_t)t * K + k], num_rows, status) : -1;
    raw[k] = (on && p >= 0) ? *(reinterpret_cast<const uint4*>(rows + (size_t)p * H) + v) : make_uint4(0, 0, 0, 0);
  }
  float2 g[4];
  {
    const uint4 gu = on ? __ldg(reinterpret_cast<const uint4*>(gamma + 8 * v)) : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&gu);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(gh[q]);
      g[q] = make_float2(1.f + f.x, 1.f + f.y);  // gain centre added in fp32
    }
  }
  {
    float ss[kFinFewMaxK];
#pragma unroll
    for (int k = 0; k < kFinFewMaxK; ++k) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[k]);
      float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = __bfloat1622float2(h[q]);
        const float2 a = weight_before_norm ? fmul2(f, g[q]) : f;
        s2 = ffma2(a, a, s2);
      }
      ss[k] = s2.x + s2.y;
    }
    float4* dst = reinterpret_cast<float4*>(&part[v][0]);
    dst[0] = make_float4(ss[0], ss[1], ss[2], ss[3]);
    dst[1] = make_float4(ss[4], ss[5], ss[6], ss[7]);
  }
  __syncthreads();
  for (int k = warp; k < K; k += nwarps) {
    // route k: the threads' shares in a fixed order
    float ss = 0.f;
    for (int i = lane; i < (int)blockDim.x; i += 32) ss += part[i][k];
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, d);
    const int p = e2p[(size_t)t * K + k];
    if (lane == 0)
      coef[k] = (p >= 0 && p < num_rows) ? topk_w[(size_t)t * K + k] / sqrtf(ss / (float)H + eps) : 0.f;
  }
  __syncthreads();
  if (!on) return;
  float2 acc[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.f, 0.f);
#pragma unroll
  for (int k = 0; k < kFinFewMaxK; ++k) {
    const float c = k < K ? coef[k] : 0.f;
    const float2 ck = make_float2(c, c);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[k]);
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = ffma2(__bfloat1622float2(h[q]), ck, acc[q]);
  }
  uint4 o;
  __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 r = fmul2(acc[q], g[q]);
    oh[q] = __floats2bfloat162_rn(r.x, r.y);
  }
  *reinterpret_cast<uint4*>(out + (size_t)t * H + 8 * v) = o;
}

cudaError_t launch_finalize_parts(const void* const* parts, int nparts, int num_rows, const int32_t* e2p,
                                  const float* w, const void* gamma, float eps,
                                  int weight_before_norm, int T, int K, int H, void* out,
                                  int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (nparts < 1 || nparts > kMaxParts) return cudaErrorInvalidValue;
  RowParts rp{};
  rp.n = nparts;
  for (int i = 0; i < nparts; ++i) rp.p[i] = reinterpret_cast<const __nv_bfloat16*>(parts[i]);
  const int vpt = ceil_div(H / 8, kFinThreads);
  auto gp = reinterpret_cast<const __nv_bfloat16*>(gamma);
  auto op = reinterpret_cast<__nv_bfloat16*>(out);
  cudaError_t err = cudaSuccess;
  const size_t staged = (size_t)K * H * 2;
  // few tokens: the latency of one reduction round matters more than bandwidth
  if (nparts == 1 && T <= kFinFewMaxTokens && K <= kFinFewMaxK && H <= 8 * kFinFewMaxThreads)
    return launch_kernel(finalize_few_kernel, dim3(T), dim3((H / 8 + 31) / 32 * 32), 0, stream, true,
                         reinterpret_cast<const __nv_bfloat16*>(parts[0]), num_rows, e2p, w, gp, eps,
                         weight_before_norm, K, H, op, status);
  const int ring_slots = (int)std::min<size_t>(kFinRingMaxSlots, (size_t)kFinRingBytes / ((size_t)H * 2));
  const int ring_vpt = ceil_div(H / 8, kFinRingThreads);
  const int parts_slots = (int)std::min<size_t>(kFinRingMaxSlots, (size_t)kFinRingPartsBytes / ((size_t)H * 2));
  if (nparts > 1 && T >= kFinRingMinTokens && parts_slots >= 2 && ring_vpt <= 5) {
    static int psms = 0;
    if (psms == 0) {
      int dev = 0, n = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 148;
      psms = n;
    }
    const int grid = std::min(T, kFinRingPartsCtas * psms);
    const size_t smem = (size_t)parts_slots * H * 2;
#define MOE_FIN_RING_PARTS(n)                                                                                   \
  case n:                                                                                                       \
    err = ensure_smem_limit(reinterpret_cast<const void*>(finalize_ring_parts_kernel<n>), kFinRingPartsBytes);   \
    if (err == cudaSuccess)                                                                                     \
      err = launch_kernel(finalize_ring_parts_kernel<n>, dim3(grid), dim3(kFinRingThreads + 32), smem, stream,   \
                          true, rp, e2p, w, gp, eps, weight_before_norm, T, K, H, num_rows, parts_slots, op,     \
                          status);                                                                              \
    return err;
    switch (ring_vpt) {
      MOE_FIN_RING_PARTS(1)
      MOE_FIN_RING_PARTS(2)
      MOE_FIN_RING_PARTS(3)
      MOE_FIN_RING_PARTS(4)
      MOE_FIN_RING_PARTS(5)
      default:
        return cudaErrorInvalidValue;
    }
#undef MOE_FIN_RING_PARTS
  }
  if (nparts == 1 && T >= kFinRingMinTokens && ring_slots >= 2 && ring_vpt <= 5) {
    auto rows = reinterpret_cast<const __nv_bfloat16*>(parts[0]);
    static int sms = 0;
    if (sms == 0) {
      int dev = 0, n = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 148;
      sms = n;
    }
    const int grid = std::min(T, kFinRingCtas * sms);
    const size_t smem = (size_t)ring_slots * H * 2;
#define MOE_FIN_RING(n)                                                                                       \
  case n:                                                                                                     \
    err = ensure_smem_limit(reinterpret_cast<const void*>(finalize_ring_kernel<n>), kFinRingBytes);            \
    if (err == cudaSuccess)                                                                                   \
      err = launch_kernel(finalize_ring_kernel<n>, dim3(grid), dim3(kFinRingThreads + 32), smem, stream, true, \
                          rows, e2p, w, gp, eps, weight_before_norm, T, K, H, num_rows, ring_slots, op,        \
                          status);                                                                            \
    return err;
    switch (ring_vpt) {
      MOE_FIN_RING(1)
      MOE_FIN_RING(2)
      MOE_FIN_RING(3)
      MOE_FIN_RING(4)
      MOE_FIN_RING(5)
      default:
        return cudaErrorInvalidValue;
    }
#undef MOE_FIN_RING
  }
  if (nparts == 1 && K <= kFinMaxK && staged <= (size_t)kFinStagedMaxBytes && vpt <= 5) {
    auto rows = reinterpret_cast<const __nv_bfloat16*>(parts[0]);
#define MOE_FIN_STAGED(n)                                                                       \
  case n:                                                                                       \
    err = ensure_smem_limit(reinterpret_cast<const void*>(finalize_staged_kernel<n>),            \
                            kFinStagedMaxBytes);                                                  \
    if (err == cudaSuccess)                                                                     \
      err = launch_kernel(finalize_staged_kernel<n>, dim3(T), dim3(kFinThreads), staged, stream,  \
                          true, rows, e2p, w, gp, eps, weight_before_norm, K, H, num_rows, op, status);            \
    return err;
    switch (vpt) {
      MOE_FIN_STAGED(1)
      MOE_FIN_STAGED(2)
      MOE_FIN_STAGED(3)
      MOE_FIN_STAGED(4)
      MOE_FIN_STAGED(5)
      default:
        return cudaErrorInvalidValue;
    }
#undef MOE_FIN_STAGED
  }
#define MOE_FIN_CASE(n)                                                                     \
  case n:                                                                                   \
    err = launch_kernel(finalize_kernel<n, (n <= 2 ? kFinChunk : n <= 4 ? 4 : 2)>, dim3(T),            \
                        dim3(kFinThreads), 0, stream, true, rp, e2p, w, gp, eps,                 \
                        weight_before_norm, K, H, num_rows, op, status);                         \
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
  return err;
}

}  // namespace moe

namespace moe {
cudaError_t launch_finalize(const void* rows, int num_rows, const int32_t* e2p, const float* w,
                            const void* gamma, float eps, int weight_before_norm, int T, int K, int H,
                            void* out, int32_t* status, cudaStream_t stream) {
  const void* parts[1] = {rows};
  return launch_finalize_parts(parts, 1, num_rows, e2p, w, gamma, eps, weight_before_norm, T, K, H, out, status,
                               stream);
}
}  // namespace moe

namespace moe {

// The finalize when GEMM2's epilogue already produced each route row's sums
// of squares (row_ss [num_rows][H / 32], fp32 partials over 32 columns, gain
// weighted for the weight-before-norm reading): every route's coefficient
// w[t, k] / sqrt(mean + eps) is known before any row is read, so the rows
// stream through once with no reduction between a row's load and its use.
// One CTA per token: route k's H / 32 partials are summed by 16 lanes of
// one warp, as float4s (lane j takes float4s j, j + 16, ..., adding .x, .y,
// .z, .w in turn; then an xor butterfly over the 16 lanes), the order the
// finalize_sumsq_units_kernel uses too; then
// every thread takes 8-element vectors of the hidden dimension, issues the
// loads of all of its routes' vectors at once (up to eight in flight), and
// accumulates coef_k * r_k in fp32; out = bf16(g * sum), g = 1 + gamma, in
// both readings.
constexpr int kFinSsThreads = 256;

__global__ void __launch_bounds__(kFinSsThreads) finalize_sumsq_kernel(
    const __nv_bfloat16* __restrict__ rows, const float* __restrict__ row_ss, int num_rows,
    const int32_t* __restrict__ e2p, const float* __restrict__ topk_w, const __nv_bfloat16* __restrict__ gamma,
    float eps, int K, int H, __nv_bfloat16* __restrict__ out, int32_t* status) {
  __shared__ float coef[kFinMaxK];
  __shared__ int32_t rowp[kFinMaxK];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int G4 = H / 128;
  // routes 16 r + 2 warp + (lane >> 4), over the 16 lanes lane & 15
  for (int k0 = 0; k0 < K; k0 += 2 * (kFinSsThreads / 32)) {
    const int k = k0 + 2 * warp + (lane >> 4), j = lane & 15;
    int p = -1;
    if (k < K) {
      p = e2p[(size_t)t * K + k];
      if (p < -1 || p >= num_rows) {
        if (j == 0) record_status(status, MOE_ERR_INVALID_ROUTE);
        p = -1;
      }
    }
    const float4* src = reinterpret_cast<const float4*>(row_ss + (size_t)(p >= 0 ? p : 0) * (H / 32));
    float ss = 0.f;
    if (p >= 0)
      for (int m = j; m < G4; m += 16) {
        const float4 x = src[m];
        ss += x.x;
        ss += x.y;
        ss += x.z;
        ss += x.w;
      }
#pragma unroll
    for (int d = 1; d < 16; d <<= 1) ss += __shfl_xor_sync(0xFFFFFFFFu, ss, d);
    if (k < K && j == 0) {
      rowp[k] = p;
      coef[k] = p >= 0 ? topk_w[(size_t)t * K + k] / sqrtf(ss / (float)H + eps) : 0.f;
    }
  }
  __syncthreads();
  const int nvec = H / 8;
  for (int v = threadIdx.x; v < nvec; v += kFinSsThreads) {
    float2 acc[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.f, 0.f);
    for (int k0 = 0; k0 < K; k0 += 8) {
      uint4 raw[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int k = k0 + c;
        const int p = k < K ? rowp[k] : -1;
        raw[c] = p >= 0 ? __ldcs(reinterpret_cast<const uint4*>(rows + (size_t)p * H) + v) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int k = k0 + c;
        if (k >= K) break;
        const float2 ck = make_float2(coef[k], coef[k]);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[c]);
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = ffma2(__bfloat1622float2(h[q]), ck, acc[q]);
      }
    }
    const uint4 gu = *reinterpret_cast<const uint4*>(gamma + 8 * v);
    const __nv_bfloat162* gh = reinterpret_cast<const __nv_bfloat162*>(&gu);
    uint4 o;
    __nv_bfloat162* oh = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 gf = __bfloat1622float2(gh[q]);
      const float2 r = fmul2(acc[q], make_float2(1.f + gf.x, 1.f + gf.y));  // gain centre added in fp32
      oh[q] = __floats2bfloat162_rn(r.x, r.y);
    }
    *reinterpret_cast<uint4*>(out + (size_t)t * H + 8 * v) = o;
  }
}

// The same finalize for K <= 8 in units of (token, 1024 columns), four warps
// each (finalize_units.cuh): a persistent grid walks the units, reading the next
// unit's routing while it finishes the current one, so that no CTA waits
// through a coefficient phase with nothing else in flight.
__global__ void __launch_bounds__(32 * kFinUnitWarps) finalize_sumsq_units_kernel(FinArgs a, int T) {
  __shared__ float coef[kFinUnitMaxK];
  pdl_wait();
  pdl_trigger();
  constexpr int kThreads = 32 * kFinUnitWarps;
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int slices = (a.H / 8 + kThreads - 1) / kThreads, n = T * slices;
  int u = blockIdx.x;
  FinPre f{};
  if (u < n) f = fin_prepare(a, u / slices, (u % slices) * kThreads + 32 * wi + lane, lane);
  while (u < n) {
    const int un = u + gridDim.x;
    FinPre g{};
    if (un < n) g = fin_prepare(a, un / slices, (un % slices) * kThreads + 32 * wi + lane, lane);
    fin_finish_inl(a, f, lane, wi, coef, kThreads);
    fin_bar_sync(kThreads);  // every warp has read coef before the next unit writes it
    f = g;
    u = un;
  }
}

cudaError_t launch_finalize_sumsq(const void* rows, const float* row_ss, int num_rows, const int32_t* e2p,
                                  const float* w, const void* gamma, float eps, int T, int K, int H, void* out,
                                  int32_t* status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (K > kFinMaxK) return cudaErrorInvalidValue;
  if (K <= kFinUnitMaxK) {
    FinArgs a;
    a.rows = reinterpret_cast<const __nv_bfloat16*>(rows);
    a.row_ss = row_ss;
    a.e2p = e2p;
    a.w = w;
    a.gamma = reinterpret_cast<const __nv_bfloat16*>(gamma);
    a.out = reinterpret_cast<__nv_bfloat16*>(out);
    a.status = status;
    a.eps = eps;
    a.K = K;
    a.H = H;
    a.num_rows = num_rows;
    static int sms = 0;
    if (sms == 0) {
      int dev = 0, n = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        n = 148;
      sms = n;
    }
    static int per_sm = 0;
    if (per_sm == 0) {
      int b = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, finalize_sumsq_units_kernel, 32 * kFinUnitWarps, 0) !=
              cudaSuccess ||
          b < 1)
        b = 4;
      per_sm = b;
    }
    const long long units = (long long)T * ((H / 8 + 32 * kFinUnitWarps - 1) / (32 * kFinUnitWarps));
    const long long slots = (long long)sms * per_sm;
    const int grid = (int)(units < slots ? units : slots);
    return launch_kernel(finalize_sumsq_units_kernel, dim3(grid), dim3(32 * kFinUnitWarps), 0, stream, true, a, T);
  }
  return launch_kernel(finalize_sumsq_kernel, dim3(T), dim3(kFinSsThreads), 0, stream, true,
                       reinterpret_cast<const __nv_bfloat16*>(rows), row_ss, num_rows, e2p, w,
                       reinterpret_cast<const __nv_bfloat16*>(gamma), eps, K, H,
                       reinterpret_cast<__nv_bfloat16*>(out), status);
}

}  // namespace moe
