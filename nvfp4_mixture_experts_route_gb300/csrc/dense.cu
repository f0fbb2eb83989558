// The MoE pooler and unpooler around the expert block (the model page: the
// MoE's `pooler` ReplicatedLinear(hidden_size, moe_hidden_size, bias=False,
// quant_config=None) before the experts and `unpooler` back after them):
// plain bf16 projections y = x . w^T with fp32 accumulation and one bf16
// rounding, on the 5th-generation tensor cores (tcgen05.mma kind::f16).
//
// Tiling (swapped, as for the decode GEMMs): the MMA's M = 128 rows are output
// features (weight rows), N = a tile of tokens (32, 64, 128 or 256 by T);
// a unit is (token tile, 128-feature tile, K slice). Few tokens give few
// (token, feature) tiles, so K is split into slices until there are about
// four units per CTA; each slice then writes an fp32 partial [slice][T][Dout]
// and dense_reduce_kernel sums the slices in order and rounds once.
//
// Persistent, warp-specialised kernel, one or two CTAs per SM, 6 warps: warp 0 lane 0
// is the TMA producer (per stage of K = 64 elements: a 128 x 128 B weight box
// and an N x 128 B token box, both 128-byte swizzled, on one mbarrier), warp 1
// lane 0 issues 4 MMAs of K = 16 per stage and commits the stage back, warps
// 2-5 are the epilogue (TMEM lane quadrant w % 4); two accumulator buffers.
// Every mbarrier wait is bounded (1 s); on a timeout the CTA records
// MOE_ERR_TIMEOUT, stops, drains its copies and MMAs, frees its tensor memory
// and exits.
#include "common.cuh"

namespace moe {

constexpr int kDThreads = 192;
constexpr int kDMaxStages = 8;
constexpr uint32_t kDWBytes = 128 * 128;  // weight box per stage

struct DenseParams {
  __nv_bfloat16* y;  // [T, Dout] when slices == 1
  float* part;       // [slices, T, Dout] otherwise
  int32_t* status;
  int T, Din, Dout, slices;
};

// Token tiles of up to 64 run two CTAs per SM (two TMA producers and MMA
// issuers streaming weights), larger ones one.
__host__ __device__ constexpr int dense_ctas(int n) { return n <= 64 ? 2 : 1; }
__host__ __device__ constexpr uint32_t dense_stage_bytes(int n) { return kDWBytes + (uint32_t)n * 128; }
__host__ __device__ constexpr int dense_stages(int n) {
  const int st = ((dense_ctas(n) == 1 ? 232448 : 115456) - 1024) / (int)dense_stage_bytes(n);
  return st > kDMaxStages ? kDMaxStages : st;
}
__host__ __device__ constexpr size_t dense_smem_bytes(int n) {
  return 1024 + (size_t)dense_stages(n) * dense_stage_bytes(n);
}

// Instruction descriptor for kind::f16: fp32 accumulator (bits [4,6) = 1),
// A and B bf16 (format 1 in [7,10) and [10,13)), both K-major, N >> 3 in
// [17,23), M >> 4 in [24,29).
__host__ __device__ constexpr uint32_t idesc_bf16(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int N>
__global__ void __launch_bounds__(kDThreads, dense_ctas(N))
    dense_bf16_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const DenseParams p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kDMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kDMaxStages];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  pdl_wait();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) pdl_trigger();

  constexpr int ST = dense_stages(N);
  constexpr uint32_t ncols = 2 * N;  // two accumulator buffers
  const int tiles_w = p.Dout / 128, tiles_t = (p.T + N - 1) / N;
  const int per_slice = tiles_w * tiles_t;
  const int n_units = per_slice * p.slices;
  if ((int)blockIdx.x >= n_units) return;
  const int KC = p.Din / 64;                               // K = 64 stages along Din
  const int spc = (KC + p.slices - 1) / p.slices;          // stages per slice
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sW = sbase, sX = sW + ST * kDWBytes;

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&accf_bar[b]), 1);
      mbar_init(smem_u32(&acce_bar[b]), 4);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      int it = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x) {
        const int slice = u / per_slice, rem = u % per_slice;
        const int tt = rem / tiles_w, mt = rem % tiles_w;
        const int k0 = slice * spc, k1 = min(KC, k0 + spc);
        for (int kc = k0; kc < k1; ++kc, ++it) {
          const int s = it % ST, round = it / ST;
          if (round > 0 &&
              !mbar_wait(smem_u32(&empty_bar[s]), (round - 1) & 1, &abort_flag, p.status)) {
            stop = true;
            break;
          }
          const uint32_t fb = smem_u32(&full_bar[s]);
          mbar_arrive_expect_tx(fb, dense_stage_bytes(N));
          tma_load_2d(sW + s * kDWBytes, &tmW, fb, kc * 128, mt * 128);
          tma_load_2d(sX + s * (uint32_t)N * 128, &tmX, fb, kc * 128, tt * N);
        }
      }
      for (int j = max(0, it - ST); j < it; ++j)
        mbar_wait_cleanup(smem_u32(&full_bar[j % ST]), (j / ST) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ----------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, N);
      const uint64_t w_desc0 = smem_desc(sW, 16, 1024, 2);
      const uint64_t x_desc0 = smem_desc(sX, 16, 1024, 2);
      int it = 0, uc = 0;
      bool stop = false;
      for (int u = blockIdx.x; u < n_units && !stop; u += gridDim.x, ++uc) {
        const int b = uc & 1, use = uc >> 1;
        if (use > 0 && !mbar_wait(smem_u32(&acce_bar[b]), (use - 1) & 1, &abort_flag, p.status))
          break;
        tc_fence_after();
        const int slice = u / per_slice;
        const int k0 = slice * spc, k1 = min(KC, k0 + spc);
        const uint32_t dacc = tmem + (uint32_t)(b * N);
        for (int kc = k0; kc < k1; ++kc, ++it) {
          const int s = it % ST, round = it / ST;
          if (!mbar_wait(smem_u32(&full_bar[s]), round & 1, &abort_flag, p.status)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint64_t wd = w_desc0 + ((s * kDWBytes) >> 4), xd = x_desc0 + ((s * (uint32_t)N * 128) >> 4);
#pragma unroll
          for (int j = 0; j < 4; ++j)  // K = 16 bf16 = 32 bytes per MMA
            tc_mma_bf16(dacc, wd + 2 * j, xd + 2 * j, idesc, (kc > k0 || j > 0) ? 1u : 0u);
          tc_commit(smem_u32(&empty_bar[s]));
        }
        if (stop) break;
        tc_commit(smem_u32(&accf_bar[b]));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;
    int uc = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++uc) {
      const int b = uc & 1, use = uc >> 1;
      const bool ok = mbar_wait(smem_u32(&accf_bar[b]), use & 1, &abort_flag, p.status);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      const int slice = u / per_slice, rem = u % per_slice;
      const int tt = rem / tiles_w, mt = rem % tiles_w;
      const int o = mt * 128 + 32 * q + lane;  // this lane's output feature
      const uint32_t taddr = tmem + (uint32_t)(b * N) + ((uint32_t)(32 * q) << 16);
      for (int c0 = 0; c0 < N; c0 += 32) {
        float v[32];
        tmem_ld32(taddr + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int t = tt * N + c0 + i;
          if (t < p.T) {
            if (p.slices == 1)
              p.y[(size_t)t * p.Dout + o] = __float2bfloat16_rn(v[i]);
            else
              p.part[((size_t)slice * p.T + t) * p.Dout + o] = v[i];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acce_bar[b]));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) {
      tc_commit(smem_u32(&drain_bar));
      mbar_wait_cleanup(smem_u32(&drain_bar), 0);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// y[i] = bf16(sum over slices s = 0, 1, ... of part[s][i]), four elements per thread.
__global__ void __launch_bounds__(256) dense_reduce_kernel(const float* __restrict__ part, int slices,
                                                           long long n, __nv_bfloat16* __restrict__ y) {
  pdl_wait();
  pdl_trigger();
  for (long long i = 4 * (blockIdx.x * (long long)blockDim.x + threadIdx.x); i < n;
       i += 4ll * gridDim.x * blockDim.x) {
    float4 acc = *reinterpret_cast<const float4*>(part + i);
    for (int s = 1; s < slices; ++s) {
      const float4 v = *reinterpret_cast<const float4*>(part + (size_t)s * n + i);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(y + i) = o;
  }
}

int dense_tile_n(int T) { return T <= 32 ? 32 : T <= 64 ? 64 : T <= 128 ? 128 : 256; }

static int dense_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 148;
  return n;
}

// K slices: few (token, feature) tiles cannot keep every SM streaming
// weights, so Din is split until there are about four units per SM (the
// persistent CTAs then finish within a unit of each other), each slice
// keeping at least 4 stages of K = 64; the count is then trimmed so that no
// slice is empty (slices * stages-per-slice covers Din exactly once).
int dense_slices(int T, int Din, int Dout, int nsm) {
  const int n = dense_tile_n(T);
  const int base = ((T + n - 1) / n) * (Dout / 128);
  const int KC = Din / 64;
  int s = 1;
  while (base * s < 4 * dense_ctas(n) * nsm && KC / (s * 2) >= 4) s *= 2;
  const int spc = (KC + s - 1) / s;
  return (KC + spc - 1) / spc;
}

int dense_slices_here(int T, int Din, int Dout) { return dense_slices(T, Din, Dout, dense_sm_count()); }

template <int N>
static cudaError_t launch_dense_n(const CUtensorMap& tw, const CUtensorMap& tx, const DenseParams& p,
                                  cudaStream_t stream) {
  auto kern = dense_bf16_kernel<N>;
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), (int)dense_smem_bytes(N));
  if (err != cudaSuccess) return err;
  const long long units = (long long)((p.T + N - 1) / N) * (p.Dout / 128) * p.slices;
  const int slots = dense_ctas(N) * dense_sm_count();
  const int grid = (int)(units < slots ? units : slots);
  return launch_kernel(kern, dim3(grid), dim3(kDThreads), dense_smem_bytes(N), stream, true, tw, tx, p);
}

int launch_dense_bf16(const void* x, const void* w, int T, int Din, int Dout, void* y, void* ws,
                      int32_t* status, cudaStream_t stream, const char** why) {
  CUtensorMap tw, tx;
  const int n = dense_tile_n(T);
  if (encode_rows_map(&tw, w, (uint64_t)Din * 2, (uint64_t)Dout, 128) != CUDA_SUCCESS ||
      encode_rows_map(&tx, x, (uint64_t)Din * 2, (uint64_t)T, (uint32_t)n) != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled failed for the dense projection";
    return MOE_ERR_CUDA;
  }
  DenseParams p{};
  p.y = reinterpret_cast<__nv_bfloat16*>(y);
  p.part = reinterpret_cast<float*>(ws);
  p.status = status;
  p.T = T;
  p.Din = Din;
  p.Dout = Dout;
  p.slices = dense_slices(T, Din, Dout, dense_sm_count());
  cudaError_t err;
  switch (n) {
    case 32: err = launch_dense_n<32>(tw, tx, p, stream); break;
    case 64: err = launch_dense_n<64>(tw, tx, p, stream); break;
    case 128: err = launch_dense_n<128>(tw, tx, p, stream); break;
    default: err = launch_dense_n<256>(tw, tx, p, stream); break;
  }
  if (err == cudaSuccess && p.slices > 1) {
    const long long total = (long long)T * Dout;
    long long g = (total / 4 + 255) / 256;
    if (g > 152 * 8) g = 152 * 8;
    err = launch_kernel(dense_reduce_kernel, dim3((int)(g < 1 ? 1 : g)), dim3(256), 0, stream, true,
                        (const float*)p.part, p.slices, total, p.y);
  }
  if (err != cudaSuccess) {
    *why = cudaGetErrorString(err);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
