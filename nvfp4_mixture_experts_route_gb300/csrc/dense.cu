// The MoE pooler and unpooler around the expert block (the model page: the
// MoE's `pooler` ReplicatedLinear(hidden_size, moe_hidden_size, bias=False,
// quant_config=None) before the experts and `unpooler` back after them):
// plain bf16 projections y = x . w^T with fp32 accumulation and one bf16
// rounding, on the 5th-generation tensor cores (tcgen05.mma kind::f16).
//
// Tiling (swapped, as for the decode GEMMs): the MMA's M = 128 rows are output
// features (weight rows), N = a tile of tokens (32, 64, 128 or 256 by T);
// a tile is (token tile, 128-feature tile) over all of Din.
//
// Many tiles: each CTA takes whole tiles in turn. Few tiles (few tokens)
// cannot keep every SM streaming weights, so the work is split stream-K
// style: the (tile, K = 64 step) space, tile-major, is cut into one
// contiguous, equal range per CTA. A range covers the end of one tile, any
// number of whole tiles and the start of another; a whole tile is stored
// directly, a partial one as an fp32 partial in the CTA's first or last
// slot of the workspace. Per (tile, TMEM lane quadrant) a counter collects
// the partial segments' epilogue warps; the warp that completes it sums the
// tile's partials in CTA order (deterministic), rounds once to bf16, stores
// and resets the counter. No second kernel.
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
  __nv_bfloat16* y;  // [T, Dout]
  float* part;       // stream-K: [grid][2][N][128] fp32 partials
  int32_t* ctr;      // stream-K: [tiles][4] arrival counters, zero on entry
  int32_t* status;
  int T, Din, Dout, streamk;
};

// The segments one CTA works through, in order: (tile, first and one past
// the last K = 64 step of it). Whole tiles in turn (u = c, c + G, ...), or,
// stream-K, the CTA's contiguous share [c W / G, (c + 1) W / G) of the
// W = tiles * KC steps.
struct SegIter {
  long long x, end;
  int u, tiles, KC, G;
  bool streamk;
  __device__ SegIter(int c, int G_, int tiles_, int KC_, bool sk) : tiles(tiles_), KC(KC_), G(G_), streamk(sk) {
    const long long W = (long long)tiles * KC;
    u = c;
    x = sk ? (long long)c * W / G : 0;
    end = sk ? (long long)(c + 1) * W / G : 0;
  }
  __device__ bool next(int& tile, int& k0, int& k1) {
    if (!streamk) {
      if (u >= tiles) return false;
      tile = u;
      k0 = 0;
      k1 = KC;
      u += G;
      return true;
    }
    if (x >= end) return false;
    tile = (int)(x / KC);
    k0 = (int)(x - (long long)tile * KC);
    const long long e = min(end, (long long)(tile + 1) * KC);
    k1 = (int)(e - (long long)tile * KC);
    x = e;
    return true;
  }
};

// The CTA whose stream-K share holds step x: the largest c with
// floor(c W / G) <= x.
__device__ __forceinline__ int streamk_cta_of(long long x, long long W, int G) {
  return (int)(((x + 1) * G + W - 1) / W) - 1;
}

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
  const int tiles = tiles_w * tiles_t;
  const int KC = p.Din / 64;  // K = 64 stages along Din
  const bool sk = p.streamk != 0;
  const int G = gridDim.x;
  if (!sk && (int)blockIdx.x >= tiles) return;
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
      SegIter seg(blockIdx.x, G, tiles, KC, sk);
      int tile, k0, k1;
      while (!stop && seg.next(tile, k0, k1)) {
        const int tt = tile / tiles_w, mt = tile % tiles_w;
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
      SegIter seg(blockIdx.x, G, tiles, KC, sk);
      int tile, k0, k1;
      while (!stop && seg.next(tile, k0, k1)) {
        const int b = uc & 1, use = uc >> 1;
        ++uc;
        if (use > 0 && !mbar_wait(smem_u32(&acce_bar[b]), (use - 1) & 1, &abort_flag, p.status))
          break;
        tc_fence_after();
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
    const long long W = (long long)tiles * KC;
    const int first_tile = sk ? (int)((long long)blockIdx.x * W / G / KC) : 0;
    int uc = 0;
    SegIter seg(blockIdx.x, G, tiles, KC, sk);
    int tile, k0, k1;
    while (seg.next(tile, k0, k1)) {
      const int b = uc & 1, use = uc >> 1;
      ++uc;
      const bool ok = mbar_wait(smem_u32(&accf_bar[b]), use & 1, &abort_flag, p.status);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      const int tt = tile / tiles_w, mt = tile % tiles_w;
      const int r = 32 * q + lane;      // this lane's row of the feature tile
      const int o = mt * 128 + r;       // its output feature
      const int nt = min(N, p.T - tt * N);  // real tokens in the tile
      const uint32_t taddr = tmem + (uint32_t)(b * N) + ((uint32_t)(32 * q) << 16);
      const bool whole = k0 == 0 && k1 == KC;
      float* slot = p.part + ((size_t)blockIdx.x * 2 + (tile == first_tile ? 0 : 1)) * (size_t)N * 128;
      for (int c0 = 0; c0 < nt; c0 += 32) {
        float v[32];
        tmem_ld32(taddr + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int t = c0 + i;
          if (t < nt) {
            if (whole)
              p.y[(size_t)(tt * N + t) * p.Dout + o] = __float2bfloat16_rn(v[i]);
            else
              slot[(size_t)t * 128 + r] = v[i];
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acce_bar[b]));
      if (!whole) {
        // This warp's rows of the partial are stored; the warp that brings the
        // (tile, quadrant) count to the tile's segment count sums them all.
        const int c_first = streamk_cta_of((long long)tile * KC, W, G);
        const int c_last = streamk_cta_of((long long)(tile + 1) * KC - 1, W, G);
        __threadfence();
        __syncwarp();
        int old = 0;
        if (lane == 0) old = atomicAdd(p.ctr + tile * 4 + q, 1);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == c_last - c_first) {
          __threadfence();
          // CTA c's slot for this tile: its first (0) or its last (1)
          auto slot_of = [&](int c) {
            const int ft = (int)((long long)c * W / G / KC);
            return p.part + ((size_t)c * 2 + (tile == ft ? 0 : 1)) * (size_t)N * 128 + r;
          };
          for (int t0 = 0; t0 < nt; t0 += 8) {
            // sum over c = c_first, c_first + 1, ... in that order; the loads
            // of up to 8 CTAs x 8 tokens are issued before their adds
            float acc[8];
            const float* s0 = slot_of(c_first);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = t0 + i < nt ? __ldcg(s0 + (size_t)(t0 + i) * 128) : 0.0f;
            for (int c = c_first + 1; c <= c_last; c += 8) {
              float v[8][8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float* sj = slot_of(min(c + j, c_last));
#pragma unroll
                for (int i = 0; i < 8; ++i)
                  v[j][i] = c + j <= c_last && t0 + i < nt ? __ldcg(sj + (size_t)(t0 + i) * 128) : 0.0f;
              }
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (c + j <= c_last) {
#pragma unroll
                  for (int i = 0; i < 8; ++i) acc[i] += v[j][i];
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i)
              if (t0 + i < nt) p.y[(size_t)(tt * N + t0 + i) * p.Dout + o] = __float2bfloat16_rn(acc[i]);
          }
          if (lane == 0) p.ctr[tile * 4 + q] = 0;
        }
      }
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

int dense_tile_n(int T) { return T <= 32 ? 32 : T <= 64 ? 64 : T <= 128 ? 128 : 256; }

static int dense_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 148;
  return n;
}

// The launch plan: tiles, whether they are split stream-K (fewer than four
// tiles per CTA slot: whole tiles would leave CTAs idle or uneven), the grid,
// and the workspace (256-byte-aligned counters, then the partial slots).
struct DensePlan {
  int n, tiles, KC, grid;
  bool streamk;
  size_t ctr_bytes, ws_bytes;
};

static DensePlan dense_plan(int T, int Din, int Dout, int nsm) {
  DensePlan d{};
  d.n = dense_tile_n(T);
  d.tiles = ((T + d.n - 1) / d.n) * (Dout / 128);
  d.KC = Din / 64;
  const int slots = dense_ctas(d.n) * nsm;
  d.streamk = d.tiles < 4 * slots;
  const long long W = (long long)d.tiles * d.KC;
  d.grid = d.streamk ? (int)(W < slots ? W : slots) : (d.tiles < slots ? d.tiles : slots);
  if (d.streamk) {
    d.ctr_bytes = ((size_t)d.tiles * 4 * sizeof(int32_t) + 255) / 256 * 256;
    d.ws_bytes = d.ctr_bytes + (size_t)d.grid * 2 * d.n * 128 * sizeof(float);
  }
  return d;
}

size_t dense_workspace_here(int T, int Din, int Dout) {
  return T > 0 ? dense_plan(T, Din, Dout, dense_sm_count()).ws_bytes : 0;
}

template <int N>
static cudaError_t launch_dense_n(const CUtensorMap& tw, const CUtensorMap& tx, const DenseParams& p, int grid,
                                  cudaStream_t stream) {
  auto kern = dense_bf16_kernel<N>;
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), (int)dense_smem_bytes(N));
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(grid), dim3(kDThreads), dense_smem_bytes(N), stream, true, tw, tx, p);
}

int launch_dense_bf16(const void* x, const void* w, int T, int Din, int Dout, void* y, void* ws,
                      int32_t* status, cudaStream_t stream, const char** why) {
  CUtensorMap tw, tx;
  const DensePlan d = dense_plan(T, Din, Dout, dense_sm_count());
  if (encode_rows_map(&tw, w, (uint64_t)Din * 2, (uint64_t)Dout, 128) != CUDA_SUCCESS ||
      encode_rows_map(&tx, x, (uint64_t)Din * 2, (uint64_t)T, (uint32_t)d.n) != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled failed for the dense projection";
    return MOE_ERR_CUDA;
  }
  DenseParams p{};
  p.y = reinterpret_cast<__nv_bfloat16*>(y);
  p.status = status;
  p.T = T;
  p.Din = Din;
  p.Dout = Dout;
  p.streamk = d.streamk ? 1 : 0;
  cudaError_t err = cudaSuccess;
  if (d.streamk) {
    p.ctr = reinterpret_cast<int32_t*>(ws);
    p.part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(ws) + d.ctr_bytes);
    // The counters must start at zero; the kernel leaves them zero again,
    // but a caller's fresh or reused workspace is cleared here all the same.
    err = cudaMemsetAsync(ws, 0, (size_t)d.tiles * 4 * sizeof(int32_t), stream);
  }
  if (err == cudaSuccess) {
    switch (d.n) {
      case 32: err = launch_dense_n<32>(tw, tx, p, d.grid, stream); break;
      case 64: err = launch_dense_n<64>(tw, tx, p, d.grid, stream); break;
      case 128: err = launch_dense_n<128>(tw, tx, p, d.grid, stream); break;
      default: err = launch_dense_n<256>(tw, tx, p, d.grid, stream); break;
    }
  }
  if (err != cudaSuccess) {
    *why = cudaGetErrorString(err);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
