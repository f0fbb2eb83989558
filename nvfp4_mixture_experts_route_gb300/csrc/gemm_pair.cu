// Steps a3-a5 at prefill sizes in the pair form: GEMM1 + SwiGLU + NVFP4
// requantization of the intermediate (the same arithmetic as the
// grouped_gemm_kernel's GEMM1 epilogue) for 128-row route tiles, with
// tcgen05.mma.cta_group::2 over clusters of two CTAs on two SMs.
//
// Work unit: a pair of consecutive route tiles of one expert (the second
// absent when the expert has an odd number of tiles) against 256 prepared
// w13 rows (16 gate/up granules: 128 intermediate columns). One MMA of
// M = 256 (rank r's 128 route rows as A rows 128 r .. 128 r + 127) by
// N = 256 (rank r's smem holds weight rows 128 r .. 128 r + 127) by K = 64;
// each CTA's tensor memory holds its 128 rows x 256 columns of the
// accumulator. Per K = 64 step: one MMA and three scale-atom copies (the
// route tile's atom and both 128-row weight atoms, into both CTAs' tensor
// memory), so one instruction stream feeds two SMs with twice the rows per
// instruction of the single-CTA kernel.
//
// Per CTA: warp 0 lane 0 loads the CTA's half of every stage (its route
// box and route scale atoms, its 128 weight rows, both weight scale halves)
// by TMA tensor loads whose bytes all complete on rank 0's full barrier of
// the stage (rank 1's in the pair form of the load), so rank 0 sees a stage
// complete only when both halves have landed; warp 1 of rank 0 issues
// (converged, lane 0 under a predicate); warps 2..9 are the epilogue of the
// CTA's own accumulator rows. Rank 0's commits arrive on both CTAs' barriers:
// the stage's empty barrier (each producer refills its own half) and, after a
// unit, the accumulator-full barrier. Both CTAs' epilogue warps hand the
// accumulator back on rank 0's acce barrier. A ring of kStages stages;
// tensor memory: 256 accumulator columns plus 48 scale columns per stage.
// Every wait is bounded (1 s, MOE_ERR_TIMEOUT); a cluster barrier precedes
// the teardown so that neither CTA frees what the other may still touch.
#include "common.cuh"
#include "layout.cuh"

namespace moe {

namespace gpair {
constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr int kStages = 5;
constexpr uint32_t kBox = 128 * 128;                     // 128 rows x 128 bytes (K = 256)
constexpr uint32_t kSfa = 4 * kAtomBytes;                // a route tile's 4 atoms of a stage
constexpr uint32_t kSfb = 8 * kAtomBytes;                // both weight halves' 4 atoms
constexpr int kMaxPairs = 1024;                          // route tiles a launch may hold
constexpr uint32_t kSmem = 1024 + kStages * (2 * kBox + kSfa + kSfb) + kMaxPairs * 8;  // + pair list and experts
constexpr uint32_t kTmemCols = 512;
static_assert(256 + kStages * 48 <= (int)kTmemCols, "pair GEMM1 tensor memory");
static_assert(kSmem <= 232448, "pair GEMM1 shared memory");
}  // namespace gpair

struct PairGemmParams {
  const uint8_t* w_sf;   // prepared weight scale atoms [E][rows_w/128][K/64][512]
  const uint8_t* a_sf;   // route operand scale atoms [tiles][K/64][512]
  const float* s0;       // g1_alphas
  const float* s1;       // g1_scale_c
  const float* a2_gscale;
  const int32_t* tile_expert;
  const int32_t* tile_row_limit;
  const int32_t* totals;
  uint8_t* hq;           // intermediate codes [P][I/2]
  uint8_t* hq_sf;        // intermediate scale atoms [tiles][I/64][512]
  int32_t* status;
  int K, rows_w, I, max_tiles, num_experts;  // contraction length, weight rows per expert
};

// The pair-start route tiles (the first tile of each expert's consecutive
// pairs) in ascending order, by one warp: a tile starts a pair when its
// distance from the first tile of its expert's run is even. starts[i] is the
// tile, with kHasPeer set when the next tile belongs to the same expert;
// experts[i] its expert. Every lane loads its tiles' experts first
// (kMaxPairs / 32 of them at most), so that the scan waits for one round of
// loads, not one per 32 tiles, and the units read only shared memory after.
constexpr int kHasPeer = 1 << 30;
__device__ __forceinline__ int build_pair_starts(const int32_t* tile_expert, int ntiles, int* starts, int* experts,
                                                 int lane) {
  constexpr int kPer = gpair::kMaxPairs / 32;
  int ex[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int t = 32 * i + lane;
    ex[i] = t < ntiles ? __ldcg(tile_expert + t) : -2;
  }
  int count = 0, carry_start = 0, prev_e = -1;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int base = 32 * i;
    if (base >= ntiles) break;
    const int t = base + lane;
    const bool valid = t < ntiles;
    const int e = ex[i];
    int e_prev = __shfl_up_sync(0xFFFFFFFFu, e, 1);
    if (lane == 0) e_prev = prev_e;
    const bool run_start = valid && (t == 0 || e != e_prev);
    const uint32_t rs = __ballot_sync(0xFFFFFFFFu, run_start);
    const uint32_t upto = lane == 31 ? rs : (rs & ((2u << lane) - 1u));
    const int start = upto ? base + (31 - __clz(upto)) : carry_start;
    const bool ps = valid && ((t - start) & 1) == 0;
    // the expert of tile t + 1 (lane 31: the first tile of the next 32)
    int e_next = __shfl_down_sync(0xFFFFFFFFu, e, 1);
    const int e_wrap = __shfl_sync(0xFFFFFFFFu, i + 1 < kPer ? ex[i + 1 < kPer ? i + 1 : i] : -2, 0);
    if (lane == 31) e_next = e_wrap;
    const bool peer = t + 1 < ntiles && e_next == e;
    const uint32_t pm = __ballot_sync(0xFFFFFFFFu, ps);
    const int at = count + __popc(pm & ((1u << lane) - 1u));
    if (ps) {
      starts[at] = t | (peer ? kHasPeer : 0);
      experts[at] = e;
    }
    count += __popc(pm);
    carry_start = __shfl_sync(0xFFFFFFFFu, start, 31);
    prev_e = __shfl_sync(0xFFFFFFFFu, e, 31);
  }
  return count;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(gpair::kThreads, 1)
    gemm1_pair_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmWsf, const __grid_constant__ CUtensorMap tmAsf,
                     const PairGemmParams p) {
  using namespace gpair;
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kStages];   // rank 0: both CTAs' halves of the stage landed
  __shared__ __align__(8) uint64_t empty_bar[kStages];  // the stage's MMAs completed (rank 0's commit)
  __shared__ __align__(8) uint64_t accf_bar;            // the unit's accumulator is complete
  __shared__ __align__(8) uint64_t acce_bar;            // rank 0: both CTAs' epilogues read it out
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag, npairs_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sW = sbase;                    // weight boxes
  const uint32_t sA = sW + kStages * kBox;      // route boxes
  const uint32_t sSFA = sA + kStages * kBox;    // route scale atoms
  const uint32_t sSFB = sSFA + kStages * kSfa;  // weight scale atoms (both halves)
  int* starts = reinterpret_cast<int*>(dsmem + (sSFB + kStages * kSfb - smem_u32(dsmem)));
  int* experts = starts + kMaxPairs;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&accf_bar), 1);
    mbar_init(smem_u32(&acce_bar), 2 * kEpiWarps);
    mbar_init(smem_u32(&drain_bar), 1);
    abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmWsf);
    tma_prefetch_desc(&tmAsf);
  }
  pdl_wait();
  const int ntiles = min(max(__ldcg(p.totals), 0), p.max_tiles);
  if (warp == 2) {
    const int n = build_pair_starts(p.tile_expert, ntiles, starts, experts, lane);
    if (lane == 0) npairs_s = n;
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&tmem_slot), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers are initialised before any remote arrive or commit
  tc_fence_after();
  if (tid == 0) pdl_trigger();
  const uint32_t tmem = tmem_slot;
  const int npairs = npairs_s;
  const int KC = p.K / 64, nks = p.K / 256;
  const int tw = p.rows_w / 256;  // units per pair (256 weight rows each)
  const int n_units = npairs * tw;
  const int cl = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  // unit u: pair u / tw (weight tile fastest, so that the clusters working
  // at the same time share the route pair in L2), weight rows 256 (u % tw)
  // An expert id outside [0, E) (a corrupt routing table) reads as expert 0
  // for the loads, so that every address stays in range and every role
  // still walks the same stages, and the unit's results are not stored.
  auto unit_tiles = [&](int u, int& w, int& e, int& mine, int& peer, bool& bad) {
    const int pi = u / tw;
    w = u - pi * tw;
    const int v = starts[pi];
    const int t0 = v & (kHasPeer - 1);
    peer = (v & kHasPeer) ? t0 + 1 : -1;  // rank 1's tile
    e = experts[pi];
    mine = rank == 0 ? t0 : peer;
    bad = e < 0 || e >= p.num_experts;
    if (bad) e = 0;
  };
  const uint32_t t_sfa = tmem + 256;
  const uint32_t t_sfb = t_sfa + kStages * 16;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      int it = 0;
      bool stop = false;
      const int wrows_per_e = p.rows_w / 128;  // 128-row weight tiles per expert
      for (int u = cl; u < n_units && !stop; u += ncl) {
        int w, e, mine, peer;
        bool bad;
        unit_tiles(u, w, e, mine, peer, bad);
        if (bad && rank == 0) record_status(p.status, MOE_ERR_INVALID_ROUTE);
        // rank 0 expects both halves' bytes; rank 1's route half is absent
        // when its tile is (an odd last tile of the expert)
        const int wrow = e * p.rows_w + 256 * w + 128 * (int)rank;
        // atom rows (128 bytes, 4 per atom) of the two weight halves and of the route tile, at K step 0
        const int wsf_row0 = ((e * wrows_per_e + 2 * w) * KC) * 4, wsf_row1 = wsf_row0 + KC * 4;
        const int asf_row = mine >= 0 ? mine * KC * 4 : 0;
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int s = it % kStages, round = it / kStages;
          if (round > 0 && !mbar_wait(smem_u32(&empty_bar[s]), (round - 1) & 1, &abort_flag, p.status)) {
            stop = true;
            break;
          }
          const uint32_t fb = smem_u32(&full_bar[s]);
          if (rank == 0) {
            const uint32_t half0 = kBox + kSfb + (mine >= 0 ? kBox + kSfa : 0u);
            const uint32_t half1 = kBox + kSfb + (peer >= 0 ? kBox + kSfa : 0u);
            mbar_arrive_expect_tx(fb, half0 + half1);
            tma_load_2d(sW + s * kBox, &tmW, fb, ks * 128, wrow);
            tma_load_2d(sSFB + s * kSfb, &tmWsf, fb, 0, wsf_row0 + 16 * ks);
            tma_load_2d(sSFB + s * kSfb + kSfa, &tmWsf, fb, 0, wsf_row1 + 16 * ks);
            if (mine >= 0) {
              tma_load_2d(sA + s * kBox, &tmA, fb, ks * 128, mine * 128);
              tma_load_2d(sSFA + s * kSfa, &tmAsf, fb, 0, asf_row + 16 * ks);
            }
          } else {
            const uint32_t fb0 = cluster_map(fb, 0);  // rank 0's full barrier of the stage
            tma_load_2d_pair(sW + s * kBox, &tmW, fb0, ks * 128, wrow);
            tma_load_2d_pair(sSFB + s * kSfb, &tmWsf, fb0, 0, wsf_row0 + 16 * ks);
            tma_load_2d_pair(sSFB + s * kSfb + kSfa, &tmWsf, fb0, 0, wsf_row1 + 16 * ks);
            if (mine >= 0) {
              tma_load_2d_pair(sA + s * kBox, &tmA, fb0, ks * 128, mine * 128);
              tma_load_2d_pair(sSFA + s * kSfa, &tmAsf, fb0, 0, asf_row + 16 * ks);
            }
          }
        }
      }
      // rank 0: the copies still in flight (both halves complete on its
      // barriers) land before either CTA passes the teardown's cluster barrier
      if (rank == 0)
        for (int j = max(0, it - kStages); j < it; ++j)
          mbar_wait_cleanup(smem_u32(&full_bar[j % kStages]), (j / kStages) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // --------------------------- MMA issuer (rank 0) ---------------------------
    // (rank 1's warp 1 has nothing to do: rank 0 issues for both CTAs)
    if (rank == 0) {
      constexpr uint32_t idesc = idesc_nvf4(256, 256);
      const uint64_t w_desc0 = smem_desc(sW, 16, 1024, 2), a_desc0 = smem_desc(sA, 16, 1024, 2);
      const uint64_t sfa_desc0 = smem_desc(sSFA, 0, 128, 0), sfb_desc0 = smem_desc(sSFB, 0, 128, 0);
      int it = 0, uc = 0;
      bool stop = false;
      for (int u = cl; u < n_units && !stop; u += ncl, ++uc) {
        if (uc > 0) {
          const bool ok = mbar_wait_cluster(smem_u32(&acce_bar), (uc - 1) & 1, &abort_flag, p.status);
          if (!__all_sync(0xFFFFFFFFu, ok)) break;
        }
        tc_fence_after();
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          const bool ok = mbar_wait(smem_u32(&full_bar[s]), ph, &abort_flag, p.status);
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t fa = t_sfa + s * 16, fbc = t_sfb + s * 32;
          const uint64_t sad = sfa_desc0 + ((s * kSfa) >> 4), sbd = sfb_desc0 + ((s * kSfb) >> 4);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            pair_copy_atom(fa + 4 * j, sad + j * (kAtomBytes >> 4));
            pair_copy_atom(fbc + 8 * j, sbd + j * (kAtomBytes >> 4));
            pair_copy_atom(fbc + 8 * j + 4, sbd + (4 + j) * (kAtomBytes >> 4));
          }
          const uint64_t ad = a_desc0 + ((s * kBox) >> 4), wd = w_desc0 + ((s * kBox) >> 4);
#pragma unroll
          for (int j = 0; j < 4; ++j)  // A = route rows, B = weight rows; 32 bytes (K = 64) per step
            pair_mma(tmem, ad + ((32 * j) >> 4), wd + ((32 * j) >> 4), idesc, fa + 4 * j, fbc + 8 * j,
                     (ks | j) != 0);
          pair_commit_both(smem_u32(&empty_bar[s]));
        }
        if (stop) break;
        pair_commit_both(smem_u32(&accf_bar));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue ------------------------------
    // Warp w reads TMEM lane quadrant w % 4 (32 route rows) and columns
    // 128 h .. 128 h + 127 (h = which of the quadrant's two warps): granules
    // 4 h .. 4 h + 3 of the unit, i.e. intermediate columns
    // 128 w + 64 h .. + 63 of its rows.
    const int q = warp & 3, h = (warp - 2) >> 2;
    const float a2g = *p.a2_gscale;
    int uc = 0;
    for (int u = cl; u < n_units; u += ncl, ++uc) {
      const bool ok = mbar_wait_warp(smem_u32(&accf_bar), uc & 1, &abort_flag, p.status);
      if (!ok) break;
      tc_fence_after();
      int w, e, mine, peer;
      bool bad;
      unit_tiles(u, w, e, mine, peer, bad);
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16) + 128 * h;
      uint32_t acc[4][32];
#pragma unroll
      for (int k = 0; k < 4; ++k) tmem_ld32_async(taddr + 32 * k, acc[k]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(smem_u32(&acce_bar));
        else  // the accumulator's columns are in registers (tcgen05.wait::ld above)
          mbar_arrive_cluster_relaxed(smem_u32(&acce_bar), 0);
      }
      if (mine >= 0 && !bad) {
        const float s0 = p.s0[e], s1 = p.s1[e];
        const int r = mine * 128 + 32 * q + lane;  // permuted route row
        uint32_t cw[8], sf4 = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float hv[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g = s0 * __uint_as_float(acc[k][i]);
            const float up = s1 * __uint_as_float(acc[k][16 + i]);
            hv[i] = __fdividef(g, 1.0f + __expf(-g)) * up;  // SiLU(gate) * up
          }
          uint2 codes;
          uint32_t sfc;
          quant16(hv, a2g, codes, sfc);
          cw[2 * k] = codes.x;
          cw[2 * k + 1] = codes.y;
          sf4 |= sfc << (8 * k);
        }
        uint4* dst = reinterpret_cast<uint4*>(p.hq + (size_t)r * (p.I / 2) + 64 * w + 32 * h);
        dst[0] = make_uint4(cw[0], cw[1], cw[2], cw[3]);
        dst[1] = make_uint4(cw[4], cw[5], cw[6], cw[7]);
        // blocks 8 w + 4 h .. + 3: one aligned 4-byte group of the row's atom
        *reinterpret_cast<uint32_t*>(p.hq_sf + act_sf_offset(r, 8 * w + 4 * h, 128, p.I / 64, 1)) = sf4;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (rank == 0 && warp == 1) {
    // one more commit tracks every tcgen05 op issued (on a timeout too)
    pair_commit(smem_u32(&drain_bar));
    if (lane == 0) mbar_wait_cleanup(smem_u32(&drain_bar), 0);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // rank 0's MMAs are done with rank 1's memory; no remote arrive is pending
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

static int even_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 2)
    n = 148;
  return n & ~1;
}

// Whether the pair form takes a GEMM1 of this shape: 128-row route tiles,
// K (= H) and the weight rows per expert (2I) multiples of 256.
bool gemm_pair_fits(int tile_m, int K, int rows_w, int max_tiles) {
  return tile_m == 128 && K % 256 == 0 && rows_w % 256 == 0 && max_tiles <= gpair::kMaxPairs && max_tiles > 0;
}

static cudaError_t launch_gemm_pair(const CUtensorMap& tmW, const CUtensorMap& tmA, PairGemmParams& p, int E,
                                    cudaStream_t stream, bool pdl) {
  CUtensorMap tmWsf, tmAsf;
  const uint64_t kc_bytes = (uint64_t)(p.K / 64) * kAtomBytes;
  p.num_experts = E;
  if (encode_atoms_map(&tmWsf, p.w_sf, (uint64_t)E * (p.rows_w / 128) * kc_bytes, 16) != CUDA_SUCCESS ||
      encode_atoms_map(&tmAsf, p.a_sf, (uint64_t)p.max_tiles * kc_bytes, 16) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  auto kern = gemm1_pair_kernel;
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), (int)gpair::kSmem);
  if (err != cudaSuccess) return err;
  return launch_kernel(kern, dim3(even_sm_count()), dim3(gpair::kThreads), gpair::kSmem, stream, pdl, tmW, tmA,
                       tmWsf, tmAsf, p);
}


cudaError_t launch_gemm1_pair(const CUtensorMap& tmW, const CUtensorMap& tmA, const uint8_t* w_sf,
                              const uint8_t* a_sf, const float* g1_alphas, const float* g1_scale_c,
                              const float* a2_gscale, const int32_t* tile_expert, const int32_t* tile_row_limit,
                              const int32_t* totals, uint8_t* hq, uint8_t* hq_sf, int E, int H, int I,
                              int max_tiles, int32_t* status, cudaStream_t stream, bool pdl) {
  PairGemmParams p{};
  p.w_sf = w_sf;
  p.a_sf = a_sf;
  p.s0 = g1_alphas;
  p.s1 = g1_scale_c;
  p.a2_gscale = a2_gscale;
  p.tile_expert = tile_expert;
  p.tile_row_limit = tile_row_limit;
  p.totals = totals;
  p.hq = hq;
  p.hq_sf = hq_sf;
  p.status = status;
  p.K = H;
  p.rows_w = 2 * I;
  p.I = I;
  p.max_tiles = max_tiles;
  return launch_gemm_pair(tmW, tmA, p, E, stream, pdl);
}

}  // namespace moe
