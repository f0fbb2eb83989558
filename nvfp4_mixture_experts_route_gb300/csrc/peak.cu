// moe_fp4_mma_rate: the dense NVFP4 tensor-core rate of this GPU, measured
// with the same instruction the expert GEMMs issue
// (tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X, M = 128,
// K = 64 per instruction, fp32 accumulation in tensor memory).
//
// Operands stay in shared memory (no global loads), so the launch measures
// the tensor pipe and the issuing thread, not memory: a dense GEMM of
// M = 128 * CTAs, N, K = 64 * MMAs per CTA whose operand tiles are reused.
// One thread per CTA issues everything, in K = 256 stages as the expert GEMMs
// do: optionally the stage's scale-factor copies into tensor memory
// (tcgen05.cp 32x128b.warpx4, one per 128 rows of each operand per K = 64
// step), then the stage's MMAs, then one tcgen05.commit to the stage's
// mbarrier; a stage's tensor-memory scale columns are rewritten only after
// the commit of their previous use has arrived (a ring of stages). Variants
// separate the cost of the MMAs, of the scale copies and of the commits, and
// of the issue form: lane 0 alone running the issue loops, or the whole warp
// running them converged with lane 0 issuing under a predicate.
//
// Every wait is bounded (1 s) and reports MOE_ERR_TIMEOUT; no trap.
#include "common.cuh"
#include "layout.cuh"

namespace moe {

// Tensor-memory columns: the accumulator (N) plus scale columns -- per stage
// of MPC MMAs, 4 columns for A's atom and 4 per 128 rows of B -- for every
// ring stage when copied per stage, or for one K = 256 stage loaded once.
__host__ __device__ constexpr int rate_sf_cols(int n, int sfcp, int mpc, int ring) {
  return (sfcp ? ring * mpc : 4) * 4 * (1 + n / 128);
}
__host__ __device__ constexpr uint32_t rate_tmem_cols(int n, int sfcp, int mpc, int ring) {
  uint32_t c = 32;
  while ((int)c < n + rate_sf_cols(n, sfcp, mpc, ring)) c <<= 1;
  return c;
}

// One tcgen05.cp of a 128-row x 32-byte shared-memory matrix into 128 lanes
// x 8 columns (no replication): the cost of a wider copy, timed against the
// 512-byte 32x128b.warpx4 atoms. WI: issued by lane 0 of a converged warp.
template <bool WI>
__device__ __forceinline__ void tc_copy_128x256b_f(uint32_t taddr, uint64_t desc) {
  if constexpr (WI)
    asm volatile(
        "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
        "@e tcgen05.cp.cta_group::1.128x256b [%0], %1;\n\t}" ::"r"(taddr),
        "l"(desc)
        : "memory");
  else
    asm volatile("tcgen05.cp.cta_group::1.128x256b [%0], %1;" ::"r"(taddr), "l"(desc) : "memory");
}
// Shared memory: one 128-byte-swizzled K = 256 chunk of A (128 rows) and of
// B (N rows), and four K = 64 steps of scale atoms for each.
__host__ __device__ constexpr uint32_t rate_smem_bytes(int n) {
  return 1024 + 128 * 128 + (uint32_t)n * 128 + 4 * kAtomBytes * (1 + n / 128);
}

// SFCP: 0 scales copied once; 1 copied every stage by the MMA thread; 2 by
// a second warp's lane 0, which commits each stage's copies to a barrier the
// MMA thread waits on (the expert GEMM1's scale-copy warp); 3 by two more
// warps, one for A's atoms and one for B's; 4 every stage by the MMA thread
// with 128x256b copies (two K = 64 steps each) for both operands; 5 the same
// for A only. Modes 4 and 5 time the copies only: the scale values are all
// the same, so the columns' layout does not matter to the MMAs here.
__host__ __device__ constexpr int rate_threads(int sfcp) { return sfcp == 2 ? 64 : sfcp == 3 ? 96 : 32; }

template <int N, int SFCP, int MPC, int RING, bool WI>
__global__ void __launch_bounds__(rate_threads(SFCP)) fp4_mma_rate_kernel(int stages, int32_t* status) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t bar[RING];
  __shared__ __align__(8) uint64_t sfa_ready[RING];
  __shared__ __align__(8) uint64_t sfb_ready[RING];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t cp_drain[2];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  constexpr int S = N / 128;  // scale atoms of B per K = 64 step
  constexpr int SL = SFCP ? MPC : 4;  // K = 64 steps whose scales a column slot holds
  constexpr uint32_t ncols = rate_tmem_cols(N, SFCP, MPC, RING);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t sA = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sB = sA + 128 * 128;
  const uint32_t sSFA = sB + N * 128;
  const uint32_t sSFB = sSFA + 4 * kAtomBytes;
  uint8_t* base = dsmem + (sA - smem_u32(dsmem));

  // Operand bytes: any e2m1 codes do (every code is finite); scales 0x38 =
  // 1.0 in e4m3. Written through the generic proxy, read by the tensor core.
  const uint32_t op_bytes = 128 * 128 + N * 128;
  if (warp == 0) {
    for (uint32_t i = lane * 4; i < op_bytes; i += 128)
      *reinterpret_cast<uint32_t*>(base + i) = (i * 2654435761u) ^ 0x5A3C9617u;
    for (uint32_t i = op_bytes + lane * 4; i < op_bytes + 4 * kAtomBytes * (1 + S); i += 128)
      *reinterpret_cast<uint32_t*>(base + i) = 0x38383838u;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) {
      for (int r = 0; r < RING; ++r) {
        mbar_init(smem_u32(&bar[r]), 1);
        mbar_init(smem_u32(&sfa_ready[r]), 1);
        mbar_init(smem_u32(&sfb_ready[r]), 1);
      }
      mbar_init(smem_u32(&drain_bar), 1);
      mbar_init(smem_u32(&cp_drain[0]), 1);
      mbar_init(smem_u32(&cp_drain[1]), 1);
      abort_flag = 0;
      fence_barrier_init();
    }
    __syncwarp();
    tmem_alloc(smem_u32(&tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t t_sf = tmem + N;

  if (WI || lane == 0) {
    constexpr uint32_t idesc = idesc_nvf4(128, N);
    const uint64_t a_desc = smem_desc(sA, 16, 1024, 2), b_desc = smem_desc(sB, 16, 1024, 2);
    const uint64_t sfa_desc = smem_desc(sSFA, 0, 128, 0), sfb_desc = smem_desc(sSFB, 0, 128, 0);
    // scale columns of step j (of ring stage r when copied per stage): A's
    // atoms of the slot's SL steps, then B's S atoms per step
    auto sfa_col = [&](int r, int j) { return t_sf + (uint32_t)(r * SL * 4 * (1 + S) + 4 * j); };
    auto sfb_col = [&](int r, int j) { return t_sf + (uint32_t)(r * SL * 4 * (1 + S) + 4 * SL + 4 * j * S); };
    auto copy_a = [&](int r, int j) {
      tc_copy_scale_atom_f<WI>(sfa_col(r, j), sfa_desc + (uint64_t)((j & 3) * (kAtomBytes >> 4)));
    };
    auto copy_b = [&](int r, int j) {
#pragma unroll
      for (int sub = 0; sub < S; ++sub)
        tc_copy_scale_atom_f<WI>(sfb_col(r, j) + 4 * sub, sfb_desc + (uint64_t)(((j & 3) * S + sub) * (kAtomBytes >> 4)));
    };
    auto copy_scales = [&](int r, int j) {
      if (SFCP >= 4) {
        // 128 rows x 32 bytes from the scale region (4 KB inside the
        // operand buffer) into the 8 columns of steps j and j + 1
        if ((j & 1) == 0) {
          tc_copy_128x256b_f<WI>(sfa_col(r, j), smem_desc(sSFA, 128, 256, 0));
          if (SFCP == 4) {
#pragma unroll
            for (int sub = 0; sub < S; ++sub) tc_copy_128x256b_f<WI>(sfb_col(r, j) + 8 * sub, smem_desc(sSFA, 128, 256, 0));
          }
        }
        if (SFCP == 5) copy_b(r, j);
        return;
      }
      copy_a(r, j);
      copy_b(r, j);
    };
    if (warp > 0) {
      // copy warp(s): stage s's columns are free once the MMAs of stage
      // s - ring (same slot) have completed
      bool do_a = SFCP == 2 || warp == 1, do_b = SFCP == 2 || warp == 2;
      for (int s = 0; s < stages; ++s) {
        const int r = s % RING;
        if (s >= RING && !mbar_wait_f<WI>(smem_u32(&bar[r]), ((s / RING) - 1) & 1, &abort_flag, status))
          break;
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < MPC; ++j) {
          if (do_a) copy_a(r, j);
          if (do_b) copy_b(r, j);
        }
        tc_commit_f<WI>(smem_u32(warp == 2 ? &sfb_ready[r] : &sfa_ready[r]));
      }
      tc_commit_f<WI>(smem_u32(&cp_drain[warp - 1]));
      mbar_wait_cleanup(smem_u32(&cp_drain[warp - 1]), 0);
    } else {
    if (!SFCP) {
#pragma unroll
      for (int j = 0; j < 4; ++j) copy_scales(0, j);  // once; ordered before the MMAs that read them
    }
    for (int s = 0; s < stages; ++s) {
      const int r = s % RING;
      const bool copy_warps = SFCP == 2 || SFCP == 3;
      if (!copy_warps && s >= RING && !mbar_wait_f<WI>(smem_u32(&bar[r]), ((s / RING) - 1) & 1, &abort_flag, status))
        break;
      if (copy_warps && !mbar_wait_f<WI>(smem_u32(&sfa_ready[r]), (s / RING) & 1, &abort_flag, status)) break;
      if (SFCP == 3 && !mbar_wait_f<WI>(smem_u32(&sfb_ready[r]), (s / RING) & 1, &abort_flag, status)) break;
      tc_fence_after();
      if (SFCP == 1 || SFCP >= 4) {
#pragma unroll
        for (int j = 0; j < MPC; ++j) copy_scales(r, j);
      }
#pragma unroll
      for (int j = 0; j < MPC; ++j) {
        const uint64_t koff = (uint64_t)((32 * (j & 3)) >> 4);
        const int rs = SFCP ? r : 0, js = SFCP ? j : (j & 3);
        tc_mma_nvf4_f<WI>(tmem, a_desc + koff, b_desc + koff, idesc, sfa_col(rs, js), sfb_col(rs, js),
                    (s | j) != 0);
      }
      tc_commit_f<WI>(smem_u32(&bar[r]));
    }
    tc_commit_f<WI>(smem_u32(&drain_bar));
    mbar_wait_cleanup(smem_u32(&drain_bar), 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, ncols);
}

template <int N, int SFCP, int MPC, int RING, bool WI>
static cudaError_t launch_rate(int grid, int smem, int stages, int32_t* status, cudaStream_t stream) {
  auto kern = fp4_mma_rate_kernel<N, SFCP, MPC, RING, WI>;
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), smem);
  if (err != cudaSuccess) return err;
  kern<<<grid, rate_threads(SFCP), smem, stream>>>(stages, status);
  return cudaGetLastError();
}

// Host check of a variant: MOE_OK, or an error code with the reason.
int fp4_mma_rate_check(int n, int sf_copies, int mpc, int ctas_per_sm, int ring, int warp_issue, int stages,
                       const char** why) {
  if (!((n == 128 || n == 256) && sf_copies >= 0 && sf_copies <= 5 && (mpc == 4 || mpc == 16) &&
        (ctas_per_sm == 1 || ctas_per_sm == 2) && (ring == 3 || ring == 5) && (warp_issue == 0 || warp_issue == 1) &&
        stages >= 1 && stages <= (1 << 24))) {
    *why = "fp4 rate: n in {128, 256}, sf_copies in 0..5, mmas_per_commit in {4, 16}, ctas_per_sm in {1, 2}, "
           "ring in {3, 5}, warp_issue in {0, 1}";
    return MOE_ERR_INVALID_ARG;
  }
  if ((n == 256 && ctas_per_sm == 2) || (sf_copies && mpc == 16) || (ring == 5 && (ctas_per_sm == 2 || !sf_copies))) {
    *why = "fp4 rate: that variant does not fit tensor memory";
    return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

// n: MMA N (128 or 256); sf_copies: scale copies once (0), every stage by
// the MMA thread (1), by one copy warp (2) or by two (3);
// mpc: MMAs per commit (4: a K = 256 stage; 16: a K = 1024 stage, only
// without per-stage copies); ctas_per_sm: 1 or 2 (2 only for n = 128, whose
// tensor memory then fits two CTAs); warp_issue: 0 lane 0 alone runs the
// issue loops, 1 the whole warp runs them converged, lane 0 issuing.
int launch_fp4_mma_rate(int n, int sf_copies, int mpc, int ctas_per_sm, int ring, int warp_issue, int stages,
                        int sms, int32_t* status, cudaStream_t stream, double* flops, const char** why) {
  const int rc = fp4_mma_rate_check(n, sf_copies, mpc, ctas_per_sm, ring, warp_issue, stages, why);
  if (rc) return rc;
  // Shared memory requested per CTA so that exactly ctas_per_sm fit an SM:
  // their tensor memory (at most 512 / ctas_per_sm columns each) then never
  // waits for another CTA's.
  const int smem = ctas_per_sm == 1 ? 160 * 1024 : 96 * 1024;
  const int grid = sms * ctas_per_sm;
  *flops = 2.0 * 128.0 * n * 64.0 * (double)mpc * (double)stages * (double)grid;
  cudaError_t err;
  const int key =
      (warp_issue ? 10000 : 0) + (n == 256 ? 1000 : 0) + (ring == 5 ? 100 : 0) + 10 * sf_copies + (mpc == 16 ? 1 : 0);
  switch (key) {
#define MOE_RATE1(k, nn, cp, mpcv, rg, wi) \
  case k: err = launch_rate<nn, cp, mpcv, rg, wi>(grid, smem, stages, status, stream); break;
#define MOE_RATE(k, nn, cp, mpcv, rg) MOE_RATE1(k, nn, cp, mpcv, rg, false) MOE_RATE1(10000 + k, nn, cp, mpcv, rg, true)
    MOE_RATE(0, 128, 0, 4, 3)
    MOE_RATE(1, 128, 0, 16, 3)
    MOE_RATE(10, 128, 1, 4, 3)
    MOE_RATE(20, 128, 2, 4, 3)
    MOE_RATE(30, 128, 3, 4, 3)
    MOE_RATE(40, 128, 4, 4, 3)
    MOE_RATE(50, 128, 5, 4, 3)
    MOE_RATE(110, 128, 1, 4, 5)
    MOE_RATE(120, 128, 2, 4, 5)
    MOE_RATE(130, 128, 3, 4, 5)
    MOE_RATE(1000, 256, 0, 4, 3)
    MOE_RATE(1001, 256, 0, 16, 3)
    MOE_RATE(1010, 256, 1, 4, 3)
    MOE_RATE(1020, 256, 2, 4, 3)
    MOE_RATE(1030, 256, 3, 4, 3)
    MOE_RATE(1040, 256, 4, 4, 3)
    MOE_RATE(1050, 256, 5, 4, 3)
    MOE_RATE(1110, 256, 1, 4, 5)
    MOE_RATE(1120, 256, 2, 4, 5)
    MOE_RATE(1130, 256, 3, 4, 5)
    MOE_RATE(1140, 256, 4, 4, 5)
    MOE_RATE(1150, 256, 5, 4, 5)
#undef MOE_RATE
#undef MOE_RATE1
    default:
      *why = "fp4 rate: variant not built";
      return MOE_ERR_UNSUPPORTED;
  }
  if (err != cudaSuccess) {
    *why = cudaGetErrorString(err);
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}


// The pair form (cta_group::2) of the same MMA stream: clusters of two CTAs,
// one CTA per SM. Both CTAs fill their operand tiles and allocate tensor
// memory together (the pair allocation is collective); rank 0 alone issues,
// as a converged warp with lane 0 issuing: M = 256 MMAs whose A rows 0-127
// come from its own shared memory and 128-255 from its peer's (the same
// offsets), each scale-atom copy into both CTAs' tensor memory, and the
// commits to its own ring barriers. A cluster barrier before the teardown
// keeps the peer's shared and tensor memory until rank 0's MMAs have landed.
// FLOPs per pair MMA: 2 * 256 * N * 64.
template <int N, int SFCP>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(32, 1) fp4_mma_pair_kernel(int stages, int32_t* status) {
  constexpr int RING = 3, MPC = 4;
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t bar[RING];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  constexpr int S = N / 128;
  constexpr int SL = SFCP ? MPC : 4;
  constexpr uint32_t ncols = rate_tmem_cols(N, SFCP, MPC, RING);
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const uint32_t sA = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sB = sA + 128 * 128;
  const uint32_t sSFA = sB + N * 128;
  const uint32_t sSFB = sSFA + 4 * kAtomBytes;
  uint8_t* base = dsmem + (sA - smem_u32(dsmem));
  const uint32_t op_bytes = 128 * 128 + N * 128;
  for (uint32_t i = lane * 4; i < op_bytes; i += 128)
    *reinterpret_cast<uint32_t*>(base + i) = (i * 2654435761u) ^ 0x5A3C9617u ^ rank;
  for (uint32_t i = op_bytes + lane * 4; i < op_bytes + 4 * kAtomBytes * (1 + S); i += 128)
    *reinterpret_cast<uint32_t*>(base + i) = 0x38383838u;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (lane == 0) {
    for (int r = 0; r < RING; ++r) mbar_init(smem_u32(&bar[r]), 1);
    mbar_init(smem_u32(&drain_bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncwarp();
  cluster_sync_all();  // both CTAs' operands and barriers are ready
  tmem_alloc_pair(smem_u32(&tmem_slot), ncols);
  tmem_relinquish_pair();
  tc_fence_before();
  __syncwarp();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t t_sf = tmem + N;
  if (rank == 0) {
    constexpr uint32_t idesc = idesc_nvf4(256, N);
    const uint64_t a_desc = smem_desc(sA, 16, 1024, 2), b_desc = smem_desc(sB, 16, 1024, 2);
    const uint64_t sfa_desc = smem_desc(sSFA, 0, 128, 0), sfb_desc = smem_desc(sSFB, 0, 128, 0);
    auto sfa_col = [&](int r, int j) { return t_sf + (uint32_t)(r * SL * 4 * (1 + S) + 4 * j); };
    auto sfb_col = [&](int r, int j) { return t_sf + (uint32_t)(r * SL * 4 * (1 + S) + 4 * SL + 4 * j * S); };
    auto copies = [&](int r, int j) {
      pair_copy_atom(sfa_col(r, j), sfa_desc + (uint64_t)((j & 3) * (kAtomBytes >> 4)));
#pragma unroll
      for (int sub = 0; sub < S; ++sub)
        pair_copy_atom(sfb_col(r, j) + 4 * sub, sfb_desc + (uint64_t)(((j & 3) * S + sub) * (kAtomBytes >> 4)));
    };
    if (!SFCP) {
#pragma unroll
      for (int j = 0; j < 4; ++j) copies(0, j);
    }
    for (int s = 0; s < stages; ++s) {
      const int r = s % RING;
      if (s >= RING && !mbar_wait_warp(smem_u32(&bar[r]), ((s / RING) - 1) & 1, &abort_flag, status)) break;
      tc_fence_after();
      if (SFCP) {
#pragma unroll
        for (int j = 0; j < MPC; ++j) copies(r, j);
      }
#pragma unroll
      for (int j = 0; j < MPC; ++j) {
        const uint64_t koff = (uint64_t)((32 * (j & 3)) >> 4);
        const int rs = SFCP ? r : 0, js = SFCP ? j : (j & 3);
        pair_mma(tmem, a_desc + koff, b_desc + koff, idesc, sfa_col(rs, js), sfb_col(rs, js), (s | j) != 0);
      }
      pair_commit(smem_u32(&bar[r]));
    }
    pair_commit(smem_u32(&drain_bar));
    mbar_wait_cleanup(smem_u32(&drain_bar), 0);
  }
  tc_fence_before();
  __syncwarp();
  cluster_sync_all();  // the peer's tensor memory and shared memory are no longer read
  tc_fence_after();
  tmem_dealloc_pair(tmem, ncols);
}

static_assert(rate_tmem_cols(128, 1, 4, 3) <= 256 && rate_tmem_cols(128, 0, 16, 3) <= 256 &&
                  rate_tmem_cols(256, 1, 4, 5) <= 512 && rate_tmem_cols(256, 0, 16, 3) <= 512 &&
                  rate_tmem_cols(128, 1, 4, 5) <= 512,
              "a rate-probe variant overflows its tensor-memory share");
static_assert(rate_smem_bytes(256) <= 96 * 1024, "rate-probe operands overflow shared memory");

}  // namespace moe

namespace moe {
int report_error(int code, const char* fmt, ...);
}

extern "C" int moe_fp4_mma_rate(int n, int sf_copies, int mmas_per_commit, int ctas_per_sm, int ring,
                                int warp_issue, int stages, double* flops, int32_t* status, void* stream) {
  if (!flops) return moe::report_error(MOE_ERR_INVALID_ARG, "flops is null");
  const char* why = "";
  int rc = moe::fp4_mma_rate_check(n, sf_copies, mmas_per_commit, ctas_per_sm, ring, warp_issue, stages, &why);
  if (rc) return moe::report_error(rc, "%s", why);
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess || sms < 1)
    return moe::report_error(MOE_ERR_CUDA, "fp4 rate: no device (%s)", cudaGetErrorString(err));
  rc = moe::launch_fp4_mma_rate(n, sf_copies, mmas_per_commit, ctas_per_sm, ring, warp_issue, stages, sms, status,
                                          reinterpret_cast<cudaStream_t>(stream), flops, &why);
  return rc ? moe::report_error(rc, "%s", why) : MOE_OK;
}

extern "C" int moe_fp4_mma_rate_pair(int n, int sf_copies, int stages, double* flops, int32_t* status, void* stream) {
  if (!flops) return moe::report_error(MOE_ERR_INVALID_ARG, "flops is null");
  if (!((n == 128 || n == 256) && (sf_copies == 0 || sf_copies == 1) && stages >= 1 && stages <= (1 << 24)))
    return moe::report_error(MOE_ERR_INVALID_ARG, "fp4 rate pair: n in {128, 256}, sf_copies in {0, 1}, stages 1..2^24");
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess || sms < 2)
    return moe::report_error(MOE_ERR_CUDA, "fp4 rate pair: no device (%s)", cudaGetErrorString(err));
  const int grid = sms & ~1;  // one CTA per SM, clusters of two
  const int smem = 160 * 1024;  // more than half an SM's shared memory: one CTA per SM
  *flops = 2.0 * 256.0 * n * 64.0 * 4.0 * (double)stages * (double)(grid / 2);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
#define MOE_PAIR(nn, cp)                                                               \
  if (n == nn && sf_copies == cp) {                                                    \
    auto k = moe::fp4_mma_pair_kernel<nn, cp>;                                         \
    err = moe::ensure_smem_limit(reinterpret_cast<const void*>(k), smem);              \
    if (err == cudaSuccess) {                                                          \
      k<<<grid, 32, smem, st>>>(stages, status);                                       \
      err = cudaGetLastError();                                                        \
    }                                                                                  \
  }
  MOE_PAIR(128, 0)
  MOE_PAIR(128, 1)
  MOE_PAIR(256, 0)
  MOE_PAIR(256, 1)
#undef MOE_PAIR
  return err == cudaSuccess ? MOE_OK : moe::report_error(MOE_ERR_CUDA, "fp4 rate pair: %s", cudaGetErrorString(err));
}
