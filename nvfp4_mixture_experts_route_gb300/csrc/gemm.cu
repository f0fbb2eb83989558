// Steps a3-a6: the two grouped block-scaled FP4 GEMMs on the 5th-generation
// tensor cores (tcgen05.mma kind::mxf4nvf4, one ue4m3 scale per 16 elements).
//
// What they compute (the muse_moe_runner page, apply_routed: gemm1/gemm2
// weights with output1_scale_gate_scalar = g1_alphas, output1_scale_scalar =
// g1_scale_c, output2_scale_scalar = g2_alphas, do_finalize=False):
//   GEMM1  acc[r, n] = sum_k a[r, k] w13[e][n, k]     (r: a route row of expert e)
//          h = SiLU(g1_alphas[e] * acc[:, gate]) * (g1_scale_c[e] * acc[:, up])
//          hq = NVFP4(h) with a2_gscale                 (fused epilogue)
//   GEMM2  rows[r, :] = bf16(g2_alphas[e] * sum_i hq[r, i] w2[e][:, i])
//
// Tiling ("swap AB"): the MMA's M = 128 rows are weight rows, its N = tile_m
// rows are permuted route rows of one routing tile (all of one expert). A
// work unit is one (route tile tau, weight tile mt) pair over the whole K.
//
// Persistent, warp-specialised kernel, one or two CTAs per SM (tile_cfg
// below), 2 + 4 or 2 + 8 warps:
//   - warp 0 / lane 0: TMA producer. Walks this CTA's units in order and, per
//     pipeline stage (K = 256 elements = 128 bytes per row per chunk), loads
//     the 128 x 128 B weight box and the tile_m x 128 B route box (both
//     128-byte swizzled) and the stage's scale atoms for both operands (plain
//     bulk copies), all completing one mbarrier. The ring of ST stages runs
//     across unit boundaries, so HBM streaming never stops between units.
//   - warp 1: MMA issuer. Copies each stage's scale atoms into that stage's
//     own tensor-memory columns (tcgen05.cp 32x128b.warpx4), issues the
//     stage's MMAs of K = 64 into the unit's accumulator buffer, and commits
//     the stage back to the producer; after a unit's last stage it commits
//     the accumulator to the epilogue. GEMM1 runs this loop on the whole
//     warp, converged, with lane 0 issuing under a predicate (a faster
//     instruction stream where the issue rate bounds the kernel, at
//     prefill); GEMM2 and the one-launch pair run it on lane 0 alone.
//   - warps 2..: epilogue. Warp w reads TMEM lane quadrant w % 4 (32 weight
//     rows) of the finished accumulator (with 8 warps, two per quadrant split
//     the route columns), then hands the buffer back. With two accumulator
//     buffers the epilogue of unit i runs while unit i+1 streams; with one
//     (the larger tiles, whose tensor memory is split between two CTAs or
//     taken by one wide accumulator) the other CTA on the SM fills the gap.
// Units are ordered with the weight tile fastest (u -> mt = u % tiles_w,
// tau = u / tiles_w) and dealt round-robin, so the CTAs working at the same
// time share route tiles (and, for experts with many tiles, weight tiles) in
// L2. Tiles past the live count (totals[0]) are not units at all.
//
// GEMM1's epilogue: the prepared w13 puts the gate (16 rows) and up (16 rows)
// of 16 intermediate columns in one 32-row quadrant, so warp w stages
// scale * acc for its 32 rows x 32 route columns in shared memory and then
// each lane takes one route column: SwiGLU of 16 elements and one NVFP4
// block, no shuffles.
//
// Every mbarrier wait is bounded (1 s); on a timeout the CTA records
// MOE_ERR_TIMEOUT, stops issuing, drains its own copies and MMAs (bounded
// again), frees its tensor memory and exits.
#include "common.cuh"
#include "layout.cuh"

namespace moe {

constexpr int kStageK = 256;                   // K elements per pipeline stage
constexpr int kStageRowBytes = kStageK / 2;    // 128
constexpr int kWTile = 128;                    // weight rows per unit (MMA M)
constexpr uint32_t kABytes = kWTile * kStageRowBytes;  // 16 KiB
constexpr uint32_t kSfStageBytes = 4 * kAtomBytes;     // 4 K=64 steps
constexpr int kMaxStages = 8;
// Stages of its first unit's weights a CTA of the one-launch GEMMs prefetches
// into L2 while the previous kernel (the quantizer) finishes.
#ifndef MOE_HEAD_PREFETCH_STAGES
#define MOE_HEAD_PREFETCH_STAGES 4
#endif
constexpr int kHeadPrefetchStages = MOE_HEAD_PREFETCH_STAGES;
constexpr int kEpiStride = 33;  // floats per staged route column (32 + pad)

// One GEMM's operands: GEMM1 (w13 against the permuted activations, writes
// the intermediate) or GEMM2 (w2 against the intermediate, writes rows).
struct GemmSide {
  const uint8_t* w_sf;  // prepared scale atoms [E][rows_w/128][K/64][512]
  const uint8_t* b_sf;  // workspace scale atoms [tiles][K/64][S][512]
  const float* s0;      // g1_alphas (GEMM1) or g2_alphas (GEMM2)
  const float* s1;      // g1_scale_c (GEMM1)
  int rows_w, K, out_cols;
};

struct GemmParams {
  GemmSide g[2];  // [0] GEMM1, [1] GEMM2
  const int32_t* tile_expert;
  const int32_t* tile_row_limit;
  const int32_t* totals;
  const float* a2_gscale;  // GEMM1
  uint8_t* hq;             // GEMM1: intermediate codes [P][I/2]
  uint8_t* hq_sf;          // GEMM1: intermediate scale atoms [tiles][I/64][S][512]
  __nv_bfloat16* rows;     // GEMM2: [P][H]
  int32_t* done;           // both GEMMs in one grid: per route tile, zeroed by the quantizer
  int32_t* ticket;         // both GEMMs in one grid: the next unit to hand out, zeroed with done
  int32_t* status;
  int tile_m;
  // Set when the launch follows this library's previous step kernel with
  // programmatic dependent launch: the producer then loads the weights of its
  // first stages before waiting for that kernel (the weights and the routing
  // metadata are complete by then; only the route operand is not).
  int prefetch;
  // GEMM2: rows and their pitch are 32-byte aligned, so the epilogue stores
  // whole 32-byte sectors (st.global.v8)
  int rows32;
  // GEMM2, optional: the post-expert norm's sums of squares of the stored
  // bf16 rows, one fp32 partial per 32 columns (row_ss[P][H / 32]); weighted
  // by the norm's gain g = 1 + gamma when ss_wbn is set (the weight applied
  // before the norm), else plain.
  float* row_ss;
  const __nv_bfloat16* ss_gamma;
  int ss_wbn;
  // both GEMMs in one grid: the experts and the route tiles the buffers hold
  // (bounds for the head prefetch, which reads the routing as a hint)
  int num_experts, max_tiles;
  // Load the weights and their scales with an L2 evict_first policy (they
  // stream through once), so that the rows, sums and intermediate the grid
  // writes and reads again stay in L2.
  int w_evict_first;
};

// Sum over a warp's 32 lanes of each of 32 values: afterwards lane l holds
// the total of x[l] (a butterfly that halves the array at every level; 31
// shuffles, a fixed order of additions).
__device__ __forceinline__ float transpose_reduce32(float (&x)[32], int lane) {
#pragma unroll
  for (int d = 16; d >= 1; d >>= 1) {
    const bool upper = (lane & d) != 0;
#pragma unroll
    for (int i = 0; i < d; ++i) {
      const float send = upper ? x[i] : x[i + d];
      const float keep = upper ? x[i + d] : x[i];
      x[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, d);
    }
  }
  return x[0];
}

// Launch shape per route-tile size: CTAs per SM, accumulator buffers, K=256
// chunks per pipeline stage, epilogue warps and GEMM1 epilogue staging
// columns. One thread per CTA issues all of its tcgen05 copies and MMAs, and
// each instruction occupies that thread for a fixed time whatever its size
// (measured with a pipe probe, issued by lane 0 alone: about 28 ns per copy
// or MMA and 140 ns per commit; by a converged warp, lane 0 issuing, about a
// third less), so the tensor core is fed by several CTAs per SM wherever tensor
// memory and shared memory allow; the decode tiles (32 and 64 rows) run two
// CTAs per SM with a 4- or 3-stage ring (one CTA per SM: 1.5 x slower; three
// with 2-stage rings: 1-2 % slower at b = 8, 2 % at b = 64, once the weights
// are loaded evict_first). Each epilogue warp works through its accumulator
// columns as one dependent instruction stream, so the larger tiles take two
// warps per TMEM lane quadrant (8 in all) that split the route columns.
//
// route_m: the MMA's M = 128 rows are the route tile itself and N = 128 its
// weight rows (128-row tiles only; M = 128 is the MMA's full-rate shape and
// smaller route tiles need the swapped form). A lane of the accumulator is
// then a route row holding gate and up of the same intermediate columns, so
// GEMM1's epilogue needs no transposing staging buffer (its shared memory
// goes to the ring) and GEMM2 stores each route row contiguously.
struct TileCfg {
  int ctas, acc_bufs, chunks, epi_warps, epi_cols;
  bool route_m;
};
__host__ __device__ constexpr TileCfg tile_cfg(int tile_m) {
  return tile_m <= 32    ? TileCfg{2, 2, 1, 4, 16, false}
         : tile_m <= 64  ? TileCfg{2, 2, 1, 4, 16, false}
         : tile_m <= 128 ? TileCfg{2, 1, 1, 8, 32, true}
                         : TileCfg{1, 1, 1, 8, 32, false};
}
__host__ __device__ constexpr int ctas_per_sm(int tile_m) { return tile_cfg(tile_m).ctas; }
__host__ __device__ constexpr int acc_bufs_for(int tile_m) { return tile_cfg(tile_m).acc_bufs; }
__host__ __device__ constexpr int chunks_for(int tile_m) { return tile_cfg(tile_m).chunks; }
__host__ __device__ constexpr int epi_warps_for(int tile_m) { return tile_cfg(tile_m).epi_warps; }
__host__ __device__ constexpr int epi_cols_for(int tile_m) { return tile_cfg(tile_m).epi_cols; }
// Only GEMM1's swapped-form epilogue stages through shared memory (its
// SwiGLU pairs rows of two lanes); elsewhere the ring takes the room.
__host__ __device__ constexpr uint32_t epi_bytes_for(int tile_m, int kind) {
  return kind == 1 && !tile_cfg(tile_m).route_m
             ? (uint32_t)(epi_warps_for(tile_m) * epi_cols_for(tile_m) * kEpiStride * 4)
             : 0u;
}

__host__ __device__ constexpr int sf_atoms_for(int tile_m) { return (tile_m + 127) / 128; }

// Bytes of one pipeline stage: chunks_for(tile_m) K = 256 chunks of the
// weight box, the route box and both operands' scale atoms.
__host__ __device__ constexpr uint32_t stage_bytes(int tile_m) {
  return (uint32_t)chunks_for(tile_m) *
         (kABytes + (uint32_t)tile_m * kStageRowBytes +
          kSfStageBytes * (uint32_t)(1 + sf_atoms_for(tile_m)));
}

// Dynamic shared memory a CTA may take: 227 KB alone, otherwise its share of
// the SM's 228 KB less the per-CTA reserve and static storage. Tensor-memory
// columns a CTA may allocate: 512 / CTAs per SM, a power of two.
__host__ __device__ constexpr int smem_budget(int ctas) {
  return ctas == 1 ? 232448 : ctas == 2 ? 115456 : 76400;
}
__host__ __device__ constexpr int tmem_budget(int ctas) { return ctas == 1 ? 512 : ctas == 2 ? 256 : 128; }

__host__ __device__ constexpr uint32_t tmem_cols_for(int tile_m, int stages, int bufs) {
  const int need = bufs * tile_m + stages * 16 * chunks_for(tile_m) * (1 + sf_atoms_for(tile_m));
  uint32_t c = 32;
  while ((int)c < need) c <<= 1;
  return c;
}

// Pipeline depth: as many stages as the shared memory left after the
// epilogue staging holds and the CTA's tensor-memory share can give scale
// columns to.
__host__ __device__ constexpr int stages_for(int tile_m, int kind) {
  const int budget = smem_budget(ctas_per_sm(tile_m)) - 1024 - (int)epi_bytes_for(tile_m, kind);
  int st = budget / (int)stage_bytes(tile_m);
  st = st > kMaxStages ? kMaxStages : st;
  while (st > 1 && tmem_cols_for(tile_m, st, acc_bufs_for(tile_m)) >
                       (uint32_t)tmem_budget(ctas_per_sm(tile_m)))
    --st;
  return st;
}

__host__ __device__ constexpr size_t gemm_smem_bytes(int tile_m, int kind) {
  return 1024 + (size_t)stages_for(tile_m, kind) * stage_bytes(tile_m) + epi_bytes_for(tile_m, kind);
}

__host__ __device__ constexpr bool tile_fits(int t, int kind) {
  return stages_for(t, kind) >= 2 &&
         tmem_cols_for(t, stages_for(t, kind), acc_bufs_for(t)) <=
             (uint32_t)tmem_budget(ctas_per_sm(t)) &&
         gemm_smem_bytes(t, kind) <= (size_t)smem_budget(ctas_per_sm(t));
}
static_assert(tile_fits(32, 1) && tile_fits(64, 1) && tile_fits(128, 1) && tile_fits(256, 1) &&
                  tile_fits(32, 2) && tile_fits(64, 2) && tile_fits(128, 2) && tile_fits(256, 2),
              "a route-tile shape overflows its pipeline, tensor memory or shared memory budget");


// GEMM1 epilogue for COLS route columns of one accumulator: lanes write
// scale * acc (gate rows 0-15, up rows 16-31 of this quadrant) to the warp's
// staging rows, then each of the first COLS lanes takes one route column:
// SwiGLU over its 16 intermediate columns and one NVFP4 block.
template <int COLS>
__device__ __forceinline__ void gemm1_epilogue_chunk(uint32_t taddr, float* stage, int lane, float sc,
                                                     float a2g, int r0, int I, int mt, int q,
                                                     int tile_m, int S, uint8_t* hq, uint8_t* hq_sf) {
  float v[COLS];
  if (COLS == 32)
    tmem_ld32(taddr, *reinterpret_cast<float(*)[32]>(v));
  else
    tmem_ld16(taddr, *reinterpret_cast<float(*)[16]>(v));
#pragma unroll
  for (int i = 0; i < COLS; ++i) stage[i * kEpiStride + lane] = v[i] * sc;
  __syncwarp();
  if (lane < COLS) {
    float h[16];
    const float* col = stage + lane * kEpiStride;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float g = col[j], up = col[16 + j];
      h[j] = __fdividef(g, 1.0f + __expf(-g)) * up;  // SiLU(gate) * up
    }
    uint2 codes;
    uint32_t sfc;
    quant16(h, a2g, codes, sfc);
    const int r = r0 + lane;
    *reinterpret_cast<uint2*>(hq + (size_t)r * (I / 2) + 32 * mt + 8 * q) = codes;
    hq_sf[act_sf_offset(r, 4 * mt + q, tile_m, I / 64, S)] = static_cast<uint8_t>(sfc);
  }
  __syncwarp();
}

// How the MMA issuer runs (measured at T = 8192, 128-row tiles, one GB300):
// GEMM1 with the loop on the whole warp, converged, lane 0 issuing under a
// predicate, and the scale copies on that same warp: 0.694 ms, against 0.738
// with the copies on a warp of their own (either issue form) and 0.755 with
// lane 0 alone running the loop. GEMM2 measured the other way: 0.474 ms
// converged against 0.433 on lane 0 alone, and the decode pair the same
// either way, so those keep lane 0. (A converged loop in which lane 0 alone
// polled the barriers and broadcast the outcome: 0.875 ms for GEMM1.)
__host__ __device__ constexpr bool warp_issue_for(int mode) { return mode == 1; }
__host__ __device__ constexpr int gemm_threads(int mode, int tile_m) {
  return 64 + 32 * tile_cfg(tile_m).epi_warps;
}

// One instantiation per (mode, route-tile size). MODE 1 runs GEMM1 units, 2
// GEMM2 units, 3 both in one persistent grid: every CTA walks its GEMM1
// units, then its GEMM2 units, and the producer of a GEMM2 unit waits until
// the GEMM1 units of its route tile have stored their intermediate (a
// per-tile counter that every epilogue warp of those units raises after its
// stores), so a route tile's GEMM2 starts while later tiles' GEMM1 units
// still run and neither GEMM has a ramp or a tail of its own. Units are
// dealt round-robin, each CTA in order, and a waited-for GEMM1 unit is
// always earlier in its CTA's order than the GEMM2 unit waiting, so every
// wait ends once the grid's CTAs are resident (the grid never exceeds what
// fits at once). The tile's launch shape, pipeline depth and scale-atom
// count are compile-time, so the MMA issuer's per-stage loops unroll and its
// descriptors are base + constant.
// Both GEMMs in one grid: L2 prefetch of the first kHeadPrefetchStages
// stages of weights and weight scales of unit blockIdx.x, from a routing
// read before the previous kernel has completed (a hint: the route-tile
// count and the expert are bounded before any address is formed; a stale
// value only wastes the prefetch). Kept out of line so that its registers
// do not weigh on the kernel's steady-state loops.
template <int SPST>
__device__ __noinline__ void prefetch_head_hint(const CUtensorMap& tmA1, const CUtensorMap& tmA2, const GemmParams& p,
                                                int tw1, int tw2) {
  const int nt = min(max(__ldcg(p.totals), 0), p.max_tiles);
  const int u = blockIdx.x, n1h = nt * tw1;
  const int gi = u < n1h ? 0 : 1;
  const int tau = gi == 0 ? u / tw1 : (u - n1h) / tw2, mt = gi == 0 ? u % tw1 : (u - n1h) % tw2;
  const int e = tau < nt ? __ldcg(p.tile_expert + tau) : -1;
  if (e < 0 || e >= p.num_experts) return;
  const GemmSide& gs = p.g[gi];
  const int KC = gs.K / 64, tw = gi == 0 ? tw1 : tw2;
  const int nks = (KC + SPST - 1) / SPST;
  const int a_row = e * gs.rows_w + mt * kWTile;
  const uint8_t* wsf = gs.w_sf + ((size_t)e * tw + mt) * KC * kAtomBytes;
  for (int ks = 0; ks < nks && ks < kHeadPrefetchStages; ++ks) {
    const int kk = min(SPST, KC - SPST * ks);
    for (int c = 0; 4 * c < kk; ++c)
      tma_prefetch_l2_2d(gi == 0 ? &tmA1 : &tmA2, (ks * (SPST / 4) + c) * kStageRowBytes, a_row);
    bulk_prefetch_l2(wsf + (size_t)SPST * ks * kAtomBytes, (uint32_t)kk * kAtomBytes);
  }
}

template <int MODE, int TILE>
__global__ void __launch_bounds__(gemm_threads(MODE, TILE), tile_cfg(TILE).ctas)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                        const GemmParams p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t accf_bar[2];
  __shared__ __align__(8) uint64_t acce_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  // Both GEMMs in one grid: the units this CTA drew, in order, from the
  // producer to the MMA issuer and the epilogue warps.
  constexpr int kUnitQ = 8;
  __shared__ int unit_q[kUnitQ];
  __shared__ __align__(8) uint64_t uq_full[kUnitQ];
  __shared__ __align__(8) uint64_t uq_empty[kUnitQ];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // weight tiles per route tile of each GEMM, and the units: GEMM1's, then GEMM2's
  const int tw1 = MODE != 2 ? p.g[0].rows_w / kWTile : 0;
  const int tw2 = MODE != 1 ? p.g[1].rows_w / kWTile : 0;
  // Both GEMMs in one grid, launched before the previous kernel (the
  // quantizer, or the fused routing + quantizer) has completed: the route
  // tiles are read after the wait, which comes after the setup below.
  const bool late = MODE == 3 && p.prefetch;
  if (late && tid == 0) {
    // Prefetch into L2 the weights and weight scales of the first stages of
    // unit blockIdx.x (the first gridDim.x tickets are exactly units
    // [0, gridDim.x), so whichever CTA draws a unit finds its first stages in
    // L2). The routing read here is only a hint, bounded before use.
    prefetch_head_hint<4 * chunks_for(TILE)>(tmA1, tmA2, p, tw1, tw2);
  } else if (!p.prefetch) {
    pdl_wait();
    if (tid == 0) pdl_trigger();
  }
  const int ntiles_early = late ? 0 : __ldcg(p.totals);
  if (!late && (int)blockIdx.x >= ntiles_early * (tw1 + tw2)) {
    // Even an idle CTA must not let this grid complete before its
    // predecessor: the kernels after it rely on that ordering.
    if (p.prefetch) pdl_wait();
    return;
  }
  constexpr int tile_m = TILE, S = sf_atoms_for(TILE), ST = stages_for(TILE, MODE == 2 ? 2 : 1);
  constexpr int NB = acc_bufs_for(TILE), CH = chunks_for(TILE), EPW = epi_warps_for(TILE);
  constexpr bool kRouteM = tile_cfg(TILE).route_m;
  constexpr bool kWI = warp_issue_for(MODE);
  // Per stage: CH chunks of K = 256, i.e. up to 4 * CH MMA steps of K = 64.
  constexpr uint32_t b_bytes = (uint32_t)tile_m * kStageRowBytes;  // one chunk of the route box
  constexpr uint32_t a_stage = CH * kABytes, b_stage = CH * b_bytes;
  constexpr uint32_t sfa_stage = CH * kSfStageBytes, sfb_stage = CH * kSfStageBytes * S;
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sA = sbase;
  const uint32_t sB = sA + ST * a_stage;
  const uint32_t sSFA = sB + ST * b_stage;
  const uint32_t sSFB = sSFA + ST * sfa_stage;
  const uint32_t sEpi = sSFB + ST * sfb_stage;
  constexpr int steps_per_stage = 4 * CH;
  const int KC1 = MODE != 2 ? p.g[0].K / 64 : 0, KC2 = MODE != 1 ? p.g[1].K / 64 : 0;
  const int nks1 = (KC1 + steps_per_stage - 1) / steps_per_stage;
  const int nks2 = (KC2 + steps_per_stage - 1) / steps_per_stage;
  constexpr uint32_t ncols = tmem_cols_for(tile_m, ST, NB);
  // completions a route tile's GEMM1 units report when their intermediate is stored
  const int done_target = tw1 * EPW;

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&accf_bar[b]), 1);
      mbar_init(smem_u32(&acce_bar[b]), EPW);
    }
    mbar_init(smem_u32(&drain_bar), 1);
    for (int q = 0; q < kUnitQ; ++q) {
      mbar_init(smem_u32(&uq_full[q]), 1);
      mbar_init(smem_u32(&uq_empty[q]), 1 + EPW);  // the MMA issuer and every epilogue warp
    }
    abort_flag = 0;
    fence_barrier_init();
    if (MODE != 2) {
      tma_prefetch_desc(&tmA1);
      tma_prefetch_desc(&tmB1);
    }
    if (MODE != 1) {
      tma_prefetch_desc(&tmA2);
      tma_prefetch_desc(&tmB2);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (late) {
    // Units come from the ticket, so a CTA with none to do simply draws a
    // ticket past the end and runs through to the teardown.
    pdl_wait();
    if (tid == 0) pdl_trigger();
  }
  const int ntiles = late ? __ldcg(p.totals) : ntiles_early;
  const int n1 = ntiles * tw1;
  const int n_units = n1 + ntiles * tw2;
  // unit u -> (GEMM 0 or 1, route tile, weight tile)
  auto unit_of = [&](int u, int& gi, int& tau, int& mt) {
    if constexpr (MODE != 2) {
      if (MODE == 1 || u < n1) {
        gi = 0;
        tau = u / tw1;
        mt = u % tw1;
        return;
      }
    }
    if constexpr (MODE != 1) {
      gi = 1;
      tau = (u - n1) / tw2;
      mt = (u - n1) % tw2;
    }
  };

  const uint32_t t_sfa = tmem + (uint32_t)(NB * tile_m);
  const uint32_t t_sfb = t_sfa + ST * 16 * CH;

  if (warp == 0) {
    // ------------------------------ producer ------------------------------
    if (lane == 0) {
      int it = 0;
      bool stop = false;
      // With p.prefetch the route-operand half of the first stages (at most
      // ST of them) is held back until the previous kernel has completed.
      bool waited = !p.prefetch;
      int held = 0;
      int held_s[kMaxStages], held_ks[kMaxStages], held_tau[kMaxStages], held_kk[kMaxStages],
          held_gi[kMaxStages];
      auto load_route_half = [&](int s, int ks, int tau, int kk, int gi) {
        const uint32_t fb = smem_u32(&full_bar[s]);
        const int KC = gi == 0 ? KC1 : KC2;
        const CUtensorMap* tmB = gi == 0 ? &tmB1 : &tmB2;
        const uint8_t* bsf = p.g[gi].b_sf + (size_t)tau * KC * S * kAtomBytes;
        for (int c = 0; 4 * c < kk; ++c)
          tma_load_2d(sB + s * b_stage + c * b_bytes, tmB, fb, (ks * CH + c) * kStageRowBytes,
                      tau * tile_m);
        bulk_load(sSFB + s * sfb_stage, bsf + (size_t)steps_per_stage * ks * S * kAtomBytes,
                  (uint32_t)kk * S * kAtomBytes, fb);
      };
      auto release_held = [&]() {
        pdl_wait();
        pdl_trigger();
        for (int h = 0; h < held; ++h)
          load_route_half(held_s[h], held_ks[h], held_tau[h], held_kk[h], held_gi[h]);
        held = 0;
        waited = true;
      };
      // Units are drawn from a ticket (below), known only after the previous
      // kernel has completed: the grid's prologue waited for it.
      if constexpr (MODE == 3) waited = true;
      const uint64_t w_pol = p.w_evict_first ? l2_policy_evict_first() : 0;
      // MODE 3: the ticket this CTA holds next (drawn one unit ahead, so that
      // the atomic's latency overlaps the current unit's loads)
      int next = MODE == 3 ? atomicAdd(p.ticket, 1) : 0;
      for (int n = 0; !stop; ++n) {
        int u;
        if constexpr (MODE == 3) {
          // A unit is handed out only to a running CTA, in unit order (all
          // GEMM1 units before any GEMM2 unit): every GEMM1 unit a GEMM2 unit
          // waits for is already held by a running CTA that reaches it
          // without waiting on anything, so the waits end whatever else
          // holds the GPU's SMs.
          u = next < n_units ? next : -1;
          const int q = n % kUnitQ;
          if (n >= kUnitQ &&
              !mbar_wait(smem_u32(&uq_empty[q]), ((n / kUnitQ) - 1) & 1, &abort_flag, p.status)) {
            stop = true;
            break;
          }
          unit_q[q] = u;
          mbar_arrive(smem_u32(&uq_full[q]));
          if (u < 0) break;
          next = atomicAdd(p.ticket, 1);
        } else {
          u = blockIdx.x + n * gridDim.x;
          if (u >= n_units) break;
        }
        int gi, tau, mt;
        unit_of(u, gi, tau, mt);
        const GemmSide& gs = p.g[gi];
        const int KC = gi == 0 ? KC1 : KC2, nks = gi == 0 ? nks1 : nks2, tw = gi == 0 ? tw1 : tw2;
        const CUtensorMap* tmA = gi == 0 ? &tmA1 : &tmA2;
        const int e = __ldcg(p.tile_expert + tau);
        const int a_row = e * gs.rows_w + mt * kWTile;
        const uint8_t* wsf = gs.w_sf + ((size_t)e * tw + mt) * KC * kAtomBytes;
        if (MODE == 3 && gi == 1) {
          // This route tile's intermediate must be complete: its GEMM1 units
          // (drawn earlier, by running CTAs) report through p.done.
          if (!waited) release_held();
          if (!wait_counter_at_least(p.done + tau, done_target, &abort_flag, p.status)) {
            stop = true;
            break;
          }
          // the intermediate was stored through the generic proxy; the loads
          // below read it through the async proxy
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        for (int ks = 0; ks < nks; ++ks, ++it) {
          const int s = it % ST, round = it / ST;
          if (round > 0) {
            if (!waited) release_held();
            if (!mbar_wait(smem_u32(&empty_bar[s]), (round - 1) & 1, &abort_flag, p.status)) {
              stop = true;
              break;
            }
          }
          const int kk = min(steps_per_stage, KC - steps_per_stage * ks);
          const uint32_t nc = (uint32_t)(kk + 3) / 4;  // chunks in this stage
          const uint32_t fb = smem_u32(&full_bar[s]);
          mbar_arrive_expect_tx(fb, nc * (kABytes + b_bytes) + (uint32_t)kk * kAtomBytes * (1 + S));
          if (p.w_evict_first) {
            for (int c = 0; c < (int)nc; ++c)
              tma_load_2d_hint(sA + s * a_stage + c * kABytes, tmA, fb, (ks * CH + c) * kStageRowBytes, a_row,
                               w_pol);
            bulk_load_hint(sSFA + s * sfa_stage, wsf + (size_t)steps_per_stage * ks * kAtomBytes,
                           (uint32_t)kk * kAtomBytes, fb, w_pol);
          } else {
            for (int c = 0; c < (int)nc; ++c)
              tma_load_2d(sA + s * a_stage + c * kABytes, tmA, fb, (ks * CH + c) * kStageRowBytes,
                          a_row);
            bulk_load(sSFA + s * sfa_stage, wsf + (size_t)steps_per_stage * ks * kAtomBytes,
                      (uint32_t)kk * kAtomBytes, fb);
          }
          if (waited) {
            load_route_half(s, ks, tau, kk, gi);
          } else {
            held_s[held] = s;
            held_ks[held] = ks;
            held_tau[held] = tau;
            held_kk[held] = kk;
            held_gi[held] = gi;
            ++held;
          }
        }
      }
      if (!waited) release_held();
      // Wait for the copies still in flight (normally all consumed already).
      for (int j = max(0, it - ST); j < it; ++j)
        mbar_wait_cleanup(smem_u32(&full_bar[j % ST]), (j / ST) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ----------------------------
    // kWI: the whole warp runs the loop, converged, and lane 0 issues;
    // otherwise lane 0 alone runs it.
    if (kWI || lane == 0) {
      constexpr uint32_t idesc = idesc_nvf4(kWTile, (uint32_t)tile_m);
      // Descriptors of stage 0's first K = 64 step; another stage or step adds
      // its byte offset >> 4 to the start-address field (shared-memory
      // addresses are below 2^18, so the 14-bit field never carries).
      const uint64_t a_desc0 = smem_desc(sA, 16, 1024, 2);
      const uint64_t b_desc0 = smem_desc(sB, 16, 1024, 2);
      const uint64_t sfa_desc0 = smem_desc(sSFA, 0, 128, 0);
      const uint64_t sfb_desc0 = smem_desc(sSFB, 0, 128, 0);
      int s = 0, uc = 0;
      uint32_t phase = 0;  // ring position: stage s, its current full phase
      bool stop = false;
      for (int n = 0; !stop; ++n) {
        int u;
        if constexpr (MODE == 3) {
          const int q = n % kUnitQ;
          if (!mbar_wait_f<kWI>(smem_u32(&uq_full[q]), (n / kUnitQ) & 1, &abort_flag, p.status)) break;
          u = *reinterpret_cast<volatile int*>(&unit_q[q]);
          if constexpr (kWI) __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&uq_empty[q]));
          if (u < 0) break;
        } else {
          u = blockIdx.x + n * gridDim.x;
          if (u >= n_units) break;
        }
        const int gi = u < n1 ? 0 : 1;
        const int KC = gi == 0 ? KC1 : KC2, nks = gi == 0 ? nks1 : nks2;
        const int b = uc % NB, use = uc / NB;
        if (use > 0 &&
            !mbar_wait_f<kWI>(smem_u32(&acce_bar[b]), (use - 1) & 1, &abort_flag, p.status))
          break;
        tc_fence_after();
        const uint32_t dacc = tmem + (uint32_t)(b * tile_m);
        for (int ks = 0; ks < nks; ++ks) {
          if (!mbar_wait_f<kWI>(smem_u32(&full_bar[s]), phase, &abort_flag, p.status)) {
            stop = true;
            break;
          }
          tc_fence_after();
          const int kk = min(steps_per_stage, KC - steps_per_stage * ks);
          // Scale-factor addresses of the MMA must be 4-column aligned: each
          // K=64 step gets its own 4-column group per operand.
          const uint32_t fa = t_sfa + s * 16 * CH, fbc = t_sfb + s * 16 * CH * S;
          const uint64_t ad = a_desc0 + ((s * a_stage) >> 4), bd = b_desc0 + ((s * b_stage) >> 4);
          const uint64_t sad = sfa_desc0 + ((s * sfa_stage) >> 4);
          const uint64_t sbd = sfb_desc0 + ((s * sfb_stage) >> 4);
#pragma unroll
          for (int j = 0; j < steps_per_stage; ++j) {
            if (j < kk) {
              tc_copy_scale_atom_f<kWI>(fa + 4 * j, sad + j * (kAtomBytes >> 4));
#pragma unroll
              for (int sub = 0; sub < S; ++sub)
                tc_copy_scale_atom_f<kWI>(fbc + 4 * (j * S + sub), sbd + (j * S + sub) * (kAtomBytes >> 4));
            }
          }
#pragma unroll
          for (int j = 0; j < steps_per_stage; ++j) {
            if (j < kk) {
              // step j: chunk j / 4 of the stage, 32 bytes (K = 64) per step in it
              const uint32_t a_off = ((j >> 2) * kABytes + 32 * (j & 3)) >> 4;
              const uint32_t b_off = ((j >> 2) * b_bytes + 32 * (j & 3)) >> 4;
              if constexpr (kRouteM)  // A = route rows, B = weight rows
                tc_mma_nvf4_f<kWI>(dacc, bd + b_off, ad + a_off, idesc, fbc + 4 * j * S, fa + 4 * j,
                            (ks | j) != 0);
              else  // A = weight rows, B = route rows
                tc_mma_nvf4_f<kWI>(dacc, ad + a_off, bd + b_off, idesc, fa + 4 * j, fbc + 4 * j * S,
                            (ks | j) != 0);
            }
          }
          tc_commit_f<kWI>(smem_u32(&empty_bar[s]));
          if (++s == ST) {
            s = 0;
            phase ^= 1u;
          }
        }
        if (stop) break;
        tc_commit_f<kWI>(smem_u32(&accf_bar[b]));
        ++uc;
      }
    }
    __syncwarp();
  } else {
    // ------------------------------ epilogue ------------------------------
    const int q = warp & 3;         // TMEM lane quadrant of this warp
    const int half = (warp - 2) >> 2;  // which of the quadrant's warps (EPW = 8)
    constexpr int kSplit = EPW / 4;    // warps per quadrant
    // this warp's staging rows: epi_cols_for(tile_m) route columns of 33 floats
    float* stage = reinterpret_cast<float*>(dsmem + (sEpi - smem_u32(dsmem))) +
                   (warp - 2) * epi_cols_for(tile_m) * kEpiStride;
    int uc = 0;
    for (int n = 0;; ++n) {
      int u;
      if constexpr (MODE == 3) {
        const int q = n % kUnitQ;
        u = -2;
        if (lane == 0 && mbar_wait(smem_u32(&uq_full[q]), (n / kUnitQ) & 1, &abort_flag, p.status)) {
          u = *reinterpret_cast<volatile int*>(&unit_q[q]);
          mbar_arrive(smem_u32(&uq_empty[q]));
        }
        u = __shfl_sync(0xFFFFFFFFu, u, 0);
        if (u < 0) break;
      } else {
        u = blockIdx.x + n * gridDim.x;
        if (u >= n_units) break;
      }
      const int b = uc % NB, use = uc / NB;
      const bool ok = mbar_wait(smem_u32(&accf_bar[b]), use & 1, &abort_flag, p.status);
      __syncwarp();
      if (!ok) break;
      tc_fence_after();
      int gi, tau, mt;
      unit_of(u, gi, tau, mt);
      const bool g1 = MODE == 1 || (MODE == 3 && gi == 0);  // this unit is a GEMM1 unit
      const GemmSide& gs = p.g[gi];
      const int e = p.tile_expert[tau];
      const int row0 = tau * tile_m;
      const uint32_t taddr = tmem + (uint32_t)(b * tile_m) + ((uint32_t)(32 * q) << 16);
      if constexpr (kRouteM) {
        // lane = route row r; accumulator column c = weight row mt * 128 + c.
        // This warp takes the adjacent column groups cc = 2 half and
        // 2 half + 1 (32 columns each), so that a lane's results for the unit
        // are contiguous in its row: both groups are read out of TMEM, the
        // buffer goes back to the MMA issuer, and only then are they converted
        // and stored.
        static_assert(EPW == 8, "the route-rows-on-M epilogue takes two warps per quadrant");
        const int r = row0 + 32 * q + lane;
        uint32_t acc[2][32];
        tmem_ld32_async(taddr + 64 * half, acc[0]);
        tmem_ld32_async(taddr + 64 * half + 32, acc[1]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&acce_bar[b]));
        if (g1) {
          // columns 32cc..32cc+31: gate and up of intermediate columns
          // 16 (4 mt + cc) + 0..15 (the prepared w13 granules)
          const float s0 = gs.s0[e], s1 = gs.s1[e], a2g = *p.a2_gscale;
          const int I = gs.out_cols;
          uint32_t cw[4], sf2 = 0;  // the two groups' 16 code bytes and 2 scale bytes
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            float h[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float g = s0 * __uint_as_float(acc[k][i]);
              const float up = s1 * __uint_as_float(acc[k][16 + i]);
              h[i] = __fdividef(g, 1.0f + __expf(-g)) * up;  // SiLU(gate) * up
            }
            uint2 codes;
            uint32_t sfc;
            quant16(h, a2g, codes, sfc);
            cw[2 * k] = codes.x;
            cw[2 * k + 1] = codes.y;
            sf2 |= sfc << (8 * k);
          }
          // blocks 4 mt + 2 half and + 1: 16 contiguous code bytes, and two
          // adjacent scale bytes of the row's atom
          *reinterpret_cast<uint4*>(p.hq + (size_t)r * (I / 2) + 32 * mt + 16 * half) =
              make_uint4(cw[0], cw[1], cw[2], cw[3]);
          *reinterpret_cast<uint16_t*>(p.hq_sf + act_sf_offset(r, 4 * mt + 2 * half, tile_m, I / 64, S)) =
              static_cast<uint16_t>(sf2);
        } else {
          const float g2 = gs.s0[e];
          if (r < p.tile_row_limit[tau]) {
            float ss2[2] = {0.f, 0.f};  // this row's sums of squares of the two 32-column groups
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int cc = 2 * half + k;
              // the gain of these 32 columns (weight-before-norm sums of
              // squares), loaded as packed bf16 before the conversions so
              // that they hide the loads' latency
              uint4 gu[4];
              if (p.row_ss != nullptr && p.ss_wbn) {
                const uint4* src = reinterpret_cast<const uint4*>(p.ss_gamma + mt * kWTile + 32 * cc);
#pragma unroll
                for (int j = 0; j < 4; ++j) gu[j] = __ldg(src + j);
              }
              uint32_t w[16];
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(acc[k][2 * i]) * g2,
                                                                __uint_as_float(acc[k][2 * i + 1]) * g2);
                w[i] = *reinterpret_cast<const uint32_t*>(&h2);
              }
              if (p.row_ss != nullptr) {
                // of the stored (bf16) values, gain-weighted (g = 1 + gamma)
                // for the weight-before-norm reading
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
                  float a = f.x, c = f.y;
                  if (p.ss_wbn) {
                    const float2 gf = __bfloat1622float2(reinterpret_cast<const __nv_bfloat162*>(&gu[i >> 2])[i & 3]);
                    a = f.x * (1.f + gf.x);
                    c = f.y * (1.f + gf.y);
                  }
                  ss2[k] = fmaf(a, a, ss2[k]);
                  ss2[k] = fmaf(c, c, ss2[k]);
                }
              }
              __nv_bfloat16* dp = p.rows + (size_t)r * gs.out_cols + mt * kWTile + 32 * cc;
              if (p.rows32) {
#pragma unroll
                for (int i = 0; i < 2; ++i)
                  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dp + 16 * i),
                               "r"(w[8 * i]), "r"(w[8 * i + 1]), "r"(w[8 * i + 2]), "r"(w[8 * i + 3]),
                               "r"(w[8 * i + 4]), "r"(w[8 * i + 5]), "r"(w[8 * i + 6]), "r"(w[8 * i + 7])
                               : "memory");
              } else {
                uint4* dst = reinterpret_cast<uint4*>(dp);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
              }
            }
            if (p.row_ss != nullptr)
              *reinterpret_cast<float2*>(p.row_ss + (size_t)r * (gs.out_cols / 32) + 4 * mt + 2 * half) =
                  make_float2(ss2[0], ss2[1]);
          }
        }
      } else {
        if (g1) {
          const float sc = lane < 16 ? gs.s0[e] : gs.s1[e];
          const float a2g = *p.a2_gscale;
          const int I = gs.out_cols;
          const int cols = epi_cols_for(tile_m);
          for (int c0 = half * cols; c0 < tile_m; c0 += kSplit * cols) {
            if (cols == 32)
              gemm1_epilogue_chunk<32>(taddr + c0, stage, lane, sc, a2g, row0 + c0, I, mt, q, tile_m, S,
                                       p.hq, p.hq_sf);
            else
              gemm1_epilogue_chunk<16>(taddr + c0, stage, lane, sc, a2g, row0 + c0, I, mt, q, tile_m, S,
                                       p.hq, p.hq_sf);
          }
        } else {
          const float g2 = gs.s0[e];
          const int limit = p.tile_row_limit[tau];
          const int colx = mt * kWTile + 32 * q + lane;
          // this lane's column's gain (weight-before-norm sums of squares)
          const float gn = p.row_ss != nullptr && p.ss_wbn ? 1.f + __bfloat162float(p.ss_gamma[colx]) : 1.f;
          for (int c0 = half * 32; c0 < tile_m; c0 += kSplit * 32) {
            float v[32];
            tmem_ld32(taddr + c0, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int rr = row0 + c0 + i;
              const __nv_bfloat16 hv = __float2bfloat16_rn(v[i] * g2);
              if (rr < limit) p.rows[(size_t)rr * gs.out_cols + colx] = hv;
              const float y = __bfloat162float(hv) * gn;
              v[i] = y * y;
            }
            if (p.row_ss != nullptr) {
              // lane i: route row row0 + c0 + i, its 32 columns of this
              // quadrant summed over the warp's lanes
              const float tot = transpose_reduce32(v, lane);
              const int rr = row0 + c0 + lane;
              if (rr < limit) p.row_ss[(size_t)rr * (gs.out_cols / 32) + 4 * mt + q] = tot;
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&acce_bar[b]));
      }
      if (MODE == 3 && g1) {
        // This warp's share of the tile's intermediate is stored: publish it
        // to the GEMM2 units of the tile, whose TMA loads (async proxy) read
        // it (release at GPU scope).
        asm volatile("fence.proxy.async.global;" ::: "memory");
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(p.done + tau, 1);
      }
      ++uc;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // One more commit from the MMA thread tracks every tcgen05 op it issued
    // (on a timeout too); once it lands no MMA or copy still uses TMEM.
    if (lane == 0) {
      tc_commit(smem_u32(&drain_bar));
      mbar_wait_cleanup(smem_u32(&drain_bar), 0);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch.
// ---------------------------------------------------------------------------
static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
    n = 148;
  return n;
}

// CTAs of a kernel that fit on one SM at once, from its compiled resources
// and the device's per-SM limits: shared memory (each CTA also takes the
// runtime's per-block reserve), registers (allocated per warp in units of
// 256) and threads. The runtime's occupancy query answers 1 for these
// tensor-memory kernels although the SM holds as many as these limits allow
// (tensor memory itself is budgeted at compile time).
static cudaError_t resident_ctas(const void* kern, int threads, size_t dyn_smem, int* fit) {
  cudaFuncAttributes fa{};
  cudaError_t err = cudaFuncGetAttributes(&fa, kern);
  int dev = 0, smem_sm = 0, reserve = 0, regs_sm = 0, threads_sm = 0, blocks_sm = 0;
  if (err == cudaSuccess) err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&reserve, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
  if (err == cudaSuccess)
    err = cudaDeviceGetAttribute(&threads_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&blocks_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev);
  if (err != cudaSuccess) return err;
  const long long cta_smem = (long long)dyn_smem + (long long)fa.sharedSizeBytes + reserve;
  const long long warps = (threads + 31) / 32;
  const long long cta_regs = warps * (((long long)fa.numRegs * 32 + 255) / 256 * 256);
  long long n = blocks_sm;
  if (cta_smem > 0 && smem_sm / cta_smem < n) n = smem_sm / cta_smem;
  if (cta_regs > 0 && regs_sm / cta_regs < n) n = regs_sm / cta_regs;
  if (threads_sm / threads < n) n = threads_sm / threads;
  *fit = (int)n;
  return cudaSuccess;
}

template <int MODE, int TILE>
static cudaError_t launch_one(const CUtensorMap* maps, GemmParams& p, int max_tiles, cudaStream_t stream,
                              bool pdl) {
  p.prefetch = pdl ? 1 : 0;
  constexpr size_t smem = gemm_smem_bytes(TILE, MODE == 2 ? 2 : 1);
  auto kern = grouped_gemm_kernel<MODE, TILE>;
  cudaError_t err = ensure_smem_limit(reinterpret_cast<const void*>(kern), (int)smem);
  if (err != cudaSuccess) return err;
  // ctas_per_sm CTAs per SM (all resident at once); CTAs past the live unit
  // count exit at once.
  const long long units =
      (long long)max_tiles * ((MODE != 2 ? p.g[0].rows_w : 0) + (MODE != 1 ? p.g[1].rows_w : 0)) / kWTile;
  long long slots = (long long)ctas_per_sm(p.tile_m) * sm_count();
  if (MODE == 3) {
    // No more CTAs than fit at once (more would only queue behind the
    // resident ones for the tickets).
    int fit = 0;
    err = resident_ctas(reinterpret_cast<const void*>(kern), gemm_threads(MODE, TILE), smem, &fit);
    if (err != cudaSuccess) return err;
    if ((long long)fit * sm_count() < slots) slots = (long long)fit * sm_count();
    if (slots < 1) return cudaErrorInvalidConfiguration;
  }
  const int grid = (int)(units < slots ? units : slots);
  return launch_kernel(kern, dim3(grid), dim3(gemm_threads(MODE, TILE)), smem, stream, pdl, maps[0],
                       maps[1], maps[2], maps[3], p);
}

template <int MODE>
static cudaError_t launch_mode(const CUtensorMap* maps, GemmParams& p, int max_tiles, cudaStream_t stream,
                               bool pdl) {
  switch (p.tile_m) {
    case 32:
      return launch_one<MODE, 32>(maps, p, max_tiles, stream, pdl);
    case 64:
      return launch_one<MODE, 64>(maps, p, max_tiles, stream, pdl);
    case 128:
      return launch_one<MODE, 128>(maps, p, max_tiles, stream, pdl);
    default:
      return launch_one<MODE, 256>(maps, p, max_tiles, stream, pdl);
  }
}

// GEMM1's side: weights p_w13 [E*2I, H/2], route rows a [P, H/2]; writes hq.
static bool gemm1_side(GemmParams& p, CUtensorMap* ta, CUtensorMap* tb, const void* p_w13,
                       const void* p_w13_sf, const float* g1_alphas, const float* g1_scale_c,
                       const uint8_t* a_codes, const uint8_t* a_sf, int E, int H, int I, int tile_m, int P) {
  if (encode_rows_map(ta, p_w13, H / 2, (uint64_t)E * 2 * I, kWTile) != CUDA_SUCCESS ||
      encode_rows_map(tb, a_codes, H / 2, (uint64_t)P, (uint32_t)tile_m) != CUDA_SUCCESS)
    return false;
  p.g[0] = GemmSide{reinterpret_cast<const uint8_t*>(p_w13_sf), a_sf, g1_alphas, g1_scale_c, 2 * I, H, I};
  return true;
}

// GEMM2's side: weights p_w2 [E*H, I/2], route rows hq [P, I/2]; writes bf16 rows.
static bool gemm2_side(GemmParams& p, CUtensorMap* ta, CUtensorMap* tb, const void* p_w2,
                       const void* p_w2_sf, const float* g2_alphas, const uint8_t* h_codes,
                       const uint8_t* h_sf, int E, int H, int I, int tile_m, int P) {
  if (encode_rows_map(ta, p_w2, I / 2, (uint64_t)E * H, kWTile) != CUDA_SUCCESS ||
      encode_rows_map(tb, h_codes, I / 2, (uint64_t)P, (uint32_t)tile_m) != CUDA_SUCCESS)
    return false;
  p.g[1] = GemmSide{reinterpret_cast<const uint8_t*>(p_w2_sf), h_sf, g2_alphas, nullptr, H, I, H};
  return true;
}

bool gemm_pair_fits(int tile_m, int K, int rows_w, int max_tiles);
cudaError_t launch_gemm1_pair(const CUtensorMap& tmW, const CUtensorMap& tmA, const uint8_t* w_sf,
                              const uint8_t* a_sf, const float* g1_alphas, const float* g1_scale_c,
                              const float* a2_gscale, const int32_t* tile_expert, const int32_t* tile_row_limit,
                              const int32_t* totals, uint8_t* hq, uint8_t* hq_sf, int E, int H, int I,
                              int max_tiles, int32_t* status, cudaStream_t stream, bool pdl);

int launch_gemm1(const void* p_w13, const void* p_w13_sf, const float* g1_alphas,
                 const float* g1_scale_c, const float* a2_gscale, const int32_t* tile_expert,
                 const int32_t* tile_row_limit, const int32_t* totals, const uint8_t* a_codes,
                 const uint8_t* a_sf, uint8_t* h_codes, uint8_t* h_sf, int E, int H, int I,
                 int tile_m, int P, int max_tiles, int32_t* status, cudaStream_t stream, bool pdl,
                 const char** why) {
  CUtensorMap maps[4];
  GemmParams p{};
  if (!gemm1_side(p, &maps[0], &maps[1], p_w13, p_w13_sf, g1_alphas, g1_scale_c, a_codes, a_sf, E, H, I,
                  tile_m, P)) {
    *why = "cuTensorMapEncodeTiled failed for GEMM1";
    return MOE_ERR_CUDA;
  }
  // 128-row route tiles whose K and 2I are multiples of 256 (the prefill
  // shapes): the pair form (gemm_pair.cu), 0.637 against 0.695 ms at T = 8192
  if (gemm_pair_fits(tile_m, H, 2 * I, max_tiles)) {
    if (launch_gemm1_pair(maps[0], maps[1], reinterpret_cast<const uint8_t*>(p_w13_sf), a_sf, g1_alphas, g1_scale_c,
                          a2_gscale, tile_expert, tile_row_limit, totals, h_codes, h_sf, E, H, I, max_tiles, status,
                          stream, pdl) != cudaSuccess) {
      *why = "GEMM1 (pair form) launch failed";
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  maps[2] = maps[0];
  maps[3] = maps[1];
  p.tile_expert = tile_expert;
  p.tile_row_limit = tile_row_limit;
  p.totals = totals;
  p.a2_gscale = a2_gscale;
  p.hq = h_codes;
  p.hq_sf = h_sf;
  p.status = status;
  p.tile_m = tile_m;
  if (launch_mode<1>(maps, p, max_tiles, stream, pdl) != cudaSuccess) {
    *why = "GEMM1 launch failed";
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

int launch_gemm2(const void* p_w2, const void* p_w2_sf, const float* g2_alphas,
                 const int32_t* tile_expert, const int32_t* tile_row_limit, const int32_t* totals,
                 const uint8_t* h_codes, const uint8_t* h_sf, void* rows, float* row_ss,
                 const void* ss_gamma, int ss_wbn, int E, int H, int I, int tile_m, int P, int max_tiles,
                 int32_t* status, cudaStream_t stream, bool pdl, const char** why) {
  CUtensorMap maps[4];
  GemmParams p{};
  if (!gemm2_side(p, &maps[2], &maps[3], p_w2, p_w2_sf, g2_alphas, h_codes, h_sf, E, H, I, tile_m, P)) {
    *why = "cuTensorMapEncodeTiled failed for GEMM2";
    return MOE_ERR_CUDA;
  }
  maps[0] = maps[2];
  maps[1] = maps[3];
  const int rows32 = (reinterpret_cast<uintptr_t>(rows) % 32 == 0 && (size_t)H * 2 % 32 == 0) ? 1 : 0;
  // (GEMM2 in the pair form of gemm_pair.cu, measured: 0.457 against 0.432 ms
  // at T = 8192; its 8-stage units expose the accumulator hand-back that the
  // second CTA per SM of this kernel hides)
  p.tile_expert = tile_expert;
  p.tile_row_limit = tile_row_limit;
  p.totals = totals;
  p.rows = reinterpret_cast<__nv_bfloat16*>(rows);
  p.rows32 = rows32;
  p.row_ss = row_ss;
  p.ss_gamma = reinterpret_cast<const __nv_bfloat16*>(ss_gamma);
  p.ss_wbn = ss_wbn;
  p.status = status;
  p.tile_m = tile_m;
  if (launch_mode<2>(maps, p, max_tiles, stream, pdl) != cudaSuccess) {
    *why = "GEMM2 launch failed";
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Both GEMMs in one persistent grid (GEMM2 units of a route tile start once
// its GEMM1 units have stored the intermediate; done[0 .. max_tiles] -- the
// per-tile counters and the unit ticket after them -- must be zero).
int launch_gemms_fused(const void* p_w13, const void* p_w13_sf, const float* g1_alphas,
                       const float* g1_scale_c, const float* a2_gscale, const void* p_w2,
                       const void* p_w2_sf, const float* g2_alphas, const int32_t* tile_expert,
                       const int32_t* tile_row_limit, const int32_t* totals, const uint8_t* a_codes,
                       const uint8_t* a_sf, uint8_t* h_codes, uint8_t* h_sf, void* rows, float* row_ss,
                       const void* ss_gamma, int ss_wbn, int32_t* done, int E, int H, int I, int tile_m, int P,
                       int max_tiles, int32_t* status, cudaStream_t stream, bool pdl, const char** why) {
  CUtensorMap maps[4];
  GemmParams p{};
  if (!gemm1_side(p, &maps[0], &maps[1], p_w13, p_w13_sf, g1_alphas, g1_scale_c, a_codes, a_sf, E, H, I,
                  tile_m, P) ||
      !gemm2_side(p, &maps[2], &maps[3], p_w2, p_w2_sf, g2_alphas, h_codes, h_sf, E, H, I, tile_m, P)) {
    *why = "cuTensorMapEncodeTiled failed for the expert GEMMs";
    return MOE_ERR_CUDA;
  }
  p.tile_expert = tile_expert;
  p.tile_row_limit = tile_row_limit;
  p.totals = totals;
  p.a2_gscale = a2_gscale;
  p.hq = h_codes;
  p.hq_sf = h_sf;
  p.rows = reinterpret_cast<__nv_bfloat16*>(rows);
  p.rows32 = (reinterpret_cast<uintptr_t>(rows) % 32 == 0 && (size_t)H * 2 % 32 == 0) ? 1 : 0;
  p.row_ss = row_ss;
  p.ss_gamma = reinterpret_cast<const __nv_bfloat16*>(ss_gamma);
  p.ss_wbn = ss_wbn;
  p.done = done;
  p.ticket = done + max_tiles;
  p.num_experts = E;
  p.max_tiles = max_tiles;
  p.w_evict_first = 1;
  p.status = status;
  p.tile_m = tile_m;
  if (launch_mode<3>(maps, p, max_tiles, stream, pdl) != cudaSuccess) {
    *why = "expert GEMM launch failed";
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
