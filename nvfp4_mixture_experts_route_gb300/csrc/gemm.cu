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
// rows are permuted route rows of one routing tile (all of one expert). One
// CTA computes one (route tile tau, weight tile mt) pair over the whole K:
//   - warp 0 / lane 0: TMA producer. Per pipeline stage (K = 256 elements =
//     128 bytes per row): the 128 x 128 B weight box, the tile_m x 128 B
//     route box (both 128-byte swizzled), and the stage's scale atoms for both
//     operands with plain bulk copies; one mbarrier with a transaction count.
//   - warp 1 / lane 0: MMA issuer. Copies the stage's scale atoms into tensor
//     memory (tcgen05.cp 32x128b.warpx4; each stage has its own columns, so a
//     refill can never race an MMA still reading them), issues 4 MMAs of
//     K = 64 accumulating into TMEM columns [0, tile_m), and commits the stage
//     back to the producer.
//   - all 4 warps: epilogue. Warp w reads TMEM lanes [32w, 32w+32) (weight
//     rows) for every route column.
// The grid is (route tiles, weight tiles) with route tiles fastest, so the
// CTAs that share an expert's weight tile run side by side and the second
// reads it from L2. Tiles past the live count (totals[0]) exit at once.
//
// The prepared w13 interleaves gate and up rows in 16-row granules, so a
// warp's 32 lanes hold gate (lanes 0-15) and up (lanes 16-31) of the same 16
// intermediate columns: SwiGLU is one shuffle, the NVFP4 block amax four.
//
// Every mbarrier wait is bounded (1 s); on a timeout the CTA records
// MOE_ERR_TIMEOUT, drains its own copies and MMAs (bounded again), frees its
// tensor memory and exits.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "layout.cuh"

namespace moe {

constexpr int kStageK = 256;                   // K elements per pipeline stage
constexpr int kStageRowBytes = kStageK / 2;    // 128
constexpr int kWTile = 128;                    // weight rows per CTA (MMA M)
constexpr uint32_t kABytes = kWTile * kStageRowBytes;  // 16 KiB
constexpr uint32_t kSfStageBytes = 4 * kAtomBytes;     // 4 K=64 steps

struct GemmParams {
  const uint8_t* w_sf;  // prepared scale atoms [E][rows_w/128][K/64][512]
  const uint8_t* b_sf;  // workspace scale atoms [tiles][K/64][S][512]
  const int32_t* tile_expert;
  const int32_t* tile_row_limit;
  const int32_t* totals;
  const float* s0;         // g1_alphas (GEMM1) or g2_alphas (GEMM2)
  const float* s1;         // g1_scale_c (GEMM1)
  const float* a2_gscale;  // GEMM1
  uint8_t* hq;             // GEMM1: intermediate codes [P][I/2]
  uint8_t* hq_sf;          // GEMM1: intermediate scale atoms [tiles][I/64][S][512]
  __nv_bfloat16* rows;     // GEMM2: [P][H]
  int32_t* status;
  int E, rows_w, K, tile_m, S, out_cols;
};

__host__ __device__ constexpr uint32_t tmem_cols_for(int tile_m, int S, int stages) {
  const int need = tile_m + stages * 16 * (1 + S);
  uint32_t c = 32;
  while ((int)c < need) c <<= 1;
  return c;
}

__host__ __device__ constexpr size_t gemm_smem_bytes(int tile_m, int S, int stages) {
  return 1024 + (size_t)stages * (kABytes + (size_t)tile_m * kStageRowBytes +
                                  kSfStageBytes * (size_t)(1 + S));
}

// SwiGLU + NVFP4 requant of one route column; lanes 0-15 carry the gate and
// lanes 16-31 the up rows of 16 intermediate columns.
__device__ __forceinline__ void gemm1_column(float v, float sc, float a2g, int lane, uint8_t* hq_row,
                                             uint8_t* hq_sf_byte) {
  const float x = v * sc;
  const float o = __shfl_xor_sync(0xffffffffu, x, 16);
  const float gate = lane < 16 ? x : o;
  const float up = lane < 16 ? o : x;
  const float h = gate / (1.0f + expf(-gate)) * up;
  float a = fabsf(h);
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 8));
  const float s = (a * a2g) / 6.0f;
  const uint32_t sfc = f32_to_e4m3(s);
  const float sfv = e4m3_to_f32(sfc);
  const float inv = sfv > 0.f ? a2g / sfv : 0.f;
  const float t = h * inv;
  const float tn = __shfl_down_sync(0xffffffffu, t, 1);
  uint32_t byte = f32x2_to_e2m1x2(t, tn);
  if (!(sfv > 0.f)) byte = 0;
  const bool even = !(lane & 1);
  uint32_t lo = (even && lane < 8) ? byte << (8 * (lane >> 1)) : 0u;
  uint32_t hi = (even && lane >= 8 && lane < 16) ? byte << (8 * ((lane - 8) >> 1)) : 0u;
  lo |= __shfl_xor_sync(0xffffffffu, lo, 2);
  hi |= __shfl_xor_sync(0xffffffffu, hi, 2);
  lo |= __shfl_xor_sync(0xffffffffu, lo, 4);
  hi |= __shfl_xor_sync(0xffffffffu, hi, 4);
  lo |= __shfl_xor_sync(0xffffffffu, lo, 8);
  hi |= __shfl_xor_sync(0xffffffffu, hi, 8);
  if (lane == 0) {
    *reinterpret_cast<uint2*>(hq_row) = make_uint2(lo, hi);
    *hq_sf_byte = static_cast<uint8_t>(sfc);
  }
}

template <int KIND, int ST>
__global__ void __launch_bounds__(128, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  extern __shared__ uint8_t dsmem[];
  __shared__ __align__(8) uint64_t full_bar[ST];
  __shared__ __align__(8) uint64_t empty_bar[ST];
  __shared__ __align__(8) uint64_t acc_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tau = blockIdx.x, mt = blockIdx.y;
  if (tau >= p.totals[0]) return;
  const int e = p.tile_expert[tau];
  if (e < 0 || e >= p.E) {
    if (tid == 0) record_status(p.status, MOE_ERR_INVALID_ROUTE);
    return;
  }

  const int tile_m = p.tile_m, S = p.S;
  const uint32_t b_bytes = (uint32_t)tile_m * kStageRowBytes;
  const uint32_t sbase = (smem_u32(dsmem) + 1023u) & ~1023u;
  const uint32_t sA = sbase;
  const uint32_t sB = sA + ST * kABytes;
  const uint32_t sSFA = sB + ST * b_bytes;
  const uint32_t sSFB = sSFA + ST * kSfStageBytes;
  const int KC = p.K / 64;
  const int nks = (KC + 3) / 4;
  const uint32_t ncols = tmem_cols_for(tile_m, S, ST);

  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    mbar_init(smem_u32(&acc_bar), 1);
    abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&tmem_slot), ncols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t t_sfa = tmem + (uint32_t)tile_m;
  const uint32_t t_sfb = t_sfa + ST * 16;

  if (warp == 0) {
    if (lane == 0) {
      const int a_row = e * p.rows_w + mt * kWTile;
      const uint8_t* wsf = p.w_sf + ((size_t)e * (p.rows_w / kWTile) + mt) * KC * kAtomBytes;
      const uint8_t* bsf = p.b_sf + (size_t)tau * KC * S * kAtomBytes;
      int issued = 0;
      for (int ks = 0; ks < nks; ++ks) {
        const int s = ks % ST, round = ks / ST;
        if (round > 0 &&
            !mbar_wait(smem_u32(&empty_bar[s]), (round - 1) & 1, &abort_flag, p.status))
          break;
        const int kk = min(4, KC - 4 * ks);
        const uint32_t fb = smem_u32(&full_bar[s]);
        mbar_arrive_expect_tx(fb, kABytes + b_bytes + (uint32_t)kk * kAtomBytes * (1 + S));
        tma_load_2d(sA + s * kABytes, &tmA, fb, ks * kStageRowBytes, a_row);
        tma_load_2d(sB + s * b_bytes, &tmB, fb, ks * kStageRowBytes, tau * tile_m);
        bulk_load(sSFA + s * kSfStageBytes, wsf + (size_t)4 * ks * kAtomBytes,
                  (uint32_t)kk * kAtomBytes, fb);
        bulk_load(sSFB + s * kSfStageBytes * S, bsf + (size_t)4 * ks * S * kAtomBytes,
                  (uint32_t)kk * S * kAtomBytes, fb);
        ++issued;
      }
      // Wait for the copies still in flight (normally all landed already).
      for (int ks = max(0, issued - ST); ks < issued; ++ks)
        mbar_wait_cleanup(smem_u32(&full_bar[ks % ST]), (ks / ST) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = idesc_nvf4(kWTile, (uint32_t)tile_m);
      for (int ks = 0; ks < nks; ++ks) {
        const int s = ks % ST, round = ks / ST;
        if (!mbar_wait(smem_u32(&full_bar[s]), round & 1, &abort_flag, p.status)) break;
        tc_fence_after();
        const int kk = min(4, KC - 4 * ks);
        const uint32_t fa = t_sfa + s * 16, fbc = t_sfb + s * 16 * S;
        const uint32_t sfa_smem = sSFA + s * kSfStageBytes;
        const uint32_t sfb_smem = sSFB + s * kSfStageBytes * S;
        for (int j = 0; j < kk; ++j) {
          tc_copy_scale_atom(fa + 4 * j, smem_desc(sfa_smem + j * kAtomBytes, 0, 128, 0));
          for (int sub = 0; sub < S; ++sub)
            tc_copy_scale_atom(fbc + 4 * (j * S + sub),
                               smem_desc(sfb_smem + (j * S + sub) * kAtomBytes, 0, 128, 0));
        }
        for (int j = 0; j < kk; ++j) {
          const uint64_t ad = smem_desc(sA + s * kABytes + 32 * j, 16, 1024, 2);
          const uint64_t bd = smem_desc(sB + s * b_bytes + 32 * j, 16, 1024, 2);
          tc_mma_nvf4(tmem, ad, bd, idesc, fa + 4 * j, fbc + 4 * j * S, (ks | j) != 0);
        }
        tc_commit(smem_u32(&empty_bar[s]));
      }
      tc_commit(smem_u32(&acc_bar));
    }
    __syncwarp();
  }

  // ---------------- epilogue: TMEM -> registers -> global ----------------
  const bool ok = mbar_wait(smem_u32(&acc_bar), 0, &abort_flag, p.status);
  __syncwarp();  // the tcgen05.ld below are warp-collective
  tc_fence_after();
  if (ok && !abort_flag) {
    const uint32_t taddr = tmem + ((uint32_t)(32 * warp) << 16);
    const int row0 = tau * tile_m;
    if (KIND == 1) {
      const float sc = lane < 16 ? p.s0[e] : p.s1[e];
      const float a2g = *p.a2_gscale;
      const int I = p.out_cols, kco = I / 64;
      const int kb = 4 * mt + warp;  // intermediate 16-block of this warp
      for (int c0 = 0; c0 < tile_m; c0 += 16) {
        float v[16];
        tmem_ld16(taddr + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = row0 + c0 + i;
          gemm1_column(v[i], sc, a2g, lane, p.hq + (size_t)r * (I / 2) + 32 * mt + 8 * warp,
                       p.hq_sf + act_sf_offset(r, kb, tile_m, kco, S));
        }
      }
    } else {
      const float g2 = p.s0[e];
      const int limit = p.tile_row_limit[tau];
      const int col = mt * kWTile + 32 * warp + lane;
      for (int c0 = 0; c0 < tile_m; c0 += 16) {
        float v[16];
        tmem_ld16(taddr + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int r = row0 + c0 + i;
          if (r < limit) p.rows[(size_t)r * p.out_cols + col] = __float2bfloat16_rn(v[i] * g2);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    // Every MMA this CTA issued has completed once acc_bar has (it tracks all
    // of them); normally this returns at once.
    mbar_wait_cleanup(smem_u32(&acc_bar), 0);
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, ncols);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch.
// ---------------------------------------------------------------------------
// cuTensorMapEncodeTiled is a driver API entry; it is looked up through the
// runtime so that the library does not link libcuda (and loads on hosts
// without a driver). The lookup is done once per process.
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }();
  return fn;
}

static CUresult encode_rows_map(CUtensorMap* map, const void* base, uint64_t row_bytes,
                                uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)kStageRowBytes, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

constexpr int kStages = 4;

template <int KIND>
static cudaError_t launch_one(const CUtensorMap& ta, const CUtensorMap& tb, const GemmParams& p,
                              int max_tiles, cudaStream_t stream) {
  const size_t smem = gemm_smem_bytes(p.tile_m, p.S, kStages);
  auto kern = grouped_gemm_kernel<KIND, kStages>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  dim3 grid(max_tiles, p.rows_w / kWTile);
  kern<<<grid, 128, smem, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

// GEMM1: weights p_w13 [E*2I, H/2], route rows a [P, H/2]; writes hq.
int launch_gemm1(const void* p_w13, const void* p_w13_sf, const float* g1_alphas,
                 const float* g1_scale_c, const float* a2_gscale, const int32_t* tile_expert,
                 const int32_t* tile_row_limit, const int32_t* totals, const uint8_t* a_codes,
                 const uint8_t* a_sf, uint8_t* h_codes, uint8_t* h_sf, int E, int H, int I,
                 int tile_m, int P, int max_tiles, int32_t* status, cudaStream_t stream,
                 const char** why) {
  CUtensorMap ta, tb;
  if (encode_rows_map(&ta, p_w13, H / 2, (uint64_t)E * 2 * I, kWTile) != CUDA_SUCCESS ||
      encode_rows_map(&tb, a_codes, H / 2, (uint64_t)P, (uint32_t)tile_m) != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled failed for GEMM1";
    return MOE_ERR_CUDA;
  }
  GemmParams p{};
  p.w_sf = reinterpret_cast<const uint8_t*>(p_w13_sf);
  p.b_sf = a_sf;
  p.tile_expert = tile_expert;
  p.tile_row_limit = tile_row_limit;
  p.totals = totals;
  p.s0 = g1_alphas;
  p.s1 = g1_scale_c;
  p.a2_gscale = a2_gscale;
  p.hq = h_codes;
  p.hq_sf = h_sf;
  p.status = status;
  p.E = E;
  p.rows_w = 2 * I;
  p.K = H;
  p.tile_m = tile_m;
  p.S = sf_atoms_per_tile(tile_m);
  p.out_cols = I;
  if (launch_one<1>(ta, tb, p, max_tiles, stream) != cudaSuccess) {
    *why = "GEMM1 launch failed";
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// GEMM2: weights p_w2 [E*H, I/2], route rows hq [P, I/2]; writes bf16 rows.
int launch_gemm2(const void* p_w2, const void* p_w2_sf, const float* g2_alphas,
                 const int32_t* tile_expert, const int32_t* tile_row_limit, const int32_t* totals,
                 const uint8_t* h_codes, const uint8_t* h_sf, void* rows, int E, int H, int I,
                 int tile_m, int P, int max_tiles, int32_t* status, cudaStream_t stream,
                 const char** why) {
  CUtensorMap ta, tb;
  if (encode_rows_map(&ta, p_w2, I / 2, (uint64_t)E * H, kWTile) != CUDA_SUCCESS ||
      encode_rows_map(&tb, h_codes, I / 2, (uint64_t)P, (uint32_t)tile_m) != CUDA_SUCCESS) {
    *why = "cuTensorMapEncodeTiled failed for GEMM2";
    return MOE_ERR_CUDA;
  }
  GemmParams p{};
  p.w_sf = reinterpret_cast<const uint8_t*>(p_w2_sf);
  p.b_sf = h_sf;
  p.tile_expert = tile_expert;
  p.tile_row_limit = tile_row_limit;
  p.totals = totals;
  p.s0 = g2_alphas;
  p.rows = reinterpret_cast<__nv_bfloat16*>(rows);
  p.status = status;
  p.E = E;
  p.rows_w = H;
  p.K = I;
  p.tile_m = tile_m;
  p.S = sf_atoms_per_tile(tile_m);
  p.out_cols = H;
  if (launch_one<2>(ta, tb, p, max_tiles, stream) != cudaSuccess) {
    *why = "GEMM2 launch failed";
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
