// The extern "C" entry points of libmoe_nvfp4.so (declared and documented in
// include/moe_nvfp4.h): host-side argument checks, the workspace layout, and
// the kernel launches on the caller's stream.
#include <cstdarg>
#include <cstdio>
#include <string>

#include "common.cuh"
#include "layout.cuh"

namespace moe {
cudaError_t launch_route_permute(const int32_t*, int, int, int, int, int, int, int32_t*, int32_t*,
                                 int32_t*, int32_t*, int32_t*, int32_t*, int32_t*, int32_t*,
                                 cudaStream_t);
size_t route_smem_bytes(int E);
int route_kernel_count(int T, int K, int E);
cudaError_t launch_quantize_permute(const void*, const void*, const void*, const float*,
                                    const int32_t*, const int32_t*, const int32_t*, int, int, int,
                                    int, int, int, uint8_t*, uint8_t*, int32_t*, int32_t*, cudaStream_t);
cudaError_t launch_act_scales_io(int, uint8_t*, uint8_t*, int, int, int, cudaStream_t);
bool route_quantize_fits(int T, int K, int E);
cudaError_t launch_route_quantize(const int32_t*, int, int, int, int, int, int, int32_t*, int32_t*, int32_t*,
                                  int32_t*, int32_t*, int32_t*, int32_t*, const void*, const void*, const void*,
                                  const float*, int, uint8_t*, uint8_t*, int32_t*, int32_t*, cudaStream_t);
cudaError_t launch_prepare_weights(const void*, const void*, const void*, const void*, int, int,
                                   int, void*, void*, void*, void*, cudaStream_t);
cudaError_t launch_finalize(const void*, int, const int32_t*, const float*, const void*, float, int,
                            int, int, int, void*, int32_t*, cudaStream_t);
cudaError_t launch_finalize_parts(const void* const*, int, int, const int32_t*, const float*, const void*,
                                  float, int, int, int, int, void*, int32_t*, cudaStream_t);
cudaError_t launch_musespark1x_routing(const float*, const float*, const uint8_t*, int, int, int, float,
                                       float, int32_t*, float*, cudaStream_t);
cudaError_t launch_rmsnorm_nvfp4(const void*, const void*, float, const float*, int, int, void*, void*,
                                 cudaStream_t);
cudaError_t launch_rmsnorm_nvfp4_permuted(const void*, const void*, float, const float*, const int32_t*,
                                          const int32_t*, const int32_t*, const int32_t*, int, int, int, int, int,
                                          int, uint8_t*, uint8_t*, cudaStream_t);
int launch_gemm1(const void*, const void*, const float*, const float*, const float*,
                 const int32_t*, const int32_t*, const int32_t*, const uint8_t*, const uint8_t*,
                 uint8_t*, uint8_t*, int, int, int, int, int, int, int32_t*, cudaStream_t, bool,
                 const char**);
int launch_gemm2(const void*, const void*, const float*, const int32_t*, const int32_t*,
                 const int32_t*, const uint8_t*, const uint8_t*, void*, float*, const void*, int, int, int,
                 int, int, int, int, int32_t*, cudaStream_t, bool, const char**);
int launch_gemms_fused(const void*, const void*, const float*, const float*, const float*, const void*,
                       const void*, const float*, const int32_t*, const int32_t*, const int32_t*,
                       const uint8_t*, const uint8_t*, uint8_t*, uint8_t*, void*, float*, const void*, int,
                       int32_t*, int, int, int, int, int, int, int32_t*, cudaStream_t, bool, const char**);
cudaError_t launch_finalize_sumsq(const void*, const float*, int, const int32_t*, const float*, const void*,
                                  float, int, int, int, void*, int32_t*, cudaStream_t);
int launch_dense_bf16(const void*, const void*, int, int, int, void*, void*, int32_t*, cudaStream_t,
                      const char**);
size_t dense_workspace_here(int, int, int);
int launch_selftest_wait(uint64_t, int32_t*, int32_t*, cudaStream_t);
int launch_selftest_counter(uint64_t, const int32_t*, int32_t*, int32_t*, cudaStream_t);
int launch_selftest_occupy(int, int, uint64_t, cudaStream_t);
}  // namespace moe

namespace {

thread_local std::string g_last_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t err, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(err));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_tile(int tile_m) {
  return tile_m == 32 || tile_m == 64 || tile_m == 128 || tile_m == 256;
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct RouteDims {
  int P = 0, MT = 0;
};

int route_dims(int T, int K, int E, int tile_m, RouteDims* d) {
  if (T < 0 || K < 1 || K > 64 || E < 1 || E > 1024)
    return fail(MOE_ERR_INVALID_ARG, "bad routing shape T=%d K=%d E=%d", T, K, E);
  if (!valid_tile(tile_m)) return fail(MOE_ERR_UNSUPPORTED, "tile_m %d not in {32,64,128,256}", tile_m);
  const long long R = (long long)T * K;
  if (R > (1ll << 24)) return fail(MOE_ERR_UNSUPPORTED, "too many routes (%lld)", R);
  const long long F = R < E ? R : E;
  const long long P = (long long)tile_m * (F + (R - F) / tile_m);
  d->P = (int)P;
  d->MT = (int)(P / tile_m);
  return MOE_OK;
}

// Workspace of the expert body: permuted NVFP4 activations and the quantized
// intermediate (codes row-major, scales as per-tile atoms; see quant.cu).
// Counters after the per-route-tile ones: the one-launch GEMMs' unit ticket.
constexpr int kDoneExtra = 1;

struct WsLayout {
  size_t a_codes = 0, a_sf = 0, h_codes = 0, h_sf = 0, done = 0, total = 0;
  int P = 0, MT = 0;
};

int ws_layout(int T, int K, int E, int H, int I, int tile_m, WsLayout* w) {
  RouteDims d;
  int rc = route_dims(T, K, E, tile_m, &d);
  if (rc) return rc;
  if (H < 128 || I < 64 || H % 128 || I % 64)
    return fail(MOE_ERR_UNSUPPORTED, "hidden %d and intermediate %d must be multiples of 128 and 64", H, I);
  w->P = d.P;
  w->MT = d.MT;
  const size_t S = (size_t)moe::sf_atoms_per_tile(tile_m);
  size_t off = 0;
  w->a_codes = off;
  off = round_up(off + (size_t)d.P * (H / 2), 1024);
  w->a_sf = off;
  off = round_up(off + (size_t)d.MT * (H / 64) * S * moe::kAtomBytes, 1024);
  w->h_codes = off;
  off = round_up(off + (size_t)d.P * (I / 2), 1024);
  w->h_sf = off;
  off = round_up(off + (size_t)d.MT * (I / 64) * S * moe::kAtomBytes, 1024);
  // per route tile: GEMM1 completions the fused GEMM2 units wait for, then
  // the fused GEMMs' unit ticket
  w->done = off;
  off = round_up(off + (size_t)(d.MT + kDoneExtra) * sizeof(int32_t), 1024);
  w->total = off;
  return MOE_OK;
}

int check_ws(const void* ws, size_t ws_bytes, const WsLayout& L) {
  if (L.total && ws == nullptr) return fail(MOE_ERR_INVALID_ARG, "workspace is null");
  if (!aligned(ws, 1024)) return fail(MOE_ERR_INVALID_ARG, "workspace must be 1024-byte aligned");
  if (ws_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE, "workspace %zu bytes, need %zu", ws_bytes, L.total);
  return MOE_OK;
}

int check_route(const moe_route* r) {
  if (!r || !r->permuted_to_token || !r->tile_expert || !r->tile_row_limit || !r->totals)
    return fail(MOE_ERR_INVALID_ARG, "routing metadata pointer is null");
  return MOE_OK;
}

int check_weights(const moe_weights* w, bool gemm1) {
  if (!w) return fail(MOE_ERR_INVALID_ARG, "weights are null");
  if (gemm1) {
    if (!w->w13 || !w->w13_sf || !w->g1_alphas || !w->g1_scale_c)
      return fail(MOE_ERR_INVALID_ARG, "GEMM1 weight pointer is null");
    if (!aligned(w->w13, 16) || !aligned(w->w13_sf, 16))
      return fail(MOE_ERR_INVALID_ARG, "w13 / w13_sf must be 16-byte aligned");
  } else {
    if (!w->w2 || !w->w2_sf || !w->g2_alphas)
      return fail(MOE_ERR_INVALID_ARG, "GEMM2 weight pointer is null");
    if (!aligned(w->w2, 16) || !aligned(w->w2_sf, 16))
      return fail(MOE_ERR_INVALID_ARG, "w2 / w2_sf must be 16-byte aligned");
  }
  return MOE_OK;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

namespace moe {
// Record an error for moe_last_error() from another translation unit.
int report_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}
}  // namespace moe

extern "C" {

const char* moe_last_error(void) { return g_last_error.c_str(); }

int moe_abi_version(void) { return 5; }

int moe_device_reads_host(const void* p) {
  if (!p) return 0;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // an unregistered pointer is an answer, not an error
    return 0;
  }
  return (a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeManaged) && a.devicePointer == p ? 1 : 0;
}

int moe_prepared_sizes(int E, int H, int I, size_t out_bytes[4]) {
  if (!out_bytes) return fail(MOE_ERR_INVALID_ARG, "out_bytes is null");
  if (E < 1 || H < 1 || I < 1) return fail(MOE_ERR_INVALID_ARG, "bad shape E=%d H=%d I=%d", E, H, I);
  if (H % 128 || I % 64)
    return fail(MOE_ERR_UNSUPPORTED, "hidden %d and intermediate %d must be multiples of 128 and 64",
                H, I);
  out_bytes[0] = (size_t)E * 2 * I * (H / 2);
  out_bytes[1] = (size_t)E * 2 * I * (H / 16);
  out_bytes[2] = (size_t)E * H * (I / 2);
  out_bytes[3] = (size_t)E * H * (I / 16);
  return MOE_OK;
}

int moe_prepare_weights(const void* w13, const void* w13_sf, const void* w2, const void* w2_sf,
                        int E, int H, int I, void* p_w13, void* p_w13_sf, void* p_w2,
                        void* p_w2_sf, void* stream) {
  size_t sz[4];
  int rc = moe_prepared_sizes(E, H, I, sz);
  if (rc) return rc;
  const void* ptrs[8] = {w13, w13_sf, w2, w2_sf, p_w13, p_w13_sf, p_w2, p_w2_sf};
  for (const void* p : ptrs) {
    if (!p) return fail(MOE_ERR_INVALID_ARG, "weight pointer is null");
    if (!aligned(p, 16)) return fail(MOE_ERR_INVALID_ARG, "weight pointers must be 16-byte aligned");
  }
  cudaError_t err = moe::launch_prepare_weights(w13, w13_sf, w2, w2_sf, E, H, I, p_w13, p_w13_sf,
                                                p_w2, p_w2_sf, as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_prepare_weights");
}

int moe_route_sizes(int T, int K, int E, int tile_m, int* max_padded_rows, int* max_tiles) {
  RouteDims d;
  int rc = route_dims(T, K, E, tile_m, &d);
  if (rc) return rc;
  if (max_padded_rows) *max_padded_rows = d.P;
  if (max_tiles) *max_tiles = d.MT;
  return MOE_OK;
}

int moe_route_kernels(int T, int K, int E) {
  RouteDims d;
  int rc = route_dims(T, K, E, 32, &d);
  if (rc) return rc;
  return moe::route_kernel_count(T, K, E);
}

int moe_experts_kernels(int tile_m) {
  if (tile_m != 32 && tile_m != 64 && tile_m != 128 && tile_m != 256)
    return fail(MOE_ERR_UNSUPPORTED, "tile_m must be 32, 64, 128 or 256");
  return tile_m <= 64 ? 2 : 3;
}

int moe_route_permute(const int32_t* topk_ids, int T, int K, int E, int tile_m,
                      int32_t* expert_counts, int32_t* expert_offsets,
                      int32_t* expanded_to_permuted, int32_t* permuted_to_token,
                      int32_t* tile_expert, int32_t* tile_row_limit, int32_t* totals,
                      int32_t* status, void* stream) {
  RouteDims d;
  int rc = route_dims(T, K, E, tile_m, &d);
  if (rc) return rc;
  if (!expert_counts || !expert_offsets || !totals || (T > 0 && (!topk_ids || !expanded_to_permuted)) ||
      (d.P > 0 && (!permuted_to_token || !tile_expert || !tile_row_limit)))
    return fail(MOE_ERR_INVALID_ARG, "routing buffer is null");
  cudaError_t err = moe::launch_route_permute(topk_ids, T, K, E, tile_m, d.P, d.MT, expert_counts,
                                              expert_offsets, expanded_to_permuted,
                                              permuted_to_token, tile_expert, tile_row_limit,
                                              totals, status, as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_route_permute");
}

int moe_experts_workspace_size(int T, int K, int E, int H, int I, int tile_m, size_t* ws_bytes) {
  WsLayout L;
  int rc = ws_layout(T, K, E, H, I, tile_m, &L);
  if (rc) return rc;
  if (!ws_bytes) return fail(MOE_ERR_INVALID_ARG, "ws_bytes is null");
  *ws_bytes = L.total;
  return MOE_OK;
}

int moe_experts_quantize(const void* x, const void* a, const void* a_sf, const float* a1_gscale,
                         const moe_route* r, int T, int H, int I, int E, int K, int tile_m,
                         void* ws, size_t ws_bytes, int32_t* status, void* stream) {
  WsLayout L;
  int rc = ws_layout(T, K, E, H, I, tile_m, &L);
  if (rc) return rc;
  if ((rc = check_ws(ws, ws_bytes, L)) || (rc = check_route(r))) return rc;
  if (L.P == 0) return MOE_OK;
  if (x) {
    if (!a1_gscale) return fail(MOE_ERR_INVALID_ARG, "a1_gscale is null");
    if (!aligned(x, 16)) return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
  } else {
    if (!a || !a_sf) return fail(MOE_ERR_INVALID_ARG, "give x, or a and a_sf");
    if (!aligned(a, 16) || !aligned(a_sf, 4))
      return fail(MOE_ERR_INVALID_ARG, "a must be 16-byte and a_sf 4-byte aligned");
  }
  if (!r->expanded_to_permuted) return fail(MOE_ERR_INVALID_ARG, "route expanded_to_permuted is null");
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  cudaError_t err = moe::launch_quantize_permute(
      x, x ? nullptr : a, x ? nullptr : a_sf, a1_gscale, r->expanded_to_permuted, r->tile_row_limit,
      r->totals, T, K, H, tile_m, L.P, L.MT + kDoneExtra, base + L.a_codes, base + L.a_sf,
      reinterpret_cast<int32_t*>(base + L.done), status, as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_experts_quantize");
}

// pdl: launch the GEMM as a programmatic dependent of the kernel before it,
// which must be this library's own step kernel launched in the same call
// (the GEMM then loads weights before that kernel has completed).
static int experts_gemm1(const moe_weights* w, const float* a2_gscale, const moe_route* r, int T,
                         int H, int I, int E, int K, int tile_m, void* ws, size_t ws_bytes,
                         int32_t* status, void* stream, bool pdl) {
  WsLayout L;
  int rc = ws_layout(T, K, E, H, I, tile_m, &L);
  if (rc) return rc;
  if ((rc = check_ws(ws, ws_bytes, L)) || (rc = check_route(r)) || (rc = check_weights(w, true)))
    return rc;
  if (!a2_gscale) return fail(MOE_ERR_INVALID_ARG, "a2_gscale is null");
  if (L.P == 0) return MOE_OK;
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  const char* why = "";
  rc = moe::launch_gemm1(w->w13, w->w13_sf, w->g1_alphas, w->g1_scale_c, a2_gscale, r->tile_expert,
                         r->tile_row_limit, r->totals, base + L.a_codes, base + L.a_sf,
                         base + L.h_codes, base + L.h_sf, E, H, I, tile_m, L.P, L.MT, status,
                         as_stream(stream), pdl, &why);
  return rc ? fail(rc, "%s", why) : MOE_OK;
}

int moe_experts_gemm1(const moe_weights* w, const float* a2_gscale, const moe_route* r, int T,
                      int H, int I, int E, int K, int tile_m, void* ws, size_t ws_bytes,
                      int32_t* status, void* stream) {
  return experts_gemm1(w, a2_gscale, r, T, H, I, E, K, tile_m, ws, ws_bytes, status, stream, false);
}

// The post-expert norm's sums of squares, fused into GEMM2's epilogue when
// row_ss is set (gamma and the norm reading then given too).
struct SumSq {
  float* row_ss = nullptr;
  const void* gamma = nullptr;
  int wbn = 0;
};

static int experts_gemm2(const moe_weights* w, const moe_route* r, int T, int H, int I, int E,
                         int K, int tile_m, void* gemm2_rows, void* ws, size_t ws_bytes,
                         int32_t* status, void* stream, bool pdl, SumSq ss = SumSq()) {
  WsLayout L;
  int rc = ws_layout(T, K, E, H, I, tile_m, &L);
  if (rc) return rc;
  if ((rc = check_ws(ws, ws_bytes, L)) || (rc = check_route(r)) || (rc = check_weights(w, false)))
    return rc;
  if (L.P == 0) return MOE_OK;
  if (!gemm2_rows || !aligned(gemm2_rows, 16))
    return fail(MOE_ERR_INVALID_ARG, "gemm2_rows must be non-null and 16-byte aligned");
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  const char* why = "";
  rc = moe::launch_gemm2(w->w2, w->w2_sf, w->g2_alphas, r->tile_expert, r->tile_row_limit,
                         r->totals, base + L.h_codes, base + L.h_sf, gemm2_rows, ss.row_ss, ss.gamma, ss.wbn, E,
                         H, I, tile_m, L.P, L.MT, status, as_stream(stream), pdl, &why);
  return rc ? fail(rc, "%s", why) : MOE_OK;
}

int moe_experts_gemm2(const moe_weights* w, const moe_route* r, int T, int H, int I, int E, int K,
                      int tile_m, void* gemm2_rows, void* ws, size_t ws_bytes, int32_t* status,
                      void* stream) {
  return experts_gemm2(w, r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes, status, stream, false);
}

// Both GEMMs as one persistent grid. pdl as for the split GEMMs;
// zero_counters: clear the per-tile completion counters and the unit ticket
// first (one memset; the quantizer already leaves them zero inside
// moe_nvfp4_experts).
static int experts_fused(const moe_weights* w, const float* a2_gscale, const moe_route* r, int T, int H,
                         int I, int E, int K, int tile_m, void* gemm2_rows, void* ws, size_t ws_bytes,
                         int32_t* status, void* stream, bool pdl, bool zero_counters, SumSq ss = SumSq()) {
  WsLayout L;
  int rc = ws_layout(T, K, E, H, I, tile_m, &L);
  if (rc) return rc;
  if ((rc = check_ws(ws, ws_bytes, L)) || (rc = check_route(r)) || (rc = check_weights(w, true)) ||
      (rc = check_weights(w, false)))
    return rc;
  if (!a2_gscale) return fail(MOE_ERR_INVALID_ARG, "a2_gscale is null");
  if (L.P == 0) return MOE_OK;
  if (!gemm2_rows || !aligned(gemm2_rows, 16))
    return fail(MOE_ERR_INVALID_ARG, "gemm2_rows must be non-null and 16-byte aligned");
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  if (zero_counters) {
    const cudaError_t err =
        cudaMemsetAsync(base + L.done, 0, (size_t)(L.MT + kDoneExtra) * sizeof(int32_t), as_stream(stream));
    if (err != cudaSuccess) return cuda_fail(err, "moe_experts_gemms");
  }
  const char* why = "";
  rc = moe::launch_gemms_fused(w->w13, w->w13_sf, w->g1_alphas, w->g1_scale_c, a2_gscale, w->w2, w->w2_sf,
                               w->g2_alphas, r->tile_expert, r->tile_row_limit, r->totals,
                               base + L.a_codes, base + L.a_sf, base + L.h_codes, base + L.h_sf, gemm2_rows,
                               ss.row_ss, ss.gamma, ss.wbn, reinterpret_cast<int32_t*>(base + L.done), E, H, I,
                               tile_m, L.P, L.MT, status,
                               as_stream(stream), pdl, &why);
  return rc ? fail(rc, "%s", why) : MOE_OK;
}

int moe_experts_gemms(const moe_weights* w, const float* a2_gscale, const moe_route* r, int T, int H,
                      int I, int E, int K, int tile_m, void* gemm2_rows, void* ws, size_t ws_bytes,
                      int32_t* status, void* stream) {
  return experts_fused(w, a2_gscale, r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes, status, stream,
                       false, true);
}

static int experts_body(const moe_weights* w, const void* x, const void* a, const void* a_sf,
                        const float* a1_gscale, const float* a2_gscale, const moe_route* r, int T, int H,
                        int I, int E, int K, int tile_m, void* gemm2_rows, void* ws, size_t ws_bytes,
                        int32_t* status, void* stream, SumSq ss) {
  int rc = check_weights(w, true);
  if (rc || (rc = check_weights(w, false))) return rc;
  rc = moe_experts_quantize(x, a, a_sf, a1_gscale, r, T, H, I, E, K, tile_m, ws, ws_bytes, status,
                            stream);
  if (rc) return rc;
  // Decode-sized route tiles (tile_m <= 64): both GEMMs run as one
  // persistent grid, a programmatic dependent of the quantizer that starts
  // streaming its first weight stages while the quantizer drains; a route
  // tile's GEMM2 units start once its GEMM1 units have stored the
  // intermediate (the quantizer zeroed their counters), so GEMM2 has no ramp
  // of its own. Prefill tiles issue-bound on the tensor pipe gain nothing
  // from that and keep two launches, each a programmatic dependent of the
  // kernel before it.
  if (moe_experts_kernels(tile_m) == 3) {
    rc = experts_gemm1(w, a2_gscale, r, T, H, I, E, K, tile_m, ws, ws_bytes, status, stream, true);
    if (rc) return rc;
    return experts_gemm2(w, r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes, status, stream, true, ss);
  }
  return experts_fused(w, a2_gscale, r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes, status, stream,
                       true, false, ss);
}

// The sums-of-squares arguments of the *_sumsq entry points, checked.
static int sumsq_args(const void* gamma, int weight_before_norm, float* row_sumsq, SumSq* ss) {
  if (!row_sumsq || !aligned(row_sumsq, 16)) return fail(MOE_ERR_INVALID_ARG, "row_sumsq must be 16-byte aligned");
  if (weight_before_norm && (!gamma || !aligned(gamma, 16)))
    return fail(MOE_ERR_INVALID_ARG, "gamma must be given, 16-byte aligned, with weight_before_norm");
  ss->row_ss = row_sumsq;
  ss->gamma = gamma;
  ss->wbn = weight_before_norm ? 1 : 0;
  return MOE_OK;
}

int moe_experts_gemm2_sumsq(const moe_weights* w, const moe_route* r, int T, int H, int I, int E, int K,
                            int tile_m, void* gemm2_rows, const void* gamma, int weight_before_norm,
                            float* row_sumsq, void* ws, size_t ws_bytes, int32_t* status, void* stream) {
  SumSq ss;
  const int rc = sumsq_args(gamma, weight_before_norm, row_sumsq, &ss);
  if (rc) return rc;
  return experts_gemm2(w, r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes, status, stream, false, ss);
}

int moe_experts_gemms_sumsq(const moe_weights* w, const float* a2_gscale, const moe_route* r, int T, int H,
                            int I, int E, int K, int tile_m, void* gemm2_rows, const void* gamma,
                            int weight_before_norm, float* row_sumsq, void* ws, size_t ws_bytes,
                            int32_t* status, void* stream) {
  SumSq ss;
  const int rc = sumsq_args(gamma, weight_before_norm, row_sumsq, &ss);
  if (rc) return rc;
  return experts_fused(w, a2_gscale, r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes, status, stream, false,
                       true, ss);
}

int moe_nvfp4_experts(const moe_weights* w, const void* x, const void* a, const void* a_sf,
                      const float* a1_gscale, const float* a2_gscale, const moe_route* r, int T,
                      int H, int I, int E, int K, int tile_m, void* gemm2_rows, void* ws,
                      size_t ws_bytes, int32_t* status, void* stream) {
  return experts_body(w, x, a, a_sf, a1_gscale, a2_gscale, r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes,
                      status, stream, SumSq());
}

// Routing and the expert body in one call: with few routes and decode-sized
// route tiles the routing runs inside the input quantizer (one kernel, then
// the one-launch GEMMs as its programmatic dependent); otherwise the routing
// kernels, then moe_nvfp4_experts.
static bool routed_fused(int T, int K, int E, int tile_m) {
  return T > 0 && moe::route_quantize_fits(T, K, E) && moe_experts_kernels(tile_m) == 2;
}

int moe_routed_experts_kernels(int T, int K, int E, int tile_m) {
  RouteDims d;
  int rc = route_dims(T, K, E, tile_m, &d);
  if (rc) return rc;
  if (routed_fused(T, K, E, tile_m)) return 2;
  return moe::route_kernel_count(T, K, E) + (d.P > 0 ? moe_experts_kernels(tile_m) : 0);
}

// moe_nvfp4_experts_routed: routing inside the quantizer when routed_fused,
// else the routing kernels then experts_body.
static int routed_body(const moe_weights* w, const int32_t* topk_ids, const void* x, const void* a,
                       const void* a_sf, const float* a1_gscale, const float* a2_gscale, int T, int H, int I,
                       int E, int K, int tile_m, int32_t* expert_counts, int32_t* expert_offsets,
                       int32_t* expanded_to_permuted, int32_t* permuted_to_token, int32_t* tile_expert,
                       int32_t* tile_row_limit, int32_t* totals, void* gemm2_rows, void* ws, size_t ws_bytes,
                       int32_t* status, void* stream) {
  WsLayout L;
  int rc = ws_layout(T, K, E, H, I, tile_m, &L);
  if (rc || (rc = check_weights(w, true)) || (rc = check_weights(w, false))) return rc;
  const moe_route r{permuted_to_token, tile_expert, tile_row_limit, totals, expanded_to_permuted};
  if (!routed_fused(T, K, E, tile_m)) {
    rc = moe_route_permute(topk_ids, T, K, E, tile_m, expert_counts, expert_offsets, expanded_to_permuted,
                           permuted_to_token, tile_expert, tile_row_limit, totals, status, stream);
    if (rc) return rc;
    return experts_body(w, x, a, a_sf, a1_gscale, a2_gscale, &r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes,
                        status, stream, SumSq());
  }
  if (!expert_counts || !expert_offsets || !topk_ids || !expanded_to_permuted || !permuted_to_token ||
      !tile_expert || !tile_row_limit || !totals)
    return fail(MOE_ERR_INVALID_ARG, "routing buffer is null");
  if ((rc = check_ws(ws, ws_bytes, L))) return rc;
  if (x) {
    if (!a1_gscale) return fail(MOE_ERR_INVALID_ARG, "a1_gscale is null");
    if (!aligned(x, 16)) return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
  } else {
    if (!a || !a_sf) return fail(MOE_ERR_INVALID_ARG, "give x, or a and a_sf");
    if (!aligned(a, 16) || !aligned(a_sf, 4))
      return fail(MOE_ERR_INVALID_ARG, "a must be 16-byte and a_sf 4-byte aligned");
  }
  if (!a2_gscale) return fail(MOE_ERR_INVALID_ARG, "a2_gscale is null");
  if (!gemm2_rows || !aligned(gemm2_rows, 16))
    return fail(MOE_ERR_INVALID_ARG, "gemm2_rows must be non-null and 16-byte aligned");
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  cudaError_t err = moe::launch_route_quantize(
      topk_ids, T, K, E, tile_m, L.P, L.MT, expert_counts, expert_offsets, expanded_to_permuted, permuted_to_token,
      tile_expert, tile_row_limit, totals, x, x ? nullptr : a, x ? nullptr : a_sf, a1_gscale, H, base + L.a_codes,
      base + L.a_sf, reinterpret_cast<int32_t*>(base + L.done), status, as_stream(stream));
  if (err != cudaSuccess) return cuda_fail(err, "routing + input quantization");
  return experts_fused(w, a2_gscale, &r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes, status, stream, true,
                       false);
}

int moe_nvfp4_experts_routed(const moe_weights* w, const int32_t* topk_ids, const void* x, const void* a,
                             const void* a_sf, const float* a1_gscale, const float* a2_gscale, int T, int H,
                             int I, int E, int K, int tile_m, int32_t* expert_counts, int32_t* expert_offsets,
                             int32_t* expanded_to_permuted, int32_t* permuted_to_token, int32_t* tile_expert,
                             int32_t* tile_row_limit, int32_t* totals, void* gemm2_rows, void* ws,
                             size_t ws_bytes, int32_t* status, void* stream) {
  return routed_body(w, topk_ids, x, a, a_sf, a1_gscale, a2_gscale, T, H, I, E, K, tile_m, expert_counts,
                     expert_offsets, expanded_to_permuted, permuted_to_token, tile_expert, tile_row_limit, totals,
                     gemm2_rows, ws, ws_bytes, status, stream);
}

// The whole block: the routing kernels, the expert body with the sums of
// squares fused into GEMM2, then the finalize from them. (Routing inside the
// quantizer, as moe_nvfp4_experts_routed does, measured no faster here.)
int moe_moe_block_kernels(int T, int K, int E, int tile_m) {
  const int n = moe_route_kernels(T, K, E);
  if (n < 0) return n;
  const int b = moe_experts_kernels(tile_m);
  if (b < 0) return b;
  RouteDims d;
  int rc = route_dims(T, K, E, tile_m, &d);
  if (rc) return rc;
  return n + (d.P > 0 ? b + 1 : 0);
}

int moe_nvfp4_moe_block(const moe_weights* w, const int32_t* topk_ids, const float* topk_weights, const void* x,
                        const void* a, const void* a_sf, const float* a1_gscale, const float* a2_gscale,
                        const void* gamma, float eps, int weight_before_norm, int T, int H, int I, int E, int K,
                        int tile_m, int32_t* expert_counts, int32_t* expert_offsets, int32_t* expanded_to_permuted,
                        int32_t* permuted_to_token, int32_t* tile_expert, int32_t* tile_row_limit,
                        int32_t* totals, void* gemm2_rows, float* row_sumsq, void* out, void* ws, size_t ws_bytes,
                        int32_t* status, void* stream) {
  WsLayout L;
  int rc = ws_layout(T, K, E, H, I, tile_m, &L);
  if (rc) return rc;
  if (H > 16384) return fail(MOE_ERR_UNSUPPORTED, "hidden %d above 16384", H);
  if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
  if (T > 0 && (!topk_weights || !gamma || !out || !aligned(gamma, 16) || !aligned(out, 16)))
    return fail(MOE_ERR_INVALID_ARG, "topk_weights, gamma and out must be given; gamma and out 16-byte aligned");
  SumSq ss;
  if ((rc = sumsq_args(gamma, weight_before_norm, row_sumsq, &ss))) return rc;
  if ((rc = check_weights(w, true)) || (rc = check_weights(w, false)) || (rc = check_ws(ws, ws_bytes, L)))
    return rc;
  if (L.P > 0) {  // what the body checks, before anything is enqueued
    if (x) {
      if (!a1_gscale) return fail(MOE_ERR_INVALID_ARG, "a1_gscale is null");
      if (!aligned(x, 16)) return fail(MOE_ERR_INVALID_ARG, "x must be 16-byte aligned");
    } else {
      if (!a || !a_sf) return fail(MOE_ERR_INVALID_ARG, "give x, or a and a_sf");
      if (!aligned(a, 16) || !aligned(a_sf, 4))
        return fail(MOE_ERR_INVALID_ARG, "a must be 16-byte and a_sf 4-byte aligned");
    }
    if (!a2_gscale) return fail(MOE_ERR_INVALID_ARG, "a2_gscale is null");
    if (!gemm2_rows || !aligned(gemm2_rows, 16))
      return fail(MOE_ERR_INVALID_ARG, "gemm2_rows must be non-null and 16-byte aligned");
  }
  rc = moe_route_permute(topk_ids, T, K, E, tile_m, expert_counts, expert_offsets, expanded_to_permuted,
                         permuted_to_token, tile_expert, tile_row_limit, totals, status, stream);
  if (rc || L.P == 0) return rc;
  const moe_route r{permuted_to_token, tile_expert, tile_row_limit, totals, expanded_to_permuted};
  rc = experts_body(w, x, a, a_sf, a1_gscale, a2_gscale, &r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes, status,
                    stream, ss);
  if (rc) return rc;
  return moe_post_expert_finalize_sumsq(gemm2_rows, row_sumsq, L.P, expanded_to_permuted, topk_weights, gamma, eps,
                                        T, K, H, out, status, stream);
}

int moe_nvfp4_experts_sumsq(const moe_weights* w, const void* x, const void* a, const void* a_sf,
                            const float* a1_gscale, const float* a2_gscale, const moe_route* r, int T, int H,
                            int I, int E, int K, int tile_m, void* gemm2_rows, const void* gamma,
                            int weight_before_norm, float* row_sumsq, void* ws, size_t ws_bytes,
                            int32_t* status, void* stream) {
  SumSq ss;
  const int rc = sumsq_args(gamma, weight_before_norm, row_sumsq, &ss);
  if (rc) return rc;
  return experts_body(w, x, a, a_sf, a1_gscale, a2_gscale, r, T, H, I, E, K, tile_m, gemm2_rows, ws, ws_bytes,
                      status, stream, ss);
}

int moe_experts_export(int which, const void* ws, size_t ws_bytes, int T, int H, int I, int E,
                       int K, int tile_m, void* codes, void* scales, void* stream) {
  WsLayout L;
  int rc = ws_layout(T, K, E, H, I, tile_m, &L);
  if (rc) return rc;
  if ((rc = check_ws(ws, ws_bytes, L))) return rc;
  if (which != 0 && which != 1) return fail(MOE_ERR_INVALID_ARG, "which must be 0 or 1");
  if (L.P == 0) return MOE_OK;
  if (!codes || !scales) return fail(MOE_ERR_INVALID_ARG, "codes / scales are null");
  // Every one of the max_padded_rows rows is copied; rows past totals[1]
  // hold whatever the workspace held.
  uint8_t* base = const_cast<uint8_t*>(reinterpret_cast<const uint8_t*>(ws));
  const int Kc = which ? I : H;
  cudaError_t err = cudaMemcpyAsync(codes, base + (which ? L.h_codes : L.a_codes),
                                    (size_t)L.P * (Kc / 2), cudaMemcpyDeviceToDevice,
                                    as_stream(stream));
  if (err == cudaSuccess)
    err = moe::launch_act_scales_io(1, base + (which ? L.h_sf : L.a_sf),
                                    reinterpret_cast<uint8_t*>(scales), Kc, tile_m, L.P,
                                    as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_experts_export");
}

int moe_experts_import(int which, const void* codes, const void* scales, int T, int H, int I,
                       int E, int K, int tile_m, void* ws, size_t ws_bytes, void* stream) {
  WsLayout L;
  int rc = ws_layout(T, K, E, H, I, tile_m, &L);
  if (rc) return rc;
  if ((rc = check_ws(ws, ws_bytes, L))) return rc;
  if (which != 0 && which != 1) return fail(MOE_ERR_INVALID_ARG, "which must be 0 or 1");
  if (L.P == 0) return MOE_OK;
  if (!codes || !scales) return fail(MOE_ERR_INVALID_ARG, "codes / scales are null");
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  const int Kc = which ? I : H;
  cudaError_t err = cudaMemcpyAsync(base + (which ? L.h_codes : L.a_codes), codes,
                                    (size_t)L.P * (Kc / 2), cudaMemcpyDeviceToDevice,
                                    as_stream(stream));
  if (err == cudaSuccess)
    err = moe::launch_act_scales_io(0, base + (which ? L.h_sf : L.a_sf),
                                    const_cast<uint8_t*>(reinterpret_cast<const uint8_t*>(scales)),
                                    Kc, tile_m, L.P, as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_experts_import");
}

int moe_post_expert_finalize(const void* rows, int num_rows, const int32_t* expanded_to_permuted,
                             const float* topk_weights, const void* gamma, float eps,
                             int weight_before_norm, int T, int K, int H, void* out,
                             int32_t* status, void* stream) {
  if (T < 0 || K < 1 || H < 8 || H % 8 || H > 16384 || num_rows < 0)
    return fail(MOE_ERR_INVALID_ARG, "bad finalize shape T=%d K=%d H=%d rows=%d", T, K, H, num_rows);
  if (T == 0) return MOE_OK;
  if ((num_rows > 0 && !rows) || !expanded_to_permuted || !topk_weights || !gamma || !out)
    return fail(MOE_ERR_INVALID_ARG, "finalize pointer is null");
  if (!aligned(rows, 16) || !aligned(gamma, 16) || !aligned(out, 16))
    return fail(MOE_ERR_INVALID_ARG, "rows / gamma / out must be 16-byte aligned");
  if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
  cudaError_t err = moe::launch_finalize(rows, num_rows, expanded_to_permuted, topk_weights, gamma, eps,
                                         weight_before_norm, T, K, H, out, status, as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_post_expert_finalize");
}

int moe_post_expert_finalize_sumsq(const void* rows, const float* row_sumsq, int num_rows,
                                   const int32_t* expanded_to_permuted, const float* topk_weights,
                                   const void* gamma, float eps, int T, int K, int H, void* out,
                                   int32_t* status, void* stream) {
  if (T < 0 || K < 1 || K > 64 || H < 128 || H % 128 || H > 16384 || num_rows < 0)
    return fail(MOE_ERR_INVALID_ARG, "bad finalize shape T=%d K=%d H=%d rows=%d", T, K, H, num_rows);
  if (T == 0) return MOE_OK;
  if ((num_rows > 0 && (!rows || !row_sumsq)) || !expanded_to_permuted || !topk_weights || !gamma || !out)
    return fail(MOE_ERR_INVALID_ARG, "finalize pointer is null");
  if (!aligned(rows, 16) || !aligned(gamma, 16) || !aligned(out, 16) || !aligned(row_sumsq, 16))
    return fail(MOE_ERR_INVALID_ARG, "rows / row_sumsq / gamma / out must be 16-byte aligned");
  if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
  cudaError_t err = moe::launch_finalize_sumsq(rows, row_sumsq, num_rows, expanded_to_permuted, topk_weights,
                                               gamma, eps, T, K, H, out, status, as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_post_expert_finalize_sumsq");
}

int moe_post_expert_finalize_tp(const void* const* rows_parts, int nparts, int num_rows,
                                const int32_t* expanded_to_permuted, const float* topk_weights,
                                const void* gamma, float eps, int weight_before_norm, int T, int K,
                                int H, void* out, int32_t* status, void* stream) {
  if (T < 0 || K < 1 || H < 8 || H % 8 || H > 16384 || num_rows < 0)
    return fail(MOE_ERR_INVALID_ARG, "bad finalize shape T=%d K=%d H=%d rows=%d", T, K, H, num_rows);
  if (nparts < 1 || nparts > 16) return fail(MOE_ERR_UNSUPPORTED, "nparts %d not in [1, 16]", nparts);
  if (T == 0) return MOE_OK;
  if (!rows_parts || !expanded_to_permuted || !topk_weights || !gamma || !out)
    return fail(MOE_ERR_INVALID_ARG, "finalize pointer is null");
  for (int i = 0; i < nparts; ++i)
    if (!rows_parts[i] || !aligned(rows_parts[i], 16))
      return fail(MOE_ERR_INVALID_ARG, "row part %d is null or not 16-byte aligned", i);
  if (!aligned(gamma, 16) || !aligned(out, 16))
    return fail(MOE_ERR_INVALID_ARG, "gamma / out must be 16-byte aligned");
  if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
  cudaError_t err = moe::launch_finalize_parts(rows_parts, nparts, num_rows, expanded_to_permuted, topk_weights,
                                               gamma, eps, weight_before_norm, T, K, H, out, status,
                                               as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_post_expert_finalize_tp");
}

int moe_musespark1x_routing(const float* logits, const float* expert_bias, const uint8_t* is_padding, int T,
                            int E, int K, float route_scale, float eps, int32_t* topk_ids,
                            float* topk_weights, void* stream) {
  if (T < 0 || E < 1 || E > 1024 || K < 1 || K > 32 || K > E)
    return fail(MOE_ERR_INVALID_ARG, "bad routing shape T=%d E=%d K=%d (E <= 1024, K <= min(32, E))", T,
                E, K);
  if (T == 0) return MOE_OK;
  if (!logits || !expert_bias || !topk_ids || !topk_weights)
    return fail(MOE_ERR_INVALID_ARG, "routing pointer is null");
  if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
  cudaError_t err = moe::launch_musespark1x_routing(logits, expert_bias, is_padding, T, E, K, route_scale, eps,
                                                    topk_ids, topk_weights, as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_musespark1x_routing");
}

int moe_rmsnorm_nvfp4_quant(const void* x, const void* gamma, float eps, const float* gscale, int T, int H,
                            void* a, void* a_sf, void* stream) {
  if (T < 0 || H < 16 || H % 16) return fail(MOE_ERR_INVALID_ARG, "bad shape T=%d H=%d", T, H);
  if (T == 0) return MOE_OK;
  if (!x || !gamma || !gscale || !a || !a_sf) return fail(MOE_ERR_INVALID_ARG, "pointer is null");
  if (!aligned(x, 16) || !aligned(gamma, 16) || !aligned(a, 8))
    return fail(MOE_ERR_INVALID_ARG, "x / gamma must be 16-byte and a 8-byte aligned");
  if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
  cudaError_t err = moe::launch_rmsnorm_nvfp4(x, gamma, eps, gscale, T, H, a, a_sf, as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_rmsnorm_nvfp4_quant");
}

int moe_experts_norm_quantize(const void* x, const void* gamma, float eps, const float* a1_gscale,
                              const moe_route* r, int T, int H, int I, int E, int K, int tile_m, void* ws,
                              size_t ws_bytes, int32_t* status, void* stream) {
  (void)status;
  WsLayout L;
  int rc = ws_layout(T, K, E, H, I, tile_m, &L);
  if (rc) return rc;
  if ((rc = check_ws(ws, ws_bytes, L)) || (rc = check_route(r))) return rc;
  if (L.P == 0) return MOE_OK;
  if (!x || !gamma || !a1_gscale) return fail(MOE_ERR_INVALID_ARG, "x / gamma / a1_gscale is null");
  if (!aligned(x, 16) || !aligned(gamma, 16))
    return fail(MOE_ERR_INVALID_ARG, "x and gamma must be 16-byte aligned");
  if (!(eps >= 0.f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  if (!r->expanded_to_permuted) return fail(MOE_ERR_INVALID_ARG, "route expanded_to_permuted is null");
  cudaError_t err = moe::launch_rmsnorm_nvfp4_permuted(
      x, gamma, eps, a1_gscale, r->permuted_to_token, r->expanded_to_permuted, r->tile_row_limit, r->totals, T, K,
      H, tile_m, L.P, L.MT, base + L.a_codes, base + L.a_sf, as_stream(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_experts_norm_quantize");
}

}  // extern "C"

static int dense_shape(int T, int Din, int Dout) {
  if (T < 0 || Din < 64 || Dout < 128 || Din % 64 || Dout % 128)
    return fail(MOE_ERR_UNSUPPORTED, "dense shape: need Din %% 64 == 0, Dout %% 128 == 0 (T=%d Din=%d Dout=%d)",
                T, Din, Dout);
  return MOE_OK;
}

extern "C" int moe_dense_bf16_workspace_size(int T, int Din, int Dout, size_t* ws_bytes) {
  int rc = dense_shape(T, Din, Dout);
  if (rc) return rc;
  if (!ws_bytes) return fail(MOE_ERR_INVALID_ARG, "ws_bytes is null");
  *ws_bytes = moe::dense_workspace_here(T, Din, Dout);
  return MOE_OK;
}

extern "C" int moe_dense_bf16(const void* x, const void* w, int T, int Din, int Dout, void* y,
                              void* ws, size_t ws_bytes, int32_t* status, void* stream) {
  size_t need = 0;
  int rc = moe_dense_bf16_workspace_size(T, Din, Dout, &need);
  if (rc) return rc;
  if (T == 0) return MOE_OK;
  if (!x || !w || !y) return fail(MOE_ERR_INVALID_ARG, "dense x, w or y is null");
  if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 16))
    return fail(MOE_ERR_INVALID_ARG, "dense x, w and y must be 16-byte aligned");
  if (need > 0 && (!ws || ws_bytes < need || !aligned(ws, 16)))
    return fail(MOE_ERR_WORKSPACE, "dense workspace: need %zu bytes, 16-byte aligned", need);
  const char* why = "";
  rc = moe::launch_dense_bf16(x, w, T, Din, Dout, y, ws, status, as_stream(stream), &why);
  return rc ? fail(rc, "%s", why) : MOE_OK;
}

extern "C" int moe_selftest_wait_timeout(uint64_t limit_ns, int32_t* status, int32_t* result,
                                         void* stream) {
  if (!status || !result) return fail(MOE_ERR_INVALID_ARG, "status and result are required");
  if (limit_ns < 1000ull || limit_ns > 1000000000ull)
    return fail(MOE_ERR_INVALID_ARG, "limit_ns must be within [1 us, 1 s]");
  const int rc = moe::launch_selftest_wait(limit_ns, status, result, as_stream(stream));
  return rc ? fail(rc, "self-test launch failed") : MOE_OK;
}

extern "C" int moe_selftest_counter_timeout(uint64_t limit_ns, const int32_t* counter, int32_t* status,
                                            int32_t* result, void* stream) {
  if (!counter || !status || !result) return fail(MOE_ERR_INVALID_ARG, "counter, status and result are required");
  if (!aligned(counter, 4)) return fail(MOE_ERR_INVALID_ARG, "counter must be 4-byte aligned");
  if (limit_ns < 1000ull || limit_ns > 1000000000ull)
    return fail(MOE_ERR_INVALID_ARG, "limit_ns must be within [1 us, 1 s]");
  const int rc = moe::launch_selftest_counter(limit_ns, counter, status, result, as_stream(stream));
  return rc ? fail(rc, "self-test launch failed") : MOE_OK;
}

extern "C" int moe_selftest_occupy(int ctas, int smem_bytes, uint64_t ns, void* stream) {
  if (ctas < 1 || ctas > 65535 || smem_bytes < 0 || smem_bytes > 227 * 1024)
    return fail(MOE_ERR_INVALID_ARG, "occupy: ctas in [1, 65535], smem_bytes in [0, 227 KB]");
  if (ns > 2000000000ull) return fail(MOE_ERR_INVALID_ARG, "occupy: ns must be at most 2 s");
  const int rc = moe::launch_selftest_occupy(ctas, smem_bytes, ns, as_stream(stream));
  return rc ? fail(rc, "occupy launch failed") : MOE_OK;
}
