/*
 * moe_nvfp4.h -- C ABI of libmoe_nvfp4.so: the routed NVFP4 mixture-of-experts
 * expert block with the MuseSpark1x post-expert finalize, for GB300 (sm_103a).
 *
 * The block (vLLM "muse_moe_runner" page: MuseSparkTrtLlmNvFp4Experts
 * .apply_routed and MusePostExpertFinalize; "flashinfer_ops" page:
 * FlashInferOps.slot / nvfp4_arguments / gemm2_rows; "expert_tp" page:
 * StockNvfp4 and the module docstring; "model" page: MuseSpark1xMoE):
 *
 *   a1  a    = NVFP4(x) with the fp32 global scale a1_gscale
 *   a2  routing metadata: per-expert histogram, permuted and padded rows
 *   a3  acc  = a . w13[e]^T  (block-scaled FP4, fp32 accumulate)
 *       gate = g1_alphas[e] * acc[:, 0:I],  up = g1_scale_c[e] * acc[:, I:2I]
 *   a4  h    = SiLU(gate) * up
 *   a5  hq   = NVFP4(h) with a2_gscale
 *   a6  rows = bf16(g2_alphas[e] * hq . w2[e]^T)
 *   a7  out[t] = bf16( sum_k w[t,k] * RMSNorm(rows[p(t,k)]) ), fp32 norm
 *       output and fp32 sum; zero-centred gamma (weight 1 + gamma)
 *
 * Conventions for every entry point:
 *   - Pointers are device memory owned by the caller unless stated; scalar
 *     arguments (sizes, eps, flags) are host values.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Every call only enqueues work on it: no allocation, no host
 *     synchronisation, no host read of device data.
 *   - The return value is MOE_OK or a negative MOE_ERR_* code for errors
 *     found on the host (arguments, sizes, a failed launch); nothing is
 *     enqueued when a call returns an error. moe_last_error() then gives the
 *     reason (thread-local, valid until the next failing call).
 *   - Data-dependent errors found on the device (an expert id out of range,
 *     a bounded wait that gave up) are recorded in the optional caller-owned
 *     `int32_t* status` word: the first error code wins (atomic
 *     compare-and-swap from 0). The library never clears it: zero it before
 *     the calls and read it after synchronising. A kernel that records an
 *     error leaves the outputs it could not compute unspecified.
 *   - No kernel traps, asserts or waits without a bound.
 *
 * Number formats: e2m1 values packed two per byte, the even element in the
 * low nibble; e4m3 ("fn") block scales, one per 16 consecutive elements along
 * K; bf16 activations; fp32 scalars.
 */
#ifndef MOE_NVFP4_H
#define MOE_NVFP4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,   /* null pointer, bad size, misaligned buffer */
  MOE_ERR_UNSUPPORTED = -2,   /* shape the layout/kernels cannot hold      */
  MOE_ERR_WORKSPACE = -3,     /* workspace smaller than the size query     */
  MOE_ERR_CUDA = -4,          /* a CUDA runtime / driver call failed       */
  MOE_ERR_TIMEOUT = -5,       /* device: a bounded wait gave up            */
  MOE_ERR_INVALID_ROUTE = -6, /* device: topk id >= E or < -1              */
};

/* Reason for the last error returned on this thread ("" if none). */
const char* moe_last_error(void);

/* ABI version, bumped on any incompatible change. */
int moe_abi_version(void);

/* 1 if kernels of this library may read and write the host memory at p
 * through p itself (page-locked or managed memory that the current device
 * maps at the same address, as unified addressing gives cudaHostAlloc
 * memory), else 0. Callers use it before passing host pointers as step
 * inputs or outputs (zero-copy serving); no error is recorded. */
int moe_device_reads_host(const void* p);

/* ------------------------------------------------------------------------
 * Weight preparation (runs once per layer, at load).
 *
 * Raw weights (the expert_tp page, StockNvfp4 shapes, block scales
 * unswizzled):
 *   w13    uint8 [E, 2I, H/2]   rows [0, I) gate (w1), rows [I, 2I) up (w3)
 *   w13_sf e4m3  [E, 2I, H/16]
 *   w2     uint8 [E, H, I/2]
 *   w2_sf  e4m3  [E, H, I/16]
 *
 * Prepared layout written by moe_prepare_weights (this library's own, not
 * the pages' TRT-LLM layout):
 *   p_w13    uint8 [E, 2I, H/2]: prepared row r holds raw row
 *              16*(r/32) + r%32           if r%32 < 16  (gate)
 *              I + 16*(r/32) + r%32 - 16  otherwise     (up)
 *            so every 32-row group holds the gate and up rows of the same
 *            16 intermediate columns (the GEMM1 epilogue pairs them in one
 *            warp). Bytes inside a row are unchanged.
 *   p_w13_sf uint8 [E, 2I/128, H/64, 512]: scale atoms. Byte
 *              (e, mt, kc, 16*m0 + 4*m1 + c), m0 < 32, m1 < 4, c < 4,
 *            holds the scale of prepared row 128*mt + 32*m1 + m0 for the
 *            16-element block 4*kc + c. One atom is what one tcgen05.cp
 *            (32x128b, warpx4) moves into tensor memory for one K=64 MMA of
 *            128 rows.
 *   p_w2     uint8 [E, H, I/2]: w2 unchanged.
 *   p_w2_sf  uint8 [E, H/128, I/64, 512]: the same atoms over w2_sf.
 *
 * Layout identity (the expert_tp page's requirement for free TP cuts): for
 * tp with I' = I/tp, I' % 64 == 0 and H % 128 == 0, intermediate slice r of
 * the prepared tensors -- p_w13 rows [2rI', 2(r+1)I'), p_w13_sf row tiles
 * [2rI'/128, 2(r+1)I'/128), p_w2 bytes [rI'/2, (r+1)I'/2) of every row,
 * p_w2_sf k-atoms [rI'/64, (r+1)I'/64) -- is byte for byte
 * moe_prepare_weights of the raw slice.
 *
 * Requires H % 128 == 0 and I % 64 == 0 (else MOE_ERR_UNSUPPORTED).
 * ---------------------------------------------------------------------- */

/* Bytes of the four prepared tensors: {p_w13, p_w13_sf, p_w2, p_w2_sf}. */
int moe_prepared_sizes(int E, int H, int I, size_t out_bytes[4]);

/* Write the prepared layout. Inputs and outputs must not overlap; every
 * pointer 16-byte aligned. */
int moe_prepare_weights(const void* w13, const void* w13_sf, const void* w2,
                        const void* w2_sf, int E, int H, int I, void* p_w13,
                        void* p_w13_sf, void* p_w2, void* p_w2_sf,
                        void* stream);

/* ------------------------------------------------------------------------
 * Routing metadata (step a2; the flashinfer_ops page, FlashInferOps.slot).
 *
 * R = T*K routes, route j = t*K + k. tile_m in {32, 64, 128, 256}; E in
 * [1, 1024].
 *   expert_counts[E]        routes per expert
 *   expert_offsets[E+1]     exclusive prefix of the padded counts
 *                           ceil(count/tile_m)*tile_m; [E] = total padded
 *   expanded_to_permuted[R] permuted row of route j; -1 if topk_ids[j] == -1
 *   permuted_to_token[P]    token of a permuted row; -1 on padding rows and
 *                           on every row past the total
 *   tile_expert[MT]         expert of tile tau (rows [tau*tile_m,
 *                           (tau+1)*tile_m)); -1 past the live tiles
 *   tile_row_limit[MT]      offsets[e] + counts[e] of that expert; -1 past
 *   totals[2]               {live tiles, total padded rows}
 * with P = max_padded_rows = tile_m*(F + (R-F)/tile_m), F = min(E, R) (the
 * flashinfer_ops page's gemm2_rows bound) and MT = max_tiles = P/tile_m.
 * Inside an expert, routes take rows in ascending j: the result is unique
 * and deterministic. topk_ids of -1 mean "not routed" (expert parallel marks
 * remote experts so); ids < -1 or >= E record MOE_ERR_INVALID_ROUTE in
 * *status and leave the metadata unspecified. T == 0 is valid.
 * ---------------------------------------------------------------------- */

int moe_route_sizes(int T, int K, int E, int tile_m, int* max_padded_rows,
                    int* max_tiles);

/* Kernels moe_route_permute enqueues for this shape: 1 (one CTA, few
 * routes) or 3 (count / scan / scatter over segments of about 2048 routes,
 * from T*K >= 4096). Returns the count, or a negative status for a bad shape. */
int moe_route_kernels(int T, int K, int E);

int moe_route_permute(const int32_t* topk_ids, int T, int K, int E,
                      int tile_m, int32_t* expert_counts,
                      int32_t* expert_offsets, int32_t* expanded_to_permuted,
                      int32_t* permuted_to_token, int32_t* tile_expert,
                      int32_t* tile_row_limit, int32_t* totals,
                      int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Experts (steps a1, a3-a6; the muse_moe_runner page, apply_routed with
 * do_finalize=False, and the flashinfer_ops page, nvfp4_arguments).
 * ---------------------------------------------------------------------- */

typedef struct moe_weights {
  const void* w13;         /* prepared uint8 [E, 2I, H/2]            */
  const void* w13_sf;      /* prepared uint8 [E, 2I/128, H/64, 512]  */
  const void* w2;          /* prepared uint8 [E, H, I/2]             */
  const void* w2_sf;       /* prepared uint8 [E, H/128, I/64, 512]   */
  const float* g1_alphas;  /* fp32 [E]: gate scale ("output1_scale_gate_scalar") */
  const float* g1_scale_c; /* fp32 [E]: up scale ("output1_scale_scalar"); holds
                              no 1/a2 -- the requant applies a2_gscale */
  const float* g2_alphas;  /* fp32 [E]: GEMM2 scale ("output2_scale_scalar") */
} moe_weights;

typedef struct moe_route {
  const int32_t* permuted_to_token;    /* [max_padded_rows] */
  const int32_t* tile_expert;          /* [max_tiles] */
  const int32_t* tile_row_limit;       /* [max_tiles] */
  const int32_t* totals;               /* [2] */
  const int32_t* expanded_to_permuted; /* [T, K]; read by the input quantizer, which
                                          quantizes each token once and writes it to
                                          the rows of its routes; an entry outside
                                          [-1, max_padded_rows) is skipped and
                                          recorded as MOE_ERR_INVALID_ROUTE in status */
} moe_route;

/* Kernels moe_nvfp4_experts enqueues for this route-tile size: 2 (the
 * quantizer and one persistent launch of both GEMMs, tile_m <= 64) or 3
 * (the quantizer, GEMM1, GEMM2). Returns the count, or a negative status
 * for an unsupported tile_m. */
int moe_experts_kernels(int tile_m);

/* Workspace bytes moe_nvfp4_experts needs (the permuted NVFP4 activations,
 * the quantized intermediate and one completion counter per route tile;
 * contents opaque). */
int moe_experts_workspace_size(int T, int K, int E, int H, int I, int tile_m,
                               size_t* ws_bytes);

/* The whole expert body: a1 quantization into permuted order, GEMM1 with
 * the SwiGLU + NVFP4 requant epilogue, GEMM2 (for tile_m <= 64 both GEMMs
 * in one persistent launch, where a GEMM2 tile starts once every GEMM1 tile
 * of its route tile has written its intermediate). Give either x (bf16 [T, H]) or
 * a pre-quantized a (uint8 [T, H/2]) with a_sf (e4m3 [T, H/16], row-major,
 * as scaled_fp4_quant(..., is_sf_swizzled_layout=False) returns it) and
 * pass NULL for the other. a1_gscale, a2_gscale: device fp32 [1].
 * gemm2_rows: bf16 [max_padded_rows, H]; only rows < totals[1] that carry a
 * route are written (the flashinfer_ops page trims to gemm2_rows; padding
 * rows are never read by the finalize). Requires H % 128 == 0,
 * I % 64 == 0 (every expert-TP slice the prepared layout admits), tile_m in
 * {32, 64, 128, 256}; every device pointer 16-byte
 * aligned; ws at least moe_experts_workspace_size bytes, 1024-byte
 * aligned. */
int moe_nvfp4_experts(const moe_weights* w, const void* x, const void* a,
                      const void* a_sf, const float* a1_gscale,
                      const float* a2_gscale, const moe_route* r, int T,
                      int H, int I, int E, int K, int tile_m,
                      void* gemm2_rows, void* ws, size_t ws_bytes,
                      int32_t* status, void* stream);

/* Routing and the whole expert body in one call (steps a2, a1, a3-a6 as the
 * flashinfer_ops page's FlashInferOps.slot runs them: metadata, then the
 * experts): the result of
 * moe_route_permute (same buffers, same contents, readable after the call,
 * e.g. by the finalize) followed by moe_nvfp4_experts on that route. With few
 * routes (T*K <= 2048, E <= 256) and tile_m <= 64 the routing runs inside the
 * input quantizer: every CTA of that kernel computes the routing in its own
 * shared memory and the first also writes it out, so the step has no kernel
 * boundary between routing and quantization (2 kernels in all, see
 * moe_routed_experts_kernels). Otherwise it enqueues the routing kernels and
 * then moe_nvfp4_experts. Arguments as for those two entry points; an invalid
 * expert id is reported in status as moe_route_permute reports it. */
int moe_nvfp4_experts_routed(const moe_weights* w, const int32_t* topk_ids,
                             const void* x, const void* a, const void* a_sf,
                             const float* a1_gscale, const float* a2_gscale,
                             int T, int H, int I, int E, int K, int tile_m,
                             int32_t* expert_counts, int32_t* expert_offsets,
                             int32_t* expanded_to_permuted,
                             int32_t* permuted_to_token, int32_t* tile_expert,
                             int32_t* tile_row_limit, int32_t* totals,
                             void* gemm2_rows, void* ws, size_t ws_bytes,
                             int32_t* status, void* stream);

/* Kernels moe_nvfp4_experts_routed enqueues for these sizes (a negative
 * status for invalid ones). */
int moe_routed_experts_kernels(int T, int K, int E, int tile_m);

/* The whole routed expert block in one call (steps a1-a7: the
 * muse_moe_runner page's apply_routed with do_finalize=False followed by
 * MusePostExpertFinalize): routing, the expert body with
 * the post-expert norm's sums of squares fused into GEMM2's epilogue
 * (moe_nvfp4_experts_sumsq), and the finalize from those sums
 * (moe_post_expert_finalize_sumsq): out bf16 [T, H]. The result equals, bit
 * for bit, moe_route_permute, then moe_nvfp4_experts_sumsq, then
 * moe_post_expert_finalize_sumsq on the same buffers (the routing buffers,
 * gemm2_rows and row_sumsq [max_padded_rows, H/32] fp32 hold what those
 * calls leave). For tile_m <= 64: the routing kernel, then the input
 * quantizer, one persistent launch of both GEMMs and the finalize, each a
 * programmatic dependent of the kernel before it (moe_moe_block_kernels). topk_weights fp32
 * [T, K]; gamma bf16 [H] (zero-centred gain, 16-byte aligned), eps,
 * weight_before_norm as for moe_post_expert_finalize; out 16-byte aligned;
 * the rest as for moe_nvfp4_experts_routed. */
int moe_nvfp4_moe_block(const moe_weights* w, const int32_t* topk_ids,
                        const float* topk_weights, const void* x, const void* a,
                        const void* a_sf, const float* a1_gscale,
                        const float* a2_gscale, const void* gamma, float eps,
                        int weight_before_norm, int T, int H, int I, int E,
                        int K, int tile_m, int32_t* expert_counts,
                        int32_t* expert_offsets, int32_t* expanded_to_permuted,
                        int32_t* permuted_to_token, int32_t* tile_expert,
                        int32_t* tile_row_limit, int32_t* totals,
                        void* gemm2_rows, float* row_sumsq, void* out,
                        void* ws, size_t ws_bytes, int32_t* status,
                        void* stream);

/* Kernels moe_nvfp4_moe_block enqueues for these sizes (a negative status
 * for invalid ones). */
int moe_moe_block_kernels(int T, int K, int E, int tile_m);

/* moe_nvfp4_experts with the first half of the post-expert norm fused into
 * GEMM2's epilogue: besides the bf16 rows it writes, for every route row,
 * the sums of squares of its stored values over each 32 columns,
 *   row_sumsq[p][c] = sum_{j < 32} (g[32c + j] * rows[p][32c + j])^2
 * with g = 1 + float(gamma) when weight_before_norm != 0 (the weight applied
 * before the norm) and g = 1 otherwise. row_sumsq: fp32
 * [max_padded_rows, H/32], 16-byte aligned; only the rows GEMM2 writes get
 * values. gamma: bf16 [H], 16-byte aligned (may be NULL with
 * weight_before_norm = 0). moe_post_expert_finalize_sumsq then finalizes
 * from it without a reduction pass over the rows. Everything else as
 * moe_nvfp4_experts. */
int moe_nvfp4_experts_sumsq(const moe_weights* w, const void* x, const void* a,
                            const void* a_sf, const float* a1_gscale,
                            const float* a2_gscale, const moe_route* r, int T,
                            int H, int I, int E, int K, int tile_m,
                            void* gemm2_rows, const void* gamma,
                            int weight_before_norm, float* row_sumsq, void* ws,
                            size_t ws_bytes, int32_t* status, void* stream);

/* The same body in its three launches, for timing one step alone. Called
 * in this order on one stream they equal moe_nvfp4_experts. */
int moe_experts_quantize(const void* x, const void* a, const void* a_sf,
                         const float* a1_gscale, const moe_route* r, int T,
                         int H, int I, int E, int K, int tile_m, void* ws,
                         size_t ws_bytes, int32_t* status, void* stream);
int moe_experts_gemm1(const moe_weights* w, const float* a2_gscale,
                      const moe_route* r, int T, int H, int I, int E, int K,
                      int tile_m, void* ws, size_t ws_bytes, int32_t* status,
                      void* stream);
int moe_experts_gemm2(const moe_weights* w, const moe_route* r, int T, int H,
                      int I, int E, int K, int tile_m, void* gemm2_rows,
                      void* ws, size_t ws_bytes, int32_t* status,
                      void* stream);

/* GEMM1 and GEMM2 as the one persistent launch moe_nvfp4_experts uses for
 * tile_m <= 64 (any supported tile_m is accepted): after
 * moe_experts_quantize it equals moe_experts_gemm1 followed by
 * moe_experts_gemm2, bit for bit. It first clears the workspace's per-tile
 * completion counters (one memset of 4 bytes per route tile), so it may be
 * called again on the same quantized workspace. Arguments as for
 * moe_experts_gemm1 and moe_experts_gemm2. */
int moe_experts_gemms(const moe_weights* w, const float* a2_gscale,
                      const moe_route* r, int T, int H, int I, int E, int K,
                      int tile_m, void* gemm2_rows, void* ws, size_t ws_bytes,
                      int32_t* status, void* stream);

/* moe_experts_gemm2 and moe_experts_gemms with the sums of squares of
 * moe_nvfp4_experts_sumsq fused into GEMM2's epilogue (arguments as there). */
int moe_experts_gemm2_sumsq(const moe_weights* w, const moe_route* r, int T,
                            int H, int I, int E, int K, int tile_m,
                            void* gemm2_rows, const void* gamma,
                            int weight_before_norm, float* row_sumsq, void* ws,
                            size_t ws_bytes, int32_t* status, void* stream);
int moe_experts_gemms_sumsq(const moe_weights* w, const float* a2_gscale,
                            const moe_route* r, int T, int H, int I, int E,
                            int K, int tile_m, void* gemm2_rows,
                            const void* gamma, int weight_before_norm,
                            float* row_sumsq, void* ws, size_t ws_bytes,
                            int32_t* status, void* stream);

/* Copy a quantized operand out of / into the workspace, in permuted row
 * order with row-major scales: which = 0 for the activations a (codes
 * uint8 [max_padded_rows, H/2], scales e4m3 [max_padded_rows, H/16]),
 * which = 1 for the intermediate hq ([max_padded_rows, I/2] and
 * [max_padded_rows, I/16]). moe_experts_import followed by
 * moe_experts_gemm2 runs GEMM2 on a given intermediate. In the activations,
 * padding rows (permuted_to_token == -1) have zero scales and unspecified
 * codes, which contribute exactly zero to every product; rows past
 * totals[1] are unspecified. */
int moe_experts_export(int which, const void* ws, size_t ws_bytes, int T,
                       int H, int I, int E, int K, int tile_m, void* codes,
                       void* scales, void* stream);
int moe_experts_import(int which, const void* codes, const void* scales,
                       int T, int H, int I, int E, int K, int tile_m,
                       void* ws, size_t ws_bytes, void* stream);

/* moe_nvfp4_experts without a workspace argument: it allocates nothing.
 *
 * The pages have no counterpart of this entry point. It exists for callers
 * that cannot allocate device memory at the point of the call: code
 * recorded into a CUDA graph capture (cudaMalloc is not allowed while a
 * stream is being captured), latency-critical serving loops that must not
 * reach the allocator (a cudaMalloc may synchronise the device), and
 * plug-ins whose host framework owns all device memory and hands them
 * none. Instead of a caller buffer it uses one fixed array of
 * moe_noalloc_scratch_bytes() bytes (32 MiB) that the library defines in
 * device memory; every GPU that loads the library holds that array until
 * the process exits. Shapes whose workspace (moe_experts_workspace_size)
 * is larger are refused with MOE_ERR_WORKSPACE before anything is enqueued.
 * The workspace size depends only on the shape, not on the routing: compare
 * moe_experts_workspace_size with moe_noalloc_scratch_bytes(). At H = 5120,
 * I = 2048, E = 128, top-8 and tile_m = 32 that admits up to 287 tokens
 * (tile_m = 128: 8 tokens; the padded-row bound grows with the tile).
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and keeps it; make that
 * first call before any stream capture. The address is looked up again
 * when the device's context has changed since (after a cudaDeviceReset),
 * so make the first call after a reset outside a capture too. Every other argument, the outputs
 * and the status word behave as in moe_nvfp4_experts, and the caller still
 * owns x / a / a_sf, the routing metadata and gemm2_rows. All calls share
 * the one array: two calls whose work overlaps on the GPU (different
 * streams without ordering between them) race and give undefined results.
 * Nothing in the array has to start at zero: every byte a call reads has
 * been written earlier in the same call. */
int moe_nvfp4_experts_noalloc(const moe_weights* w, const void* x, const void* a,
                              const void* a_sf, const float* a1_gscale,
                              const float* a2_gscale, const moe_route* r, int T,
                              int H, int I, int E, int K, int tile_m,
                              void* gemm2_rows, int32_t* status, void* stream);

/* Size in bytes of the array moe_nvfp4_experts_noalloc uses. */
size_t moe_noalloc_scratch_bytes(void);

/* ------------------------------------------------------------------------
 * Post-expert finalize (step a7; the muse_moe_runner page,
 * MusePostExpertFinalize.__call__(unfinalized, out), _finalize_native,
 * _finalize_chunk, _effective_weight; the model page's post_expert_norm).
 *
 *   out[t] = bf16( sum_{k < K} w[t,k] * N(rows[p(t,k)]) ),  p = -1 adds 0
 *   g = 1 + float(gamma)            (gain centre added in fp32)
 *   weight_before_norm != 0:  u = g*r,  N = u * rsqrt(mean(u^2) + eps)
 *   weight_before_norm == 0:  N = g * r * rsqrt(mean(r^2) + eps)
 * all in fp32 over the full hidden size H, summed over k in order 0..K-1.
 * rows: bf16 [num_rows, H] (GEMM2 rows); expanded_to_permuted int32
 * [T, K]; topk_weights fp32 [T, K]; gamma bf16 [H]; out bf16 [T, H]
 * (caller-owned, may not alias rows). H % 8 == 0, H <= 16384, num_rows >= 0;
 * T == 0 is valid. An expanded_to_permuted entry outside [-1, num_rows)
 * records MOE_ERR_INVALID_ROUTE in *status (optional device word) and that
 * route is skipped as if it were -1: no row outside the buffer is read.
 * ---------------------------------------------------------------------- */
int moe_post_expert_finalize(const void* rows, int num_rows,
                             const int32_t* expanded_to_permuted,
                             const float* topk_weights, const void* gamma,
                             float eps, int weight_before_norm, int T, int K,
                             int H, void* out, int32_t* status, void* stream);

/* The finalize from moe_nvfp4_experts_sumsq's output: each route's norm
 * coefficient w[t,k] / sqrt(sum_c row_sumsq[p][c] / H + eps) (the H/32
 * partials summed in a fixed order) and then
 *   out[t] = bf16( g * sum_k coef_k * rows[p(t,k)] ),  g = 1 + float(gamma),
 * equal to moe_post_expert_finalize in the reading row_sumsq was made with,
 * up to the order of the fp32 sums. rows bf16 [num_rows, H], row_sumsq fp32
 * [num_rows, H/32], both 16-byte aligned; H % 128 == 0, H <= 16384,
 * K <= 64; the row bound and status word as for moe_post_expert_finalize. */
int moe_post_expert_finalize_sumsq(const void* rows, const float* row_sumsq,
                                   int num_rows,
                                   const int32_t* expanded_to_permuted,
                                   const float* topk_weights, const void* gamma,
                                   float eps, int T, int K, int H, void* out,
                                   int32_t* status, void* stream);

/* Expert-TP tail (the expert_tp page: with expert tensor parallelism every
 * rank computes K-partial GEMM2 rows over its intermediate slice, and they
 * are summed -- "FP32 sum, one BF16 rounding" -- before the per-route norm;
 * the muse_moe_runner page's TP finalize fuses that sum into the norm).
 * rows_parts is a HOST array of nparts (1..16) device pointers to bf16
 * [num_rows, H] row buffers indexed alike; each route's row is
 * bf16(sum_r float(part_r[p])) and then finalized exactly as
 * moe_post_expert_finalize does (the same row bound and status word). With
 * nparts = 1 it equals moe_post_expert_finalize. */
int moe_post_expert_finalize_tp(const void* const* rows_parts, int nparts,
                                int num_rows,
                                const int32_t* expanded_to_permuted,
                                const float* topk_weights, const void* gamma,
                                float eps, int weight_before_norm, int T, int K,
                                int H, void* out, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Steps that feed the block (the model page, MuseSpark1xMoE).
 * ---------------------------------------------------------------------- */

/* MuseSpark1x routing from fp32 router logits [T, E] (fused_musespark1x_routing:
 * sigmoid scores, an fp32 expert bias [E] that only steers the choice,
 * sum-renormalised weights with division eps, route_scale; no groups):
 *   s = sigmoid(logits); chosen = the K largest s + bias, the lower expert
 *   index first on equal values; w = s[chosen] / (sum + eps) * route_scale.
 * topk_ids int32 [T, K] in choice order, topk_weights fp32 [T, K]. Tokens
 * with is_padding[t] != 0 (optional uint8 [T]) get ids -1 and weights 0.
 * E <= 1024, K <= min(32, E). */
int moe_musespark1x_routing(const float* logits, const float* expert_bias,
                            const uint8_t* is_padding, int T, int E, int K,
                            float route_scale, float eps, int32_t* topk_ids,
                            float* topk_weights, void* stream);

/* Pre-expert RMSNorm fused into the NVFP4 input quantization
 * (norm_quant_trtllm_nvfp4; the norm's weight applied after normalising):
 *   y = x / sqrt(mean(x^2) + eps) * (1 + gamma),  (a, a_sf) = NVFP4(y, gscale)
 * x bf16 [T, H], gamma bf16 [H] (zero-centred), gscale device fp32 [1];
 * y stays fp32 and is quantized like moe_experts_quantize. Outputs a uint8
 * [T, H/2] and a_sf e4m3 [T, H/16] row-major (scaled_fp4_quant's layout). */
int moe_rmsnorm_nvfp4_quant(const void* x, const void* gamma, float eps,
                            const float* gscale, int T, int H, void* a,
                            void* a_sf, void* stream);

/* The same, written straight into the expert body's workspace in permuted
 * order: a drop-in replacement for moe_experts_quantize when the block's
 * input is the pooled, not yet normalised activation. */
int moe_experts_norm_quantize(const void* x, const void* gamma, float eps,
                              const float* a1_gscale, const moe_route* r, int T,
                              int H, int I, int E, int K, int tile_m, void* ws,
                              size_t ws_bytes, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Pooler / unpooler (the model page: the MoE block's `pooler`
 * ReplicatedLinear(hidden_size, moe_hidden_size, bias=False,
 * quant_config=None) before the experts, `unpooler` back after them):
 *   y[t, o] = bf16( sum_i x[t, i] * w[o, i] )   (fp32 accumulation)
 * x bf16 [T, Din] row-major, w bf16 [Dout, Din] row-major (the Linear
 * weight), y bf16 [T, Dout]. Din % 64 == 0, Dout % 128 == 0, every pointer
 * 16-byte aligned. For few tokens the (output tile, K) work is split evenly
 * over the CTAs; tiles split between CTAs leave fp32 partials and arrival
 * counters in ws, and the last arrival sums the partials in a fixed order
 * (deterministic) inside the same kernel. The call clears the counters
 * (one memset of at most a few KB) before the kernel, so ws needs no
 * initialisation; its contents are opaque. ws may be NULL when
 * moe_dense_bf16_workspace_size reports 0. T == 0 is valid.
 * ---------------------------------------------------------------------- */
int moe_dense_bf16_workspace_size(int T, int Din, int Dout, size_t* ws_bytes);

int moe_dense_bf16(const void* x, const void* w, int T, int Din, int Dout, void* y,
                   void* ws, size_t ws_bytes, int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Dense NVFP4 tensor-core rate of this GPU, for the roofline of the
 * compute-bound (prefill) expert GEMMs. The pages print no throughput; this
 * measures the instruction the expert GEMMs issue
 * (tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X, M = 128,
 * K = 64, e2m1 operands with ue4m3 scales per 16 elements, fp32 accumulate in
 * tensor memory) on operands held in shared memory: every CTA (ctas_per_sm per
 * SM, on every SM) issues `stages` stages of mmas_per_commit MMAs of N = n,
 * each stage ending in one tcgen05.commit, `ring` (3 or 5) stages in flight.
 * sf_copies selects how the scale factors reach tensor memory: 0 once before
 * the loop; 1 every stage as the expert GEMMs copy them (tcgen05.cp
 * 32x128b.warpx4, one per 128 rows of each operand per K = 64 step) by the
 * MMA thread itself; 2 by a second warp that hands each stage over through an
 * mbarrier; 3 by two more warps, one per operand; 4 every stage by the MMA
 * thread with 128x256b copies (two K = 64 steps per copy) for both operands;
 * 5 the same for A only. Modes 4 and 5 time the copies, not a scale layout:
 * every scale byte is 1.0 here. warp_issue selects how the issuing warps run
 * their loops: 0 lane 0 alone; 1 the whole warp, converged, with lane 0
 * issuing each tcgen05 instruction under a predicate (the expert GEMM1's
 * form). Supported: n = 128 (ctas_per_sm 1 or 2) or
 * 256 (ctas_per_sm 1); mmas_per_commit 4, or 16 with sf_copies = 0; ring 5
 * only with ctas_per_sm = 1 and sf_copies != 0; warp_issue 0 or 1; stages
 * 1 .. 2^24. *flops
 * (host) receives the launch's FLOPs,
 * 2 * 128 * n * 64 * mmas_per_commit * stages * CTAs; time the launch with
 * events on `stream`. A wait that gives up records MOE_ERR_TIMEOUT in *status
 * (optional device word). Operands and outputs are scratch inside the kernel.
 * ---------------------------------------------------------------------- */
int moe_fp4_mma_rate(int n, int sf_copies, int mmas_per_commit, int ctas_per_sm,
                     int ring, int warp_issue, int stages, double* flops,
                     int32_t* status, void* stream);

/* The pair form of the same measurement: tcgen05.mma.cta_group::2 (M = 256
 * across the two CTAs of a cluster, on two SMs, A rows 128-255 read from the
 * peer CTA's shared memory), one CTA per SM on an even number of SMs. Rank 0
 * of each pair issues `stages` stages of 4 MMAs of N = n (128 or 256), with
 * the scale atoms copied once (sf_copies 0) or every stage into both CTAs'
 * tensor memory (1: tcgen05.cp.cta_group::2 32x128b.warpx4, one per 128 rows
 * of A's and of B's scales per K = 64 step), a ring of 3 stages in flight.
 * *flops (host) receives 2 * 256 * n * 64 * 4 * stages * pairs. Waits are
 * bounded and report MOE_ERR_TIMEOUT in *status (optional device word);
 * other arguments outside the ranges return MOE_ERR_INVALID_ARG. */
int moe_fp4_mma_rate_pair(int n, int sf_copies, int stages, double* flops,
                          int32_t* status, void* stream);

/* ------------------------------------------------------------------------
 * Self-test of the failure path: runs the library's bounded mbarrier wait on
 * a barrier that nothing completes, with limit_ns (1 us .. 1 s). On return
 * (after a stream sync) *status holds MOE_ERR_TIMEOUT and result[0..1] == {1, 1}:
 * the waiting thread gave up at the limit, a second waiter (whose own limit
 * is 1 s) through the CTA's abort flag, after result[2] microseconds.
 * result is int32 [3]. No trap, no hang; the context stays usable.
 * ---------------------------------------------------------------------- */
int moe_selftest_wait_timeout(uint64_t limit_ns, int32_t* status, int32_t* result,
                              void* stream);

/* The same for the completion-counter wait of the one-launch expert GEMMs
 * (a GEMM2 unit polling the count of its route tile's finished GEMM1
 * units): both waiters poll *counter for a value of at least 1. counter is
 * a caller-owned device int32 that stays 0 (4-byte aligned); status, result
 * and the outcome are as for moe_selftest_wait_timeout. */
int moe_selftest_counter_timeout(uint64_t limit_ns, const int32_t* counter,
                                 int32_t* status, int32_t* result, void* stream);

/* Holds SMs the way another stream's kernel would, for testing that the
 * library's kernels finish while other work occupies part of the GPU: ctas
 * CTAs of one warp, each with smem_bytes (<= 227 KB) of dynamic shared memory
 * so that nothing else fits beside it on its SM, each exiting after ns
 * nanoseconds (at most 2 s) of spinning on the global timer. */
int moe_selftest_occupy(int ctas, int smem_bytes, uint64_t ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_NVFP4_H */
