// moe_nvfp4_experts_noalloc: the expert body (moe_nvfp4_experts) with its
// workspace in a fixed device array of this library instead of a
// caller-provided buffer, for callers that cannot allocate device memory.
#include <cstddef>
#include <mutex>

#include "common.cuh"

namespace moe {
int report_error(int code, const char* fmt, ...);
}

namespace {

// Largest workspace the no-allocation entry point can serve. The workspace
// size depends only on the shape (moe_experts_workspace_size), never on the
// routing: at H = 5120, I = 2048, E = 128, top-8 and tile_m = 32 a batch of 8
// tokens needs 11 MB, 64 tokens 24 MB, and up to 287 tokens fit. Every GPU
// that loads the library holds this array until the process exits.
constexpr size_t kScratchBytes = size_t(32) << 20;
// The array is 256-byte aligned; up to 768 bytes are skipped to give the
// workspace the 1024-byte alignment moe_nvfp4_experts asks for.
constexpr size_t kAlignSlack = 1024;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes + kAlignSlack];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
  CUcontext ctx;  // the context the address belongs to
  void* addr;
};
Cached g_addr[kMaxDevices] = {};

// The calling thread's current context, through the driver entry point the
// runtime hands out (the library does not link libcuda); null if unknown.
CUcontext current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = []() -> PFN_cuCtxGetCurrent_v4000 {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f);
  }();
  CUcontext c = nullptr;
  if (fn == nullptr || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

// Device address of g_scratch on the current device, looked up on the first
// call and again whenever the device's context has changed since (a
// cudaDeviceReset tears the module down with its context; the array then
// lives at a new address). In host code `g_scratch` names a host-side
// shadow, not the device array, so it must never be passed to a kernel
// directly.
int scratch_address(void** out) {
  int dev = -1;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return moe::report_error(MOE_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(err));
  if (dev < 0 || dev >= kMaxDevices)
    return moe::report_error(MOE_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  const CUcontext ctx = current_context();
  if (g_addr[dev].addr == nullptr || ctx == nullptr || ctx != g_addr[dev].ctx) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_scratch);
    if (err != cudaSuccess || p == nullptr)
      return moe::report_error(MOE_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(err));
    // the lookup makes the device's primary context current if it was not
    g_addr[dev] = Cached{current_context(), p};
  }
  *out = g_addr[dev].addr;
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_noalloc_scratch_bytes(void) { return kScratchBytes; }

int moe_nvfp4_experts_noalloc(const moe_weights* w, const void* x, const void* a, const void* a_sf,
                              const float* a1_gscale, const float* a2_gscale, const moe_route* r,
                              int T, int H, int I, int E, int K, int tile_m, void* gemm2_rows,
                              int32_t* status, void* stream) {
  size_t need = 0;
  int rc = moe_experts_workspace_size(T, K, E, H, I, tile_m, &need);
  if (rc != MOE_OK) return rc;
  if (need > kScratchBytes)
    return moe::report_error(MOE_ERR_WORKSPACE,
                             "this shape needs %zu bytes of workspace; the no-allocation entry "
                             "point holds %zu (use moe_nvfp4_experts with your own buffer)",
                             need, kScratchBytes);
  void* base = nullptr;
  rc = scratch_address(&base);
  if (rc != MOE_OK) return rc;
  const uintptr_t b = reinterpret_cast<uintptr_t>(base);
  void* ws = reinterpret_cast<void*>((b + kAlignSlack - 1) & ~uintptr_t(kAlignSlack - 1));
  return moe_nvfp4_experts(w, x, a, a_sf, a1_gscale, a2_gscale, r, T, H, I, E, K, tile_m,
                           gemm2_rows, ws, kScratchBytes, status, stream);
}

}  // extern "C"
