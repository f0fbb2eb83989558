// moe_selftest_wait_timeout: the bounded-wait path every pipelined kernel of
// the library uses (mbar_wait), run on an mbarrier that nothing completes,
// with a caller-chosen short limit. Warp 0's lane 0 waits until the limit
// runs out, records MOE_ERR_TIMEOUT in the status word and raises the CTA's
// abort flag; warp 1's lane 0, waiting on the same barrier, must then give
// up through the flag (it records nothing). result[0..1] = 1 for each waiter
// that gave up, result[2] = microseconds the second one waited. Nothing traps
// or hangs: the kernel returns and the context stays usable.
#include "common.cuh"

namespace moe {

__global__ void selftest_wait_kernel(uint64_t limit_ns, int32_t* status, int32_t* result) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);  // one arrival expected, none will come
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    // warp 1 waits with the full 1 s limit: the abort flag should end it long
    // before; result[2] is how long it waited (microseconds)
    const uint64_t limit = warp == 0 ? limit_ns : kWaitLimitNs;
    const uint64_t t0 = global_timer_ns();
    const bool ok = mbar_wait(smem_u32(&bar), 0, &abort_flag, warp == 0 ? status : nullptr, limit);
    result[warp] = ok ? 0 : 1;
    if (warp == 1) result[2] = (int32_t)((global_timer_ns() - t0) / 1000u);
  }
}

// The same for the completion-counter wait (wait_counter_at_least) the
// one-launch expert GEMMs use between GEMM1 and GEMM2 units: both waiters
// poll a counter the caller keeps at 0 for a target of 1.
__global__ void selftest_counter_kernel(uint64_t limit_ns, const int32_t* counter, int32_t* status,
                                        int32_t* result) {
  __shared__ int abort_flag;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    const uint64_t limit = warp == 0 ? limit_ns : kWaitLimitNs;
    const uint64_t t0 = global_timer_ns();
    const bool ok = wait_counter_at_least(counter, 1, &abort_flag, warp == 0 ? status : nullptr, limit);
    result[warp] = ok ? 0 : 1;
    if (warp == 1) result[2] = (int32_t)((global_timer_ns() - t0) / 1000u);
  }
}

// Holds SMs for a while, as another stream's kernel would: every CTA keeps
// `smem` bytes of dynamic shared memory (so that nothing else fits beside
// it on its SM) and thread 0 spins on the global timer until ns have passed
// (at most 2 s), then the CTA exits.
__global__ void selftest_occupy_kernel(uint64_t ns) {
  extern __shared__ uint8_t held[];
  if (threadIdx.x == 0) {
    const uint64_t t0 = global_timer_ns();
    while (global_timer_ns() - t0 < ns) __nanosleep(1000);
    held[0] = 0;
  }
}

int launch_selftest_occupy(int ctas, int smem, uint64_t ns, cudaStream_t stream) {
  if (ensure_smem_limit(reinterpret_cast<const void*>(selftest_occupy_kernel), 227 * 1024) != cudaSuccess)
    return MOE_ERR_CUDA;
  selftest_occupy_kernel<<<ctas, 32, smem, stream>>>(ns);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_selftest_counter(uint64_t limit_ns, const int32_t* counter, int32_t* status, int32_t* result,
                            cudaStream_t stream) {
  selftest_counter_kernel<<<1, 64, 0, stream>>>(limit_ns, counter, status, result);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_selftest_wait(uint64_t limit_ns, int32_t* status, int32_t* result, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 64, 0, stream>>>(limit_ns, status, result);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
