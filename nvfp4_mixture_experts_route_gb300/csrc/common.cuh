// Shared device helpers for libmoe_nvfp4: status reporting, bounded
// mbarrier waits, TMA and tcgen05 (5th-generation tensor core) PTX wrappers
// for sm_103a, and the NVFP4 conversions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <utility>

#include "../../include/moe_nvfp4.h"

namespace moe {

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device. The limit set is remembered per (kernel, device), so that
// later launches that need no more (including ones recorded into a CUDA
// graph) make no attribute call; a launch that needs more raises it again.
inline cudaError_t ensure_smem_limit(const void* func, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> limit;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(mu);
  auto it = limit.find({func, dev});
  if (it != limit.end() && it->second >= bytes) return cudaSuccess;
  err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  // Ask for the largest shared-memory carveout: the kernels that come here
  // size their CTAs per SM from the whole 228 KB.
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                               (int)cudaSharedmemCarveoutMaxShared);
  if (err == cudaSuccess) limit[{func, dev}] = bytes;
  return err;
}

// ---------------------------------------------------------------------------
// Status word: the first device-side error wins.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void record_status(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch. A kernel launched with the programmatic
// stream-serialization attribute may start while the previous kernel on the
// stream drains; it must call pdl_wait() before it touches anything that
// kernel writes (or reads and this kernel overwrites). pdl_wait() returns once
// the previous kernel has completed and its memory is visible; without the
// attribute it returns at once. pdl_trigger() lets the next kernel be
// scheduled early; this library calls it only after its own pdl_wait(), so
// that everything before the previous kernel is complete when the next one
// starts.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kern` on `stream`, with the programmatic stream-serialization
// attribute when `pdl` is set.
template <typename... Params, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t stream, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Shared-memory addresses and mbarriers.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Every wait on the device gives up after this long and reports
// MOE_ERR_TIMEOUT; nothing in a correct launch waits more than microseconds.
constexpr uint64_t kWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

// Wait for phase `parity` of an mbarrier. Returns false (after recording
// MOE_ERR_TIMEOUT and raising *abort) if the wait ran out or another thread
// of the CTA already gave up. try_wait itself suspends the thread until the
// phase completes or a short hardware time limit passes, so the loop re-polls
// without sleeping (a sleep would delay the wake-up on the pipeline's
// critical path); the abort flag and the clock are read every 16 polls.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int32_t* status, uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        record_status(status, MOE_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// The same wait with acquire at cluster scope, for an mbarrier that the
// other CTA of a cluster arrives on (release at cluster scope).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  int32_t* status) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((n & 15u) == 0) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        record_status(status, MOE_ERR_TIMEOUT);
        *abort = 1;
        return false;
      }
    }
  }
}

// mbar_wait by every lane of a converged warp, with one outcome for all of
// them (false if any lane gave up), so that a warp-converged issue loop stays
// converged.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int* abort,
                                               int32_t* status) {
  const bool ok = mbar_wait(bar, parity, abort, status);
  return __all_sync(0xFFFFFFFFu, ok);
}

template <bool W>
__device__ __forceinline__ bool mbar_wait_f(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* status) {
  if constexpr (W)
    return mbar_wait_warp(bar, parity, abort, status);
  else
    return mbar_wait(bar, parity, abort, status);
}

// Bounded wait until the int32 *counter (global memory, raised by other CTAs
// after a GPU-scope release) is at least target: acquire loads at GPU scope,
// a short sleep between polls after the first eight. Gives up through the
// CTA's abort flag, or after limit_ns recording MOE_ERR_TIMEOUT and raising
// the flag; returns whether the count was reached.
__device__ __forceinline__ bool wait_counter_at_least(const int32_t* counter, int32_t target,
                                                      volatile int* abort, int32_t* status,
                                                      uint64_t limit_ns = kWaitLimitNs) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t n = 0;; ++n) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    if (v >= target) return true;
    if (*abort) return false;
    if (n >= 8) __nanosleep(64);
    if ((n & 15u) == 15u && global_timer_ns() - t0 > limit_ns) {
      record_status(status, MOE_ERR_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

// Bounded wait used only on the clean-up path (no status update).
__device__ __forceinline__ void mbar_wait_cleanup(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) return;
    __nanosleep(256);
  }
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies) and plain bulk copies, global -> shared.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// The pair form of the same load: the box lands in this CTA's shared memory
// and its bytes complete on an mbarrier of either CTA of the pair (`bar` is a
// shared::cluster address, e.g. from mapa), so that one CTA's barrier can
// count both CTAs' halves of a stage.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar_cluster,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
// The shared::cluster address of the variable at local shared offset `addr`
// in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// The same loads with an L2 eviction policy (a createpolicy value): data
// that streams through once is marked evict_first, so that what was written
// during the launch and is read again soon stays in L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x,
                                                 int32_t y, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                               uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// Prefetch one box of a tensor map, or a contiguous range (16-byte multiple),
// from global memory into L2 only (no shared-memory destination, nothing to
// wait for).
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, block-scaled FP4 MMA, copies and loads.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address >> 4 in
// bits [0,14), leading byte offset >> 4 in [16,30), stride byte offset >> 4
// in [32,46), descriptor version 1 in [46,48), base offset 0, swizzle mode in
// [61,64) (0 none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 0x7u) << 61;
  return d;
}

// Copy one 512-byte scale atom (32 rows x 16 bytes, no swizzle) into four
// tensor-memory columns, replicated over the four 32-lane quadrants.
__device__ __forceinline__ void tc_copy_scale_atom(uint32_t taddr, uint64_t desc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(desc)
               : "memory");
}

// D[tmem] (+)= A[smem] . B[smem]^T with e2m1 operands and one ue4m3 scale
// per 16 K-elements from tensor memory; M = 128, K = 64 per instruction.
__device__ __forceinline__ void tc_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// Make the mbarrier track completion of every tcgen05 op this thread issued.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Warp-converged forms of the three above: the whole warp executes them with
// the same operands in every lane, and lane 0 issues the instruction under a
// predicate inside the asm instead of behind a lane-0 branch. The issuing
// thread is still lane 0 (its tcgen05.commit tracks what it issued). An issue
// loop run this way by a converged warp measured 1.3-1.7x the instruction
// rate of the same loop run by lane 0 alone.
#define MOE_LANE0_PRED \
  "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
__device__ __forceinline__ void tcw_copy_scale_atom(uint32_t taddr, uint64_t desc) {
  asm volatile(MOE_LANE0_PRED "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
               "l"(desc)
               : "memory");
}
__device__ __forceinline__ void tcw_mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(MOE_LANE0_PRED
               ".reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "@e tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
               " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d_tmem),
               "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
               : "memory");
}
__device__ __forceinline__ void tcw_commit(uint32_t bar) {
  asm volatile(MOE_LANE0_PRED
               "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
               : "memory");
}
#undef MOE_LANE0_PRED

// The issue form chosen at compile time: W = warp-converged (tcw_*), else
// the calling thread alone (tc_*).
template <bool W>
__device__ __forceinline__ void tc_copy_scale_atom_f(uint32_t taddr, uint64_t desc) {
  if constexpr (W)
    tcw_copy_scale_atom(taddr, desc);
  else
    tc_copy_scale_atom(taddr, desc);
}
template <bool W>
__device__ __forceinline__ void tc_mma_nvf4_f(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
  if constexpr (W)
    tcw_mma_nvf4(d_tmem, adesc, bdesc, idesc, sfa_tmem, sfb_tmem, accumulate);
  else
    tc_mma_nvf4(d_tmem, adesc, bdesc, idesc, sfa_tmem, sfb_tmem, accumulate);
}
template <bool W>
__device__ __forceinline__ void tc_commit_f(uint32_t bar) {
  if constexpr (W)
    tcw_commit(bar);
  else
    tc_commit(bar);
}

// ---------------------------------------------------------------------------
// The pair form (cta_group::2): two CTAs of a cluster, on two SMs, share one
// MMA of M = 256 (A rows 0-127 from rank 0's shared memory, 128-255 from rank
// 1's, the same offsets); each CTA's tensor memory holds its 128 rows of the
// accumulator. Tensor memory is allocated and freed by one warp of each CTA
// together; rank 0 issues the copies, MMAs and commits. Every tcgen05
// instruction of a kernel that uses the pair form takes cta_group::2.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of both CTAs: release what this CTA wrote, acquire the peer's.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Issued by lane 0 of a converged warp (the predicate is set inside the asm).
#define MOE_PAIR_PRED \
  "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
__device__ __forceinline__ void pair_copy_atom(uint32_t taddr, uint64_t desc) {
  asm volatile(MOE_PAIR_PRED "@e tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr), "l"(desc)
               : "memory");
}
__device__ __forceinline__ void pair_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                         uint32_t acc) {
  asm volatile(MOE_PAIR_PRED
               ".reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "@e tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X"
               " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" ::"r"(d),
               "l"(a), "l"(b), "r"(idesc), "r"(acc), "r"(sfa), "r"(sfb)
               : "memory");
}
// Commit to this CTA's mbarrier.
__device__ __forceinline__ void pair_commit(uint32_t bar) {
  asm volatile(MOE_PAIR_PRED "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                   bar)
               : "memory");
}
// Commit to the mbarrier at the same offset in both CTAs of the pair.
__device__ __forceinline__ void pair_commit_both(uint32_t bar) {
  asm volatile(MOE_PAIR_PRED
               "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
               " [%0], %1;\n\t}" ::"r"(bar),
               "h"((uint16_t)3)
               : "memory");
}
#undef MOE_PAIR_PRED
// Arrive (release at cluster scope) on the mbarrier at local offset `bar` in
// the shared memory of cluster CTA `rank`.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar, uint32_t rank) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n\t}" ::"r"(bar),
      "r"(rank)
      : "memory");
}
// The same arrive without release semantics: for a hand-off that orders no
// memory, only tensor-memory reads that tcgen05.wait::ld has already
// completed (a release at cluster scope costs the arriving thread about
// 0.7 us).
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t bar, uint32_t rank) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\t"
      "mapa.shared::cluster.u32 ra, %0, %1;\n\t"
      "mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [ra];\n\t}" ::"r"(bar),
      "r"(rank)
      : "memory");
}

// Instruction descriptor for kind::mxf4nvf4: A and B e2m1 (format 1) in bits
// [7,10) and [10,13), both K-major, N >> 3 in [17,23), scale type ue4m3 (0)
// in bit 23, M >> 4 in [24,29), scale-factor ids 0, dense K = 64.
__host__ __device__ constexpr uint32_t idesc_nvf4(uint32_t M, uint32_t N) {
  return (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// 32 lanes x 32 bit, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// The same load without the wait: the registers are valid only after
// tmem_wait_ld(), which lets one warp have several loads in flight.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------------------
// NVFP4 conversions (PTX cvt with round-to-nearest-even and saturation).
// ---------------------------------------------------------------------------
// e4m3 code of a non-negative fp32 value (satfinite).
__device__ __forceinline__ uint32_t f32_to_e4m3(float v) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(v));
  return r & 0xFFu;
}

// fp32 value of an e4m3 code (exact: every e4m3 value is an fp16 value).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint32_t h2;
  uint16_t in = static_cast<uint16_t>(code & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
}

// Two e2m1 codes in one byte: `lo` in bits [0,4), `hi` in bits [4,8).
__device__ __forceinline__ uint32_t f32x2_to_e2m1x2(float lo, float hi) {
  uint16_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "mov.b16 %0, {t, 0};\n\t}"
      : "=h"(r)
      : "f"(hi), "f"(lo));
  return r & 0xFFu;
}

// NVFP4 of one 16-element block with global scale g; same arithmetic as the
// input quantization (s = amax*g/6, sf = e4m3(s), q = e2m1(v * g/sf)).
__device__ __forceinline__ void quant16(const float (&v)[16], float g, uint2& codes,
                                        uint32_t& sf_code) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  sf_code = f32_to_e4m3((amax * g) / 6.0f);
  const float sfv = e4m3_to_f32(sf_code);
  uint32_t lo = 0, hi = 0;
  if (sfv > 0.f) {
    const float inv = g / sfv;
#pragma unroll
    for (int i = 0; i < 8; i += 2) lo |= f32x2_to_e2m1x2(v[i] * inv, v[i + 1] * inv) << (4 * i);
#pragma unroll
    for (int i = 0; i < 8; i += 2)
      hi |= f32x2_to_e2m1x2(v[8 + i] * inv, v[9 + i] * inv) << (4 * i);
  }
  codes = make_uint2(lo, hi);
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// Tensor maps (host).
// ---------------------------------------------------------------------------
// cuTensorMapEncodeTiled is a driver API entry; it is looked up through the
// runtime so that the library does not link libcuda (and loads on hosts
// without a driver). The lookup is done once per process.
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// A [rows, row_bytes] byte matrix read in 128-byte-wide, box_rows-high,
// 128-byte-swizzled boxes (the K-major operand tiles of the tcgen05 GEMMs).
inline CUresult encode_rows_map(CUtensorMap* map, const void* base, uint64_t row_bytes,
                                uint64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {row_bytes, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {128u, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
            elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}


// Scale-atom arrays as a 2D uint8 tensor of 128-byte rows (4 rows per
// 512-byte atom), boxes of box_rows rows, no swizzle: a TMA tensor load of
// 16 rows brings the 4 atoms of a K = 256 stage.
inline CUresult encode_atoms_map(CUtensorMap* map, const void* base, uint64_t bytes, uint32_t box_rows) {
  auto fn = encode_fn();
  if (fn == nullptr) return CUDA_ERROR_NOT_FOUND;
  const cuuint64_t dims[2] = {128u, bytes / 128u};
  const cuuint64_t strides[1] = {128u};
  const cuuint32_t box[2] = {128u, box_rows};
  const cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Packed fp32x2 arithmetic (one instruction for two lanes of the pair):
// d = a * b + c and d = a * b, each element rounded as its scalar form.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)),
        "l"(*reinterpret_cast<unsigned long long*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<unsigned long long*>(&a)), "l"(*reinterpret_cast<unsigned long long*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

}  // namespace moe
