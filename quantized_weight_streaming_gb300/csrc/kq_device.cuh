// Device helpers of libkq: shared-memory barriers (mbarrier), 1-D bulk copies
// (cp.async.bulk, the TMA engine without a tensor map) and bounded waits.
//
// Every wait in the library is bounded: after about one second of spinning
// it gives up, records KQ_ERR_TIMEOUT in the translation unit's device status
// word and returns false, so that a kernel never hangs the GPU.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace kq {

// Cycles a bounded wait spins before it gives up (about 1 s at 2 GHz).
constexpr long long kWaitLimitCycles = 2000000000LL;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// try_wait with a suspend-time hint: a thread whose phase is not complete is
// suspended (for at most kSuspendNs, woken when the phase completes) instead of
// returning at once, so waiting warps do not take issue slots from working ones.
constexpr uint32_t kSuspendNs = 20000;
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity), "r"(kSuspendNs)
      : "memory");
  return done != 0;
}

// Waits (suspended between checks) for the phase with the given parity to
// complete; false after about one second.
__device__ __forceinline__ bool mbar_wait_suspend(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait_suspend(bar, parity)) return true;
  long long start = clock64();
  while (!mbar_try_wait_suspend(bar, parity)) {
    if (clock64() - start > kWaitLimitCycles) return false;
  }
  return true;
}

// Waits for the phase with the given parity to complete; false once
// limit_cycles SM clock cycles have passed (about one second by default).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  long long limit_cycles = kWaitLimitCycles) {
  if (mbar_try_wait(bar, parity)) return true;
  long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - start > limit_cycles) return false;
  }
  return true;
}

// Programmatic dependent launch: waits until the grid launched before this
// one on the stream has completed and its writes are visible.  A kernel
// launched with the programmatic-serialization attribute may start (and run
// its prologue) while that grid is still running; launched without it, this
// returns at once.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Lets the grid launched after this one on the stream as a programmatic
// dependent begin: its CTAs take SMs as this grid's CTAs exit and run their
// prologue, then wait in grid_dependency_wait until this grid has completed.
// Every kernel of the library waits before its first global access, so the
// trigger can come as early as right after that wait.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches kernel k as a programmatic dependent of the stream's previous
// kernel (the kernel must call grid_dependency_wait before reading that
// kernel's outputs).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_dependent(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                    Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}

// L2 policy for data read exactly once (the weight stream): evict first.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Global -> shared bulk copy completing on `bar` (bytes and addresses multiples
// of 16).  The destination is this CTA's shared memory.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
      "%4;" ::"r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Named barrier among `count` threads (multiple of 32), id 1..15.
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace kq

namespace kq {

// 2-D tiled TMA load (cp.async.bulk.tensor) of the box at element coordinates
// (x, y) of the tensor map at `tmap` (a CUtensorMap in param or global memory)
// into this CTA's shared memory, completing on `bar`.  x is the innermost
// coordinate; callers keep x * element size a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const void* tmap, int32_t x, int32_t y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

}  // namespace kq
