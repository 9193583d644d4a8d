// Read-only streaming control kernel of libkq.
//
// A decode GEMV can at best read each weight byte once at the rate the memory
// system delivers bytes into an SM.  This kernel measures that rate on the
// data path the GEMV kernels use, with no arithmetic in the way: one
// persistent CTA per SM, a producer warp issuing bulk asynchronous copies
// (cp.async.bulk, L2 evict-first) into a ring of shared-memory stages, and
// sixteen consumer warps that read every 16-byte word of each stage back from
// shared memory, fold it into an XOR and free the stage.  The achieved rate is
// the in-harness ceiling that the GEMV kernels' bandwidth is measured against
// (the weight-bandwidth argument of "Kipp Benchmarks", "Decode is
// weight-bandwidth-bound"; the Bonsai page's measured practical ceiling of a
// read-only streaming kernel, section 8).
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {

constexpr int kCtlConsumerWarps = 16;
constexpr int kCtlThreads = 32 * (kCtlConsumerWarps + 1);
constexpr int kCtlMaxSmem = 227 * 1024;

__device__ unsigned int g_control_status = 0;

__device__ __forceinline__ int64_t min_i64(int64_t a, int64_t b) { return a < b ? a : b; }

// Bytes [c * stage_bytes, min(bytes, (c + 1) * stage_bytes)) form chunk c;
// CTA b streams chunks [nchunks * b / grid, nchunks * (b + 1) / grid).
__global__ void __launch_bounds__(kCtlThreads, 1)
    stream_read_kernel(const uint8_t* __restrict__ src, int64_t bytes, int stage_bytes, int stages,
                       uint32_t* __restrict__ sink) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * stage_bytes);
  uint64_t* empty = full + stages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + stages);
  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kCtlConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int64_t nchunks = (bytes + stage_bytes - 1) / stage_bytes;
  const int64_t cb = nchunks * blockIdx.x / gridDim.x, ce = nchunks * (blockIdx.x + 1) / gridDim.x;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      int64_t t = 0;
      for (int64_t c = cb; c < ce; ++c, ++t) {
        const int s = (int)(t % stages);
        const uint32_t par = (uint32_t)((t / stages) & 1);
        if (*abort_flag || !mbar_wait_bounded(&empty[s], par ^ 1u)) {
          *abort_flag = 1;
          atomicOr(&g_control_status, 1u << KQ_ERR_TIMEOUT);
          break;
        }
        const int64_t off = c * stage_bytes;
        const uint32_t len = (uint32_t)min_i64(stage_bytes, bytes - off);
        mbar_arrive_expect_tx(&full[s], len);
        bulk_g2s(smem + (size_t)s * stage_bytes, src + off, len, &full[s], policy);
      }
      // never leave the CTA with copies in flight
      for (int64_t u = t - 1; u >= 0 && u >= t - stages; --u)
        (void)mbar_wait_bounded(&full[u % stages], (uint32_t)((u / stages) & 1));
    }
    return;
  }

  const int cw = warp - 1;
  uint32_t acc = 0;
  int64_t t = 0;
  for (int64_t c = cb; c < ce; ++c, ++t) {
    const int s = (int)(t % stages);
    const uint32_t par = (uint32_t)((t / stages) & 1);
    if (*abort_flag) continue;
    if (!mbar_wait_bounded(&full[s], par)) {
      *abort_flag = 1;
      atomicOr(&g_control_status, 1u << KQ_ERR_TIMEOUT);
      continue;
    }
    const int64_t off = c * stage_bytes;
    const int words = (int)(min_i64(stage_bytes, bytes - off) / 16);
    const uint4* p = reinterpret_cast<const uint4*>(smem + (size_t)s * stage_bytes);
    for (int i = cw * 32 + lane; i < words; i += kCtlConsumerWarps * 32) {
      const uint4 v = p[i];
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (*abort_flag) return;
#pragma unroll
  for (int mk = 16; mk; mk >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, mk);
  if (lane == 0 && acc) atomicXor(sink, acc);
}

// Self-test of the bounded waits: one thread waits on an mbarrier whose phase
// nothing completes, with the library's bounded wait and a short limit, and
// records KQ_ERR_TIMEOUT as every kernel of the library does when a wait
// runs out.  No fault, no hang: the wait gives up and the kernel returns.
__global__ void wait_selftest_kernel(long long limit_cycles) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    if (!mbar_wait_bounded(&bar, 0, limit_cycles)) atomicOr(&g_control_status, 1u << KQ_ERR_TIMEOUT);
  }
}

int read_control_status(int clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_control_status, sizeof(v)) != cudaSuccess) return -1;
  if (clear) {
    unsigned int z = 0;
    cudaMemcpyToSymbol(g_control_status, &z, sizeof(z));
  }
  return (int)v;
}

}  // namespace kq

using namespace kq;

extern "C" int kq_stream_read(const void* d_src, int64_t bytes, int32_t stage_bytes, int32_t stages,
                              uint32_t* d_sink, void* stream) {
  clear_error();
  if (!d_src || !d_sink) return fail(KQ_ERR_INVALID_ARG, "NULL source or sink");
  if (bytes < 16 || bytes % 16 != 0) return fail(KQ_ERR_SHAPE, "bytes = %lld (a positive multiple of 16)", (long long)bytes);
  if (stage_bytes < 1024 || stage_bytes > 98304 || stage_bytes % 16 != 0)
    return fail(KQ_ERR_INVALID_ARG, "stage_bytes = %d (a multiple of 16 in [1024, 98304])", stage_bytes);
  if (stages < 1 || stages > 8) return fail(KQ_ERR_INVALID_ARG, "stages = %d (1..8)", stages);
  const size_t smem = (size_t)stages * (size_t)stage_bytes + 2 * (size_t)stages * 8 + 16;
  if (smem > (size_t)kCtlMaxSmem)
    return fail(KQ_ERR_INVALID_ARG, "ring of %zu bytes of shared memory with its barriers (at most %d)", smem,
                kCtlMaxSmem);
  if (!aligned16(d_src) || !aligned16(d_sink)) return fail(KQ_ERR_ALIGNMENT, "source or sink not 16-byte aligned");
  int dev = 0, sms = 0;
  KQ_CUDA_TRY(cudaGetDevice(&dev));
  KQ_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(stream_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kCtlMaxSmem);
  });
  if (attr_err != cudaSuccess) return fail(KQ_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));
  const int64_t nchunks = (bytes + stage_bytes - 1) / stage_bytes;
  const int grid = (int)std::min<int64_t>(nchunks, sms);
  stream_read_kernel<<<grid, kCtlThreads, smem, (cudaStream_t)stream>>>(static_cast<const uint8_t*>(d_src), bytes,
                                                                       stage_bytes, stages, d_sink);
  KQ_CUDA_TRY(cudaGetLastError());
  return KQ_OK;
}

extern "C" int kq_selftest_bounded_wait(int64_t limit_cycles, void* stream) {
  clear_error();
  if (limit_cycles < 1 || limit_cycles > kWaitLimitCycles)
    return fail(KQ_ERR_INVALID_ARG, "limit_cycles = %lld (1 .. %lld)", (long long)limit_cycles,
                (long long)kWaitLimitCycles);
  wait_selftest_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((long long)limit_cycles);
  KQ_CUDA_TRY(cudaGetLastError());
  return KQ_OK;
}
