// The one-launch Q8_0 GEMV for small matrices ("Kipp Benchmarks", the
// batch-1 Q8_0 matvec of decode; the Q8_0 format as the Kipp architecture
// page defines it: blocks of 32 int8 codes with one fp16 scale).
//
// A small matrix (a few MB) spreads too little work per SM for the
// streaming kernel's fixed path (the shared-memory ring, its barriers and
// the copies' first round trip) and its K splits' second pass to pay off.
// Here each warp owns one row and loads it straight into registers, 16 bytes
// per lane at a time, all of the row's loads in flight at once; the CTA
// stages the activation in shared memory meanwhile.  No K split: one launch
// per call, and each output is one warp's sum in a fixed order.  The CTA is
// small enough to start beside the kernel ahead of it, and it has L2 fetch
// its rows while it waits for that kernel.
//
//   y[r] = sum_b d[r][b] * sum_{j in b} q[r][j] * x[j]
//
// Lane l takes the 16-byte granules g = l, l + 32, ... of its row (half a
// 32-code block each); it adds d * (its granule's dot product, two chains
// of eight FMAs) in granule order, and the warp adds the 32 lane sums with a
// fixed butterfly.  An int8 code becomes an exact float by a byte permute
// into the mantissa of 2^23 and one subtract.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {
namespace direct {

constexpr int kWarps = 8;                    // rows per CTA
constexpr int kThreads = 32 * kWarps;
constexpr int kMaxGranules = 8;              // per lane: k up to 32 x 8 x 16 = 4096
constexpr int64_t kMaxK = 32 * kMaxGranules * 16;

// the four int8 codes of word w as exact floats: each, biased by 128, is the low
// byte of the mantissa of 2^23, and the subtract takes 2^23 + 128 off again
__device__ __forceinline__ void codes4(uint32_t w, float (&f)[4]) {
  const uint32_t u = w ^ 0x80808080u;  // q + 128 in each byte
#pragma unroll
  for (int j = 0; j < 4; ++j)
    f[j] = __int_as_float((int)__byte_perm(u, 0x4B000000u, 0x7650u | (uint32_t)j)) - 8388736.0f;  // 2^23 + 128
}

// IO16: the fp16 chain (fp16 x in, fp16 y out, fp32 accumulation rounded
// once at the end).
template <bool IO16>
__global__ void __launch_bounds__(kThreads) q8_0_gemv_kernel(const int8_t* __restrict__ codes,
                                                             const __half* __restrict__ scales, int64_t n, int k,
                                                             int64_t sstride, const void* __restrict__ x,
                                                             void* __restrict__ y) {
  // The activation, k floats, as float4 q of granule g at [q * (k / 16) + g]:
  // the lanes of a warp, on consecutive granules, read consecutive entries.
  extern __shared__ float4 xs4[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  const int ngran = k / 16;
  const bool live = row < n;
  // Launched as a programmatic dependent, the CTA may start while the kernel
  // ahead still runs: it asks L2 for its row's codes (a prefetch, which
  // returns no data: L2 is where that kernel's writes land, so the loads
  // after the wait still see them), then reads nothing before that kernel
  // has completed.
  if (live && lane == 0)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(codes + row * (int64_t)k), "r"((uint32_t)k)
                 : "memory");
  grid_dependency_wait();
  allow_dependent_launch();

  // the row's codes and scales, all in flight before the activation staging
  uint4 cw[kMaxGranules];
  float d[kMaxGranules];
  const uint4* crow = reinterpret_cast<const uint4*>(codes + (live ? row : 0) * (int64_t)k);
  const __half* srow = scales + (live ? row : 0) * sstride;
#pragma unroll
  for (int i = 0; i < kMaxGranules; ++i) {
    const int g = lane + 32 * i;
    if (live && g < ngran) {
      cw[i] = __ldcs(crow + g);
      d[i] = __half2float(__ldg(srow + (g >> 1)));
    } else {
      cw[i] = make_uint4(0u, 0u, 0u, 0u);
      d[i] = 0.f;
    }
  }
  for (int t = threadIdx.x; t < k / 4; t += kThreads) {
    float4 v;
    if constexpr (IO16) {
      const uint2 h = __ldcg(reinterpret_cast<const uint2*>(x) + t);
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
      const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
      v = make_float4(a.x, a.y, b.x, b.y);
    } else {
      v = __ldcg(reinterpret_cast<const float4*>(x) + t);
    }
    xs4[(t & 3) * ngran + (t >> 2)] = v;
  }
  __syncthreads();
  if (!live) return;

  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxGranules; ++i) {
    const int g = lane + 32 * i;
    if (g < ngran) {
      const uint32_t wv[4] = {cw[i].x, cw[i].y, cw[i].z, cw[i].w};
      float p0 = 0.f, p1 = 0.f;  // codes 0-7 and 8-15 of the granule
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float4 xa = xs4[(2 * h) * ngran + g], xb = xs4[(2 * h + 1) * ngran + g];
        float f0[4], f1[4];
        codes4(wv[2 * h], f0);
        codes4(wv[2 * h + 1], f1);
        float& p = h ? p1 : p0;
        p = fmaf(f0[0], xa.x, p);
        p = fmaf(f0[1], xa.y, p);
        p = fmaf(f0[2], xa.z, p);
        p = fmaf(f0[3], xa.w, p);
        p = fmaf(f1[0], xb.x, p);
        p = fmaf(f1[1], xb.y, p);
        p = fmaf(f1[2], xb.z, p);
        p = fmaf(f1[3], xb.w, p);
      }
      acc = fmaf(d[i], p0 + p1, acc);
    }
  }
#pragma unroll
  for (int mk = 16; mk; mk >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, mk);
  if (lane == 0) {
    if constexpr (IO16)
      static_cast<__half*>(y)[row] = __float2half_rn(acc);
    else
      static_cast<float*>(y)[row] = acc;
  }
}

}  // namespace direct

bool gemv_direct_applies(const kq_qmat* W, int64_t m) {
  return m == 1 && W->fmt == KQ_Q8_0 && W->k <= direct::kMaxK && W->n * W->k <= kGemvDirectMaxBytes;
}

int gemv_direct(const kq_qmat* W, const void* d_x, void* d_y, bool io16, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  const dim3 grid((unsigned)((W->n + direct::kWarps - 1) / direct::kWarps)), block(direct::kThreads);
  const size_t smem = (size_t)W->k * sizeof(float);
  const int8_t* codes = static_cast<const int8_t*>(W->codes);
  const __half* scales = static_cast<const __half*>(W->scales);
  const int64_t ss = scale_stride(KQ_Q8_0, W->k);
  if (io16)
    KQ_CUDA_TRY(launch_dependent(direct::q8_0_gemv_kernel<true>, grid, block, smem, st, codes, scales, W->n,
                                 (int)W->k, ss, d_x, d_y));
  else
    KQ_CUDA_TRY(launch_dependent(direct::q8_0_gemv_kernel<false>, grid, block, smem, st, codes, scales, W->n,
                                 (int)W->k, ss, d_x, d_y));
  return KQ_OK;
}

}  // namespace kq
