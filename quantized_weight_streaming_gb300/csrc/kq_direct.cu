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
#include "kq_stream.cuh"

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

// ---------------------------------------------------------------------------
// PQ2_0 ("Bonsai 2 27B": ternary g128 codes, the weights folded with the
// blockwise Hadamard R of section 4.2, so y = W' (R x); the ternary matvec of
// section 8.5 with the -1 folded into the sum of x').
//
// A CTA owns kSlabs slabs of 16 rows; each slab's K is cut into kParts parts,
// one warp per (slab, part).  The CTA first rotates the whole x itself (each
// warp takes every kWarps-th 128-block) into a B table of fp16 high and low
// parts, then each warp runs mma.sync.m16n8k16 over its part with the codes
// loaded straight from global memory into registers; the parts of a row are
// added in part order through shared memory.
//
// The tensor-core scheme is the streaming kernel's: a 2-bit code masked in
// place inside its 16-bit half is the exact fp16 denormal c * 2^(s-24) for
// bit position s <= 10 (s = 10 only for c <= 2, which ternary codes are);
// one AND per two codes builds an A register, one shift by 4 brings the
// pairs at bits 12 and 14 down to 8 and 10.  B holds x' * 2^-E (E the
// block's exponent) times 2^(14-s), split into high and low fp16 parts in
// columns 0 and 1, so a block's 8 MMAs give C = sum c x' 2^(-10-E), and
//     y += d * (2^(10+E) * C - sum_{j in block} x'_j).
// Word layout: thread (g = lane/4, t = lane%4) loads words 2t and 2t+1 of
// each 8-word block row of rows g and g+8 (one 8-byte load each, the four
// threads of a row covering its 32 bytes), and word group q of a block is
// word 2t+q of thread t, so every MMA stays inside one block.
// ---------------------------------------------------------------------------
namespace pq {

constexpr int kSlabs = 5;   // 16-row slabs per CTA
constexpr int kParts = 3;   // K parts per slab
constexpr int kWarps = kSlabs * kParts;
constexpr int kThreads = 32 * kWarps;
constexpr int kRows = 16 * kSlabs;
constexpr int kMaxBlk = 14;  // 128-blocks per part: k up to 3 x 14 x 128 = 5376
constexpr int64_t kMaxK = (int64_t)kParts * kMaxBlk * 128;
constexpr int64_t kMaxCodeBytes = 16ll << 20;

// shared memory: per-warp scratch (one block of x'), the B table (4 bytes per
// position), per block 2^(10+E) and sum x', and the parts' partial outputs
__host__ __device__ constexpr size_t scratch_bytes() { return (size_t)kWarps * 128 * 4; }
__host__ __device__ constexpr size_t smem_bytes(int64_t k) {
  return scratch_bytes() + (size_t)k * 4 + 2 * (size_t)(k / 128) * 4 + (size_t)(kParts - 1) * kRows * 4;
}

// the denormal bit position of register `reg` of MMA j (0: word elements 2j
// and 2j+8; 1: 2j+1 and 2j+9), after the shift for j = 3
__device__ __forceinline__ int pair_bit(int j, int reg) { return j < 3 ? 4 * j + 2 * reg : 8 + 2 * reg; }

// B table entry of (block b, word group q, MMA j, column n: 0 high / 1 low,
// thread t)
__device__ __forceinline__ int btab_index(int b, int q, int j, int n, int t) {
  return (((b * 2 + q) * 4 + j) * 2 + n) * 4 + t;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  return (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// IO16: the fp16 chain (fp16 x, x' rounded to fp16 right after the
// transform, fp16 y rounded once at the end).
template <bool IO16>
__global__ void __launch_bounds__(kThreads, 1) pq2_0_gemv_kernel(const uint32_t* __restrict__ codes,
                                                                 const __half* __restrict__ scales, int64_t n,
                                                                 int k, int64_t sstride,
                                                                 const void* __restrict__ x, void* __restrict__ y) {
  extern __shared__ __align__(16) uint8_t sm[];
  const int nblk = k / 128;
  float* scratch_all = reinterpret_cast<float*>(sm);
  uint2* btab = reinterpret_cast<uint2*>(sm + scratch_bytes());
  float* fx = reinterpret_cast<float*>(sm + scratch_bytes() + (size_t)k * 4);
  float* sx = fx + nblk;
  float* comb = sx + nblk;  // [kParts - 1][kRows]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slab = warp % kSlabs, part = warp / kSlabs;
  const int g = lane >> 2, t = lane & 3;
  const int64_t wpr = k / 16;  // code words per row
  const int64_t row0 = (int64_t)blockIdx.x * kRows + slab * 16;
  const int64_t rA = row0 + g, rB = row0 + g + 8;
  const bool liveA = rA < n, liveB = rB < n;

  // Launched as a programmatic dependent: the slab's rows are asked of L2
  // first (a prefetch returns no data, and L2 is where the kernel ahead
  // writes), then nothing is read before that kernel has completed.
  if (part == 0 && lane < 16 && row0 + lane < n)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(codes + (row0 + lane) * wpr),
                 "r"((uint32_t)(k / 4))
                 : "memory");
  grid_dependency_wait();
  allow_dependent_launch();

  // this part's blocks [b0, b1); their codes and scales for rows g and g+8
  const int per = (nblk + kParts - 1) / kParts;
  const int b0 = part * per, b1 = min(nblk, b0 + per);
  uint2 cA[kMaxBlk], cB[kMaxBlk];
  float dA[kMaxBlk], dB[kMaxBlk];
#pragma unroll
  for (int i = 0; i < kMaxBlk; ++i) {
    const int b = b0 + i;
    cA[i] = cB[i] = make_uint2(0u, 0u);
    dA[i] = dB[i] = 0.f;
    if (b < b1) {
      if (liveA) {
        cA[i] = __ldcs(reinterpret_cast<const uint2*>(codes + rA * wpr + 8 * b) + t);
        dA[i] = __half2float(__ldg(scales + rA * sstride + b));
      }
      if (liveB) {
        cB[i] = __ldcs(reinterpret_cast<const uint2*>(codes + rB * wpr + 8 * b) + t);
        dB[i] = __half2float(__ldg(scales + rB * sstride + b));
      }
    }
  }

  // x' = R x per block, its exponent and sum, and its B table entries
  float* scratch = scratch_all + warp * 128;
  const float inv_sqrt128 = 0.08838834764831845f;
  for (int b = warp; b < nblk; b += kWarps) {
    float v[4];
    if constexpr (IO16) {
      const uint2 h = __ldcg(reinterpret_cast<const uint2*>(static_cast<const __half*>(x) + 128 * b + 4 * lane));
      const float2 p0 = __half22float2(*reinterpret_cast<const __half2*>(&h.x));
      const float2 p1 = __half22float2(*reinterpret_cast<const __half2*>(&h.y));
      v[0] = p0.x;
      v[1] = p0.y;
      v[2] = p1.x;
      v[3] = p1.y;
    } else {
      const float4 f = __ldcg(reinterpret_cast<const float4*>(static_cast<const float*>(x) + 128 * b + 4 * lane));
      v[0] = f.x;
      v[1] = f.y;
      v[2] = f.z;
      v[3] = f.w;
    }
    fwht128_lane4(v, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      v[i] = IO16 ? __half2float(__float2half_rn(v[i] * inv_sqrt128)) : v[i] * inv_sqrt128;
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
    for (int mk = 16; mk; mk >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, mk));
    // block exponent E with amax < 2^(E+1), clamped to [-100, 100]
    int e = amax > 0.f ? ((__float_as_int(amax) >> 23) & 0xFF) - 127 : 0;
    if (amax > 0.f && e == -127) e = -126;  // denormal block maximum
    e = max(-100, min(100, e));
    const float unscale = pow2f(-e);
    float s = v[0] + v[1] + v[2] + v[3];
#pragma unroll
    for (int mk = 16; mk; mk >>= 1) s += __shfl_xor_sync(0xffffffffu, s, mk);
    __syncwarp();
    *reinterpret_cast<float4*>(scratch + 4 * lane) =
        make_float4(v[0] * unscale, v[1] * unscale, v[2] * unscale, v[3] * unscale);
    __syncwarp();
    // lane (q, j, tt) builds the high and low entries of word 2 tt + q for MMA j
    const int tt = lane & 3, j = (lane >> 2) & 3, q = lane >> 4;
    const float* xw = scratch + 16 * (2 * tt + q);
    const float s0 = pow2f(14 - pair_bit(j, 0)), s1 = pow2f(14 - pair_bit(j, 1));
    const float u0 = xw[2 * j] * s0, u1 = xw[2 * j + 8] * s0, u2 = xw[2 * j + 1] * s1, u3 = xw[2 * j + 9] * s1;
    const float h0 = __half2float(__float2half_rn(u0)), h1 = __half2float(__float2half_rn(u1));
    const float h2 = __half2float(__float2half_rn(u2)), h3 = __half2float(__float2half_rn(u3));
    btab[btab_index(b, q, j, 0, tt)] = make_uint2(pack_half2(h0, h1), pack_half2(h2, h3));
    btab[btab_index(b, q, j, 1, tt)] = make_uint2(pack_half2(u0 - h0, u1 - h1), pack_half2(u2 - h2, u3 - h3));
    if (lane == 0) {
      sx[b] = s;
      fx[b] = pow2f(10 + e);
    }
  }
  __syncthreads();

  // B column g of the fragment: 0 (high) or 1 (low); lanes g >= 2 read
  // column 0 again, their products land in output columns nobody reads
  const int ncol = g < 2 ? g : 0;
  float accA = 0.f, accB = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxBlk; ++i) {
    const int b = b0 + i;
    if (b < b1) {
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};  // word groups 0 and 1
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t wa = q ? cA[i].y : cA[i].x, wb = q ? cB[i].y : cB[i].x;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t xa = j < 3 ? wa : wa >> 4, xb = j < 3 ? wb : wb >> 4;
          const uint32_t m0 = 0x00030003u << pair_bit(j, 0), m1 = 0x00030003u << pair_bit(j, 1);
          const uint2 bf = btab[btab_index(b, q, j, ncol, t)];
          if (q)
            mma_16816(c1, xa & m0, xb & m0, xa & m1, xb & m1, bf.x, bf.y);
          else
            mma_16816(c0, xa & m0, xb & m0, xa & m1, xb & m1, bf.x, bf.y);
        }
      }
      // columns 0 and 1 (high and low) of rows g and g+8 sit in thread t = 0
      const float F = fx[b], S = sx[b];
      accA = fmaf(dA[i], fmaf(F, (c0[0] + c0[1]) + (c1[0] + c1[1]), -S), accA);
      accB = fmaf(dB[i], fmaf(F, (c0[2] + c0[3]) + (c1[2] + c1[3]), -S), accB);
    }
  }

  // the parts of each row, added in part order
  if (part > 0 && t == 0) {
    comb[(part - 1) * kRows + slab * 16 + g] = accA;
    comb[(part - 1) * kRows + slab * 16 + g + 8] = accB;
  }
  __syncthreads();
  if (part == 0 && t == 0) {
#pragma unroll
    for (int p = 1; p < kParts; ++p) {
      accA += comb[(p - 1) * kRows + slab * 16 + g];
      accB += comb[(p - 1) * kRows + slab * 16 + g + 8];
    }
    if constexpr (IO16) {
      if (liveA) static_cast<__half*>(y)[rA] = __float2half_rn(accA);
      if (liveB) static_cast<__half*>(y)[rB] = __float2half_rn(accB);
    } else {
      if (liveA) static_cast<float*>(y)[rA] = accA;
      if (liveB) static_cast<float*>(y)[rB] = accB;
    }
  }
}

}  // namespace pq

}  // namespace direct

// PQ2_0: the page's 128-block rotation without signs, on the default
// (mma.sync) consumer
static bool pq2_0_direct_applies(const kq_qmat* W, int64_t m) {
  return m == 1 && W->fmt == KQ_PQ2_0 && W->had_block == 128 && W->signs == nullptr && W->k <= direct::pq::kMaxK &&
         W->n * (W->k / 4) <= direct::pq::kMaxCodeBytes && kq_get_pq2_0_consumer() == KQ_PQ2_0_MMA_SYNC;
}

bool gemv_direct_applies(const kq_qmat* W, int64_t m) {
  return (m == 1 && W->fmt == KQ_Q8_0 && W->k <= direct::kMaxK && W->n * W->k <= kGemvDirectMaxBytes) ||
         pq2_0_direct_applies(W, m);
}

int gemv_direct(const kq_qmat* W, const void* d_x, void* d_y, bool io16, void* stream) {
  cudaStream_t st = (cudaStream_t)stream;
  if (W->fmt == KQ_PQ2_0) {
    namespace P = direct::pq;
    const dim3 grid((unsigned)((W->n + P::kRows - 1) / P::kRows)), block(P::kThreads);
    const size_t smem = P::smem_bytes(W->k);
    const uint32_t* codes = static_cast<const uint32_t*>(W->codes);
    const __half* scales = static_cast<const __half*>(W->scales);
    const int64_t ss = scale_stride(KQ_PQ2_0, W->k);
    if (io16)
      KQ_CUDA_TRY(launch_dependent(P::pq2_0_gemv_kernel<true>, grid, block, smem, st, codes, scales, W->n, (int)W->k,
                                   ss, d_x, d_y));
    else
      KQ_CUDA_TRY(launch_dependent(P::pq2_0_gemv_kernel<false>, grid, block, smem, st, codes, scales, W->n,
                                   (int)W->k, ss, d_x, d_y));
    return KQ_OK;
  }
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
