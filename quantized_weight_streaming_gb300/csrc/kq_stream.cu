// The weight-streaming kernels of libkq: batch-1 GEMV, small-M GEMM and the
// decode-step driver, for the Q8_0 and PQ2_0 block formats.
//
// Decode is bound by streaming every weight once per token ("Kipp
// Benchmarks", "Decode is weight-bandwidth-bound"); the kernel therefore does
// nothing but keep HBM busy and dequantize in registers:
//
//  * One persistent CTA per SM: warp 0 is the producer, eight consumer warps
//    compute.  The producer copies tiles of 16 weight rows (codes plane plus
//    scales plane) into a ring of shared-memory stages with 1-D bulk copies
//    (cp.async.bulk, completion counted on an mbarrier, L2 evict-first since
//    every weight byte is read exactly once).
//  * Work is a list of items (matrix, 16-row group, K split).  Each CTA owns a
//    contiguous run of items, so it changes matrices rarely; every item walks
//    its K range in chunks (one chunk per stage).
//  * When a CTA starts an item of a new (matrix, split), its consumer warps
//    stage the activation slice in shared memory.  For PQ2_0 this prologue
//    applies the blockwise normalised Walsh-Hadamard transform (x' = R x,
//    "Bonsai 2 27B - ternary g128 + blockwise Hadamard", section 4.2) in
//    registers and warp shuffles, fused into the load.
//  * Q8_0 dot: sum_b d_b sum_j q_j x_j with the int8 code turned into an fp32
//    integer by a byte permute into the mantissa of 2^23 and one subtract.
//  * PQ2_0 dot: sum_b d_b (sum_j c_j x'_j - sum_j x'_j) with c in {0,1,2}
//    (the ternary value is c-1; the -1 is folded into a precomputed activation
//    sum, an idea the Bonsai page, section 8.5, uses on Metal).  A 2-bit code
//    masked in place inside its 32-bit word IS an fp32 denormal c * 4^j *
//    2^-149, so one AND per code produces the FMA operand; the activation is
//    pre-scaled by the matching power of two in the prologue, which keeps the
//    arithmetic exact up to fp32 rounding of the sums.
//  * Each output row is reduced across lanes with shuffles in a fixed order;
//    with K splits, partials land in the workspace and a second pass adds them
//    in split order.  Results never depend on the grid size.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <vector>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {

// ---- geometry ---------------------------------------------------------------
constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kTileRows = 16;                            // rows per tile
constexpr int kRowsPerWarp = kTileRows / kConsumerWarps;  // 2
constexpr int kStageCodeBytes = 24576;                   // codes bytes per stage (1536 per row)
constexpr int kStageScaleBytes = kTileRows * 96;          // up to 48 scales per row
constexpr int kStageBytes = kStageCodeBytes + kStageScaleBytes;
constexpr int kStages = 5;
constexpr int kXMax = 18432;                             // activation floats staged per item (all m)
constexpr int kGranMax = kXMax / 32;                     // PQ2_0 per-granule side arrays
constexpr size_t kSmemBytes =
    (size_t)kStages * kStageBytes + (size_t)kXMax * 4 + 2 * (size_t)kGranMax * 4 + 2 * kStages * 8 + 16;

__device__ unsigned int g_stream_status = 0;
__device__ __forceinline__ void stream_flag(int status) { atomicOr(&g_stream_status, 1u << status); }

// One matrix of the work list.
struct Job {
  const uint8_t* codes;
  const uint16_t* scales;
  const float* x;  // m rows, row stride k
  float* y;        // m rows, row stride ldy (splits == 1)
  float* ws;       // [splits][m][n] partials (splits > 1)
  int64_t n, k, ldy;
  int64_t x_off, y_off;  // offsets into the packed activation / output (decode plan)
  int64_t item_begin;    // first global item of this job
  int64_t items;       // row_groups * splits
  int32_t sstride;     // scales row stride (halves)
  int32_t row_groups;
  int32_t splits;
  int32_t split_k;  // weights per split (multiple of the alignment unit)
  int32_t chunk_k;  // weights per tile (multiple of the alignment unit)
};

struct Params {
  Job job0;                // used when jobs == nullptr
  const Job* jobs;         // device table (decode plan)
  const float* x_base;     // packed activations (decode plan)
  float* y_base;           // packed outputs (decode plan)
  const int64_t* bounds;   // per-CTA item ranges [bounds[c], bounds[c+1]) (plan), or nullptr
  int32_t njobs;
  int64_t total_items;
};

template <int FMT>
struct Fmt;
template <>
struct Fmt<KQ_Q8_0> {
  static constexpr int kBlock = 32;
  static constexpr int kCodesPerByte = 1;
  static constexpr int kAlign = 256;    // split / chunk unit: 32 granules of 8 codes, 8 scales
  static constexpr int kCodesPerGran = 8;
};
template <>
struct Fmt<KQ_PQ2_0> {
  static constexpr int kBlock = 128;
  static constexpr int kCodesPerByte = 4;
  static constexpr int kAlign = 1024;   // 32 granules of 32 codes, 8 scales
  static constexpr int kCodesPerGran = 32;
};

// Item -> (job, row group, split).  Items of a job are split-major.
struct ItemCursor {
  int32_t j = -1;
  Job job;
  __device__ void seek(const Params& p, int64_t item) {
    if (p.jobs == nullptr) {
      if (j < 0) {
        job = p.job0;
        j = 0;
      }
      return;
    }
    if (j >= 0 && item >= job.item_begin && item < job.item_begin + job.items) return;
    if (j < 0) j = 0;
    while (true) {
      const Job& cand = p.jobs[j];
      if (item >= cand.item_begin + cand.items) {
        ++j;
        continue;
      }
      if (item < cand.item_begin) {
        --j;
        continue;
      }
      break;
    }
    job = p.jobs[j];
    job.x = p.x_base + job.x_off;
    job.y = p.y_base + job.y_off;
  }
};

__device__ __forceinline__ void cta_range(const Params& p, int64_t& b, int64_t& e) {
  if (p.bounds) {
    b = p.bounds[blockIdx.x];
    e = p.bounds[blockIdx.x + 1];
  } else {
    b = p.total_items * blockIdx.x / gridDim.x;
    e = p.total_items * (blockIdx.x + 1) / gridDim.x;
  }
}

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }  // e in [-126, 127]

// Position of code j (0..15) of a 32-bit word in the masked-denormal view:
// codes 0..11 are masked in place (bits 2j), codes 12..15 after a shift by 24.
__device__ __forceinline__ int code_bitpos(int j) { return j < 12 ? 2 * j : 2 * (j - 12); }

// ---------------------------------------------------------------------------
// Activation prologue: stage x[m][kbeg, kend) of the current job.
// ---------------------------------------------------------------------------
template <int FMT, int M>
__device__ void stage_activation(const Job& job, int64_t kbeg, int64_t kend, float* xbuf, float* fx, float* sx,
                                 int cw, int lane) {
  const int len = (int)(kend - kbeg);
  if (FMT == KQ_Q8_0) {
    for (int m = 0; m < M; ++m) {
      const float4* src = reinterpret_cast<const float4*>(job.x + (int64_t)m * job.k + kbeg);
      float4* dst = reinterpret_cast<float4*>(xbuf + m * len);
      for (int i = cw * 32 + lane; i < len / 4; i += kConsumerWarps * 32) dst[i] = src[i];
    }
  } else {
    const int nblk = len / 128;
    const float inv_sqrt128 = 0.08838834764831845f;
    for (int t = cw; t < M * nblk; t += kConsumerWarps) {
      const int m = t / nblk, b = t % nblk;
      float4 f = *reinterpret_cast<const float4*>(job.x + (int64_t)m * job.k + kbeg + b * 128 + 4 * lane);
      float v[4] = {f.x, f.y, f.z, f.w};
      // fast Walsh-Hadamard transform, natural (Sylvester) order: strides 1, 2 in registers ...
      float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
      v[0] = a0 + a2;
      v[2] = a0 - a2;
      v[1] = a1 + a3;
      v[3] = a1 - a3;
      // ... strides 4 .. 64 across lanes
#pragma unroll
      for (int mk = 1; mk < 32; mk <<= 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float q = __shfl_xor_sync(0xffffffffu, v[i], mk);
          v[i] = (lane & mk) ? (q - v[i]) : (v[i] + q);
        }
      }
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[i] *= inv_sqrt128;
        amax = fmaxf(amax, fabsf(v[i]));
      }
#pragma unroll
      for (int mk = 16; mk; mk >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, mk));
      // block exponent E with amax < 2^(E+1), clamped to [-100, 100]
      int e = amax > 0.f ? ((__float_as_int(amax) >> 23) & 0xFF) - 127 : 0;
      if (amax > 0.f && e == -127) e = -126;  // denormal block maximum
      e = max(-100, min(100, e));
      const float unscale = pow2f(-e);
      float s = v[0] + v[1] + v[2] + v[3];
#pragma unroll
      for (int mk = 1; mk < 8; mk <<= 1) s += __shfl_xor_sync(0xffffffffu, s, mk);
      float4 o;
      float* op = &o.x;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = (4 * lane + i) & 15;  // code index inside its 32-bit word
        op[i] = (v[i] * unscale) * pow2f(126 - code_bitpos(j));
      }
      *reinterpret_cast<float4*>(xbuf + m * len + b * 128 + 4 * lane) = o;
      if ((lane & 7) == 0) {
        const int g = m * (len / 32) + b * 4 + lane / 8;
        sx[g] = s;
        fx[g] = pow2f(23 + e);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Consumer math for one stage.
// ---------------------------------------------------------------------------
template <int M>
__device__ __forceinline__ void q8_0_tile(const uint8_t* st_codes, const uint16_t* st_scales, int kc, int sp,
                                          int rows, int xoff, int xlen, const float* xbuf, int cw, int lane,
                                          float (&acc)[kRowsPerWarp][M]) {
  const int G = kc / 8;
  for (int g = lane; g < G; g += 32) {
    float4 xa[M], xb[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float4* xp = reinterpret_cast<const float4*>(xbuf + m * xlen + xoff + g * 8);
      xa[m] = xp[0];
      xb[m] = xp[1];
    }
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int row = cw * kRowsPerWarp + r;
      if (row >= rows) break;
      const uint2 c = *reinterpret_cast<const uint2*>(st_codes + row * kc + g * 8);
      const float d = __half2float(__ushort_as_half(st_scales[row * sp + g / 4]));
      const uint32_t u0 = c.x ^ 0x80808080u, u1 = c.y ^ 0x80808080u;
      constexpr float kMagic = 8388736.0f;  // 2^23 + 128
      float q[8];
      q[0] = __int_as_float(__byte_perm(u0, 0x4B000000u, 0x7540)) - kMagic;
      q[1] = __int_as_float(__byte_perm(u0, 0x4B000000u, 0x7541)) - kMagic;
      q[2] = __int_as_float(__byte_perm(u0, 0x4B000000u, 0x7542)) - kMagic;
      q[3] = __int_as_float(__byte_perm(u0, 0x4B000000u, 0x7543)) - kMagic;
      q[4] = __int_as_float(__byte_perm(u1, 0x4B000000u, 0x7540)) - kMagic;
      q[5] = __int_as_float(__byte_perm(u1, 0x4B000000u, 0x7541)) - kMagic;
      q[6] = __int_as_float(__byte_perm(u1, 0x4B000000u, 0x7542)) - kMagic;
      q[7] = __int_as_float(__byte_perm(u1, 0x4B000000u, 0x7543)) - kMagic;
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float p = q[0] * xa[m].x;
        p = fmaf(q[1], xa[m].y, p);
        p = fmaf(q[2], xa[m].z, p);
        p = fmaf(q[3], xa[m].w, p);
        p = fmaf(q[4], xb[m].x, p);
        p = fmaf(q[5], xb[m].y, p);
        p = fmaf(q[6], xb[m].z, p);
        p = fmaf(q[7], xb[m].w, p);
        acc[r][m] = fmaf(d, p, acc[r][m]);
      }
    }
  }
}

// 16 codes of one word against 16 pre-scaled activations.
__device__ __forceinline__ float ternary_word(uint32_t w, const float* xt, float a) {
#pragma unroll
  for (int j = 0; j < 12; ++j) a = fmaf(__uint_as_float(w & (3u << (2 * j))), xt[j], a);
  const uint32_t h = w >> 24;
#pragma unroll
  for (int j = 12; j < 16; ++j) a = fmaf(__uint_as_float(h & (3u << (2 * (j - 12)))), xt[j], a);
  return a;
}

template <int M>
__device__ __forceinline__ void pq2_0_tile(const uint8_t* st_codes, const uint16_t* st_scales, int kc, int sp,
                                           int rows, int xoff, int xlen, const float* xbuf, const float* fx,
                                           const float* sx, int cw, int lane, float (&acc)[kRowsPerWarp][M]) {
  const int G = kc / 32;       // granules of 32 codes (two words, 8 bytes) per row
  const int pitch = kc / 4;    // code bytes per row in the stage
  const int gl = xlen / 32;    // granules per activation row in the side arrays
  for (int g = lane; g < G; g += 32) {
    uint2 c[kRowsPerWarp];
    float d[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int row = cw * kRowsPerWarp + r;
      const int rr = row < rows ? row : 0;
      c[r] = *reinterpret_cast<const uint2*>(st_codes + rr * pitch + g * 8);
      d[r] = __half2float(__ushort_as_half(st_scales[rr * sp + g / 4]));
    }
    float a[kRowsPerWarp][M];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) a[r][m] = 0.f;
#pragma unroll
    for (int wi = 0; wi < 2; ++wi) {
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float xt[16];
        const float4* xp = reinterpret_cast<const float4*>(xbuf + m * xlen + xoff + g * 32 + wi * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float4 t = xp[i];
          xt[4 * i] = t.x;
          xt[4 * i + 1] = t.y;
          xt[4 * i + 2] = t.z;
          xt[4 * i + 3] = t.w;
        }
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) a[r][m] = ternary_word(wi ? c[r].y : c[r].x, xt, a[r][m]);
      }
    }
    const int gi = (xoff / 32) + g;
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float f = fx[m * gl + gi], s = sx[m * gl + gi];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) acc[r][m] = fmaf(d[r], fmaf(f, a[r][m], -s), acc[r][m]);
    }
  }
}

// ---------------------------------------------------------------------------
// The persistent streaming kernel.
// ---------------------------------------------------------------------------
template <int FMT, int M>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const __grid_constant__ Params p) {
  using F = Fmt<FMT>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  float* xbuf = reinterpret_cast<float*>(smem + (size_t)kStages * kStageBytes);
  float* fx = xbuf + kXMax;
  float* sx = fx + kGranMax;
  uint64_t* full = reinterpret_cast<uint64_t*>(sx + kGranMax);
  uint64_t* empty = full + kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kStages);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  int64_t ib, ie;
  cta_range(p, ib, ie);

  if (warp == 0) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      ItemCursor cur;
      int64_t tile = 0;
      bool ok = true;
      for (int64_t item = ib; item < ie && ok; ++item) {
        cur.seek(p, item);
        const Job& job = cur.job;
        const int64_t local = item - job.item_begin;
        const int split = (int)(local / job.row_groups);
        const int rg = (int)(local % job.row_groups);
        const int64_t row0 = (int64_t)rg * kTileRows;
        const int rows = (int)min64(kTileRows, job.n - row0);
        const int64_t kbeg = (int64_t)split * job.split_k;
        const int64_t kend = min64(job.k, kbeg + job.split_k);
        const int64_t rowbytes = job.k / F::kCodesPerByte;
        for (int64_t k0 = kbeg; k0 < kend; k0 += job.chunk_k, ++tile) {
          const int kc = (int)min64(job.chunk_k, kend - k0);
          const int cbytes = kc / F::kCodesPerByte;
          const int sp = ((kc / F::kBlock) + 7) & ~7;
          const int s = (int)(tile % kStages);
          const uint32_t par = (uint32_t)((tile / kStages) & 1);
          if (*abort_flag || !mbar_wait_bounded(&empty[s], par ^ 1u)) {
            *abort_flag = 1;
            stream_flag(KQ_ERR_TIMEOUT);
            ok = false;
            break;
          }
          uint8_t* st = stages + (size_t)s * kStageBytes;
          uint8_t* st_scales = st + rows * cbytes;
          mbar_arrive_expect_tx(&full[s], (uint32_t)(rows * (cbytes + 2 * sp)));
          if (kc == job.k) {
            bulk_g2s(st, job.codes + row0 * rowbytes, (uint32_t)(rows * cbytes), &full[s], policy);
            bulk_g2s(st_scales, job.scales + row0 * job.sstride, (uint32_t)(rows * 2 * sp), &full[s], policy);
          } else {
            for (int r = 0; r < rows; ++r) {
              bulk_g2s(st + r * cbytes, job.codes + (row0 + r) * rowbytes + k0 / F::kCodesPerByte, (uint32_t)cbytes,
                       &full[s], policy);
              bulk_g2s(st_scales + r * 2 * sp, job.scales + (row0 + r) * job.sstride + k0 / F::kBlock,
                       (uint32_t)(2 * sp), &full[s], policy);
            }
          }
        }
      }
      // Never leave the CTA with copies in flight: wait for the last stages issued.
      for (int64_t t = tile - 1; t >= 0 && t >= tile - kStages; --t)
        (void)mbar_wait_bounded(&full[t % kStages], (uint32_t)((t / kStages) & 1));
    }
    return;
  }

  // -------------------------------- consumers --------------------------------
  const int cw = warp - 1;
  ItemCursor cur;
  int32_t cached_job = -1, cached_split = -1;
  int64_t tile = 0;
  for (int64_t item = ib; item < ie; ++item) {
    cur.seek(p, item);
    const Job& job = cur.job;
    const int64_t local = item - job.item_begin;
    const int split = (int)(local / job.row_groups);
    const int rg = (int)(local % job.row_groups);
    const int64_t row0 = (int64_t)rg * kTileRows;
    const int rows = (int)min64(kTileRows, job.n - row0);
    const int64_t kbeg = (int64_t)split * job.split_k;
    const int64_t kend = min64(job.k, kbeg + job.split_k);
    const int xlen = (int)(kend - kbeg);
    if (cur.j != cached_job || split != cached_split) {
      named_barrier(1, kConsumerWarps * 32);  // everyone is done with the previous slice
      stage_activation<FMT, M>(job, kbeg, kend, xbuf, fx, sx, cw, lane);
      named_barrier(1, kConsumerWarps * 32);
      cached_job = cur.j;
      cached_split = split;
    }
    float acc[kRowsPerWarp][M];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) acc[r][m] = 0.f;

    // After an abort every warp keeps walking the item list (so the named
    // barriers above stay matched) but waits for and computes nothing.
    for (int64_t k0 = kbeg; k0 < kend; k0 += job.chunk_k, ++tile) {
      const int kc = (int)min64(job.chunk_k, kend - k0);
      const int cbytes = kc / F::kCodesPerByte;
      const int sp = ((kc / F::kBlock) + 7) & ~7;
      const int s = (int)(tile % kStages);
      const uint32_t par = (uint32_t)((tile / kStages) & 1);
      if (*abort_flag) continue;
      if (!mbar_wait_bounded(&full[s], par)) {
        *abort_flag = 1;
        stream_flag(KQ_ERR_TIMEOUT);
        continue;
      }
      const uint8_t* st = stages + (size_t)s * kStageBytes;
      const uint16_t* st_scales = reinterpret_cast<const uint16_t*>(st + rows * cbytes);
      const int xoff = (int)(k0 - kbeg);
      if (FMT == KQ_Q8_0)
        q8_0_tile<M>(st, st_scales, kc, sp, rows, xoff, xlen, xbuf, cw, lane, acc);
      else
        pq2_0_tile<M>(st, st_scales, kc, sp, rows, xoff, xlen, xbuf, fx, sx, cw, lane, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (*abort_flag) continue;

    // fixed-order lane reduction, then one write per (row, m)
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
#pragma unroll
      for (int m = 0; m < M; ++m) {
        float v = acc[r][m];
#pragma unroll
        for (int mk = 16; mk; mk >>= 1) v += __shfl_xor_sync(0xffffffffu, v, mk);
        acc[r][m] = v;
      }
    }
    if (lane == 0) {
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = cw * kRowsPerWarp + r;
        if (row < rows) {
#pragma unroll
          for (int m = 0; m < M; ++m) {
            if (job.splits == 1)
              job.y[(int64_t)m * job.ldy + row0 + row] = acc[r][m];
            else
              job.ws[((int64_t)split * M + m) * job.n + row0 + row] = acc[r][m];
          }
        }
      }
    }
  }
}

// Second pass of split-K: y[m][row] = sum over splits in split order.
__global__ void reduce_splits_kernel(const float* __restrict__ ws, float* __restrict__ y, int64_t n, int64_t ldy,
                                     int m, int splits) {
  const int64_t total = (int64_t)m * n;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t mm = i / n, row = i % n;
    float s = ws[mm * n + row];
    for (int sp = 1; sp < splits; ++sp) s += ws[((int64_t)sp * m + mm) * n + row];
    y[mm * ldy + row] = s;
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

struct Geometry {
  int32_t splits, split_k, chunk_k, row_groups;
};

static int64_t align_unit(int fmt) { return fmt == KQ_Q8_0 ? Fmt<KQ_Q8_0>::kAlign : Fmt<KQ_PQ2_0>::kAlign; }
static int64_t chunk_max(int fmt) { return fmt == KQ_Q8_0 ? kStageCodeBytes / kTileRows : kStageCodeBytes / kTileRows * 4; }

// Splits and chunks of one matrix for m activation rows.  requested = 0 means
// as few splits as the activation staging allows.
static Geometry make_geometry(int fmt, int64_t n, int64_t k, int64_t m, int requested) {
  Geometry g;
  const int64_t unit = align_unit(fmt);
  int64_t max_split = std::max<int64_t>(unit, (kXMax / m) / unit * unit);
  int64_t splits = std::max<int64_t>(requested > 0 ? requested : 1, (k + max_split - 1) / max_split);
  int64_t split_k = round_up((k + splits - 1) / splits, unit);
  split_k = std::min(split_k, max_split);
  splits = (k + split_k - 1) / split_k;
  int64_t nchunks = (split_k + chunk_max(fmt) - 1) / chunk_max(fmt);
  int64_t chunk_k = round_up((split_k + nchunks - 1) / nchunks, unit);
  chunk_k = std::min(chunk_k, chunk_max(fmt));
  g.splits = (int32_t)splits;
  g.split_k = (int32_t)split_k;
  g.chunk_k = (int32_t)chunk_k;
  g.row_groups = (int32_t)((n + kTileRows - 1) / kTileRows);
  return g;
}

static int device_sms(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  return KQ_OK;
}

template <int FMT, int M>
static int launch_stream(const Params& p, int grid, cudaStream_t st) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(stream_kernel<FMT, M>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
    configured = true;
  }
  stream_kernel<FMT, M><<<grid, kThreads, kSmemBytes, st>>>(p);
  KQ_CUDA_TRY(cudaGetLastError());
  return KQ_OK;
}

static int launch_any(int fmt, int m, const Params& p, int grid, cudaStream_t st) {
  if (fmt == KQ_Q8_0) {
    switch (m) {
      case 1: return launch_stream<KQ_Q8_0, 1>(p, grid, st);
      case 2: return launch_stream<KQ_Q8_0, 2>(p, grid, st);
      case 3: return launch_stream<KQ_Q8_0, 3>(p, grid, st);
      case 4: return launch_stream<KQ_Q8_0, 4>(p, grid, st);
    }
  } else {
    switch (m) {
      case 1: return launch_stream<KQ_PQ2_0, 1>(p, grid, st);
      case 2: return launch_stream<KQ_PQ2_0, 2>(p, grid, st);
      case 3: return launch_stream<KQ_PQ2_0, 3>(p, grid, st);
      case 4: return launch_stream<KQ_PQ2_0, 4>(p, grid, st);
    }
  }
  return fail(KQ_ERR_UNSUPPORTED, "m = %d", m);
}

constexpr int kMaxRowsPerLaunch = 4;
constexpr int64_t kMaxM = 64;

static size_t splitk_ws_bytes(const kq_qmat* W, int64_t m, int splits) {
  int64_t mm = min64(m, kMaxRowsPerLaunch);
  Geometry g = make_geometry(W->fmt, W->n, W->k, mm, splits);
  return g.splits > 1 ? (size_t)g.splits * (size_t)mm * (size_t)W->n * sizeof(float) : 0;
}

static int gemm_impl(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int splits, void* d_ws,
                     size_t ws_bytes, void* stream, int expect_fmt) {
  if (int s = check_qmat(W, expect_fmt)) return s;
  if (m < 1 || m > kMaxM) return fail(KQ_ERR_SHAPE, "m = %lld outside [1, %lld]", (long long)m, (long long)kMaxM);
  if (splits < 0) return fail(KQ_ERR_INVALID_ARG, "splits = %d", splits);
  if (!d_X || !d_Y) return fail(KQ_ERR_INVALID_ARG, "NULL activation or output");
  if (!aligned16(d_X) || !aligned16(d_Y)) return fail(KQ_ERR_ALIGNMENT, "x or y not 16-byte aligned");
  const size_t need = splitk_ws_bytes(W, m, splits);
  if (need > 0 && (d_ws == nullptr || ws_bytes < need))
    return fail(KQ_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, d_ws ? ws_bytes : (size_t)0);
  if (need > 0 && !aligned16(d_ws)) return fail(KQ_ERR_ALIGNMENT, "workspace not 16-byte aligned");
  int sms = 0;
  if (int s = device_sms(&sms)) return s;
  cudaStream_t st = (cudaStream_t)stream;
  for (int64_t m0 = 0; m0 < m; m0 += kMaxRowsPerLaunch) {
    const int mm = (int)min64(kMaxRowsPerLaunch, m - m0);
    Geometry g = make_geometry(W->fmt, W->n, W->k, mm, splits);
    Params p{};
    Job& j = p.job0;
    j.codes = (const uint8_t*)W->codes;
    j.scales = (const uint16_t*)W->scales;
    j.x = d_X + m0 * W->k;
    j.y = d_Y + m0 * W->n;
    j.ws = (float*)d_ws;
    j.n = W->n;
    j.k = W->k;
    j.ldy = W->n;
    j.item_begin = 0;
    j.items = (int64_t)g.row_groups * g.splits;
    j.sstride = (int32_t)scale_stride(W->fmt, W->k);
    j.row_groups = g.row_groups;
    j.splits = g.splits;
    j.split_k = g.split_k;
    j.chunk_k = g.chunk_k;
    p.jobs = nullptr;
    p.bounds = nullptr;
    p.njobs = 1;
    p.total_items = j.items;
    const int grid = (int)min64(j.items, sms);
    if (int s = launch_any(W->fmt, mm, p, grid, st)) return s;
    if (g.splits > 1) {
      const int64_t tot = (int64_t)mm * W->n;
      const int rgrid = (int)min64((tot + 255) / 256, (int64_t)sms * 8);
      reduce_splits_kernel<<<rgrid, 256, 0, st>>>((const float*)d_ws, d_Y + m0 * W->n, W->n, W->n, mm, g.splits);
      KQ_CUDA_TRY(cudaGetLastError());
    }
  }
  return KQ_OK;
}

int read_stream_status(int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_stream_status, sizeof(v));
  if (e != cudaSuccess) return -1;
  if (clear) {
    unsigned int z = 0;
    cudaMemcpyToSymbol(g_stream_status, &z, sizeof(z));
  }
  return (int)v;
}

int read_prep_status(int clear);  // kq_prep.cu

}  // namespace kq

// -----------------------------------------------------------------------------
// Decode plan
// -----------------------------------------------------------------------------
struct kq_plan {
  int fmt = 0;
  int64_t count = 0;
  int64_t x_floats = 0, y_floats = 0, weight_bytes = 0;
  int grid = 0;
  int64_t total_items = 0;
  std::vector<kq::Job> host_jobs;
  kq::Job* d_jobs = nullptr;  // device copy of host_jobs
  int64_t* d_bounds = nullptr;
};

using namespace kq;

extern "C" {

size_t kq_gemv_workspace_bytes(const kq_qmat* W, int64_t m) {
  if (check_qmat(W, -1) != KQ_OK || m < 1) return 0;
  return splitk_ws_bytes(W, m, 0);
}

size_t kq_gemm_splitk_workspace_bytes(const kq_qmat* W, int64_t m, int32_t splits) {
  if (check_qmat(W, -1) != KQ_OK || m < 1 || splits < 0) return 0;
  return splitk_ws_bytes(W, m, splits);
}

int kq_gemv_q8_0(const kq_qmat* W, const float* d_x, float* d_y, void* d_ws, size_t ws_bytes, void* stream) {
  clear_error();
  return gemm_impl(W, d_x, 1, d_y, 0, d_ws, ws_bytes, stream, KQ_Q8_0);
}

int kq_gemv_pq2_0(const kq_qmat* W, const float* d_x, float* d_y, void* d_ws, size_t ws_bytes, void* stream) {
  clear_error();
  return gemm_impl(W, d_x, 1, d_y, 0, d_ws, ws_bytes, stream, KQ_PQ2_0);
}

int kq_gemm_small_m(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, void* d_ws, size_t ws_bytes,
                    void* stream) {
  clear_error();
  return gemm_impl(W, d_X, m, d_Y, 0, d_ws, ws_bytes, stream, -1);
}

int kq_gemm_splitk(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int32_t splits, void* d_ws,
                   size_t ws_bytes, void* stream) {
  clear_error();
  return gemm_impl(W, d_X, m, d_Y, splits, d_ws, ws_bytes, stream, -1);
}

int kq_decode_plan_create(const kq_qmat* mats, int64_t count, kq_plan** out) {
  clear_error();
  if (!mats || !out) return fail(KQ_ERR_INVALID_ARG, "NULL pointer");
  if (count < 1) return fail(KQ_ERR_SHAPE, "count = %lld", (long long)count);
  *out = nullptr;
  const int fmt = mats[0].fmt;
  for (int64_t i = 0; i < count; ++i) {
    if (int s = check_qmat(&mats[i], -1)) return fail(s, "matrix %lld: %s", (long long)i, kq_last_error());
    if (mats[i].fmt != fmt) return fail(KQ_ERR_UNSUPPORTED, "matrix %lld: mixed formats in one plan", (long long)i);
    if (mats[i].k > kXMax) return fail(KQ_ERR_UNSUPPORTED, "matrix %lld: k = %lld > %d", (long long)i,
                                       (long long)mats[i].k, kXMax);
  }
  int sms = 0;
  if (int s = device_sms(&sms)) return s;
  kq_plan* p = new kq_plan();
  p->fmt = fmt;
  p->count = count;
  std::vector<double> item_bytes;
  int64_t items = 0;
  for (int64_t i = 0; i < count; ++i) {
    const kq_qmat& W = mats[i];
    Geometry g = make_geometry(fmt, W.n, W.k, 1, 1);
    Job j{};
    j.codes = (const uint8_t*)W.codes;
    j.scales = (const uint16_t*)W.scales;
    j.x = nullptr;
    j.y = nullptr;
    j.x_off = p->x_floats;
    j.y_off = p->y_floats;
    j.ws = nullptr;
    j.n = W.n;
    j.k = W.k;
    j.ldy = W.n;
    j.item_begin = items;
    j.items = g.row_groups;
    j.sstride = (int32_t)scale_stride(fmt, W.k);
    j.row_groups = g.row_groups;
    j.splits = 1;
    j.split_k = (int32_t)W.k;
    j.chunk_k = g.chunk_k;
    p->host_jobs.push_back(j);
    const double rb = (double)code_row_bytes(fmt, W.k) + 2.0 * j.sstride;
    for (int32_t r = 0; r < g.row_groups; ++r)
      item_bytes.push_back(rb * (double)min64(kTileRows, W.n - (int64_t)r * kTileRows));
    items += g.row_groups;
    p->x_floats += W.k;
    p->y_floats += W.n;
    p->weight_bytes += kq_codes_bytes(fmt, W.n, W.k) + W.n * (W.k / block_of(fmt)) * 2;
  }
  p->total_items = items;
  p->grid = (int)min64(items, sms);
  // byte-balanced contiguous item ranges, one per CTA
  std::vector<int64_t> bounds(p->grid + 1, items);
  double total = 0;
  for (double b : item_bytes) total += b;
  bounds[0] = 0;
  double accum = 0;
  int c = 1;
  for (int64_t it = 0; it < items && c < p->grid; ++it) {
    accum += item_bytes[(size_t)it];
    while (c < p->grid && accum >= total * c / p->grid) bounds[c++] = it + 1;
  }
  for (; c < p->grid; ++c) bounds[c] = items;
  bounds[p->grid] = items;
  cudaError_t e = cudaMalloc(&p->d_jobs, sizeof(Job) * (size_t)count);
  if (e == cudaSuccess) e = cudaMalloc(&p->d_bounds, sizeof(int64_t) * (size_t)(p->grid + 1));
  if (e == cudaSuccess)
    e = cudaMemcpy(p->d_bounds, bounds.data(), sizeof(int64_t) * (size_t)(p->grid + 1), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(p->d_jobs, p->host_jobs.data(), sizeof(Job) * (size_t)count, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaFree(p->d_jobs);
    cudaFree(p->d_bounds);
    delete p;
    return fail(KQ_ERR_CUDA, "plan allocation: %s", cudaGetErrorString(e));
  }
  *out = p;
  return KQ_OK;
}

int kq_decode_plan_sizes(const kq_plan* plan, int64_t* x_floats, int64_t* y_floats, int64_t* weight_bytes) {
  clear_error();
  if (!plan) return fail(KQ_ERR_INVALID_ARG, "NULL plan");
  if (x_floats) *x_floats = plan->x_floats;
  if (y_floats) *y_floats = plan->y_floats;
  if (weight_bytes) *weight_bytes = plan->weight_bytes;
  return KQ_OK;
}

size_t kq_decode_workspace_bytes(const kq_plan* plan) {
  (void)plan;
  return 0;
}

int kq_decode_step(kq_plan* plan, const float* d_x_packed, float* d_y_packed, void* d_ws, size_t ws_bytes,
                   void* stream) {
  clear_error();
  (void)d_ws;
  (void)ws_bytes;
  if (!plan) return fail(KQ_ERR_INVALID_ARG, "NULL plan");
  if (!d_x_packed || !d_y_packed) return fail(KQ_ERR_INVALID_ARG, "NULL activation or output");
  if (!aligned16(d_x_packed) || !aligned16(d_y_packed)) return fail(KQ_ERR_ALIGNMENT, "x or y not 16-byte aligned");
  cudaStream_t st = (cudaStream_t)stream;
  Params p{};
  p.jobs = plan->d_jobs;
  p.x_base = d_x_packed;
  p.y_base = d_y_packed;
  p.bounds = plan->d_bounds;
  p.njobs = (int32_t)plan->count;
  p.total_items = plan->total_items;
  if (plan->fmt == KQ_Q8_0) return launch_stream<KQ_Q8_0, 1>(p, plan->grid, st);
  return launch_stream<KQ_PQ2_0, 1>(p, plan->grid, st);
}

void kq_decode_plan_destroy(kq_plan* plan) {
  if (!plan) return;
  cudaFree(plan->d_jobs);
  cudaFree(plan->d_bounds);
  delete plan;
}

int kq_kernel_binary_version(int* version) {
  clear_error();
  if (!version) return fail(KQ_ERR_INVALID_ARG, "NULL pointer");
  cudaFuncAttributes a{};
  KQ_CUDA_TRY(cudaFuncGetAttributes(&a, stream_kernel<KQ_PQ2_0, 1>));
  *version = a.binaryVersion;
  return KQ_OK;
}

int kq_device_status(int clear) {
  clear_error();
  KQ_CUDA_TRY(cudaDeviceSynchronize());
  int a = read_stream_status(clear), b = read_prep_status(clear);
  if (a < 0 || b < 0) return fail(KQ_ERR_CUDA, "reading the device status word failed");
  const unsigned v = (unsigned)a | (unsigned)b;
  if (v & (1u << KQ_ERR_TIMEOUT)) return fail(KQ_ERR_TIMEOUT, "a bounded device wait expired");
  if (v & (1u << KQ_ERR_NONFINITE)) return fail(KQ_ERR_NONFINITE, "non-finite weight met on the device");
  if (v & (1u << KQ_ERR_RANGE)) return fail(KQ_ERR_RANGE, "scale overflowed fp16 on the device");
  return KQ_OK;
}

}  // extern "C"
