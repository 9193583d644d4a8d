// The weight-streaming kernels of libkq: batch-1 GEMV, small-M GEMM and the
// decode-step driver, for the Q8_0 and PQ2_0 block formats.
//
// Decode is bound by streaming every weight once per token ("Kipp
// Benchmarks", "Decode is weight-bandwidth-bound"); the kernel does nothing
// but keep HBM busy and dequantize in registers:
//
//  * One persistent CTA per SM: warp 0 is the producer, sixteen consumer
//    warps compute.  A tile is 256 bytes of codes per row (256 Q8_0 weights,
//    1024 PQ2_0 weights or 512 SCALE4 weights) plus the row's fp16 scales of
//    those weights: 128 rows for Q8_0 in a ring of four shared-memory
//    stages, 256 rows for PQ2_0 and SCALE4 in a ring of two.  The producer
//    brings each tile in with 2-D TMA loads (cp.async.bulk.tensor over tensor
//    maps of the row-major planes; rows past n and columns past k come back
//    as zeros), completion counted on an mbarrier, L2 evict-first since every
//    weight byte is read exactly once.
//  * Work is a list of items (matrix, 128-row block, K split).  Each CTA owns
//    a contiguous run of items, so it changes matrices rarely; an item walks
//    its K range one 256-byte chunk (one tile) at a time.
//  * Q8_0 consumers: warp w owns rows 8w..8w+7 of every tile and lane l the
//    l-th 8-byte granule of each row (8 weights), the granule's activations
//    loaded once (conflict-free 16-byte loads from a swizzled layout) and
//    reused by the eight rows.  The int8 code becomes an fp32 integer by a
//    byte permute into the mantissa of 2^23 and one subtract; rows go in
//    pairs through the fp32 pair instructions (FADD2 / FFMA2), so one
//    instruction converts or multiplies the codes of two rows.
//  * When a CTA starts an item of a new (matrix, split), its consumers stage
//    the activation slice in shared memory.  For PQ2_0 this prologue applies
//    the blockwise normalised Walsh-Hadamard transform (x' = R x, "Bonsai 2
//    27B - ternary g128 + blockwise Hadamard", section 4.2) in registers and
//    warp shuffles, fused into the load.
//  * PQ2_0 consumers run on the tensor cores (mma.sync m16n8k16, fp16 in,
//    fp32 accumulate): warp w owns 64 rows (four 16-row slabs) and a quarter
//    of the tile's K, so each B fragment it loads serves four slabs.  A
//    2-bit code masked in place inside its 32-bit word is the exact fp16
//    subnormal c * 2^(s-24): one AND per two codes builds an A register.  B
//    holds x' as an fp16 high/low pair scaled per block by 2^(14-s-E); the
//    ternary -1 is folded into a precomputed per-block activation sum, as
//    the Bonsai page, section 8.5, does on Metal: y += d (2^(10+E) C - sum x').
//  * Each output is reduced across lanes with shuffles in a fixed order; with
//    K splits, partials land in the workspace and a second pass adds them in
//    split order.  Results never depend on the grid size.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>
#include <vector>

#include "kq_device.cuh"
#include "kq_internal.h"
#include "kq_stream.cuh"
#include "kq_tc.h"

namespace kq {

__device__ unsigned int g_stream_status = 0;
__device__ __forceinline__ void stream_flag(int status) { atomicOr(&g_stream_status, 1u << status); }

// A linked plan's activation slice x[kbeg, kbeg + len) (one row), alpha
// applied, as plain fp32 into dst.  A thread takes one float4 of the slice
// per pass; a cut row block of the source is the sum of its partials in slot
// order, with up to 4 of them loaded at once, so a block cut n ways costs
// ceil(n / 4) round trips rather than n.  The arithmetic equals load_x4's:
// ((p0 + p1) + ...) * alpha.
// t_first: the source row block of the thread's first float4, read by the
// caller ahead of time (see first_tile).
template <int TR>
__device__ __forceinline__ void gather_slice(const XSrc& xs, int64_t kbeg, int len, float* dst, int tid,
                                             TileOut t_first) {
  constexpr int kT = 32 * kConsumerWarps;
  constexpr int kS = 4;  // partial loads in flight
  const int n4 = len / 4;
  for (int i = tid; i < n4; i += kT) {
    const int64_t g = kbeg + 4 * (int64_t)i;
    const TileOut t = i == tid ? t_first : (xs.tiles ? xs.tiles[g / TR] : TileOut{0, 1, 0});
    float4 r;
    if (t.nseg > 1) {
      const float* pb = xs.parts + t.part + g % TR;
      r = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int q0 = 0; q0 < t.nseg; q0 += kS) {
        float4 u[kS];
#pragma unroll
        for (int q = 0; q < kS; ++q)
          if (q0 + q < t.nseg) u[q] = __ldcg(reinterpret_cast<const float4*>(pb + (int64_t)(q0 + q) * TR));
#pragma unroll
        for (int q = 0; q < kS; ++q)
          if (q0 + q < t.nseg) {
            if (q0 + q == 0) {
              r = u[q];
            } else {
              r.x += u[q].x;
              r.y += u[q].y;
              r.z += u[q].z;
              r.w += u[q].w;
            }
          }
      }
    } else {
      const float* b = xs.base + g;
      r = xs.vec4 ? __ldcg(reinterpret_cast<const float4*>(b))
                  : make_float4(__ldcg(b), __ldcg(b + 1), __ldcg(b + 2), __ldcg(b + 3));
    }
    *reinterpret_cast<float4*>(dst + 4 * i) = make_float4(r.x * xs.alpha, r.y * xs.alpha, r.z * xs.alpha, r.w * xs.alpha);
  }
}

// Waits (one thread) until every CTA has finished `stage`; false on timeout.
__device__ __forceinline__ bool wait_stage(const Params& p, int stage) {
  const int32_t* ctr = p.stage_done + stage;
  const long long start = clock64();
  while (true) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ctr) : "memory");
    if (v >= (int32_t)gridDim.x) return true;
    if (clock64() - start > kWaitLimitCycles) return false;
    __nanosleep(64);
  }
}

// Q8_0 swizzled activation layout: the 8 activations of lane l in tile chunk
// t are read as two 16-byte pieces c = 0, 1 at [t][c][l], so the 32 lanes of
// a warp read 512 contiguous bytes per load.  Index of the float4 holding
// positions p..p+3 (p % 4 == 0) of the staged slice.
__device__ __forceinline__ int q8_swz4(int p) {
  const int t = p / 256, r = p % 256;
  return t * 64 + ((r % 8) / 4) * 32 + r / 8;
}

// ---------------------------------------------------------------------------
// PQ2_0 on the tensor cores: mma.sync.m16n8k16, f16 x f16 -> f32.
//
// A (16 weight rows x 16 codes).  A 2-bit code masked in place inside a
// 16-bit half is an exact fp16 denormal c * 2^(s-24) while its bit position
// s <= 10; one AND with 0x00030003 << s therefore turns the two codes at bits
// s and 16+s of a 32-bit code word (word elements s/2 and 8+s/2) into one
// half2 A register, and one shift right by 4 brings the pairs at 12 and 14
// down to 8 and 10.  Thread (g = lane/4, t = lane%4) owns word t of every
// group of four words of rows g and g+8 and feeds all 16 of its codes to the
// four MMAs of that group: MMA j takes the pairs at s = 4j and 4j+2 (after
// the shift for j = 3), i.e. logical k (2t, 2t+1) <- word elements
// (2j, 2j+8) and (2t+8, 2t+9) <- (2j+1, 2j+9).  Per 16 codes: one shift and
// eight ANDs with immediates.
//
// B (16 codes x 8 columns): column 2m holds the high fp16 part and 2m+1 the
// low part of activation row m, x' * 2^-E (|.| < 2) scaled by 2^(14-s) to
// match its code's denormal scale; every product is c * x' * 2^(-10-E)
// exactly.  A block of 128 codes is 8 MMAs, then its scale d is applied:
//     y += d * (2^(10+E) * (C_hi + C_lo) - sum_j x'_j)
//
// The codes of a tile arrive as two 128-byte-wide TMA boxes with the 128-byte
// swizzle (16-byte chunk c of box row r stored at chunk c ^ (r % 8)), so the
// 32 lanes of a word load touch 32 distinct banks.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// denormal bit position (after the shift for j = 3) of the pair of register
// `reg` (0: elements 2j, 2j+8; 1: elements 2j+1, 2j+9) of MMA j
__host__ __device__ __forceinline__ int pair_bit(int j, int reg) { return j < 3 ? 4 * j + 2 * reg : 8 + 2 * reg; }

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  return (uint32_t)__half_as_ushort(__float2half_rn(lo)) | ((uint32_t)__half_as_ushort(__float2half_rn(hi)) << 16);
}

// B table entry (uint2) of (block b of the slice, word group q, MMA j,
// column n < 2M, thread t): 64 M entries of 8 bytes per block of 128
// positions, i.e. 4 M bytes per position, the size of M fp32 activations.
template <int M>
__device__ __forceinline__ int btab_index(int b, int q, int j, int n, int t) {
  return (((b * 2 + q) * 4 + j) * (2 * M) + n) * 4 + t;
}

// SCALE4 B table entry (uint2) of (32-block b of the slice, MMA j, column n,
// thread t): 16 M entries of 8 bytes per block, again 4 M bytes per position.
template <int M>
__device__ __forceinline__ int btab4_index(int b, int j, int n, int t) {
  return ((b * 2 + j) * (2 * M) + n) * 4 + t;
}

// ---------------------------------------------------------------------------
// Activation prologue: stage x[m][kbeg, kend) of the current job.
//  Q8_0: fp32 activations in the swizzled layout.
//  PQ2_0: blockwise Walsh-Hadamard transform, then the B table of every
//  block, plus per block the factor 2^(10+E) and the sum of x'.
// ---------------------------------------------------------------------------
// IO16: the activation is fp16, and for PQ2_0 the transformed activation is
// rounded to fp16 right after the transform (the fp16 chain).
__device__ __forceinline__ float round_f16(float v) { return __half2float(__float2half_rn(v)); }

// The source row block that holds float4 `tid` of a linked gather from kbeg
// (the plan's tables only: it can be read before the source stage is done).
template <int TR>
__device__ __forceinline__ TileOut first_tile(const XSrc& xs, int64_t kbeg, int64_t kend, int tid) {
  const int64_t g = kbeg + 4 * (int64_t)tid;
  return xs.tiles && g < kend ? xs.tiles[g / TR] : TileOut{0, 1, 0};
}

template <int FMT, int M, bool IO16 = false, bool LINKED = false>
__device__ void stage_activation(const XSrc& xs, int64_t kbeg, int64_t kend, int xlen_pad, float* xbuf, float* fx,
                                 float* sx, float* scratch, int cw, int lane, TileOut t_first = TileOut{0, 1, 0}) {
  constexpr int kTR = LINKED ? Geo<FMT>::kTileRows : 0;  // a linked source's row blocks
  const int len = (int)(kend - kbeg);
  constexpr int kT = 32 * kConsumerWarps;
  // Linked PQ2_0 / SCALE4: the slice is first gathered as fp32 into the
  // staging buffer; each warp below then reads its blocks from there and
  // rewrites the same bytes with their table entries.
  constexpr bool kGather = LINKED && FMT != KQ_Q8_0;
  static_assert(!kGather || M == 1, "linked plans have one activation row");
  if constexpr (kGather) {
    gather_slice<Geo<FMT>::kTileRows>(xs, kbeg, len, xbuf, cw * 32 + lane, t_first);
    named_barrier(1, kConsumerWarps * 32);
  }

  if (FMT == KQ_Q8_0) {
    float4* xb4 = reinterpret_cast<float4*>(xbuf);
    for (int m = 0; m < M; ++m) {
      for (int i = cw * 32 + lane; i < len / 4; i += kT)
        xb4[m * (xlen_pad / 4) + q8_swz4(4 * i)] =
            load_x4<IO16, kTR>(xs, m, kbeg + 4 * i, LINKED && i == cw * 32 + lane ? &t_first : nullptr);
    }
  } else if (FMT == KQ_SCALE4) {
    // A warp takes 128 positions (four 32-blocks, eight lanes per block) at a
    // time: per block the exponent E of its largest |x|, 8 * sum(x) (the
    // implicit zero point) and the B table entries, x * 2^-E as fp16 high and
    // low parts scaled by 2^(14-s) to match the code's bit offset s.
    uint2* btab = reinterpret_cast<uint2*>(xbuf);
    const int ngrp = (len + 127) / 128;  // the last group may hold fewer than four blocks
    for (int tt = cw; tt < M * ngrp; tt += kConsumerWarps) {
      const int m = tt / ngrp, q = tt % ngrp;
      // len is a multiple of 32: a block's eight lanes are all inside or all past the slice
      const bool inside = q * 128 + 4 * lane < len;
      const float4 f = !inside ? make_float4(0.f, 0.f, 0.f, 0.f)
                       : kGather ? *reinterpret_cast<const float4*>(xbuf + q * 128 + 4 * lane)
                                 : load_x4<IO16, kTR>(xs, m, kbeg + q * 128 + 4 * lane);
      float amax = fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w)));
      float ssum = (f.x + f.y) + (f.z + f.w);
#pragma unroll
      for (int mk = 1; mk < 8; mk <<= 1) {
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, mk));
        ssum += __shfl_xor_sync(0xffffffffu, ssum, mk);
      }
      int e = amax > 0.f ? ((__float_as_int(amax) >> 23) & 0xFF) - 127 : 0;
      if (amax > 0.f && e == -127) e = -126;
      e = max(-100, min(100, e));
      const float unscale = pow2f(-e);
      __syncwarp();
      *reinterpret_cast<float4*>(scratch + 4 * lane) =
          make_float4(f.x * unscale, f.y * unscale, f.z * unscale, f.w * unscale);
      __syncwarp();
      // lane (block bq, MMA j, thread t): word t of the block, elements 2j,
      // 2j+4 (bit offset 0) and 2j+1, 2j+5 (bit offset 4) after the shift by 8j
      const int bq = lane >> 3, j = (lane >> 2) & 1, t = lane & 3;
      const float* xw = scratch + 32 * bq + 8 * t;
      const float u0 = xw[2 * j] * 16384.f, u1 = xw[2 * j + 4] * 16384.f;
      const float u2 = xw[2 * j + 1] * 1024.f, u3 = xw[2 * j + 5] * 1024.f;
      const float h0 = __half2float(__float2half_rn(u0)), h1 = __half2float(__float2half_rn(u1));
      const float h2 = __half2float(__float2half_rn(u2)), h3 = __half2float(__float2half_rn(u3));
      const int gb = q * 4 + bq;  // block inside the slice
      if (!inside) continue;       // (no further shuffle in this iteration)
      btab[btab4_index<M>(gb, j, 2 * m, t)] = make_uint2(pack_half2(h0, h1), pack_half2(h2, h3));
      btab[btab4_index<M>(gb, j, 2 * m + 1, t)] = make_uint2(pack_half2(u0 - h0, u1 - h1), pack_half2(u2 - h2, u3 - h3));
      if ((lane & 7) == 0) {
        fx[m * (xlen_pad / 32) + gb] = pow2f(10 + e);
        sx[m * (xlen_pad / 32) + gb] = 8.f * ssum;
      }
    }
  } else {
    const int nblk = len / 128;
    uint2* btab = reinterpret_cast<uint2*>(xbuf);
    const float inv_sqrt128 = 0.08838834764831845f;
    // The page's n = 1024 rotation is H_1024 = H_8 (x) H_128 in Sylvester
    // order (index 128 a + e): H_128 on each 128-block, then H_8 across the
    // eight blocks at each position e, then 1/32.  The two passes go through
    // `raw` ([block][row][128] floats): the B-table region itself for one
    // activation row (each warp then rewrites only its own block), the upper
    // half of the buffer for more rows (the split keeps both halves apart).
    const bool h1024 = xs.had == 1024;
    float* raw = M == 1 ? xbuf : xbuf + kXMax / 2;
    if (h1024) {
      for (int tt = cw; tt < M * nblk; tt += kConsumerWarps) {
        const int m = tt / nblk, b = tt % nblk;
        float4 f;
        if constexpr (kGather)
          f = *reinterpret_cast<const float4*>(xbuf + b * 128 + 4 * lane);
        else
          f = load_x4<IO16, kTR>(xs, m, kbeg + b * 128 + 4 * lane);
        float v[4] = {f.x, f.y, f.z, f.w};
        if (xs.signs) {
          const char4 s4 = *reinterpret_cast<const char4*>(xs.signs + kbeg + b * 128 + 4 * lane);
          v[0] *= (float)s4.x;
          v[1] *= (float)s4.y;
          v[2] *= (float)s4.z;
          v[3] *= (float)s4.w;
        }
        fwht128_lane4(v, lane);
        *reinterpret_cast<float4*>(raw + ((int64_t)b * M + m) * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
      }
      named_barrier(1, kConsumerWarps * 32);
      const int cols = (nblk / 8) * M * 128;
      for (int c = cw * 32 + lane; c < cols; c += kConsumerWarps * 32) {
        const int e = c % 128, mm = (c / 128) % M, bb = c / (128 * M);
        float v[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) v[a] = raw[((int64_t)(bb * 8 + a) * M + mm) * 128 + e];
#pragma unroll
        for (int h = 1; h < 8; h <<= 1)
#pragma unroll
          for (int a = 0; a < 8; ++a)
            if (!(a & h)) {
              const float x0 = v[a], x1 = v[a + h];
              v[a] = x0 + x1;
              v[a + h] = x0 - x1;
            }
#pragma unroll
        for (int a = 0; a < 8; ++a) {
          const float r = v[a] * 0.03125f;
          raw[((int64_t)(bb * 8 + a) * M + mm) * 128 + e] = IO16 ? round_f16(r) : r;
        }
      }
      named_barrier(1, kConsumerWarps * 32);
    }
    for (int tt = cw; tt < M * nblk; tt += kConsumerWarps) {
      const int m = tt / nblk, b = tt % nblk;
      float v[4];
      if (h1024) {  // x' of this block, transformed above
        const float4 f = *reinterpret_cast<const float4*>(raw + ((int64_t)b * M + m) * 128 + 4 * lane);
        v[0] = f.x;
        v[1] = f.y;
        v[2] = f.z;
        v[3] = f.w;
      } else {
        float4 f;
        if constexpr (kGather)
          f = *reinterpret_cast<const float4*>(xbuf + b * 128 + 4 * lane);
        else
          f = load_x4<IO16, kTR>(xs, m, kbeg + b * 128 + 4 * lane);
        v[0] = f.x;
        v[1] = f.y;
        v[2] = f.z;
        v[3] = f.w;
        fwht128_lane4(v, lane);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = IO16 ? round_f16(v[i] * inv_sqrt128) : v[i] * inv_sqrt128;
      }
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
      // the normalised block goes through the warp's scratch; lane (q, j, t)
      // then builds the high and low B entries of word 4q+t for MMA j
      __syncwarp();
      *reinterpret_cast<float4*>(scratch + 4 * lane) =
          make_float4(v[0] * unscale, v[1] * unscale, v[2] * unscale, v[3] * unscale);
      __syncwarp();
      const int t = lane & 3, j = (lane >> 2) & 3, q = lane >> 4;
      const float* xw = scratch + 16 * (4 * q + t);
      const float s0 = pow2f(14 - pair_bit(j, 0)), s1 = pow2f(14 - pair_bit(j, 1));
      const float u0 = xw[2 * j] * s0, u1 = xw[2 * j + 8] * s0, u2 = xw[2 * j + 1] * s1, u3 = xw[2 * j + 9] * s1;
      const float h0 = __half2float(__float2half_rn(u0)), h1 = __half2float(__float2half_rn(u1));
      const float h2 = __half2float(__float2half_rn(u2)), h3 = __half2float(__float2half_rn(u3));
      btab[btab_index<M>(b, q, j, 2 * m, t)] = make_uint2(pack_half2(h0, h1), pack_half2(h2, h3));
      btab[btab_index<M>(b, q, j, 2 * m + 1, t)] =
          make_uint2(pack_half2(u0 - h0, u1 - h1), pack_half2(u2 - h2, u3 - h3));
      if (lane == 0) {
        const int gb = m * (xlen_pad / 128) + b;
        sx[gb] = s;
        fx[gb] = pow2f(10 + e);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// SCALE4 consumer math for one 256-row tile (512 weights per row, sixteen
// 32-blocks): warp cw takes the 64 rows of row group cw % 4 and the K quarter
// cw / 4 (four blocks).  A block of a row is one 16-byte chunk, four code
// words, word t for thread t; a 4-bit code masked in place at bit offset s of
// an fp16 half is the exact subnormal q * 2^(s-24) (s = 0 or 4), so per word
// one AND per two codes builds an A register: MMA j = 0 takes the words as
// they are, j = 1 shifted right by 8.  Per block and row:
//     y += d * (2^(10+E) * (C_hi + C_lo) - 8 * sum x)
// ---------------------------------------------------------------------------
template <int M>
__device__ __forceinline__ void scale4_tile(const uint8_t* st_codes, const uint16_t* st_scales, int rows, int ci,
                                            int nblk_valid, const float* xbuf, const float* fx, const float* sx,
                                            int xlen_pad, int cw, int lane, float (&acc)[4][2]) {
  constexpr int kRows = Geo<KQ_SCALE4>::kTileRows;
  constexpr int kSpr = Geo<KQ_SCALE4>::kScalesPerRow;
  const int rg = cw & 3, kq = cw >> 2;
  if (rg * 64 >= rows) return;
  const int g = lane >> 2, t = lane & 3;
  const int kh = kq >> 1;
  const uint8_t* base = st_codes + kh * (kRows * 128) + (rg * 64 + g) * 128 + 4 * t;
  const int g16 = g << 4;
  // B column n comes from the lanes with g = n.  Lanes with g >= 2M load
  // column 0 again: their products land only in output columns >= 2M, which
  // nobody reads, so the load needs no predicate.
  const uint2* bthread = reinterpret_cast<const uint2*>(xbuf) + (g < 2 * M ? g : 0) * 4 + t;
  const int bt0 = 4 * kq;       // first block of the quarter inside the tile row
  const int b0 = ci * 16 + bt0;  // first block inside the staged slice
  const int tm = t < M ? t : 0;
  const float4 F4 = *reinterpret_cast<const float4*>(fx + tm * (xlen_pad / 32) + b0);
  const float4 S4 = *reinterpret_cast<const float4*>(sx + tm * (xlen_pad / 32) + b0);
  const float Fv[4] = {F4.x, F4.y, F4.z, F4.w}, Sv[4] = {S4.x, S4.y, S4.z, S4.w};
#pragma unroll
  for (int bl = 0; bl < 4; ++bl) {
    if (bt0 + bl >= nblk_valid) break;
    const uint2* bb = bthread + (b0 + bl) * (2 * 2 * M * 4);
    const int off = ((((kq & 1) * 4 + bl) << 4) ^ g16);
    uint32_t w[4][2];
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4) {
      w[s4][0] = *reinterpret_cast<const uint32_t*>(base + s4 * (16 * 128) + off);
      w[s4][1] = *reinterpret_cast<const uint32_t*>(base + s4 * (16 * 128) + 8 * 128 + off);
    }
    float c[4][4];
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
      for (int e = 0; e < 4; ++e) c[s4][e] = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const uint2 bf = bb[j * (2 * M * 4)];
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const uint32_t xa = j ? w[s4][0] >> 8 : w[s4][0], xb = j ? w[s4][1] >> 8 : w[s4][1];
        mma_16816(c[s4], xa & 0x000F000Fu, xb & 0x000F000Fu, xa & 0x00F000F0u, xb & 0x00F000F0u, bf.x, bf.y);
      }
    }
    if (t < M) {
      const float F = Fv[bl], S = Sv[bl];
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const int rA = rg * 64 + s4 * 16 + g;
        const float dA = __half2float(__ushort_as_half(st_scales[rA * kSpr + bt0 + bl]));
        const float dB = __half2float(__ushort_as_half(st_scales[(rA + 8) * kSpr + bt0 + bl]));
        acc[s4][0] = fmaf(dA, fmaf(F, c[s4][0] + c[s4][1], -S), acc[s4][0]);
        acc[s4][1] = fmaf(dB, fmaf(F, c[s4][2] + c[s4][3], -S), acc[s4][1]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Q8_0 consumer math for one tile: rows 8w..8w+7, granule `lane` of chunk `ci`.
// ---------------------------------------------------------------------------
template <int M>
__device__ __forceinline__ void q8_0_tile(const uint8_t* st_codes, const uint16_t* st_scales, int rows, int ci,
                                          int xlen_pad, const float* xbuf, int cw, int lane,
                                          float (&acc)[kRowsPerWarp][M]) {
  float4 xa[M], xb[M];
#pragma unroll
  for (int m = 0; m < M; ++m) {
    const float4* xp = reinterpret_cast<const float4*>(xbuf + m * xlen_pad) + ci * 64 + lane;
    xa[m] = xp[0];
    xb[m] = xp[32];
  }
  // rows in pairs: the fp32 pair instructions (FADD2 / FFMA2) convert and
  // multiply the codes of two rows against the same activations at once
#pragma unroll
  for (int r = 0; r < kRowsPerWarp; r += 2) {
    const int row = cw * kRowsPerWarp + r;
    if (row >= rows) break;
    const uint2 c0 = *reinterpret_cast<const uint2*>(st_codes + row * kChunkBytes + lane * 8);
    const uint2 c1 = *reinterpret_cast<const uint2*>(st_codes + (row + 1) * kChunkBytes + lane * 8);
    const float2 d2 = make_float2(__half2float(__ushort_as_half(st_scales[row * 8 + lane / 4])),
                                  __half2float(__ushort_as_half(st_scales[(row + 1) * 8 + lane / 4])));
    const uint32_t u[2][2] = {{c0.x ^ 0x80808080u, c0.y ^ 0x80808080u}, {c1.x ^ 0x80808080u, c1.y ^ 0x80808080u}};
    const float2 kMagic2 = make_float2(-8388736.0f, -8388736.0f);  // -(2^23 + 128)
    float2 q[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t sel = 0x7540u + (uint32_t)(e & 3);
      q[e] = __fadd2_rn(make_float2(__int_as_float(__byte_perm(u[0][e >> 2], 0x4B000000u, sel)),
                                    __int_as_float(__byte_perm(u[1][e >> 2], 0x4B000000u, sel))),
                        kMagic2);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
      const float xv[8] = {xa[m].x, xa[m].y, xa[m].z, xa[m].w, xb[m].x, xb[m].y, xb[m].z, xb[m].w};
      float2 p = __fmul2_rn(q[0], make_float2(xv[0], xv[0]));
#pragma unroll
      for (int e = 1; e < 8; ++e) p = __ffma2_rn(q[e], make_float2(xv[e], xv[e]), p);
      const float2 a = __ffma2_rn(d2, p, make_float2(acc[r][m], acc[r + 1][m]));
      acc[r][m] = a.x;
      acc[r + 1][m] = a.y;
    }
  }
}

// ---------------------------------------------------------------------------
// PQ2_0 consumer math for one 256-row tile: warp cw takes the 64 rows of row
// group cw % 4 (four 16-row slabs) and the K quarter cw / 4 (2 blocks, 256
// codes per row), so every B fragment it loads serves four slabs and its 32
// MMAs per block form eight independent chains.  acc[s][0] / acc[s][1] are
// the partial outputs of rows g and g+8 of slab s for activation row m = t.
// ---------------------------------------------------------------------------
template <int M>
__device__ __forceinline__ void pq2_0_tile(const uint8_t* st_codes, const uint16_t* st_scales, int rows, int ci,
                                           int nblk_valid, const float* xbuf, const float* fx, const float* sx,
                                           int xlen_pad, int cw, int lane, float (&acc)[4][2]) {
  constexpr int kRows = Geo<KQ_PQ2_0>::kTileRows;
  const int rg = cw & 3, kq = cw >> 2;
  if (rg * 64 >= rows) return;
  const int g = lane >> 2, t = lane & 3;
  const int kh = kq >> 1;  // 128-byte half box holding this quarter
  // Rows g, g+8 of every slab share r % 8 = g, so the swizzled offset of word
  // t of chunk c is base + ((c ^ g) << 4) for all eight rows.
  const uint8_t* base = st_codes + kh * (kRows * 128) + (rg * 64 + g) * 128 + 4 * t;
  const int g16 = g << 4;
  // B column n comes from the lanes with g = n.  Lanes with g >= 2M load
  // column 0 again: their products land only in output columns >= 2M, which
  // nobody reads, so the load needs no predicate.
  const uint2* bthread = reinterpret_cast<const uint2*>(xbuf) + (g < 2 * M ? g : 0) * 4 + t;
  // the two blocks' activation factors and sums
  const int bt0 = 2 * kq;  // first block of the quarter inside the tile row
  const int b0 = ci * 8 + bt0;  // first block inside the staged slice
  const int tm = t < M ? t : 0;  // lanes t >= M hold no activation row
  const float2 F2 = *reinterpret_cast<const float2*>(fx + tm * (xlen_pad / 128) + b0);
  const float2 S2 = *reinterpret_cast<const float2*>(sx + tm * (xlen_pad / 128) + b0);
  __half2 dpair[4][2];  // the scales of both blocks of rows g, g+8 of each slab, loaded once
#pragma unroll
  for (int bl = 0; bl < 2; ++bl) {
    if (bt0 + bl >= nblk_valid) break;
    const uint2* bb = bthread + (b0 + bl) * (2 * 4 * 2 * M * 4);
    // one accumulator per slab: four chains of 8 MMAs, interleaved
    float c[4][4];
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4)
#pragma unroll
      for (int e = 0; e < 4; ++e) c[s4][e] = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int off = ((((kq & 1) * 4 + 2 * bl + q) << 4) ^ g16);
      uint32_t w[4][2];
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        w[s4][0] = *reinterpret_cast<const uint32_t*>(base + s4 * (16 * 128) + off);
        w[s4][1] = *reinterpret_cast<const uint32_t*>(base + s4 * (16 * 128) + 8 * 128 + off);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint2 bf = bb[(q * 4 + j) * (2 * M * 4)];
        const uint32_t m0 = 0x00030003u << pair_bit(j, 0), m1 = 0x00030003u << pair_bit(j, 1);
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          const uint32_t xa = j < 3 ? w[s4][0] : w[s4][0] >> 4, xb = j < 3 ? w[s4][1] : w[s4][1] >> 4;
          mma_16816(c[s4], xa & m0, xb & m0, xa & m1, xb & m1, bf.x, bf.y);
        }
      }
    }
    if (t < M) {
      const float F = bl ? F2.y : F2.x, S = bl ? S2.y : S2.x;
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const int rA = rg * 64 + s4 * 16 + g;
        if (bl == 0) {
          dpair[s4][0] = *reinterpret_cast<const __half2*>(st_scales + rA * 8 + bt0);
          dpair[s4][1] = *reinterpret_cast<const __half2*>(st_scales + (rA + 8) * 8 + bt0);
        }
        const float dA = bl ? __high2float(dpair[s4][0]) : __low2float(dpair[s4][0]);
        const float dB = bl ? __high2float(dpair[s4][1]) : __low2float(dpair[s4][1]);
        acc[s4][0] = fmaf(dA, fmaf(F, c[s4][0] + c[s4][1], -S), acc[s4][0]);
        acc[s4][1] = fmaf(dB, fmaf(F, c[s4][2] + c[s4][3], -S), acc[s4][1]);
      }
    }
  }
}

// Waits for the stage phase with the given parity: 0 once it completed, 1 if
// another warp has aborted the kernel meanwhile, 2 after about one second.
// The abort flag is read only while waiting, not once per tile.
__device__ __forceinline__ int stage_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return 0;
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return 1;
    if (clock64() - start > kWaitLimitCycles) return 2;
  }
  return 0;
}

// ---------------------------------------------------------------------------
// The persistent streaming kernel.
// ---------------------------------------------------------------------------
// LINKED: a linked decode plan (stages, activation sources, stage counters,
// split partials read by dependants).  The unlinked instantiation (single
// GEMV / GEMM and plans without links) compiles none of that machinery.
// IO16: the fp16 chain (fp16 activation in, fp16 output; unlinked GEMVs only).
template <int FMT, int M, bool LINKED = false, bool IO16 = false>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const __grid_constant__ Params p) {
  using F = Fmt<FMT>;
  using G = Geo<FMT>;
  constexpr int kStages = G::kStages, kStageBytes = G::kStageBytes, kTileRows = G::kTileRows;
  constexpr int kTileCodeBytes = G::kTileCodeBytes;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* xbuf = reinterpret_cast<float*>(smem + (size_t)kStages * kStageBytes);
  float* fx = xbuf + G::kXMaxF;
  float* sx = fx + G::kBlkMax;
  float* scratch_all = sx + G::kBlkMax;
  float* combine = scratch_all;  // shares the scratch region (see Geo)
  uint64_t* full = reinterpret_cast<uint64_t*>(scratch_all + G::kScratchRegion);
  uint64_t* empty = full + kStages;
  uint64_t* cfull = empty + kStages;  // [4] PQ2_0: K-quarter partials of a slab pair written
  uint64_t* cfree = cfull + 4;        // [4] PQ2_0: the slab pair's partials consumed
  volatile int* abort_flag = reinterpret_cast<volatile int*>(cfree + 4);

  const int warp = threadIdx.x / 32, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    for (int q = 0; q < 4; ++q) {
      mbar_init(&cfull[q], 3);
      mbar_init(&cfree[q], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  // Launched as a programmatic dependent, the CTA got here while the kernel
  // before it may still run: the weights, the activations and the outputs
  // are touched only after it has completed.
  grid_dependency_wait();
  allow_dependent_launch();

  const int nst = LINKED ? p.nstages : 1;

  if (warp < kProducerWarps) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kProducerRegs) : "memory");
    if (warp != 0) return;
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kConsumerRegs) : "memory");
  }
  if (warp == 0) {
    // ------------------------------- producer -------------------------------
    // The weight stream never waits for a stage: it runs ahead into the next
    // stage's tiles as far as the ring allows.
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      ItemCursor cur;
      int64_t tile = 0;
      bool ok = true;
      int32_t last_j = -1;
      for (int st = 0; st < nst && ok; ++st) {
      int64_t ib, ie;
      cta_range(p, st, ib, ie);
      for (int64_t item = ib; item < ie && ok; ++item) {
        int rb;
        int64_t kbeg, kend;
        if constexpr (LINKED) {
          const Seg& sg = p.segs[item];
          cur.use(p, sg.j);
          rb = sg.rb;
          kbeg = (int64_t)sg.c0 * F::kChunk;
          kend = min64(cur.job.k, (int64_t)sg.c1 * F::kChunk);
        } else {
          cur.next(p, item);
          rb = cur.rb;
          kbeg = (int64_t)cur.split * cur.job.split_k;
          kend = min64(cur.job.k, kbeg + cur.job.split_k);
        }
        if (cur.j != last_j) {
          prefetch_tmap(cur.mc);
          prefetch_tmap(cur.ms);
          last_j = cur.j;
        }
        for (int64_t k0 = kbeg; k0 < kend; k0 += F::kChunk, ++tile) {
          const int s = (int)(tile % kStages);
          const uint32_t par = (uint32_t)((tile / kStages) & 1);
          if (*abort_flag || !mbar_wait_bounded(&empty[s], par ^ 1u)) {
            *abort_flag = 1;
            stream_flag(KQ_ERR_TIMEOUT);
            ok = false;
            break;
          }
          uint8_t* st = stages + (size_t)s * kStageBytes;
          mbar_arrive_expect_tx(&full[s], (uint32_t)kStageBytes);
          // codes: u32 elements, x = k0 code bytes / 4; scales: u32 elements (2 fp16), x = k0 / block / 2
          const int32_t xc = (int32_t)(k0 / F::kCodesPerByte / 4);
          if (FMT == KQ_Q8_0) {
            tma_load_2d(st, cur.mc, xc, rb * kTileRows, &full[s], policy);
          } else {  // two 128-byte swizzled half boxes
            tma_load_2d(st, cur.mc, xc, rb * kTileRows, &full[s], policy);
            tma_load_2d(st + kTileRows * 128, cur.mc, xc + 32, rb * kTileRows, &full[s], policy);
          }
          tma_load_2d(st + kTileCodeBytes, cur.ms, (int32_t)(k0 / F::kBlock / 2), rb * kTileRows, &full[s], policy);
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
  const int cw = warp - kProducerWarps;
  float* scratch = scratch_all + cw * kScratchFloats;
  ItemCursor cur;
  // The staged activation slice.  Unlinked: keyed by (job, split).  Linked:
  // by the activation's key and the K range (kbeg << 16 | kend, both below
  // 2^15), so that a job sharing the activation and the range reuses it (the
  // transform memo).
  int32_t cached_key = -1;
  uint32_t cached_range = 0xFFFFFFFFu;
  int ready = -1;          // linked: every stage up to this one has finished on all CTAs
  int ring = 0;            // stage of the next tile
  uint32_t ring_par = 0;   // its phase parity
  uint32_t combines = 0;   // PQ2_0 slab-pair handoffs so far
  int xlen_pad = 0;
  for (int st = 0; st < nst; ++st) {
  int64_t ib, ie;
  cta_range(p, st, ib, ie);
  for (int64_t item = ib; item < ie; ++item) {
    // The unit of work: weights [kbeg, kend) of row block rb against the
    // staged activation slice [sbeg, send) (an unlinked item stages exactly
    // its own K range).
    int rb;
    int64_t kbeg, kend, sbeg, send;
    uint32_t range;
    int32_t nseg = 1, slot = 0;  // linked: the row block's segments (see Seg)
    int64_t part = 0;
    if constexpr (LINKED) {
      const Seg sg = p.segs[item];
      cur.use(p, sg.j);
      rb = sg.rb;
      kbeg = (int64_t)sg.c0 * F::kChunk;
      kend = min64(cur.job.k, (int64_t)sg.c1 * F::kChunk);
      sbeg = (int64_t)sg.u0 * F::kChunk;
      send = min64(cur.job.k, (int64_t)sg.u1 * F::kChunk);
      range = ((uint32_t)sg.u0 << 16) | (uint32_t)sg.u1;
      nseg = sg.nseg;
      slot = sg.slot;
      part = sg.part;
    } else {
      cur.next(p, item);
      rb = cur.rb;
      kbeg = (int64_t)cur.split * cur.job.split_k;
      kend = kbeg + min((int64_t)cur.job.split_k, cur.job.k - kbeg);
      sbeg = kbeg;
      send = kend;
      range = (uint32_t)cur.split;
    }
    const Job& job = cur.job;
    const int split = cur.split;
    const int64_t row0 = (int64_t)rb * kTileRows;
    const int rows = min(kTileRows, (int)(job.n - row0));
    const int32_t key = LINKED ? p.links[cur.j].x_key : cur.j;
    if (key != cached_key || range != cached_range) {
      const XLink lk = LINKED ? p.links[cur.j] : XLink{-1, -1, cur.j, 1.f};
      // where the activation comes from and, for a linked source, the row
      // block of this thread's first float4: plan tables only, read here so
      // that their loads overlap the wait for the source stage
      const XSrc xs = make_xsrc(p, cur.j, job, lk);
      const TileOut t_first = LINKED ? first_tile<kTileRows>(xs, sbeg, send, cw * 32 + lane) : TileOut{0, 1, 0};
      xlen_pad = (int)(((send - sbeg) + F::kChunk - 1) / F::kChunk * F::kChunk);
      if (LINKED && lk.dep_stage > ready) {  // the activation is an output of an earlier stage
        if (cw == 0 && lane == 0 && !*abort_flag && !wait_stage(p, lk.dep_stage)) {
          *abort_flag = 1;
          stream_flag(KQ_ERR_TIMEOUT);
        }
        ready = lk.dep_stage;
      }
      named_barrier(1, kConsumerWarps * 32);  // everyone is done with the previous slice
      stage_activation<FMT, M, IO16, LINKED>(xs, sbeg, send, xlen_pad, xbuf, fx, sx, scratch, cw, lane, t_first);
      named_barrier(1, kConsumerWarps * 32);
      cached_key = key;
      cached_range = range;
    }
    float acc8[FMT == KQ_Q8_0 ? kRowsPerWarp : 1][M];
    float acc4[4][2] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
    for (int r = 0; r < (FMT == KQ_Q8_0 ? kRowsPerWarp : 1); ++r)
#pragma unroll
      for (int m = 0; m < M; ++m) acc8[r][m] = 0.f;

    // After an abort every warp keeps walking the item list (so the named
    // barriers stay matched) but waits for and computes nothing.
    const int klen = (int)(send - sbeg);  // chunk ci of the loop is chunk ci of the staged slice
    const int ci0 = (int)((kbeg - sbeg) / F::kChunk);
    const int nch = (int)((kend - sbeg + F::kChunk - 1) / F::kChunk);
    for (int ci = ci0; ci < nch; ++ci) {
      const int s = ring;
      const uint32_t par = ring_par;
      if (++ring == kStages) {
        ring = 0;
        ring_par ^= 1u;
      }
      const int64_t k0 = sbeg + (int64_t)ci * F::kChunk;
      const int wr = stage_wait(&full[s], par, abort_flag);
      if (wr != 0) {  // another warp aborted (1), or this wait ran out (2)
        if (wr == 2) {
          *abort_flag = 1;
          stream_flag(KQ_ERR_TIMEOUT);
        }
        continue;
      }
      const uint8_t* st = stages + (size_t)s * kStageBytes;
      const uint16_t* st_scales = reinterpret_cast<const uint16_t*>(st + kTileCodeBytes);
      if constexpr (FMT == KQ_Q8_0) {
        // lanes whose granule lies past k have nothing to do in this chunk
        if (k0 + (int64_t)(lane + 1) * F::kGran <= send)
          q8_0_tile<M>(st, st_scales, rows, ci, xlen_pad, xbuf, cw, lane, acc8);
      } else if constexpr (FMT == KQ_SCALE4) {
        const int nblk_valid = min(16, (klen - ci * F::kChunk) / 32);
        scale4_tile<M>(st, st_scales, rows, ci, nblk_valid, xbuf, fx, sx, xlen_pad, cw, lane, acc4);
      } else {
        const int nblk_valid = min(8, (klen - ci * F::kChunk) / 128);
        pq2_0_tile<M>(st, st_scales, rows, ci, nblk_valid, xbuf, fx, sx, xlen_pad, cw, lane, acc4);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }

    do {  // the outputs (`break` skips them after an abort)
      if constexpr (FMT == KQ_Q8_0) {
        if (*abort_flag) break;
        // fixed-order lane reduction, then one write per (row, m)
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
#pragma unroll
          for (int m = 0; m < M; ++m) {
            float v = acc8[r][m];
#pragma unroll
            for (int mk = 16; mk; mk >>= 1) v += __shfl_xor_sync(0xffffffffu, v, mk);
            acc8[r][m] = v;
          }
        }
        if (lane < kRowsPerWarp) {
          const int row = cw * kRowsPerWarp + lane;
          if (row < rows) {
            float v[M];
#pragma unroll
            for (int m = 0; m < M; ++m) {
              v[m] = acc8[0][m];
#pragma unroll
              for (int r = 1; r < kRowsPerWarp; ++r)
                if (lane == r) v[m] = acc8[r][m];
            }
#pragma unroll
            for (int m = 0; m < M; ++m) {
              if (LINKED && nseg > 1) {
                p.ws_base[part + (int64_t)slot * kTileRows + row] = v[m];
              } else if (job.splits == 1) {
                if constexpr (IO16)
                  reinterpret_cast<__half*>(job.y)[(int64_t)m * job.ldy + row0 + row] = __float2half_rn(v[m]);
                else
                  job.y[(int64_t)m * job.ldy + row0 + row] = v[m];
              } else {
                job.ws[((int64_t)split * M + m) * job.n + row0 + row] = v[m];
              }
            }
          }
        }
      } else {
        // warps cw, cw + 4, cw + 8, cw + 12 hold the four K quarters of the
        // same 64 rows: the last three hand their partials over through the
        // row group's buffer and go on (they only wait, before writing, until
        // the previous handoff has been read); the first adds them in quarter
        // order and writes the outputs
        const int sp = cw & 3, kq = cw >> 2;
        float* cb = combine + sp * (3 * 32 * 8);
        const uint32_t cpar = combines & 1u;
        ++combines;
        if (*abort_flag) break;
        if (kq > 0) {
          if (!mbar_wait_bounded(&cfree[sp], cpar ^ 1u)) {
            *abort_flag = 1;
            stream_flag(KQ_ERR_TIMEOUT);
            break;
          }
          float4* dst = reinterpret_cast<float4*>(cb + ((kq - 1) * 32 + lane) * 8);
          dst[0] = make_float4(acc4[0][0], acc4[0][1], acc4[1][0], acc4[1][1]);
          dst[1] = make_float4(acc4[2][0], acc4[2][1], acc4[3][0], acc4[3][1]);
          __syncwarp();
          if (lane == 0) mbar_arrive(&cfull[sp]);
        } else {
          if (!mbar_wait_bounded(&cfull[sp], cpar)) {
            *abort_flag = 1;
            stream_flag(KQ_ERR_TIMEOUT);
            break;
          }
          const int g = lane >> 2, t = lane & 3;
          // this lane's output row of activation t (lanes t >= M write nothing)
          float* yout = (LINKED && nseg > 1)
                            ? p.ws_base + part + (int64_t)slot * kTileRows
                            : (job.splits == 1 ? job.y + (int64_t)t * job.ldy : job.ws + ((int64_t)split * M + t) * job.n) +
                                  row0;
          const int rmax = t < M ? rows - (sp * 64 + g) : 0;  // rows of this lane's set that exist
          float y8[8] = {acc4[0][0], acc4[0][1], acc4[1][0], acc4[1][1],
                         acc4[2][0], acc4[2][1], acc4[3][0], acc4[3][1]};
#pragma unroll
          for (int q = 0; q < 3; ++q) {
            const float4* src = reinterpret_cast<const float4*>(cb + (q * 32 + lane) * 8);
            const float4 v0 = src[0], v1 = src[1];
            y8[0] += v0.x;
            y8[1] += v0.y;
            y8[2] += v0.z;
            y8[3] += v0.w;
            y8[4] += v1.x;
            y8[5] += v1.y;
            y8[6] += v1.z;
            y8[7] += v1.w;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&cfree[sp]);
          if (IO16 && job.splits == 1) {  // the final output, in fp16
            __half* yh = reinterpret_cast<__half*>(job.y) + (int64_t)t * job.ldy + row0 + sp * 64 + g;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int dr = (e >> 1) * 16 + (e & 1) * 8;
              if (dr < rmax) yh[dr] = __float2half_rn(y8[e]);
            }
          } else {
            float* yl = yout + sp * 64 + g;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const int dr = (e >> 1) * 16 + (e & 1) * 8;  // slab e/2, row g or g+8
              if (dr < rmax) yl[dr] = y8[e];
            }
          }
        }
      }
    } while (0);
  }
  // linked plan: this CTA has written every output of its items of stage st
  if (LINKED) {
    named_barrier(1, kConsumerWarps * 32);
    // a release add: the CTA's writes, ordered before it by the barrier,
    // are visible to any thread that acquires the count
    if (cw == 0 && lane == 0)
      asm volatile("red.release.gpu.global.add.s32 [%0], 1;" ::"l"(p.stage_done + st) : "memory");
  }
  }

  // Linked plan: once the last stage has finished everywhere, the cut row
  // blocks' outputs are their partials added in slot order (the sums their
  // readers used), each CTA every gridDim.x-th block.
  if constexpr (LINKED) {
    if (p.n_cuts > 0) {
      if (cw == 0 && lane == 0 && !*abort_flag && !wait_stage(p, nst - 1)) {
        *abort_flag = 1;
        stream_flag(KQ_ERR_TIMEOUT);
      }
      named_barrier(1, kConsumerWarps * 32);
      if (*abort_flag) return;
      // one warp per cut block; a lane sums rows 4l .. 4l + 3 (and 4l + 128 ..)
      for (int c = blockIdx.x + gridDim.x * cw; c < p.n_cuts; c += gridDim.x * kConsumerWarps) {
        const CutOut cu = p.cuts[c];
        const float* pb = p.ws_base + cu.part;
        constexpr int kQ = kTileRows / 128;  // float4 per lane
        float4 v[kQ];
        for (int q0 = 0; q0 < cu.nseg; q0 += 4) {
          float4 u[4][kQ];
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int h = 0; h < kQ; ++h)
              if (q0 + q < cu.nseg)
                u[q][h] = __ldcg(reinterpret_cast<const float4*>(pb + (int64_t)(q0 + q) * kTileRows + 128 * h) + lane);
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int h = 0; h < kQ; ++h)
              if (q0 + q < cu.nseg) {
                if (q0 + q == 0) {
                  v[h] = u[q][h];
                } else {
                  v[h].x += u[q][h].x;
                  v[h].y += u[q][h].y;
                  v[h].z += u[q][h].z;
                  v[h].w += u[q][h].w;
                }
              }
        }
        float* y = p.y_base + cu.y;
#pragma unroll
        for (int h = 0; h < kQ; ++h) {
          const int r = 128 * h + 4 * lane;
          const float e[4] = {v[h].x, v[h].y, v[h].z, v[h].w};
#pragma unroll
          for (int d = 0; d < 4; ++d)
            if (r + d < cu.rows) y[r + d] = e[d];
        }
      }
    }
  }
}

// Second pass of split-K: y[m][row] = sum over splits in split order (OUT16:
// the sum rounded once to fp16).
template <bool OUT16 = false>
__global__ void reduce_splits_kernel(const float* __restrict__ ws, float* __restrict__ y, int64_t n, int64_t ldy,
                                     int m, int splits) {
  grid_dependency_wait();  // the partials of the kernel before (a programmatic dependent launch)
  allow_dependent_launch();
  const int64_t total = (int64_t)m * n;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t mm = i / n, row = i % n;
    float s = ws[mm * n + row];
    for (int sp = 1; sp < splits; ++sp) s += ws[((int64_t)sp * m + mm) * n + row];
    if constexpr (OUT16)
      reinterpret_cast<__half*>(y)[mm * ldy + row] = __float2half_rn(s);
    else
      y[mm * ldy + row] = s;
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

static int64_t chunk_of(int fmt) {
  return fmt == KQ_Q8_0 ? Fmt<KQ_Q8_0>::kChunk : (fmt == KQ_SCALE4 ? Fmt<KQ_SCALE4>::kChunk : Fmt<KQ_PQ2_0>::kChunk);
}

struct Geometry {
  int32_t splits, split_k, row_blocks;
};

// Splits of one matrix for m activation rows.  requested > 0 asks for that
// many splits (more if the activation staging needs them); requested = 0
// picks the count that minimises an estimate of the kernel time on `sms`
// CTAs: tiles of the busiest CTA times the time of a tile, plus the second
// pass when there is more than one split.
// The staged slice of m rows must fit kXMax floats, or half of it for the
// n = 1024 rotation with m > 1 (its transform passes use the other half).
static int64_t staging_floats(const kq_qmat* W, int64_t m) {
  return W->fmt == KQ_PQ2_0 && W->had_block == 1024 && m > 1 ? kXMax / 2 : xmax_of(W->fmt);
}

static Geometry make_geometry(int fmt, int64_t n, int64_t k, int64_t m, int requested, int sms = 0,
                              int64_t xmax = kXMax) {
  Geometry g;
  const int64_t unit = chunk_of(fmt);
  const int64_t max_split = std::max<int64_t>(unit, (xmax / m) / unit * unit);
  const int64_t min_splits = (k + max_split - 1) / max_split;
  const int64_t row_blocks = (n + tile_rows(fmt) - 1) / tile_rows(fmt);
  int64_t splits = std::max<int64_t>(requested > 0 ? requested : 1, min_splits);
  if (requested == 0 && sms > 0) {
    const int64_t chunks = (k + unit - 1) / unit;
    const double kTileUs = fmt == KQ_PQ2_0 ? 2.0 : (fmt == KQ_SCALE4 ? 1.6 : 0.75), kReduceUs = 2.5;
    double best = 1e30;
    for (int64_t s = min_splits; s <= chunks; ++s) {
      const int64_t sk = round_up((k + s - 1) / s, unit);
      if (sk > max_split) continue;
      const int64_t real = (k + sk - 1) / sk;
      const int64_t items = row_blocks * real;
      const double t = (double)((items + sms - 1) / sms) * (double)((sk + unit - 1) / unit) * kTileUs +
                       (real > 1 ? kReduceUs : 0.0);
      if (t < best - 1e-9) {
        best = t;
        splits = real;
      }
    }
  }
  int64_t split_k = std::min(round_up((k + splits - 1) / splits, unit), max_split);
  splits = (k + split_k - 1) / split_k;
  g.splits = (int32_t)splits;
  g.split_k = (int32_t)split_k;
  g.row_blocks = (int32_t)row_blocks;
  return g;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// Tensor maps of a matrix's planes, both viewed as 2-D arrays of 32-bit
// elements: codes [n][k*bits/32], box 64 x 128 (256 bytes of 128 rows) or,
// for PQ2_0, 32 x 128 with the 128-byte swizzle; scales [n][stride/2], box
// 4 x 128 (8 fp16 scales of 128 rows).
static int make_maps(const kq_qmat* W, CUtensorMap* mc, CUtensorMap* ms) {
  auto fn = encode_fn();
  if (!fn) return fail(KQ_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
  const int64_t rowbytes = code_row_bytes(W->fmt, W->k);
  const int64_t sst = scale_stride(W->fmt, W->k);
  cuuint64_t gdim[2] = {(cuuint64_t)(rowbytes / 4), (cuuint64_t)W->n};
  cuuint64_t gstride[1] = {(cuuint64_t)rowbytes};
  // Q8_0: one 256-byte box per tile row; PQ2_0: two 128-byte boxes with the
  // 128-byte swizzle (the tensor-core consumer reads columns of 8 rows)
  const bool swz = W->fmt != KQ_Q8_0;
  cuuint32_t box[2] = {swz ? 32u : (cuuint32_t)(kChunkBytes / 4), (cuuint32_t)tile_rows(W->fmt)};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(mc, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(W->codes), gdim, gstride, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KQ_ERR_CUDA, "tensor map of the codes plane: CUresult %d", (int)r);
  cuuint64_t sdim[2] = {(cuuint64_t)(sst / 2), (cuuint64_t)W->n};
  cuuint64_t sstr[1] = {(cuuint64_t)(sst * 2)};
  // one tile row's scales: chunk / block fp16 values, as 32-bit elements
  cuuint32_t sbox[2] = {(cuuint32_t)(chunk_of(W->fmt) / block_of(W->fmt) / 2), (cuuint32_t)tile_rows(W->fmt)};
  r = fn(ms, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(W->scales), sdim, sstr, sbox, es,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KQ_ERR_CUDA, "tensor map of the scales plane: CUresult %d", (int)r);
  return KQ_OK;
}

static int device_sms(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail(KQ_ERR_CUDA, "device query: %s", cudaGetErrorString(e));
  return KQ_OK;
}

// Sets the kernel's shared-memory limit and checks that it was compiled to
// the register count the setmaxnreg split assumes (once per kernel).
template <typename K>
static int prepare_kernel_once(K kernel, size_t smem, std::once_flag& once, int& status, char (&msg)[160]) {
  std::call_once(once, [&] {
    cudaFuncAttributes a{};
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&a, kernel);
    if (e != cudaSuccess) {
      status = KQ_ERR_CUDA;
      snprintf(msg, sizeof(msg), "kernel attributes: %s", cudaGetErrorString(e));
    } else if (a.numRegs != kLaunchRegs) {
      status = KQ_ERR_UNSUPPORTED;
      snprintf(msg, sizeof(msg), "stream kernel built with %d registers per thread, not %d: its register split "
               "would not fit", a.numRegs, kLaunchRegs);
    }
  });
  return status == KQ_OK ? KQ_OK : fail(status, "%s", msg);
}

template <int FMT, int M, bool IO16 = false>
static int launch_stream(const Params& p, int grid, cudaStream_t st) {
  static std::once_flag once;
  static int status = KQ_OK;
  static char msg[160];
  if (int s = prepare_kernel_once(stream_kernel<FMT, M, false, IO16>, Geo<FMT>::kSmemBytes, once, status, msg))
    return s;
  // a programmatic dependent of the stream's previous kernel: its CTAs set up
  // while that kernel's last CTAs finish
  KQ_CUDA_TRY(launch_dependent(stream_kernel<FMT, M, false, IO16>, dim3(grid), dim3(kThreads),
                               Geo<FMT>::kSmemBytes, st, p));
  return KQ_OK;
}

// The consumer of PQ2_0 products at one activation row (kq_set_pq2_0_consumer).
static std::atomic<int> g_pq2_0_consumer{KQ_PQ2_0_MMA_SYNC};
static int pq2_0_consumer() { return g_pq2_0_consumer.load(std::memory_order_relaxed); }

static int launch_any(int fmt, int m, const Params& p, int grid, cudaStream_t st, bool io16 = false) {
  if (io16) {  // the fp16 chain: one activation row
    if (m != 1) return fail(KQ_ERR_UNSUPPORTED, "fp16 activations with m = %d", m);
    if (fmt == KQ_Q8_0) return launch_stream<KQ_Q8_0, 1, true>(p, grid, st);
    if (fmt == KQ_PQ2_0) return launch_stream<KQ_PQ2_0, 1, true>(p, grid, st);
    if (fmt == KQ_SCALE4) return launch_stream<KQ_SCALE4, 1, true>(p, grid, st);
    return fail(KQ_ERR_UNSUPPORTED, "format %d", fmt);
  }
  if (fmt == KQ_PQ2_0 && m == 1 && pq2_0_consumer() == KQ_PQ2_0_TCGEN05) return launch_tcs(p, grid, st);
  if (fmt == KQ_Q8_0) {
    switch (m) {
      case 1: return launch_stream<KQ_Q8_0, 1>(p, grid, st);
      case 2: return launch_stream<KQ_Q8_0, 2>(p, grid, st);
      case 3: return launch_stream<KQ_Q8_0, 3>(p, grid, st);
      case 4: return launch_stream<KQ_Q8_0, 4>(p, grid, st);
    }
  } else if (fmt == KQ_PQ2_0) {
    switch (m) {
      case 1: return launch_stream<KQ_PQ2_0, 1>(p, grid, st);
      case 2: return launch_stream<KQ_PQ2_0, 2>(p, grid, st);
      case 3: return launch_stream<KQ_PQ2_0, 3>(p, grid, st);
      case 4: return launch_stream<KQ_PQ2_0, 4>(p, grid, st);
    }
  } else if (fmt == KQ_SCALE4) {
    switch (m) {
      case 1: return launch_stream<KQ_SCALE4, 1>(p, grid, st);
      case 2: return launch_stream<KQ_SCALE4, 2>(p, grid, st);
      case 3: return launch_stream<KQ_SCALE4, 3>(p, grid, st);
      case 4: return launch_stream<KQ_SCALE4, 4>(p, grid, st);
    }
  }
  return fail(KQ_ERR_UNSUPPORTED, "m = %d", m);
}

constexpr int kMaxRowsPerLaunch = 4;
constexpr int64_t kMaxM = 64;

static int sms_or_default() {
  int sms = 0;
  if (device_sms(&sms) != KQ_OK) {
    clear_error();
    return 0;
  }
  return sms;
}

static size_t splitk_ws_bytes(const kq_qmat* W, int64_t m, int splits) {
  if (splits == 0 && gemv_direct_applies(W, m)) return 0;
  int64_t mm = std::min<int64_t>(m, kMaxRowsPerLaunch);
  Geometry g = make_geometry(W->fmt, W->n, W->k, mm, splits, splits == 0 ? sms_or_default() : 0,
                             staging_floats(W, mm));
  return g.splits > 1 ? (size_t)g.splits * (size_t)mm * (size_t)W->n * sizeof(float) : 0;
}

static int gemm_impl(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int splits, void* d_ws,
                     size_t ws_bytes, void* stream, int expect_fmt, bool io16 = false) {
  if (int s = check_qmat(W, expect_fmt)) return s;
  if (m < 1 || m > kMaxM) return fail(KQ_ERR_SHAPE, "m = %lld outside [1, %lld]", (long long)m, (long long)kMaxM);
  if (splits < 0) return fail(KQ_ERR_INVALID_ARG, "splits = %d", splits);
  if (!d_X || !d_Y) return fail(KQ_ERR_INVALID_ARG, "NULL activation or output");
  if (!aligned16(d_X) || !aligned16(d_Y)) return fail(KQ_ERR_ALIGNMENT, "x or y not 16-byte aligned");
  // a small Q8_0 matrix at one row: the one-launch GEMV
  if (splits == 0 && gemv_direct_applies(W, m)) return gemv_direct(W, d_X, d_Y, io16, stream);
  const size_t need = splitk_ws_bytes(W, m, splits);
  if (need > 0 && (d_ws == nullptr || ws_bytes < need))
    return fail(KQ_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, d_ws ? ws_bytes : (size_t)0);
  if (need > 0 && !aligned16(d_ws)) return fail(KQ_ERR_ALIGNMENT, "workspace not 16-byte aligned");
  int sms = 0;
  if (int s = device_sms(&sms)) return s;
  Params p{};
  if (int s = make_maps(W, &p.map_codes0, &p.map_scales0)) return s;
  cudaStream_t st = (cudaStream_t)stream;
  for (int64_t m0 = 0; m0 < m; m0 += kMaxRowsPerLaunch) {
    const int mm = (int)std::min<int64_t>(kMaxRowsPerLaunch, m - m0);
    Geometry g = make_geometry(W->fmt, W->n, W->k, mm, splits, splits == 0 ? sms : 0, staging_floats(W, mm));
    // the staged activation slice (or its B table, 4 bytes per position and
    // row for PQ2_0) must fit the shared-memory buffer
    if ((int64_t)mm * g.split_k > staging_floats(W, mm))
      return fail(KQ_ERR_UNSUPPORTED, "internal: split of %d weights x %d rows exceeds the staging buffer", g.split_k, mm);
    Job& j = p.job0;
    j.x = d_X + m0 * W->k;
    j.y = d_Y + m0 * W->n;
    j.ws = (float*)d_ws;
    j.n = W->n;
    j.k = W->k;
    j.ldy = W->n;
    j.item_begin = 0;
    j.items = (int64_t)g.row_blocks * g.splits;
    j.row_blocks = g.row_blocks;
    j.splits = g.splits;
    j.split_k = g.split_k;
    j.had_block = W->had_block;
    j.signs = W->signs;
    p.jobs = nullptr;
    p.maps = nullptr;
    p.bounds = nullptr;
    p.total_items = j.items;
    const int grid = (int)std::min<int64_t>(j.items, sms);
    if (int s = launch_any(W->fmt, mm, p, grid, st, io16)) return s;
    if (g.splits > 1) {
      const int64_t tot = (int64_t)mm * W->n;
      const int rgrid = (int)std::min<int64_t>((tot + 255) / 256, (int64_t)sms * 8);
      // launched as a programmatic dependent: its launch overlaps the GEMV's tail
      if (io16)
        KQ_CUDA_TRY(launch_dependent(reduce_splits_kernel<true>, dim3(rgrid), dim3(256), 0, st, (const float*)d_ws,
                                     d_Y, W->n, W->n, mm, g.splits));
      else
        KQ_CUDA_TRY(launch_dependent(reduce_splits_kernel<false>, dim3(rgrid), dim3(256), 0, st, (const float*)d_ws,
                                     d_Y + m0 * W->n, W->n, W->n, mm, g.splits));
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

int read_prep_status(int clear);     // kq_prep.cu
int read_control_status(int clear);  // kq_control.cu

}  // namespace kq

// -----------------------------------------------------------------------------
// Decode plan
// -----------------------------------------------------------------------------
struct kq_plan {
  int fmt = 0;
  int64_t count = 0;
  int64_t x_floats = 0, y_floats = 0, weight_bytes = 0;
  int grid = 0;
  int32_t nstages = 1;
  int32_t n_split = 0;
  bool linked = false;
  int64_t total_items = 0;
  int32_t n_cuts = 0;        // linked plan: row blocks cut between CTAs
  size_t counter_bytes = 0;  // linked plan: stage counters at the start of the workspace ...
  size_t ws_bytes = 0;       // ... then the partials of the cut row blocks
  kq::Job* d_jobs = nullptr;
  CUtensorMap* d_maps = nullptr;
  int64_t* d_bounds = nullptr;
  kq::XLink* d_links = nullptr;
  kq::Seg* d_segs = nullptr;
  kq::TileOut* d_tiles = nullptr;
  kq::CutOut* d_cuts = nullptr;
};

using namespace kq;

static void destroy_plan(kq_plan* p) {
  if (!p) return;
  cudaFree(p->d_jobs);
  cudaFree(p->d_maps);
  cudaFree(p->d_bounds);
  cudaFree(p->d_links);
  cudaFree(p->d_segs);
  cudaFree(p->d_tiles);
  cudaFree(p->d_cuts);
  delete p;
}

// Checks the links of a linked plan (see kq_link in kq.h).
static int check_links(const kq_qmat* mats, const kq_link* links, int64_t count) {
  for (int64_t i = 0; i < count; ++i) {
    const kq_link& L = links[i];
    if (L.reserved != 0) return fail(KQ_ERR_INVALID_ARG, "link %lld: reserved field not 0", (long long)i);
    if (L.stage < 0 || (i > 0 && L.stage < links[i - 1].stage))
      return fail(KQ_ERR_SHAPE, "link %lld: stage %d (stages start at 0 and never decrease)", (long long)i, L.stage);
    if (L.src == KQ_SRC_PACKED) continue;
    if (L.src != KQ_SRC_INPUT_OF && L.src != KQ_SRC_OUTPUT_OF)
      return fail(KQ_ERR_INVALID_ARG, "link %lld: unknown source kind %d", (long long)i, L.src);
    if (L.of < 0 || L.of >= i)
      return fail(KQ_ERR_INVALID_ARG, "link %lld: source matrix %lld is not an earlier one", (long long)i,
                  (long long)L.of);
    const kq_qmat& S = mats[L.of];
    if (L.src == KQ_SRC_INPUT_OF) {
      if (S.k != mats[i].k)
        return fail(KQ_ERR_SHAPE, "link %lld: k = %lld differs from matrix %lld's k = %lld", (long long)i,
                    (long long)mats[i].k, (long long)L.of, (long long)S.k);
    } else {
      if (mats[i].k > S.n)
        return fail(KQ_ERR_SHAPE, "link %lld: k = %lld exceeds matrix %lld's output length %lld", (long long)i,
                    (long long)mats[i].k, (long long)L.of, (long long)S.n);
      if (links[L.of].stage >= L.stage)
        return fail(KQ_ERR_SHAPE, "link %lld: reads the output of matrix %lld of stage %d from stage %d",
                    (long long)i, (long long)L.of, links[L.of].stage, L.stage);
      if (!std::isfinite(L.alpha)) return fail(KQ_ERR_INVALID_ARG, "link %lld: alpha is not finite", (long long)i);
    }
  }
  return KQ_OK;
}

// Linked plan: the segments of every stage (see Seg).  Each CTA gets a
// contiguous run of (row block, chunk) pairs, in list order, in one of two
// ways, whichever loads the busiest CTA less (the second on a tie within 2%):
//  - equal shares of the stage's weight bytes: a chunk belongs to the CTA
//    whose share holds the chunk's middle byte (stream-K);
//  - a capacity L, as small as fits the grid: a row block that fits whole
//    into the current CTA's rest goes there, one that fits a fresh CTA opens
//    the next one, and only a row block larger than L is cut, filling each
//    CTA to L.
// The second cuts fewer row blocks (none when every CTA can take whole ones).
// A CTA's run becomes segments, one per row block it touches; a row block cut
// between CTAs gets partial slots in CTA order.
// The chunk ranges a CTA needs from one activation are merged where they
// overlap or touch, and each segment records the merged range that holds it,
// which the CTA stages once (two pieces of different row blocks, say chunks
// [14, 17) and [0, 2), stay two small slices rather than the whole K).  Fills
// each job's row blocks (tiles, from jobs[j].tile_base) and the list of cut
// row blocks.
static void build_segments(std::vector<Job>& jobs, const std::vector<XLink>& xl, const kq_link* links,
                           int64_t count, int fmt, int G, int32_t nstages, std::vector<Seg>& segs,
                           std::vector<int64_t>& bounds, std::vector<TileOut>& tiles, std::vector<CutOut>& cuts,
                           int64_t& part_floats, std::vector<char>& job_cut) {
  const int64_t unit = chunk_of(fmt);
  const int TR = tile_rows(fmt);
  bounds.assign((size_t)nstages * (G + 1), 0);
  part_floats = 0;
  job_cut.assign((size_t)count, 0);
  tiles.clear();
  for (int64_t i = 0; i < count; ++i) {
    jobs[(size_t)i].tile_base = (int64_t)tiles.size();
    tiles.resize(tiles.size() + (size_t)jobs[(size_t)i].row_blocks, TileOut{0, 1, 0});
  }
  auto chunk_bytes = [&](const Job& J, int64_t rb, int64_t c) {
    const int64_t rows = std::min<int64_t>(TR, J.n - rb * TR);
    const int64_t kk = std::min<int64_t>(unit, J.k - c * unit);
    return (double)rows * (double)(code_row_bytes(fmt, kk) + 2 * (kk / block_of(fmt)));
  };
  int64_t i0 = 0;
  for (int32_t st = 0; st < nstages; ++st) {
    int64_t i1 = i0;
    while (i1 < count && links[i1].stage == st) ++i1;
    double total = 0;
    for (int64_t i = i0; i < i1; ++i) {
      const Job& J = jobs[(size_t)i];
      const int64_t nch = (J.k + unit - 1) / unit;
      for (int64_t rb = 0; rb < J.row_blocks; ++rb)
        for (int64_t c = 0; c < nch; ++c) total += chunk_bytes(J, rb, c);
    }
    // owners of the stage's chunks in (job, row block, chunk) order
    std::vector<double> cb;     // chunk bytes
    std::vector<size_t> tile0;  // first chunk of each row block, and the end
    for (int64_t i = i0; i < i1; ++i) {
      const Job& J = jobs[(size_t)i];
      const int64_t nch = (J.k + unit - 1) / unit;
      for (int64_t rb = 0; rb < J.row_blocks; ++rb) {
        tile0.push_back(cb.size());
        for (int64_t c = 0; c < nch; ++c) cb.push_back(chunk_bytes(J, rb, c));
      }
    }
    tile0.push_back(cb.size());
    std::vector<int> own_sk(cb.size()), own_pk(cb.size());
    double cum = 0;
    for (size_t g = 0; g < cb.size(); ++g) {
      own_sk[g] = std::min(G - 1, (int)((cum + 0.5 * cb[g]) * G / total));
      cum += cb[g];
    }
    // the packing with capacity L; returns the CTAs it needs
    auto pack = [&](double L, std::vector<int>& own) {
      int cta = 0;
      double used = 0;
      for (size_t t = 0; t + 1 < tile0.size(); ++t) {
        double bt = 0;
        for (size_t g = tile0[t]; g < tile0[t + 1]; ++g) bt += cb[g];
        if (used + bt > L && bt <= L && used > 0) {  // starts a fresh CTA whole
          ++cta;
          used = 0;
        }
        for (size_t g = tile0[t]; g < tile0[t + 1]; ++g) {
          if (used + cb[g] > L && used > 0) {
            ++cta;
            used = 0;
          }
          own[g] = cta;
          used += cb[g];
        }
      }
      return cb.empty() ? 0 : cta + 1;
    };
    auto busiest = [&](const std::vector<int>& own) {
      std::vector<double> load((size_t)G, 0.0);
      for (size_t g = 0; g < cb.size(); ++g) load[(size_t)std::min(own[g], G - 1)] += cb[g];
      return cb.empty() ? 0.0 : *std::max_element(load.begin(), load.end());
    };
    double lo = total / G, hi = 0;
    for (size_t g = 0; g < cb.size(); ++g) hi = std::max(hi, cb[g]);
    hi = std::max(2.0 * lo, lo + 2 * hi);
    if (!cb.empty() && pack(hi, own_pk) <= G) {
      for (int it = 0; it < 50; ++it) {
        const double mid = 0.5 * (lo + hi);
        if (pack(mid, own_pk) <= G) hi = mid; else lo = mid;
      }
    }
    const bool packed = !cb.empty() && pack(hi, own_pk) <= G && busiest(own_pk) <= 1.02 * busiest(own_sk);
    const std::vector<int>& own = packed ? own_pk : own_sk;
    // the stage's (job, row block, chunk) runs per owning CTA
    std::vector<Seg> raw;
    std::vector<int> owner;
    size_t gi = 0;
    for (int64_t i = i0; i < i1; ++i) {
      const Job& J = jobs[(size_t)i];
      const int64_t nch = (J.k + unit - 1) / unit;
      for (int64_t rb = 0; rb < J.row_blocks; ++rb)
        for (int64_t c = 0; c < nch; ++c) {
          const int cta = own[gi++];
          if (!raw.empty() && owner.back() == cta && raw.back().j == (int32_t)i && raw.back().rb == (int32_t)rb) {
            raw.back().c1 = (int32_t)c + 1;
          } else {
            Seg g{};
            g.j = (int32_t)i;
            g.rb = (int32_t)rb;
            g.c0 = (int32_t)c;
            g.c1 = (int32_t)c + 1;
            raw.push_back(g);
            owner.push_back(cta);
          }
        }
    }
    // cut row blocks (their pieces are adjacent in raw): slots and partials
    for (size_t a = 0; a < raw.size();) {
      size_t b = a + 1;
      while (b < raw.size() && raw[b].j == raw[a].j && raw[b].rb == raw[a].rb) ++b;
      const int32_t nseg = (int32_t)(b - a);
      int64_t part = 0;
      if (nseg > 1) {
        const Job& J = jobs[(size_t)raw[a].j];
        part = part_floats;
        part_floats += (int64_t)nseg * TR;
        job_cut[(size_t)raw[a].j] = 1;
        tiles[(size_t)(J.tile_base + raw[a].rb)] = TileOut{part, nseg, 0};
        cuts.push_back(CutOut{part, J.y_off + (int64_t)raw[a].rb * TR, nseg,
                              (int32_t)std::min<int64_t>(TR, J.n - (int64_t)raw[a].rb * TR)});
      }
      for (size_t q = a; q < b; ++q) {
        raw[q].nseg = nseg;
        raw[q].slot = (int32_t)(q - a);
        raw[q].part = part;
      }
      a = b;
    }
    // per CTA, in order: the staged union of each activation's chunk ranges
    int64_t* bs = bounds.data() + (size_t)st * (G + 1);
    size_t a = 0;
    for (int c = 0; c < G; ++c) {
      bs[c] = (int64_t)segs.size();
      size_t b = a;
      while (b < raw.size() && owner[b] == c) ++b;
      for (size_t q = a; q < b; ++q) {
        const int32_t key = xl[(size_t)raw[q].j].x_key;
        std::vector<std::pair<int32_t, int32_t>> rs;
        for (size_t r = a; r < b; ++r)
          if (xl[(size_t)raw[r].j].x_key == key) rs.emplace_back(raw[r].c0, raw[r].c1);
        std::sort(rs.begin(), rs.end());
        int32_t u0 = 0, u1 = 0;
        for (size_t r = 0; r < rs.size();) {  // the merged interval holding this segment
          int32_t m0 = rs[r].first, m1 = rs[r].second;
          size_t e = r + 1;
          while (e < rs.size() && rs[e].first <= m1) m1 = std::max(m1, rs[e++].second);
          if (raw[q].c0 >= m0 && raw[q].c1 <= m1) {
            u0 = m0;
            u1 = m1;
          }
          r = e;
        }
        Seg g = raw[q];
        g.u0 = u0;
        g.u1 = u1;
        segs.push_back(g);
      }
      a = b;
    }
    bs[G] = (int64_t)segs.size();
    i0 = i1;
  }
}

// Builds a plan.  links == nullptr: every matrix reads its own packed input,
// one stage, items of whole row blocks (kq_decode_plan_create).
static int create_plan(const kq_qmat* mats, const kq_link* links, int64_t count, kq_plan** out) {
  if (!mats || !out) return fail(KQ_ERR_INVALID_ARG, "NULL pointer");
  if (count < 1) return fail(KQ_ERR_SHAPE, "count = %lld", (long long)count);
  if (count > INT32_MAX / 2) return fail(KQ_ERR_SHAPE, "count = %lld", (long long)count);
  *out = nullptr;
  const int fmt = mats[0].fmt;
  for (int64_t i = 0; i < count; ++i) {
    if (int s = check_qmat(&mats[i], -1)) return fail(s, "matrix %lld: %s", (long long)i, kq_last_error());
    if (mats[i].fmt != fmt) return fail(KQ_ERR_UNSUPPORTED, "matrix %lld: mixed formats in one plan", (long long)i);
    if (mats[i].k > xmax_of(fmt))
      return fail(KQ_ERR_UNSUPPORTED, "matrix %lld: k = %lld > %d", (long long)i, (long long)mats[i].k,
                  xmax_of(fmt));
  }
  if (links)
    if (int s = check_links(mats, links, count)) return s;
  int sms = 0;
  if (int s = device_sms(&sms)) return s;
  const int32_t nstages = links ? links[count - 1].stage + 1 : 1;
  std::vector<Job> jobs((size_t)count);
  std::vector<CUtensorMap> maps((size_t)(2 * count));
  std::vector<XLink> xl((size_t)count);
  std::vector<double> item_bytes;
  int64_t items = 0, xf = 0, yf = 0, wb = 0;
  for (int64_t i = 0; i < count; ++i) {
    const kq_qmat& W = mats[i];
    if (int s = make_maps(&W, &maps[(size_t)(2 * i)], &maps[(size_t)(2 * i + 1)])) return s;
    const int64_t row_blocks = (W.n + tile_rows(fmt) - 1) / tile_rows(fmt);
    Job& j = jobs[(size_t)i];
    j = Job{};
    j.y_off = yf;
    j.n = W.n;
    j.k = W.k;
    j.ldy = W.n;
    j.item_begin = items;
    j.items = row_blocks;
    j.row_blocks = (int32_t)row_blocks;
    j.splits = 1;
    j.split_k = (int32_t)W.k;
    j.had_block = W.had_block;
    j.signs = W.signs;
    // activation source; INPUT_OF inherits its source's, so a group shares one key
    XLink& L = xl[(size_t)i];
    const int src = links ? links[i].src : KQ_SRC_PACKED;
    if (src == KQ_SRC_PACKED) {
      j.x_off = xf;
      xf += W.k;
      L = XLink{-1, -1, (int32_t)i, 1.f};
    } else if (src == KQ_SRC_INPUT_OF) {
      j.x_off = jobs[(size_t)links[i].of].x_off;
      L = xl[(size_t)links[i].of];
    } else {
      j.x_off = 0;
      L = XLink{(int32_t)links[i].of, links[(size_t)links[i].of].stage, (int32_t)i, links[i].alpha};
    }
    const double rowbytes = (double)code_row_bytes(fmt, W.k) + 2.0 * (double)(W.k / block_of(fmt));
    for (int64_t r = 0; r < row_blocks; ++r)
      item_bytes.push_back(rowbytes * (double)std::min<int64_t>(tile_rows(fmt), W.n - r * tile_rows(fmt)));
    items += row_blocks;
    yf += W.n;
    wb += kq_codes_bytes(fmt, W.n, W.k) + W.n * (W.k / block_of(fmt)) * 2;
  }
  kq_plan* p = new kq_plan();
  p->fmt = fmt;
  p->count = count;
  p->x_floats = xf;
  p->y_floats = yf;
  p->weight_bytes = wb;
  p->nstages = nstages;
  p->linked = links != nullptr;
  std::vector<int64_t> bounds;
  std::vector<Seg> segs;
  std::vector<TileOut> tiles;
  std::vector<CutOut> cuts;
  if (p->linked) {
    const int G = sms;
    int64_t part_floats = 0;
    std::vector<char> job_cut;
    build_segments(jobs, xl, links, count, fmt, G, nstages, segs, bounds, tiles, cuts, part_floats, job_cut);
    p->grid = G;
    p->total_items = (int64_t)segs.size();
    p->n_cuts = (int32_t)cuts.size();
    p->n_split = (int32_t)std::count(job_cut.begin(), job_cut.end(), 1);
    p->counter_bytes = (size_t)round_up((int64_t)nstages * 4, 256);
    p->ws_bytes = p->counter_bytes + (size_t)part_floats * sizeof(float);
  } else {
    // Contiguous item ranges, one per CTA, by bytes.  On a full grid the
    // shares are skewed: CTA c's capacity is proportional to
    // w_c = 1 + skew * (1/2 - c / (G - 1)).  Measured on GB300 (per-CTA
    // finish stamps of one launch): with equal shares the finish time grows
    // about linearly with the CTA index, ~5% from the first CTAs to the last,
    // reproducibly, with the work of every CTA alike and whatever the order
    // in which the weights were allocated.  The skew that compensates it
    // depends on the consumer; swept on the full steps with the cut points
    // below (GB/s):
    //  - PQ2_0, Bonsai-shaped: 0.03 5094, 0.045 5110, 0.06 5137, 0.075 5128,
    //    0.09 5092;
    //  - Q8_0, Qwen-shaped: 0.06 6702, 0.09 6763, 0.12 6759, 0.15 6660;
    //  - SCALE4, Qwen-shaped: 0.06 5975, 0.09 6047, 0.12 6099, 0.15 6115.
    // The cut points minimise the largest load relative to its capacity,
    // max_c bytes_c / w_c: the least T for which filling each CTA in turn
    // with whole items up to T w_c places every item (taking each range as
    // long as it fits is optimal for a given T), found by bisection.  An
    // item holds a whole row block (up to 1.3 MB), so cutting at the
    // cumulative targets instead could leave a CTA an item above its share.
    const int pf = plane_format(fmt);
    const double deal_skew = pf == KQ_PQ2_0 ? 0.06 : (pf == KQ_Q8_0 ? 0.09 : 0.15);
    p->total_items = items;
    p->grid = (int)std::min<int64_t>(items, sms);
    const int G = p->grid;
    const double skew = G >= 128 ? deal_skew : 0.0;
    std::vector<double> wgt((size_t)G);
    double wsum = 0, total = 0, biggest = 0;
    for (int c = 0; c < G; ++c) wsum += wgt[(size_t)c] = 1.0 + skew * (0.5 - (G > 1 ? (double)c / (G - 1) : 0.0));
    for (double b : item_bytes) {
      total += b;
      biggest = std::max(biggest, b);
    }
    bounds.assign((size_t)(G + 1), items);
    bounds[0] = 0;
    // fills CTA after CTA up to T w_c; true if every item found a place
    auto fill = [&](double T, bool record) {
      int c = 0;
      double load = 0;
      for (int64_t it = 0; it < items; ++it) {
        const double b = item_bytes[(size_t)it];
        while (load + b > T * wgt[(size_t)c]) {
          if (load == 0 || c + 1 == G) return false;  // the item fits no CTA from c on
          ++c;
          if (record) bounds[(size_t)c] = it;
          load = 0;
        }
        load += b;
      }
      if (record)
        for (int r = c + 1; r <= G; ++r) bounds[(size_t)r] = items;
      return true;
    };
    double lo = total / wsum, hi = (total + (double)G * biggest) / wsum * 2.0;
    for (int r = 0; r < 64 && !fill(hi, false); ++r) hi *= 2.0;
    for (int r = 0; r < 60; ++r) {
      const double mid = 0.5 * (lo + hi);
      (fill(mid, false) ? hi : lo) = mid;
    }
    fill(hi, true);
  }
  cudaError_t e = cudaMalloc(&p->d_jobs, sizeof(Job) * (size_t)count);
  if (e == cudaSuccess) e = cudaMalloc(&p->d_maps, sizeof(CUtensorMap) * (size_t)(2 * count));
  if (e == cudaSuccess) e = cudaMalloc(&p->d_bounds, sizeof(int64_t) * bounds.size());
  if (e == cudaSuccess) e = cudaMemcpy(p->d_jobs, jobs.data(), sizeof(Job) * (size_t)count, cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(p->d_maps, maps.data(), sizeof(CUtensorMap) * (size_t)(2 * count), cudaMemcpyHostToDevice);
  if (e == cudaSuccess)
    e = cudaMemcpy(p->d_bounds, bounds.data(), sizeof(int64_t) * bounds.size(), cudaMemcpyHostToDevice);
  if (p->linked) {
    if (e == cudaSuccess) e = cudaMalloc(&p->d_links, sizeof(XLink) * (size_t)count);
    if (e == cudaSuccess) e = cudaMemcpy(p->d_links, xl.data(), sizeof(XLink) * (size_t)count, cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !segs.empty()) {
      e = cudaMalloc(&p->d_segs, sizeof(Seg) * segs.size());
      if (e == cudaSuccess) e = cudaMemcpy(p->d_segs, segs.data(), sizeof(Seg) * segs.size(), cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = cudaMalloc(&p->d_tiles, sizeof(TileOut) * tiles.size());
    if (e == cudaSuccess)
      e = cudaMemcpy(p->d_tiles, tiles.data(), sizeof(TileOut) * tiles.size(), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !cuts.empty()) {
      e = cudaMalloc(&p->d_cuts, sizeof(CutOut) * cuts.size());
      if (e == cudaSuccess) e = cudaMemcpy(p->d_cuts, cuts.data(), sizeof(CutOut) * cuts.size(), cudaMemcpyHostToDevice);
    }
  }
  if (e != cudaSuccess) {
    destroy_plan(p);
    return fail(KQ_ERR_CUDA, "plan allocation: %s", cudaGetErrorString(e));
  }
  *out = p;
  return KQ_OK;
}

template <int FMT>
static int launch_plan(const Params& p, int grid, bool cooperative, cudaStream_t st) {
  if (!cooperative)
    return FMT == KQ_PQ2_0 && pq2_0_consumer() == KQ_PQ2_0_TCGEN05 ? launch_tcs(p, grid, st)
                                                                   : launch_stream<FMT, 1>(p, grid, st);
  // The CTAs of a linked plan wait for one another (stage counters): the
  // cooperative launch guarantees that all of them are resident at once.
  static std::once_flag once;
  static int status = KQ_OK;
  static char msg[160];
  if (int s = prepare_kernel_once(stream_kernel<FMT, 1, true>, Geo<FMT>::kSmemBytes, once, status, msg)) return s;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Geo<FMT>::kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  KQ_CUDA_TRY(cudaLaunchKernelEx(&cfg, stream_kernel<FMT, 1, true>, p));
  return KQ_OK;
}

extern "C" {

// kq_gemm_small_m runs on the tensor cores from tc_min_m activation rows on
// (when k fits the tensor-core prologue), else on the streaming kernel.
static bool small_m_uses_tc(const kq_qmat* W, int64_t m) {
  return m >= tc_min_m(W->fmt) && m <= kTcMaxM && W->k <= kTcMaxK;
}

size_t kq_gemv_workspace_bytes(const kq_qmat* W, int64_t m) {
  if (check_qmat(W, -1) != KQ_OK || m < 1) return 0;
  if (small_m_uses_tc(W, m)) return tc_workspace_bytes(W, m, 0);
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

int kq_gemv_f16(const kq_qmat* W, const void* d_x, void* d_y, void* d_ws, size_t ws_bytes, void* stream) {
  clear_error();
  return gemm_impl(W, static_cast<const float*>(d_x), 1, static_cast<float*>(d_y), 0, d_ws, ws_bytes, stream, -1,
                   true);
}

int kq_gemv_scale4(const kq_qmat* W, const float* d_x, float* d_y, void* d_ws, size_t ws_bytes, void* stream) {
  clear_error();
  return gemm_impl(W, d_x, 1, d_y, 0, d_ws, ws_bytes, stream, KQ_SCALE4);
}

int kq_gemv_pq2_0(const kq_qmat* W, const float* d_x, float* d_y, void* d_ws, size_t ws_bytes, void* stream) {
  clear_error();
  return gemm_impl(W, d_x, 1, d_y, 0, d_ws, ws_bytes, stream, KQ_PQ2_0);
}

int kq_gemm_small_m(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, void* d_ws, size_t ws_bytes,
                    void* stream) {
  clear_error();
  if (int s = check_qmat(W, -1)) return s;
  if (small_m_uses_tc(W, m)) return tc_gemm(W, d_X, m, d_Y, 0, d_ws, ws_bytes, stream);
  return gemm_impl(W, d_X, m, d_Y, 0, d_ws, ws_bytes, stream, -1);
}

size_t kq_gemm_tc_workspace_bytes(const kq_qmat* W, int64_t m, int32_t splits) {
  if (check_qmat(W, -1) != KQ_OK || splits < 0 || tc_check(W, m) != KQ_OK) {
    clear_error();
    return 0;
  }
  return tc_workspace_bytes(W, m, splits);
}

int kq_gemm_tc(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int32_t splits, void* d_ws,
               size_t ws_bytes, void* stream) {
  clear_error();
  if (int s = check_qmat(W, -1)) return s;
  if (splits < 0) return fail(KQ_ERR_INVALID_ARG, "splits = %d", splits);
  return tc_gemm(W, d_X, m, d_Y, splits, d_ws, ws_bytes, stream);
}

int kq_gemm_splitk(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int32_t splits, void* d_ws,
                   size_t ws_bytes, void* stream) {
  clear_error();
  return gemm_impl(W, d_X, m, d_Y, splits, d_ws, ws_bytes, stream, -1);
}

int kq_decode_plan_create(const kq_qmat* mats, int64_t count, kq_plan** out) {
  clear_error();
  return create_plan(mats, nullptr, count, out);
}

int kq_decode_plan_create_linked(const kq_qmat* mats, const kq_link* links, int64_t count, kq_plan** out) {
  clear_error();
  if (!links) return fail(KQ_ERR_INVALID_ARG, "NULL links");
  return create_plan(mats, links, count, out);
}

int kq_decode_plan_stages(const kq_plan* plan, int32_t* stages, int32_t* split_matrices) {
  clear_error();
  if (!plan) return fail(KQ_ERR_INVALID_ARG, "NULL plan");
  if (stages) *stages = plan->nstages;
  if (split_matrices) *split_matrices = plan->n_split;
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

size_t kq_decode_workspace_bytes(const kq_plan* plan) { return plan ? plan->ws_bytes : 0; }

int kq_decode_step(kq_plan* plan, const float* d_x_packed, float* d_y_packed, void* d_ws, size_t ws_bytes,
                   void* stream) {
  clear_error();
  if (!plan) return fail(KQ_ERR_INVALID_ARG, "NULL plan");
  if ((!d_x_packed && plan->x_floats > 0) || !d_y_packed) return fail(KQ_ERR_INVALID_ARG, "NULL activation or output");
  if (!aligned16(d_x_packed) || !aligned16(d_y_packed)) return fail(KQ_ERR_ALIGNMENT, "x or y not 16-byte aligned");
  if (plan->ws_bytes > 0) {
    if (!d_ws || ws_bytes < plan->ws_bytes)
      return fail(KQ_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", plan->ws_bytes, d_ws ? ws_bytes : 0);
    if (!aligned16(d_ws)) return fail(KQ_ERR_ALIGNMENT, "workspace not 16-byte aligned");
  }
  cudaStream_t st = (cudaStream_t)stream;
  Params p{};
  p.jobs = plan->d_jobs;
  p.maps = plan->d_maps;
  p.links = plan->d_links;
  p.x_base = d_x_packed;
  p.y_base = d_y_packed;
  p.bounds = plan->d_bounds;
  p.total_items = plan->total_items;
  p.nstages = plan->nstages;
  if (plan->linked) {
    p.stage_done = static_cast<int32_t*>(d_ws);
    p.ws_base = reinterpret_cast<float*>(static_cast<uint8_t*>(d_ws) + plan->counter_bytes);
    p.segs = plan->d_segs;
    p.tiles = plan->d_tiles;
    p.cuts = plan->d_cuts;
    p.n_cuts = plan->n_cuts;
    KQ_CUDA_TRY(cudaMemsetAsync(d_ws, 0, (size_t)plan->nstages * sizeof(int32_t), st));
  }
  if (plan->fmt == KQ_Q8_0) return launch_plan<KQ_Q8_0>(p, plan->grid, plan->linked, st);
  if (plan->fmt == KQ_SCALE4) return launch_plan<KQ_SCALE4>(p, plan->grid, plan->linked, st);
  return launch_plan<KQ_PQ2_0>(p, plan->grid, plan->linked, st);
}

void kq_decode_plan_destroy(kq_plan* plan) { destroy_plan(plan); }

// ---------------------------------------------------------------------------
// Allocation-free split-K GEMM.
//
// Some callers cannot call cudaMalloc at the point where they run the
// product: code that must not allocate after start-up (a real-time serving
// loop, memory pools that forbid allocations outside their own arena, or
// callers that only hold device pointers handed to them).  For them the
// split-K partial sums live in one library-owned array in device global
// memory, reserved when the library is loaded on a device and kept until the
// process exits.
// ---------------------------------------------------------------------------
static constexpr size_t kNoAllocScratchBytes = 2u << 20;  // 2 MiB per device
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchBytes / sizeof(float)];

static std::mutex g_noalloc_mutex;
static std::vector<void*> g_noalloc_ptr;  // device address of the array, per device

// The array's device address on the current device.  In host code the
// array's name is only a host-side stand-in, so its address is looked up
// once per device (cudaGetSymbolAddress, with that device current; it
// allocates nothing) and kept.  A device reset invalidates the kept address.
static int noalloc_scratch(void** out) {
  int dev = 0;
  KQ_CUDA_TRY(cudaGetDevice(&dev));
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if ((int)g_noalloc_ptr.size() <= dev) g_noalloc_ptr.resize((size_t)dev + 1, nullptr);
  if (g_noalloc_ptr[(size_t)dev] == nullptr) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return fail(KQ_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
    g_noalloc_ptr[(size_t)dev] = ptr;
  }
  *out = g_noalloc_ptr[(size_t)dev];
  return KQ_OK;
}

size_t kq_gemm_splitk_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

int kq_gemm_splitk_noalloc(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int32_t splits, void* stream) {
  clear_error();
  if (int s = check_qmat(W, -1)) return s;
  if (m < 1 || m > kMaxM) return fail(KQ_ERR_SHAPE, "m = %lld outside [1, %lld]", (long long)m, (long long)kMaxM);
  if (splits < 0) return fail(KQ_ERR_INVALID_ARG, "splits = %d", splits);
  const size_t need = splitk_ws_bytes(W, m, splits);
  if (need > kNoAllocScratchBytes)
    return fail(KQ_ERR_WORKSPACE,
                "this split plan needs %zu bytes of scratch; the allocation-free variant has %zu (use kq_gemm_splitk "
                "with a workspace, or fewer splits)",
                need, kNoAllocScratchBytes);
  void* ws = nullptr;
  if (int s = noalloc_scratch(&ws)) return s;
  return gemm_impl(W, d_X, m, d_Y, splits, ws, kNoAllocScratchBytes, stream, -1);
}

int kq_set_pq2_0_consumer(int consumer) {
  clear_error();
  if (consumer != KQ_PQ2_0_MMA_SYNC && consumer != KQ_PQ2_0_TCGEN05)
    return fail(KQ_ERR_INVALID_ARG, "unknown PQ2_0 consumer %d", consumer);
  kq::g_pq2_0_consumer.store(consumer, std::memory_order_relaxed);
  return KQ_OK;
}

int kq_get_pq2_0_consumer(void) { return kq::g_pq2_0_consumer.load(std::memory_order_relaxed); }

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
  int a = read_stream_status(clear), b = read_prep_status(clear), c = read_tc_status(clear);
  int d = read_control_status(clear), t = read_tcs_status(clear);
  if (a < 0 || b < 0 || c < 0 || d < 0 || t < 0) return fail(KQ_ERR_CUDA, "reading the device status word failed");
  const unsigned v = (unsigned)a | (unsigned)b | (unsigned)c | (unsigned)d | (unsigned)t;
  if (v & (1u << KQ_ERR_TIMEOUT)) return fail(KQ_ERR_TIMEOUT, "a bounded device wait expired");
  if (v & (1u << KQ_ERR_NONFINITE)) return fail(KQ_ERR_NONFINITE, "non-finite weight met on the device");
  if (v & (1u << KQ_ERR_RANGE)) return fail(KQ_ERR_RANGE, "scale overflowed fp16 on the device");
  return KQ_OK;
}

}  // extern "C"
