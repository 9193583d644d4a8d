// Small-batch quantized GEMM on the 5th-generation tensor cores (tcgen05):
// Y[m][n] = X[m] . W[n] for up to 64 activation rows (X rotated per
// 128-block for PQ2_0).  With tens of activation rows the product is a real
// dense contraction (PQ2_0 at m = 64: ~390 flop per weight byte), so each
// weight chunk is unpacked once into 16-bit operands and multiplied on
// tcgen05 with fp32 accumulators in tensor memory ("Kipp Benchmarks", tensor
// matmul section: unpack a K block into a 16-bit tile, then one matrix
// multiply per block).
//
//  * Activation prologue (act_hilo_kernel): X -> blockwise normalised
//    Walsh-Hadamard transform for PQ2_0 ("Bonsai 2 27B - ternary g128 +
//    blockwise Hadamard", section 4.2) -> per-row power-of-two normalisation
//    -> an fp16 high/low matrix B[2M'][K] (row i = high part of activation
//    row i, row M'+i = its low part; M' = m rounded up to 16, extra rows
//    zero), K-major, in the caller's workspace.  hi + lo carries x to ~2^-22
//    relative.  One MMA multiplies A by both halves (N = 2M').
//  * Main kernel (tc_gemm_kernel), one persistent CTA per SM over a list of
//    items (128-row tile of W, K split), 128-weight K chunks:
//      warp 0       TMA producer: per chunk the codes of 128 rows and two
//                   64-wide 128-byte-swizzled boxes of B;
//      warp 1       allocates tensor memory and issues tcgen05.mma
//                   (kind::f16, M = 128, N = 2M', K = 16, A from tensor
//                   memory, B from shared memory) and the commits: the warp
//                   walks the list in step, one elected lane issues;
//      warps 18-19  for PQ2_0, two more issuing warps: issuer g % 3 takes
//                   the CTA's chunk g and owns accumulator buffer g % 3;
//      warps 2-9    unpack the chunk into the A operand in tensor memory
//                   (tcgen05.st): lane i of a warp owns weight row i of its
//                   quarter, each warp half of the chunk's K;
//      warps 10-17  epilogue (tcgen05.ld), each warp half of the activation
//                   columns of its lane quarter; it reads the block scales
//                   of its rows from the scales plane itself, one or two
//                   chunks ahead, so a stage is free once it has been
//                   unpacked and multiplied.
//    The A operand never touches shared memory (a 16-bit tile there would
//    cost ~4 bytes of shared-memory traffic per weight).
//  * A holds the integer code values only, exactly: q for Q8_0 (an fp16
//    integer), c - 1 for PQ2_0.  Each quantization block (32 weights for
//    Q8_0, 128 for PQ2_0) gets its own accumulator in tensor memory, and the
//    epilogue adds d_block * (hi + lo columns) into running sums held in
//    registers, scaled by the activation row's power of two at the end of
//    the item.  No weight is rounded and nothing cancels.
//  * PQ2_0 unpack: code e and code e + 8 of each 16-code word masked into
//    the two fp16 halves of a 32-bit word are the exact fp16 subnormals
//    c * 2^(s-24) (s = their bit offset, at most 8 after one shift for the
//    upper codes); one fp16 subtraction of 2^(s-24) makes them
//    (c - 1) * 2^(s-24).  The prologue scales the matching B entries by
//    2^(24-s) and permutes B's K order to the pairing, so A x B sums
//    (c - 1) x' 2^-(10+e) for every position.
//  * An issuing thread issues one instruction per 16-weight K step (8 per
//    chunk).  Measured on GB300: a thread issuing tcgen05.mma back to back
//    spends ~55-110 cycles per instruction whatever N is up to 128, so at
//    small N one thread, not the tensor pipe, would set the pace.  PQ2_0 has
//    three issuers that take whole chunks in turn and never wait for one
//    another; Q8_0 and SCALE4 keep one, as their four accumulator blocks per
//    chunk leave tensor memory for only three chunks' accumulators.  When a
//    chunk's blocks share one accumulator group (M' = 16), their MMA chains
//    are issued alternately (step t of every block, then step t + 1).
//  * The unpack -> issuer barrier is per stage slot and waited on with the
//    stage's phase right after that slot's tma_full, so an issuer that skips
//    the other issuers' chunks can never take another chunk's phase for its
//    own.
// Every wait is bounded; a timeout sets KQ_ERR_TIMEOUT in the status word,
// every role stops waiting, the producer waits (bounded) for its copies in
// flight, the MMA thread drains its work, and the tensor memory is freed
// before the kernel returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "kq_device.cuh"
#include "kq_internal.h"
#include "kq_tc.h"
#include "kq_tcgen05.cuh"

namespace kq {
namespace tc {

constexpr int kRows = 128;     // W rows per tile (MMA M)
constexpr int kChunk = 128;    // weights per K chunk
constexpr int kMaxStages = 8;  // TMA ring depth limit
constexpr int kMaxD = 4;       // accumulator buffers in tensor memory
constexpr int kDeqWarps = 8;
constexpr int kEpiWarps = 8;
constexpr int kIssuer2Warp = 2 + kDeqWarps + kEpiWarps;  // the second and third MMA issuers
constexpr int kMaxIssuers = 3;
constexpr int kThreads = 32 * (kIssuer2Warp + kMaxIssuers - 1);  // 640
constexpr int kBarBytes = 512;
constexpr size_t kSmemBytes = 232448;  // the per-CTA maximum; carved at run time
constexpr size_t kCarveBytes = kSmemBytes - 1024 /* alignment slack */ - kBarBytes;
// tensor memory: two A buffers of 64 columns (128 fp16 per row) at [0, 128),
// then the accumulators, 2M' columns each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACols = kChunk / 2;  // tensor-memory columns of one A buffer
constexpr int kMaxA = 4;                 // A buffers

// code bytes of one 128-weight chunk of a row: 128 (Q8_0), 64 (SCALE4), 32 (PQ2_0)
__host__ __device__ constexpr int chunk_row_bytes(int fmt) {
  return fmt == KQ_Q8_0 ? kChunk : (fmt == KQ_SCALE4 ? kChunk / 2 : kChunk / 4);
}
__host__ __device__ constexpr int code_chunk_bytes(int fmt) { return kRows * chunk_row_bytes(fmt); }
__host__ __device__ constexpr int b_box_bytes(int mp) { return 2 * mp * 128; }  // 64 fp16 x 2M' rows
__host__ __device__ constexpr int stage_tx_bytes(int fmt, int mp) {
  return code_chunk_bytes(fmt) + 2 * b_box_bytes(mp);
}
__host__ __device__ constexpr int stage_bytes(int fmt, int mp) { return (stage_tx_bytes(fmt, mp) + 1023) / 1024 * 1024; }
// Accumulator groups: a group holds `gb` consecutive blocks' accumulators
// (2M' columns each) under one barrier pair, so the MMA thread waits and
// commits once per group; groups rotate through d_groups() buffers.
__host__ __device__ constexpr int blocks_per_chunk(int fmt) { return fmt == KQ_PQ2_0 ? 1 : 4; }
__host__ __device__ constexpr int d_groups_for(int gb, int mp, int na = 2) {
  return (int)((kTmemCols - na * kACols) / (gb * 2 * mp)) < kMaxD ? (int)((kTmemCols - na * kACols) / (gb * 2 * mp))
                                                                  : kMaxD;
}
// A buffers (the unpack runs that many chunks ahead of the MMAs): PQ2_0 takes
// four, or three, while tensor memory still holds an accumulator buffer for
// each of its three issuers; Q8_0 and SCALE4 keep two.
__host__ __device__ constexpr int a_buffers(int fmt, int mp) {
  return blocks_per_chunk(fmt) != 1          ? 2
         : d_groups_for(1, mp, 4) >= 3       ? 4
         : d_groups_for(1, mp, 3) >= 3       ? 3
                                             : 2;
}
// largest group (4, 2 or 1 blocks, dividing the chunk's blocks) that still leaves three buffers
__host__ __device__ constexpr int group_blocks(int fmt, int mp) {
  return (blocks_per_chunk(fmt) >= 4 && d_groups_for(4, mp) >= 3)   ? 4
         : (blocks_per_chunk(fmt) >= 2 && d_groups_for(2, mp) >= 3) ? 2
                                                                     : 1;
}

__device__ unsigned int g_tc_status = 0;
__device__ __forceinline__ void tc_flag(int status) { atomicOr(&g_tc_status, 1u << status); }

struct TcParams {
  CUtensorMap map_codes;   // Q8_0: u32 [n][k/4], box 32 x 128, 128B swizzle; PQ2_0: u32 [n][k/16], box 8 x 128, 32B swizzle
  const uint16_t* scales;   // fp16 block scales [n][sstride]
  int64_t sstride;          // scales per row (a multiple of 8)
  int32_t kblocks;          // quantization blocks per row (k / block)
  CUtensorMap map_b;       // fp16 [2M'][k], box 64 x 2M', 128B swizzle
  const float* bscale;     // per activation row: the power of two the result is scaled by
  float* y;                // splits == 1: Y [m][n]; else partials [splits][m][n]
  int64_t n;
  int32_t m;       // activation rows
  int32_t mp;      // M' = m rounded up to 16
  int32_t tiles;   // 128-row tiles
  int32_t chunks;  // K chunks
  int32_t splits;  // K splits; items = splits * tiles, split-major
  int32_t stages;  // ring stages (host: as many as fit, at most kMaxStages)
};

// Position in a ring of n slots with a phase bit that flips on wrap-around.
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++slot == n) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

// ---- activation prologue ------------------------------------------------------

// PQ2_0: code pair e (codes e and e + 8 of a 16-code word) sits at bit
// offset s_e inside its fp16 half after the unpack: 2e for e <= 4, 2e - 8
// for e >= 5 (those come from the word shifted right by 8).
__host__ __device__ constexpr int pq2_0_shift(int e) { return e <= 4 ? 2 * e : 2 * e - 8; }
// K position of weight j (within its 16-weight group) in a PQ2_0 B row: even
// positions hold weights 0..7, odd positions weights 8..15.
__device__ __forceinline__ int pq2_0_pos(int j) { return j < 8 ? 2 * j : 2 * (j - 8) + 1; }
// SCALE4: a word's 4-bit codes unpack as the pairs (0,4), (1,5), (2,6),
// (3,7) of its eight weights, codes 1, 3, 5, 7 at bit offset 4 inside their
// fp16 half and codes 0, 2, 4, 6 at offset 0; weight j of an 8-group goes to
// B position 2 (j % 4) + j / 4.
__host__ __device__ constexpr int scale4_shift(int j) { return 4 * (j & 1); }
__device__ __forceinline__ int scale4_pos(int j) { return 2 * (j & 3) + (j >> 2); }

template <int FMT>
__global__ void act_hilo_kernel(const float* __restrict__ X, int m, int mp, int64_t k, __half* __restrict__ B,
                                float* __restrict__ bscale, int had, const int8_t* __restrict__ signs) {
  // one CTA per activation row i < M' (rows i >= m are zero).  Launched as a
  // programmatic dependent: X is read only after the kernel before has
  // completed; the GEMM may then launch at once and set itself up while this
  // runs (it waits for this grid's completion before reading B).
  grid_dependency_wait();
  allow_dependent_launch();
  const int i = blockIdx.x;
  __half* hi = B + (int64_t)i * k;
  __half* lo = B + (int64_t)(mp + i) * k;
  const int64_t nblk = k / 128;
  extern __shared__ float xs[];  // k floats
  __shared__ float red[32];
  if (i >= m) {
    for (int64_t j = threadIdx.x; j < k; j += blockDim.x) {
      hi[j] = __float2half_rn(0.f);
      lo[j] = __float2half_rn(0.f);
    }
    if (threadIdx.x == 0) bscale[i] = 0.f;
    return;
  }
  const float* x = X + (int64_t)i * k;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if (FMT == KQ_PQ2_0) {
    // x' = (1/sqrt(128)) H x per 128-block: butterflies of strides 1, 2 in
    // registers, 4 .. 64 across lanes (each lane holds 4 consecutive values).
    // The page's n = 1024 rotation (sign flip first) is H_8 (x) H_128 in
    // Sylvester order: the same 128-point pass unscaled, then an 8-point
    // pass across the eight 128-blocks of each 1024-block, times 1/32.
    const float inv_sqrt128 = had == 1024 ? 1.f : 0.08838834764831845f;
    for (int64_t b = warp; b < nblk; b += nwarps) {
      float4 f = *reinterpret_cast<const float4*>(x + b * 128 + 4 * lane);
      if (signs) {
        const char4 s4 = *reinterpret_cast<const char4*>(signs + b * 128 + 4 * lane);
        f.x *= (float)s4.x;
        f.y *= (float)s4.y;
        f.z *= (float)s4.z;
        f.w *= (float)s4.w;
      }
      float v[4];
      const float a0 = f.x + f.y, a1 = f.x - f.y, a2 = f.z + f.w, a3 = f.z - f.w;
      v[0] = a0 + a2;
      v[1] = a1 + a3;
      v[2] = a0 - a2;
      v[3] = a1 - a3;
#pragma unroll
      for (int mk = 1; mk < 32; mk <<= 1) {
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float q = __shfl_xor_sync(0xffffffffu, v[t], mk);
          v[t] = (lane & mk) ? (q - v[t]) : (v[t] + q);
        }
      }
      *reinterpret_cast<float4*>(xs + b * 128 + 4 * lane) =
          make_float4(v[0] * inv_sqrt128, v[1] * inv_sqrt128, v[2] * inv_sqrt128, v[3] * inv_sqrt128);
    }
    if (had == 1024) {
      __syncthreads();
      for (int64_t c = threadIdx.x; c < (k / 1024) * 128; c += blockDim.x) {
        float* col = xs + (c / 128) * 1024 + (c % 128);
        float v[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) v[a] = col[a * 128];
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
        for (int a = 0; a < 8; ++a) col[a * 128] = v[a] * 0.03125f;
      }
    }
  } else {
    for (int64_t j = threadIdx.x; j < k; j += blockDim.x) xs[j] = x[j];
  }
  __syncthreads();
  float amax = 0.f;
  for (int64_t j = threadIdx.x; j < k; j += blockDim.x) amax = fmaxf(amax, fabsf(xs[j]));
#pragma unroll
  for (int mk = 16; mk; mk >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, mk));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  if (threadIdx.x == 0) {
    float a = 0.f;
    for (int w = 0; w < nwarps; ++w) a = fmaxf(a, red[w]);
    // e = floor(log2 a) for normal a: x * 2^-e then lies in (-2, 2)
    int e = a > 0.f ? ((__float_as_int(a) >> 23) & 0xFF) - 127 : 0;
    if (FMT != KQ_Q8_0 && e > 116) tc_flag(KQ_ERR_RANGE);  // 2^(10+e) must stay a finite fp32
    // PQ2_0 and SCALE4 also scale by 2^(14-s-e) with s <= 8 and by 2^(10+e): e in [-113, 116]
    red[0] = FMT != KQ_Q8_0 ? (float)max(-113, min(116, e)) : (float)max(-126, min(126, e));
  }
  __syncthreads();
  const int e = (int)red[0];
  if (FMT == KQ_Q8_0) {
    const float unscale = __int_as_float((127 - e) << 23);  // 2^-e, exact
    for (int64_t j = threadIdx.x; j < k; j += blockDim.x) {
      const float v = xs[j] * unscale;
      const __half h = __float2half_rn(v);
      hi[j] = h;
      lo[j] = __float2half_rn(v - __half2float(h));  // v - h is exact in fp32
    }
    if (threadIdx.x == 0) bscale[i] = __int_as_float((127 + e) << 23);  // 2^e
  } else if (FMT == KQ_SCALE4) {
    // B entry of weight j: x_j 2^(14 - s - e), s the bit offset of its code, at its unpack position
    for (int64_t j = threadIdx.x; j < k; j += blockDim.x) {
      const int jj = (int)(j & 7);
      const float v = xs[j] * __int_as_float((127 + 14 - scale4_shift(jj) - e) << 23);
      const __half h = __float2half_rn(v);
      const int64_t pos = (j & ~(int64_t)7) + scale4_pos(jj);
      hi[pos] = h;
      lo[pos] = __float2half_rn(v - __half2float(h));
    }
    if (threadIdx.x == 0) bscale[i] = __int_as_float((127 + 10 + e) << 23);  // 2^(10+e)
  } else {
    // B entry of weight j: x'_j 2^(14 - s - e), s the bit offset of its code
    for (int64_t j = threadIdx.x; j < k; j += blockDim.x) {
      const int jj = (int)(j & 15), pair = jj & 7;
      const float v = xs[j] * __int_as_float((127 + 14 - pq2_0_shift(pair) - e) << 23);
      const __half h = __float2half_rn(v);
      const int64_t pos = (j & ~(int64_t)15) + pq2_0_pos(jj);
      hi[pos] = h;
      lo[pos] = __float2half_rn(v - __half2float(h));
    }
    if (threadIdx.x == 0) bscale[i] = __int_as_float((127 + 10 + e) << 23);  // 2^(10+e)
  }
}

// ---- epilogue role ------------------------------------------------------------------

// What the epilogue warps need from the kernel's set-up.
struct EpiCtx {
  uint64_t* d_full;
  uint64_t* d_empty;
  volatile int* abort_flag;
  int gb, nd, ib, ie, mp;
  uint32_t d_lane;  // this warp's lane quarter and first activation column in the accumulators
  int r, i0;        // this lane's tile row; this warp's first activation row
};

// The fp16 block scales of chunk c of a row, read past L1: four (8 bytes)
// for Q8_0 and SCALE4, one for PQ2_0.
template <int kBlocks>
struct ChunkScales {
  uint32_t w[kBlocks == 4 ? 2 : 1];
  __device__ __forceinline__ void load(const uint16_t* srow, int c) {
    if constexpr (kBlocks == 4) {
      const uint2 v = __ldcg(reinterpret_cast<const uint2*>(srow) + c);
      w[0] = v.x;
      w[1] = v.y;
    } else {
      w[0] = __ldcg(reinterpret_cast<const unsigned short*>(srow) + c);
    }
  }
  __device__ __forceinline__ float get(int b) const {
    return __half2float(__ushort_as_half((uint16_t)(w[b >> 1] >> (16 * (b & 1)))));
  }
};

// The epilogue warps: per chunk, the block scales of row r (read from the
// scales plane one chunk ahead), then per block
// d * (hi + lo) of the warp's HALF activation columns added into registers.
// The accumulator loads are batched to few tensor-memory round trips: two
// blocks per wait at HALF = 8 (their group holds all four blocks of the
// chunk), sixteen columns (hi and lo) per wait otherwise.  The epilogue never
// touches the stages.
template <int FMT, int HALF>
__device__ __forceinline__ void epilogue_role(const TcParams& p, const EpiCtx& e, int lane) {
  constexpr int kBlocks = blocks_per_chunk(FMT);
  constexpr int NI = kBlocks == 1 ? kMaxIssuers : 1;
  constexpr int kSeg = HALF >= 16 ? 16 : 8;                      // columns per load (hi and lo each)
  constexpr int kPair = (HALF == 8 && kBlocks >= 2) ? 2 : 1;     // blocks per wait
  const int MP = e.mp, gb = e.gb;
  Ring dr0;  // the accumulator buffers (one issuer)
  int g = 0;  // the chunk's place in this CTA's list (its issuer is g % NI)
  for (int item = e.ib; item < e.ie; ++item) {
    const int split = item / p.tiles, tile = item - split * p.tiles;
    const int c0 = (int)((int64_t)split * p.chunks / p.splits), c1 = (int)((int64_t)(split + 1) * p.chunks / p.splits);
    const int64_t row = (int64_t)tile * kRows + e.r;
    const bool live_row = row < p.n;
    const uint16_t* srow = p.scales + (live_row ? row : 0) * p.sstride;
    float acc[HALF];
#pragma unroll
    for (int q = 0; q < HALF; ++q) acc[q] = 0.f;
    // the scales of the next kAhead chunks are in flight (two for PQ2_0, whose
    // chunks are short; one for Q8_0 and SCALE4, whose registers are tight)
    constexpr int kAhead = kBlocks == 1 ? 2 : 1;
    ChunkScales<kBlocks> n1, n2;
    n1.load(srow, c0);
    if (kAhead > 1 && c0 + 1 < c1) n2.load(srow, c0 + 1);
    for (int c = c0; c < c1; ++c, ++g) {
      if (*e.abort_flag) continue;
      const int me = g % NI;
      // this chunk's block scales of row r; blocks past k (a ragged last chunk) weigh 0
      const ChunkScales<kBlocks> cur = n1;
      if constexpr (kAhead > 1) {
        n1 = n2;
        if (c + 2 < c1) n2.load(srow, c + 2);
      } else {
        if (c + 1 < c1) n1.load(srow, c + 1);
      }
      const int blk0 = c * kBlocks;
      float dsc[kBlocks];
#pragma unroll
      for (int b = 0; b < kBlocks; ++b) dsc[b] = live_row && blk0 + b < p.kblocks ? cur.get(b) : 0.f;
#pragma unroll
      for (int b = 0; b < kBlocks; b += kPair) {
        const int bg = b % gb;
        // one issuer: a ring over the buffers; several: buffer `me`, its (g / NI)-th use
        const int dslot = NI == 1 ? dr0.slot : me;
        const uint32_t dphase = NI == 1 ? dr0.phase : (uint32_t)((g / NI) & 1);
        if (bg == 0) {
          if (!mbar_wait_bounded(&e.d_full[dslot], dphase)) {
            *e.abort_flag = 1;
            tc_flag(KQ_ERR_TIMEOUT);
            break;
          }
          tc_fence_after();
        }
        const uint32_t t0 = e.d_lane + (uint32_t)((dslot * gb + bg) * 2 * MP);
#pragma unroll
        for (int c8 = 0; c8 < HALF; c8 += kSeg) {
          constexpr int kW = kSeg;
          const int w = HALF - c8 < kW ? HALF - c8 : kW;  // 8 or 16 columns in this segment
          float vh[kPair][kW], vl[kPair][kW];
#pragma unroll
          for (int pb = 0; pb < kPair; ++pb) {
            const uint32_t tb = t0 + (uint32_t)(pb * 2 * MP);
            if constexpr (kW == 16) {
              if (w == 16) {
                tmem_ld16(tb + (uint32_t)c8, vh[pb]);         // x high parts
                tmem_ld16(tb + (uint32_t)(MP + c8), vl[pb]);  // x low parts
                continue;
              }
            }
            tmem_ld8(tb + (uint32_t)c8, *reinterpret_cast<float(*)[8]>(vh[pb]));
            tmem_ld8(tb + (uint32_t)(MP + c8), *reinterpret_cast<float(*)[8]>(vl[pb]));
          }
          tmem_ld_wait();
#pragma unroll
          for (int pb = 0; pb < kPair; ++pb)
#pragma unroll
            for (int q = 0; q < kW; ++q)
              if (q < w) acc[c8 + q] = fmaf(dsc[b + pb], vh[pb][q] + vl[pb][q], acc[c8 + q]);
        }
        if (bg + kPair - 1 == gb - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&e.d_empty[dslot]);
          if (NI == 1) dr0.next(e.nd);
        }
      }
    }
    if (*e.abort_flag) continue;
    float* out = p.y + (int64_t)split * p.m * p.n;
#pragma unroll
    for (int q = 0; q < HALF; ++q) {
      const int i = e.i0 + q;
      if (i < p.m && live_row) out[(int64_t)i * p.n + row] = acc[q] * p.bscale[i];
    }
  }
}

// ---- main kernel ------------------------------------------------------------------

template <int FMT>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // the swizzled tiles need 1024-byte alignment
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  constexpr int kCodes = code_chunk_bytes(FMT);
  constexpr int kBlocks = blocks_per_chunk(FMT);   // quantization blocks per chunk
  constexpr int kSteps = (kChunk / 16) / kBlocks;  // 16-weight MMA steps per block
  const int MP = p.mp;
  const int nstages = p.stages;
  const int gb = group_blocks(FMT, MP);  // blocks per accumulator group
  const int na = a_buffers(FMT, MP);      // A buffers
  const uint32_t tmem_d = (uint32_t)na * kACols;  // first accumulator column
  const int nd = d_groups_for(gb, MP, na);  // accumulator groups in tensor memory
  // PQ2_0 (one block, a few accumulator columns per chunk): three MMA issuers
  // take turns by chunk (g = a chunk's place in this CTA's list); issuer
  // g % 3 owns accumulator buffer g % 3 (nd >= 3), the A buffers alternate
  // by chunk, and no issuer waits for another.  Q8_0 and SCALE4 (four blocks
  // per chunk) fill tensor memory with fewer chunks' accumulators and keep
  // one issuer over all of them.
  constexpr int NI = kBlocks == 1 ? kMaxIssuers : 1;  // MMA issuers
  const int ndi = nd / NI;                            // accumulator buffers per issuer (1 when NI > 1)
  const int sbytes = stage_bytes(FMT, MP);
  const int off_b = kCodes;  // B follows the codes (1024-byte aligned)
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kCarveBytes);
  uint64_t* tma_full = bars;                    // [kMaxStages] producer -> unpack, MMA, epilogue
  uint64_t* tma_empty = tma_full + kMaxStages;  // [kMaxStages] unpack, MMA commit, epilogue -> producer
  uint64_t* a_full = tma_empty + kMaxStages;    // [kMaxStages] unpack warps -> the chunk's issuer, per stage
  uint64_t* a_empty = a_full + kMaxStages;      // [kMaxA] MMA commit -> unpack (per A buffer)
  uint64_t* d_full = a_empty + kMaxA;               // [kMaxD] MMA commit -> epilogue
  uint64_t* d_empty = d_full + kMaxD;           // [kMaxD] epilogue warps -> MMA
  uint64_t* drain = d_empty + kMaxD;            // [kMaxIssuers] final commit of each MMA issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + kMaxIssuers);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t stage_tx = (uint32_t)stage_tx_bytes(FMT, MP);

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&tma_full[s], 1);
      mbar_init(&tma_empty[s], kDeqWarps + 1);  // codes (unpack warps), B (MMA commit)
    }
    // a_full per stage, with the stage's phase: an issuer waits on it only
    // after tma_full of the same stage and phase, which already implies that
    // the stage's previous chunk was unpacked, and the stage's next chunk
    // cannot be unpacked before this one's MMAs were issued; so no issuer,
    // however many there are, sees a phase early or late
    for (int s2 = 0; s2 < nstages; ++s2) mbar_init(&a_full[s2], kDeqWarps);
    for (int b = 0; b < na; ++b) mbar_init(&a_empty[b], 1);
    for (int b = 0; b < nd; ++b) {
      mbar_init(&d_full[b], 1);
      mbar_init(&d_empty[b], kEpiWarps);
    }
    for (int i = 0; i < kMaxIssuers; ++i) mbar_init(&drain[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (warp == 1) tmem_relinquish();
  // everything above overlaps the activation prologue; its B matrix and
  // scales are read below.  (This grid lets its dependants launch only when
  // its CTAs exit: an early trigger measured slower, the next call's prologue
  // then taking SMs while this grid still runs.)  The producer waits later,
  // for Q8_0 after it has sent off the first stages' weight codes, which the
  // prologue does not write.
  if (warp != 0) grid_dependency_wait();

  const int items = p.tiles * p.splits;
  const int ib = (int)((int64_t)items * blockIdx.x / gridDim.x);
  const int ie = (int)((int64_t)items * (blockIdx.x + 1) / gridDim.x);
  auto chunk_begin = [&](int split) { return (int)((int64_t)split * p.chunks / p.splits); };
  auto fail_wait = [&]() {
    *abort_flag = 1;
    tc_flag(KQ_ERR_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      prefetch_tmap(&p.map_codes);
      prefetch_tmap(&p.map_b);
      Ring ring;
      int issued = 0;
      bool stop = false;
      // Q8_0: the weight codes of the first stages go out before the wait for
      // the activation prologue (their stages are fresh: nothing to wait for).
      // Measured: Q8_0 M = 16 -3%; PQ2_0 +1% (its prologue is the longer one),
      // so the others wait first.
      int npre = 0;
      for (int item = ib; FMT == KQ_Q8_0 && item < ie && npre < nstages; ++item) {
        const int split = item / p.tiles, tile = item - split * p.tiles;
        const int c1 = chunk_begin(split + 1);
        for (int c = chunk_begin(split); c < c1 && npre < nstages; ++c, ++npre) {
          uint8_t* st = stages + (size_t)npre * sbytes;
          mbar_arrive_expect_tx(&tma_full[npre], stage_tx);
          tma_load_2d(st, &p.map_codes, c * (chunk_row_bytes(FMT) / 4), tile * kRows, &tma_full[npre], policy);
        }
      }
      grid_dependency_wait();
      for (int item = ib; item < ie && !stop; ++item) {
        const int split = item / p.tiles, tile = item - split * p.tiles;
        const int c1 = chunk_begin(split + 1);
        for (int c = chunk_begin(split); c < c1; ++c) {
          uint8_t* st = stages + (size_t)ring.slot * sbytes;
          uint64_t* bar = &tma_full[ring.slot];
          if (issued >= npre) {
            if (*abort_flag || !mbar_wait_bounded(&tma_empty[ring.slot], ring.phase ^ 1u)) {
              fail_wait();
              stop = true;
              break;
            }
            mbar_arrive_expect_tx(bar, stage_tx);
            tma_load_2d(st, &p.map_codes, c * (chunk_row_bytes(FMT) / 4), tile * kRows, bar, policy);
          }
          tma_load_2d(st + off_b, &p.map_b, c * kChunk, 0, bar, policy);
          tma_load_2d(st + off_b + b_box_bytes(MP), &p.map_b, c * kChunk + 64, 0, bar, policy);
          ring.next(nstages);
          ++issued;
        }
      }
      // never leave with copies in flight: wait (bounded) for the last ones,
      // walking back from the current ring position
      Ring back = ring;
      for (int j = 0; j < issued && j < nstages; ++j) {
        if (back.slot == 0) {
          back.slot = nstages - 1;
          back.phase ^= 1u;
        } else {
          --back.slot;
        }
        (void)mbar_wait_bounded(&tma_full[back.slot], back.phase);
      }
    }
  } else if (warp == 1 || warp >= kIssuer2Warp) {
    // ------------------------------ MMA issuers -------------------------------
    // The whole warp walks the list in uniform control flow and waits; one
    // elected lane issues the MMAs and commits (warp-uniform issue measured
    // about twice as fast per MMA as a loop run by lane 0 alone).
    const int me = warp == 1 ? 0 : warp - kIssuer2Warp + 1;
    if (me < NI) {
      const uint32_t idesc = idesc_f16(kRows, 2 * MP);
      Ring ring, dring, ar;  // the stage and A buffer of every chunk; this issuer's accumulator buffers
      int g = 0;
      bool stop = false;
      for (int item = ib; item < ie && !stop; ++item) {
        const int split = item / p.tiles;
        const int c0 = chunk_begin(split), c1 = chunk_begin(split + 1);
        for (int c = c0; c < c1; ++c, ++g, ring.next(nstages), ar.next(na)) {
          if (g % NI != me) continue;
          if (__any_sync(0xffffffffu, *abort_flag != 0)) {
            stop = true;
            break;
          }
          const int slot = ring.slot, ab = ar.slot;
          const bool got = mbar_wait_bounded(&tma_full[slot], ring.phase) && mbar_wait_bounded(&a_full[slot], ring.phase);
          if (!__all_sync(0xffffffffu, got)) {
            if (lane == 0) fail_wait();
            stop = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + (uint32_t)ab * kACols;
          const uint8_t* bt = stages + (size_t)slot * sbytes + off_b;
          // descriptors of the two B boxes; a K step adds its 32-byte offset (>> 4) to the start field
          const uint64_t bd0 = sw128_desc(bt), bd1 = sw128_desc(bt + b_box_bytes(MP));
          bool ok = true;
          if (kBlocks > 1 && gb == kBlocks) {
            // one accumulator group per chunk: the blocks' chains alternate
            const int dslot = me * ndi + dring.slot;
            const bool free = mbar_wait_bounded(&d_empty[dslot], dring.phase ^ 1u);
            if (!__all_sync(0xffffffffu, free)) {
              if (lane == 0) fail_wait();
              stop = true;
              break;
            }
            tc_fence_after();
            const uint32_t d0 = tmem_base + tmem_d + (uint32_t)(dslot * gb * 2 * MP);
            if (elect_one()) {
#pragma unroll
              for (int t = 0; t < kSteps; ++t)
#pragma unroll
                for (int b = 0; b < kBlocks; ++b) {
                  const int kk = b * kSteps + t;
                  const int atom = kk >> 2, sub = (kk & 3) * 32;
                  tc_mma_ts(d0 + (uint32_t)(b * 2 * MP), a_tmem + (uint32_t)(kk * 8),
                            (atom ? bd1 : bd0) + (uint64_t)(sub >> 4), idesc, t > 0 ? 1u : 0u);
                }
              tc_commit(&d_full[dslot]);
            }
            __syncwarp();
            dring.next(ndi);
          } else
          for (int b = 0; b < kBlocks; ++b) {
            const int bg = b % gb;
            const int dslot = me * ndi + dring.slot;
            if (bg == 0) {
              const bool free = mbar_wait_bounded(&d_empty[dslot], dring.phase ^ 1u);
              if (!__all_sync(0xffffffffu, free)) {
                if (lane == 0) fail_wait();
                ok = false;
                break;
              }
              tc_fence_after();
            }
            const uint32_t d_tmem = tmem_base + tmem_d + (uint32_t)((dslot * gb + bg) * 2 * MP);
            if (elect_one()) {
#pragma unroll
              for (int t = 0; t < kSteps; ++t) {
                const int kk = b * kSteps + t;
                const int atom = kk >> 2, sub = (kk & 3) * 32;
                tc_mma_ts(d_tmem, a_tmem + (uint32_t)(kk * 8), (atom ? bd1 : bd0) + (uint64_t)(sub >> 4), idesc,
                          t > 0 ? 1u : 0u);
              }
              if (bg == gb - 1) tc_commit(&d_full[dslot]);
            }
            __syncwarp();
            if (bg == gb - 1) dring.next(ndi);
          }
          if (!ok) {
            stop = true;
            break;
          }
          if (elect_one()) {
            tc_commit(&a_empty[ab]);
            tc_commit(&tma_empty[slot]);
          }
          __syncwarp();
        }
      }
      // wait until every MMA this warp issued has completed
      if (elect_one()) tc_commit(&drain[me]);
      __syncwarp();
      if (lane == 0) (void)mbar_wait_bounded(&drain[me], 0);
      __syncwarp();
    }
  } else if (warp < 2 + kDeqWarps) {
    // ------------------------------ unpack ----------------------------------
    const int quarter = warp & 3;       // tensor-memory lane quarter
    const int khalf = (warp - 2) >> 2;  // half of the chunk's K
    const int r = quarter * 32 + lane;  // weight row in the tile
    const uint32_t a_lane = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(khalf * 32);
    Ring ring, ar;  // stages; A buffers
    for (int item = ib; item < ie; ++item) {
      const int split = item / p.tiles;
      const int c0 = chunk_begin(split), c1 = chunk_begin(split + 1);
      for (int c = c0; c < c1; ++c) {
        if (!*abort_flag) {
          if (!mbar_wait_bounded(&tma_full[ring.slot], ring.phase) ||
              !mbar_wait_bounded(&a_empty[ar.slot], ar.phase ^ 1u)) {
            fail_wait();
          } else {
            tc_fence_after();
            const uint8_t* st = stages + (size_t)ring.slot * sbytes;
            const uint32_t a_tmem = a_lane + (uint32_t)ar.slot * kACols;
            if (FMT == KQ_Q8_0) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                // 16 codes: 16-byte piece 4*khalf+j of the row, at piece
                // position (4*khalf+j) ^ (r % 8) of the 128-byte swizzle
                const uint4 cw = *reinterpret_cast<const uint4*>(st + r * 128 + (((khalf * 4 + j) ^ (r & 7)) << 4));
                const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
                uint32_t o[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  // two codes, biased by 128, into the low mantissa byte of
                  // 1024: the fp16 value is 1024 + 128 + code exactly
                  const uint32_t u = w4[q >> 1] ^ 0x80808080u;
                  const uint32_t bits = __byte_perm(u, 0x64646464u, (q & 1) ? 0x7372u : 0x7170u);
                  o[q] = h2_bits(__hsub2(bits_h2(bits), __float2half2_rn(1152.f)));  // q, exact
                }
                tmem_st8(a_tmem + (uint32_t)(j * 8), o);
              }
            } else if (FMT == KQ_SCALE4) {
              // 64 codes of the row: 32 bytes (16-byte pieces 2 khalf, 2 khalf + 1)
              // of the 64-byte row, 64-byte swizzle (piece c of row r at c ^ ((r / 2) % 4))
#pragma unroll
              for (int pc = 0; pc < 2; ++pc) {
                const int piece = (2 * khalf + pc) ^ ((r >> 1) & 3);
                const uint4 cw = *reinterpret_cast<const uint4*>(st + r * 64 + piece * 16);
                const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int wh = 0; wh < 2; ++wh) {  // two words per 8 registers
                  uint32_t o[8];
#pragma unroll
                  for (int q = 0; q < 8; ++q) {
                    // pair (q % 4, q % 4 + 4) of word 2 wh + q / 4: masked in place it is
                    // c * 2^(s-24); one fp16 subtraction of 8 * 2^(s-24) makes it (c - 8) * 2^(s-24), exact
                    const uint32_t w = w4[2 * wh + (q >> 2)];
                    const int pr = q & 3;
                    const uint32_t src = pr < 2 ? w : w >> 8;
                    const uint32_t cbits = src & (0x000F000Fu << scale4_shift(pr));
                    o[q] = h2_bits(__hsub2(bits_h2(cbits), bits_h2(0x00080008u << scale4_shift(pr))));
                  }
                  tmem_st8(a_tmem + (uint32_t)(pc * 16 + wh * 8), o);
                }
              }
            } else {
              // 64 codes of the row: 16 bytes at column 16*khalf of the
              // 32-byte row, 32-byte swizzle (halves swapped on every other
              // 128 bytes)
              int off = r * 32 + khalf * 16;
              off ^= ((off >> 7) & 1) << 4;
              const uint4 cw = *reinterpret_cast<const uint4*>(st + off);
              const uint32_t w4[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
              for (int wi = 0; wi < 4; ++wi) {
                const uint32_t w = w4[wi], w8 = w >> 8;
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                  // c * 2^(s-24) - 2^(s-24) = (c - 1) * 2^(s-24), exact in fp16 subnormals
                  const uint32_t cbits = (e <= 4 ? w : w8) & (0x00030003u << pq2_0_shift(e));
                  o[e] = h2_bits(__hsub2(bits_h2(cbits), bits_h2(0x00010001u << pq2_0_shift(e))));
                }
                tmem_st8(a_tmem + (uint32_t)(wi * 8), o);
              }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
              mbar_arrive(&a_full[ring.slot]);
              mbar_arrive(&tma_empty[ring.slot]);
            }
          }
        }
        ring.next(nstages);
        ar.next(na);
      }
    }
  } else if (warp < kIssuer2Warp) {
    // ------------------------------ epilogue ------------------------------------
    const int quarter = warp & 3;                   // tensor-memory lane quarter
    const int ahalf = (warp - 2 - kDeqWarps) >> 2;  // half of the activation columns
    const int half = MP / 2;                        // 8 .. 32 activation columns per warp
    EpiCtx e;
    e.d_full = d_full;
    e.d_empty = d_empty;
    e.abort_flag = abort_flag;
    e.gb = gb;
    e.nd = nd;
    e.ib = ib;
    e.ie = ie;
    e.mp = MP;
    e.r = quarter * 32 + lane;
    e.i0 = ahalf * half;
    e.d_lane = tmem_base + ((uint32_t)(quarter * 32) << 16) + tmem_d + (uint32_t)e.i0;
    switch (half) {
      case 8:
        epilogue_role<FMT, 8>(p, e, lane);
        break;
      case 16:
        epilogue_role<FMT, 16>(p, e, lane);
        break;
      case 24:
        epilogue_role<FMT, 24>(p, e, lane);
        break;
      default:
        epilogue_role<FMT, 32>(p, e, lane);
        break;
    }
  }

  // every role ends here; then the tensor memory goes back
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// Y[i][row] = sum over splits, in split order, of the partials
__global__ void tc_reduce_kernel(const float* __restrict__ part, float* __restrict__ y, int64_t total, int splits) {
  grid_dependency_wait();  // the GEMM's partials (a programmatic dependent launch)
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total; t += (int64_t)gridDim.x * blockDim.x) {
    float acc = part[t];
    for (int s = 1; s < splits; ++s) acc += part[(int64_t)s * total + t];
    y[t] = acc;
  }
}

}  // namespace tc

// ---- host side ----------------------------------------------------------------

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
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

struct TcGeometry {
  int64_t mp = 0, nb = 0;  // M' = m rounded up to 16; B rows 2 M'
  int tiles = 0, chunks = 0, splits = 1, stages = 0;
  size_t b_bytes = 0;  // B matrix, rounded to 256
  size_t s_bytes = 0;  // per-row powers of two, rounded to 256
  size_t p_bytes = 0;  // split partials
};

// Split count: the one with the smallest modelled time, counting the chunks
// of the busiest CTA (0.4 us each), a fixed cost per item (1 us: pipeline
// fill and epilogue) and the second pass (2.5 us) when there are splits.
TcGeometry tc_geometry(const kq_qmat* W, int64_t m, int sms, int requested) {
  TcGeometry g;
  g.mp = (m + 15) / 16 * 16;
  g.nb = 2 * g.mp;
  const int fmt = W->fmt;
  g.stages = (int)std::min<int64_t>(tc::kMaxStages, (int64_t)tc::kCarveBytes / tc::stage_bytes(fmt, (int)g.mp));
  g.tiles = (int)((W->n + tc::kRows - 1) / tc::kRows);
  g.chunks = (int)((W->k + tc::kChunk - 1) / tc::kChunk);
  if (requested > 0) {
    g.splits = std::min(requested, g.chunks);
  } else {
    const int cap = std::min(g.chunks, 16);
    double best = 1e30;
    for (int s = 1; s <= cap; ++s) {
      const int64_t items = (int64_t)g.tiles * s;
      const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(items, sms > 0 ? sms : 148));
      const int64_t per_cta = (items + grid - 1) / grid;
      const int64_t chunks_per_item = (g.chunks + s - 1) / s;
      const double t = per_cta * (chunks_per_item * 0.4 + 1.0) + (s > 1 ? 2.5 : 0.0);
      if (t < best - 1e-9) {
        best = t;
        g.splits = s;
      }
    }
  }
  g.b_bytes = (size_t)round_up(g.nb * W->k * 2, 256);
  g.s_bytes = (size_t)round_up(g.mp * 4, 256);
  g.p_bytes = g.splits > 1 ? (size_t)g.splits * (size_t)m * (size_t)W->n * sizeof(float) : 0;
  return g;
}

int tc_device_sms(int* sms) {
  int dev = 0;
  KQ_CUDA_TRY(cudaGetDevice(&dev));
  KQ_CUDA_TRY(cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev));
  return KQ_OK;
}

template <int FMT>
int launch_tc(const tc::TcParams& p, int grid, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(tc::tc_gemm_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)tc::kSmemBytes);
  });
  KQ_CUDA_TRY(attr);
  // a programmatic dependent of the activation prologue: barrier set-up and
  // tensor-memory allocation overlap its tail
  KQ_CUDA_TRY(launch_dependent(tc::tc_gemm_kernel<FMT>, dim3(grid), dim3(tc::kThreads), tc::kSmemBytes, st, p));
  return KQ_OK;
}

template <int FMT>
int launch_act(const kq_qmat* W, const float* X, int m, int64_t k, int64_t mp, __half* B, float* bscale,
               cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(tc::act_hilo_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)(kTcMaxK * sizeof(float)));
  });
  KQ_CUDA_TRY(attr);
  const int bytes = (int)(k * sizeof(float));
  // a programmatic dependent of the stream's previous kernel
  KQ_CUDA_TRY(launch_dependent(tc::act_hilo_kernel<FMT>, dim3((unsigned)mp), dim3(512), (size_t)bytes, st, X, m,
                               (int)mp, k, B, bscale, (int)W->had_block, (const int8_t*)W->signs));
  return KQ_OK;
}

int encode(PFN_cuTensorMapEncodeTiled_v12000 fn, CUtensorMap* map, CUtensorMapDataType type, const void* base,
           uint64_t inner, uint64_t outer, uint64_t stride_bytes, uint32_t box_inner, uint32_t box_outer,
           CUtensorMapSwizzle swz, const char* what) {
  cuuint64_t gdim[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t gstride[1] = {(cuuint64_t)stride_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, type, 2, const_cast<void*>(base), gdim, gstride, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(KQ_ERR_CUDA, "tensor map of %s: CUresult %d", what, (int)r);
  return KQ_OK;
}

}  // namespace

int tc_check(const kq_qmat* W, int64_t m) {
  if (W->fmt != KQ_Q8_0 && W->fmt != KQ_PQ2_0 && W->fmt != KQ_SCALE4)
    return fail(KQ_ERR_UNSUPPORTED, "format %d has no tensor-core path", W->fmt);
  if (m < 1 || m > kTcMaxM) return fail(KQ_ERR_SHAPE, "m = %lld outside [1, %d]", (long long)m, kTcMaxM);
  if (W->k > kTcMaxK)
    return fail(KQ_ERR_SHAPE, "k = %lld above the tensor-core path's %d", (long long)W->k, kTcMaxK);
  return KQ_OK;
}

size_t tc_workspace_bytes(const kq_qmat* W, int64_t m, int splits) {
  int sms = 0;
  if (splits == 0 && tc_device_sms(&sms) != KQ_OK) {
    clear_error();
    sms = 0;
  }
  TcGeometry g = tc_geometry(W, m, sms, splits);
  return g.b_bytes + g.s_bytes + g.p_bytes;
}

int tc_gemm(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int splits, void* d_ws, size_t ws_bytes,
            void* stream) {
  if (int s = tc_check(W, m)) return s;
  if (!d_X || !d_Y) return fail(KQ_ERR_INVALID_ARG, "NULL activation or output");
  if (!aligned16(d_X) || !aligned16(d_Y)) return fail(KQ_ERR_ALIGNMENT, "x or y not 16-byte aligned");
  auto fn = tc_encode_fn();
  if (!fn) return fail(KQ_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled is not available from the driver");
  int sms = 0;
  if (int s = tc_device_sms(&sms)) return s;
  const TcGeometry g = tc_geometry(W, m, splits == 0 ? sms : 0, splits);
  const size_t need = g.b_bytes + g.s_bytes + g.p_bytes;
  if (!d_ws || ws_bytes < need)
    return fail(KQ_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, d_ws ? ws_bytes : (size_t)0);
  if (!aligned16(d_ws)) return fail(KQ_ERR_ALIGNMENT, "workspace not 16-byte aligned");
  if (g.stages < 2) return fail(KQ_ERR_UNSUPPORTED, "internal: %d ring stages", g.stages);
  uint8_t* ws = reinterpret_cast<uint8_t*>(d_ws);
  __half* B = reinterpret_cast<__half*>(ws);
  float* bscale = reinterpret_cast<float*>(ws + g.b_bytes);
  float* part = g.splits > 1 ? reinterpret_cast<float*>(ws + g.b_bytes + g.s_bytes) : nullptr;

  tc::TcParams p{};
  const int64_t rowbytes = code_row_bytes(W->fmt, W->k);
  const int64_t ss = scale_stride(W->fmt, W->k);
  // one chunk of a row per box row: 128 bytes (Q8_0), 64 (SCALE4), 32 (PQ2_0), each with the matching swizzle
  const uint32_t box_u32 = (uint32_t)tc::chunk_row_bytes(W->fmt) / 4;
  const CUtensorMapSwizzle cswz = W->fmt == KQ_Q8_0    ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : W->fmt == KQ_SCALE4 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                        : CU_TENSOR_MAP_SWIZZLE_32B;
  if (int s = encode(fn, &p.map_codes, CU_TENSOR_MAP_DATA_TYPE_UINT32, W->codes, rowbytes / 4, W->n, rowbytes,
                     box_u32, tc::kRows, cswz, "the codes plane"))
    return s;
  p.scales = reinterpret_cast<const uint16_t*>(W->scales);
  p.sstride = ss;
  p.kblocks = (int32_t)(W->k / (W->fmt == KQ_PQ2_0 ? 128 : 32));
  if (int s = encode(fn, &p.map_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, B, W->k, g.nb, W->k * 2, 64u, (uint32_t)g.nb,
                     CU_TENSOR_MAP_SWIZZLE_128B, "the activation matrix"))
    return s;
  p.bscale = bscale;
  p.y = g.splits > 1 ? part : d_Y;
  p.n = W->n;
  p.m = (int32_t)m;
  p.mp = (int32_t)g.mp;
  p.tiles = g.tiles;
  p.chunks = g.chunks;
  p.splits = g.splits;
  p.stages = g.stages;

  cudaStream_t st = (cudaStream_t)stream;
  const int grid = (int)std::min<int64_t>((int64_t)g.tiles * g.splits, sms);
  if (W->fmt == KQ_Q8_0) {
    if (int s = launch_act<KQ_Q8_0>(W, d_X, (int)m, W->k, g.mp, B, bscale, st)) return s;
    if (int s = launch_tc<KQ_Q8_0>(p, grid, st)) return s;
  } else if (W->fmt == KQ_SCALE4) {
    if (int s = launch_act<KQ_SCALE4>(W, d_X, (int)m, W->k, g.mp, B, bscale, st)) return s;
    if (int s = launch_tc<KQ_SCALE4>(p, grid, st)) return s;
  } else {
    if (int s = launch_act<KQ_PQ2_0>(W, d_X, (int)m, W->k, g.mp, B, bscale, st)) return s;
    if (int s = launch_tc<KQ_PQ2_0>(p, grid, st)) return s;
  }
  if (g.splits > 1) {
    const int64_t total = m * W->n;
    const int rgrid = (int)std::min<int64_t>((total + 255) / 256, (int64_t)sms * 8);
    KQ_CUDA_TRY(launch_dependent(tc::tc_reduce_kernel, dim3(rgrid), dim3(256), 0, st, (const float*)part, d_Y,
                                 total, g.splits));
  }
  return KQ_OK;
}

int read_tc_status(int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, tc::g_tc_status, sizeof(v));
  if (e != cudaSuccess) return -1;
  if (clear) {
    unsigned int z = 0;
    if (cudaMemcpyToSymbol(tc::g_tc_status, &z, sizeof(z)) != cudaSuccess) return -1;
  }
  return (int)v;
}

}  // namespace kq
