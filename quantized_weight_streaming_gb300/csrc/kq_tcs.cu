// PQ2_0 weight streaming at one activation row on the 5th-generation tensor
// cores (tcgen05): an opt-in consumer (kq_set_pq2_0_consumer) of the batch-1
// GEMV and of decode plans without links, for ternary Hadamard-rotated
// weights ("Bonsai 2 27B - ternary g128 + blockwise Hadamard", sections 3.1
// and 4.2).  Decode is bound by streaming every weight byte once ("Kipp
// Benchmarks", "Decode is weight-bandwidth-bound"); this consumer spends
// fewer integer operations per 2-bit code than the mma.sync one (5 per 16
// codes instead of 9) and moves the multiply to tcgen05.mma.
//
//  * Work list, tiles and copies are those of the streaming kernel in
//    kq_stream.cu: one persistent CTA per SM walks a contiguous run of items
//    (matrix, 256-row block, K split); a 2-stage ring receives 256 rows x 1024
//    codes per stage by two 128-byte-swizzled TMA boxes plus the tile's fp16
//    block scales.
//  * A operand (the weights), e4m3 in tensor memory.  A 2-bit code c masked
//    in place at bit 0 or bit 2 of a byte is the exact e4m3 value c * 2^-9
//    or c * 2^-7 (subnormal, or the smallest normal for c = 2 at bit 2).  Per
//    32-bit code word (16 codes) four masks and one shift give four
//    registers of four codes each: w & 0x03030303, w & 0x0C0C0C0C and the same
//    two masks of w >> 4.  Register (word m, mask c) becomes tensor-memory
//    column 4m + c of the row's lane, so byte i of that column, K position
//    16m + 4c + i of the block, holds weight 16m + 4i + c.
//  * B operand (the activation), e4m3 in shared memory.  After the blockwise
//    transform x' = R x, each 128-block is normalised by 2^-E (E the exponent
//    of its largest |x'|), multiplied by 2^(7-s) (s the code's bit offset, so
//    that A x B = c x' 2^(-E-2)) and written as four e4m3 planes v = q1 +
//    q2/16 + q3/256 + q4/4096, each plane the round-to-nearest e4m3 of the
//    previous residual times 16: relative error 2^-16, far inside the
//    1e-4 * sum|w x'| bound.  A 16-position group takes 64 bytes: one 16-byte
//    row per plane.  The MMA reads it with N = 16 through a K-major
//    descriptor without swizzle whose K core-matrix stride is 64 bytes and
//    whose 8-row-group stride is 0: rows 0-3 of a core matrix are the four
//    planes; rows 4-7 overlap the next group and rows 8-15 repeat rows 0-7,
//    all landing in accumulator columns that are never read.  So the table
//    takes 4 bytes per position, as many as the fp32 activation.
//  * Per block and half tile (128 rows) 4 MMAs (M = 128, N = 16, K = 32)
//    accumulate into that block's own accumulator, and the epilogue adds
//        y += d * (2^(E+2) * (D1 + D2/16 + D3/256 + D4/4096) - sum_j x'_j),
//    the ternary -1 folded into the block's activation sum (the Bonsai
//    page's fold, section 8.5, written from the algebra).  No weight is
//    rounded; the accumulation of each plane is fp32 on the tensor pipe.
//  * Roles: warp 0 copies (TMA); warps 1-2 issue the MMAs of the two teams;
//    warps 3-10 are two teams of four workers (team = row half, worker = the
//    tensor-memory lane quarter warp % 4).  A team's slot is 128 rows x 2
//    blocks; its workers unpack it into one of the team's two A buffers,
//    arrive on a hardware named barrier that the team's issuer waits on,
//    then run the epilogue of the team's previous slot (waiting on the
//    mbarrier its MMAs were committed to) while the issuer's elected lane
//    issues the new slot's MMAs.  Each barrier is waited on by one sequence
//    of waits taking its phases one at a time: a parity wait must never run
//    against a barrier two phases behind its target (an earlier design that
//    rotated three issuers over two accumulator buffers did, and passed a
//    wait falsely).  The issuer warps walk the list in uniform control flow
//    and one elected lane issues (warp-uniform operands measured about twice
//    as fast per MMA as a loop run by lane 0 alone).
//  * The eight workers stage the activation table whenever the CTA's
//    (matrix, split) changes, after each team ran the epilogue of its last
//    slot.  Every mbarrier wait is bounded; a timeout sets KQ_ERR_TIMEOUT and
//    every role stops waiting but keeps meeting every named barrier, the
//    producer waits for its copies in flight, the issuers drain their MMAs,
//    and the tensor memory is freed before the kernel returns.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "kq_device.cuh"
#include "kq_internal.h"
#include "kq_stream.cuh"
#include "kq_tcgen05.cuh"

namespace kq {
namespace tcs {

using G = Geo<KQ_PQ2_0>;
using F = Fmt<KQ_PQ2_0>;
using namespace kq::tc;

constexpr int kRows = G::kTileRows;                 // 256 weight rows per tile (two MMA halves)
constexpr int kStages = G::kStages;                 // TMA ring depth
constexpr int kStageBytes = G::kStageBytes;         // codes and scales of one tile
constexpr int kTileCodeBytes = G::kTileCodeBytes;   // 256 rows x 256 bytes
constexpr int kBoxBytes = kRows * 128;              // one 128-byte-wide swizzled box of the tile
constexpr int kBlocks = F::kChunk / F::kBlock;      // 128-weight blocks per tile row
// Two teams, one per row half h (128 rows, the MMA's M).  A team is four
// worker warps (one per tensor-memory lane quarter) that unpack a slot of two
// blocks (128 rows x 256 weights) into tensor memory and later run its
// epilogue, and one issuer warp.  Each team has two A buffers and two
// accumulator buffers, used by its slots in turn.
constexpr int kSlotBlocks = 2;
constexpr int kTeams = 2;
constexpr uint32_t kACols = 32 * kSlotBlocks;          // 32 columns (128 e4m3 codes per lane) per block
constexpr uint32_t kDCols = 16 * kSlotBlocks;          // N = 16 columns per block
constexpr uint32_t kTeamCols = 2 * kACols + 2 * kDCols;
constexpr uint32_t kTmemCols = 512;
static_assert(kTeams * kTeamCols <= kTmemCols, "tensor memory");
constexpr int kWorkers = 4;                            // worker warps per team
constexpr int kWarpIssuer0 = 1;                        // warps 1, 2: the teams' issuers
constexpr int kWarpWorker0 = kWarpIssuer0 + kTeams;    // warps 3..10: team (w - 3) / 4
constexpr int kWarps = kWarpWorker0 + kTeams * kWorkers;
constexpr int kThreads = 32 * kWarps;
constexpr int kStageWarps = kTeams * kWorkers;         // the warps that stage the activation table
// named barriers: 0 __syncthreads, 1 staging, 2 + 2 h + b: A buffer b of team h written
constexpr int kBarStage = 1, kBarA0 = 2;
constexpr int kPosMax = kXMax;                         // activation positions per staged slice
constexpr int kBlkMax = kPosMax / F::kBlock;
constexpr int kBlkTabBytes = F::kBlock * 4;            // 4 planes x 128 positions
// the last MMA of the last block reads the first 64 bytes past its block
// (aliased rows of the B descriptor, never summed into a read column)
constexpr int kTabBytes = kPosMax * 4 + 64;
constexpr size_t kOffTab = (size_t)kStages * kStageBytes;
constexpr size_t kOffFS = kOffTab + kTabBytes;
constexpr size_t kOffComb = kOffFS + (size_t)kBlkMax * 8;
constexpr size_t kOffScratch = kOffComb;               // (no combine buffer: a team owns its rows)
constexpr size_t kOffBars = kOffScratch + (size_t)kStageWarps * 128 * 4;
constexpr int kNumBars = 2 * kStages + 2 * kTeams + kTeams;  // full, empty, mma_done[team][buffer], drain
constexpr size_t kSmemBytes = kOffBars + (size_t)kNumBars * 8 + 16;
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(kOffTab % 16 == 0 && kOffBars % 8 == 0, "alignment");

__device__ unsigned int g_tcs_status = 0;
__device__ __forceinline__ void tcs_flag(int status) { atomicOr(&g_tcs_status, 1u << status); }
// A bounded wait expired: every role of the CTA stops waiting.
__device__ __forceinline__ void fail_wait(volatile int* abort_flag) {
  *abort_flag = 1;
  tcs_flag(KQ_ERR_TIMEOUT);
}

// e4m3 pair: hi -> bits 15:8, lo -> bits 7:0 (round to nearest even)
__device__ __forceinline__ uint32_t e4m3x2(float hi, float lo) {
  uint16_t q;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(q) : "f"(hi), "f"(lo));
  return q;
}
// the two e4m3 values of a pair back as fp32 (exact)
__device__ __forceinline__ float2 e4m3x2_to_f32(uint32_t q) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)q));
  return __half22float2(*reinterpret_cast<const __half2*>(&h));
}

// The K range [kbeg, kend) of the cursor's current item; its chunks are
// 1024 weights, the last one possibly holding fewer 128-weight blocks.
__device__ __forceinline__ void item_range(const ItemCursor& cur, int64_t& kbeg, int64_t& kend) {
  kbeg = (int64_t)cur.split * cur.job.split_k;
  kend = min64(cur.job.k, kbeg + cur.job.split_k);
}
__device__ __forceinline__ int chunk_blocks(int64_t k0, int64_t kend) {
  return (int)min64((int64_t)kBlocks, (kend - k0) / F::kBlock);
}

// Stages the activation table of x[kbeg, kbeg + len): blockwise transform
// (sign flip, 128-point FWHT, the 8-point pass of the n = 1024 rotation),
// per block the exponent E and sum of x', then the four e4m3 planes.  Run by
// the sixteen staging warps between two barriers; for the n = 1024 rotation
// the table region holds the fp32 transform in between (4 bytes per position
// either way, each warp rewriting only its own blocks).
__device__ void stage_table(const XSrc& xs, int64_t kbeg, int len, uint8_t* tab, float2* fs, float* scratch, int cw,
                            int lane) {
  const int nblk = len / F::kBlock;
  const bool h1024 = xs.had == 1024;
  float* raw = reinterpret_cast<float*>(tab);
  constexpr float kInvSqrt128 = 0.08838834764831845f;
  if (h1024) {
    for (int b = cw; b < nblk; b += kStageWarps) {
      const float4 f = load_x4(xs, 0, kbeg + b * 128 + 4 * lane);
      float v[4] = {f.x, f.y, f.z, f.w};
      if (xs.signs) {
        const char4 s4 = *reinterpret_cast<const char4*>(xs.signs + kbeg + b * 128 + 4 * lane);
        v[0] *= (float)s4.x;
        v[1] *= (float)s4.y;
        v[2] *= (float)s4.z;
        v[3] *= (float)s4.w;
      }
      fwht128_lane4(v, lane);
      *reinterpret_cast<float4*>(raw + b * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
    named_barrier(1, kStageWarps * 32);
    // H_1024 = H_8 (x) H_128: an 8-point pass across the eight 128-blocks of
    // each 1024-block at every position, then 1/32
    const int cols = (nblk / 8) * 128;
    for (int c = cw * 32 + lane; c < cols; c += kStageWarps * 32) {
      float* col = raw + (c / 128) * 1024 + (c % 128);
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
    named_barrier(1, kStageWarps * 32);
  }
  for (int b = cw; b < nblk; b += kStageWarps) {
    float v[4];
    if (h1024) {
      const float4 f = *reinterpret_cast<const float4*>(raw + b * 128 + 4 * lane);
      v[0] = f.x;
      v[1] = f.y;
      v[2] = f.z;
      v[3] = f.w;
    } else {
      const float4 f = load_x4(xs, 0, kbeg + b * 128 + 4 * lane);
      v[0] = f.x;
      v[1] = f.y;
      v[2] = f.z;
      v[3] = f.w;
      fwht128_lane4(v, lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] *= kInvSqrt128;
    }
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int mk = 16; mk; mk >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, mk));
    // block exponent E with amax < 2^(E+1), clamped to [-100, 100]
    int e = amax > 0.f ? ((__float_as_int(amax) >> 23) & 0xFF) - 127 : 0;
    if (amax > 0.f && e == -127) e = -126;  // denormal block maximum
    e = max(-100, min(100, e));
    float s = (v[0] + v[1]) + (v[2] + v[3]);
#pragma unroll
    for (int mk = 16; mk; mk >>= 1) s += __shfl_xor_sync(0xffffffffu, s, mk);
    const float unscale = pow2f(-e);
    __syncwarp();
    *reinterpret_cast<float4*>(scratch + 4 * lane) =
        make_float4(v[0] * unscale, v[1] * unscale, v[2] * unscale, v[3] * unscale);
    __syncwarp();
    // lane (m, c): word c of every plane row of group m, i.e. K positions
    // 16m + 4c + i <- weights 16m + 4i + c (i = 0..3), bit offset s = 2 (c % 2)
    const int m = lane >> 2, c = lane & 3;
    const float sc = (c & 1) ? 32.f : 128.f;  // 2^(7 - s)
    float w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = scratch[16 * m + 4 * i + c] * sc;  // |w| < 256
    uint32_t plane[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t q01 = e4m3x2(w[1], w[0]), q23 = e4m3x2(w[3], w[2]);
      plane[r] = q01 | (q23 << 16);
      if (r < 3) {  // the residual, exact in fp32, scaled into the next plane's range
        const float2 f01 = e4m3x2_to_f32(q01), f23 = e4m3x2_to_f32(q23);
        w[0] = (w[0] - f01.x) * 16.f;
        w[1] = (w[1] - f01.y) * 16.f;
        w[2] = (w[2] - f23.x) * 16.f;
        w[3] = (w[3] - f23.y) * 16.f;
      }
    }
    __syncwarp();  // the n = 1024 path read this block's fp32 values from the same bytes
    uint32_t* dst = reinterpret_cast<uint32_t*>(tab + b * kBlkTabBytes + m * 64 + 4 * c);
#pragma unroll
    for (int r = 0; r < 4; ++r) dst[r * 4] = plane[r];
    if (lane == 0) fs[b] = make_float2(pow2f(e + 2), s);
  }
}

// A worker's epilogue of its team's slot g - 1 (buffer (g - 1) % 2): wait for
// the slot's MMAs, read the four plane sums of each of its nv blocks and add
// y += d (2^(E+2) (D1 + D2/16 + D3/256 + D4/4096) - sum x') for row r.
__device__ __forceinline__ void epilogue(uint64_t* mma_done, int h, uint32_t g, volatile int* abort_flag,
                                         uint32_t lane_base, const float2* fs, int nv, int blk, float d0, float d1,
                                         float& acc) {
  const uint32_t pg = g - 1, b = pg & 1u;
  if (*abort_flag) return;
  if (!mbar_wait_suspend(&mma_done[2 * h + b], (pg >> 1) & 1u)) {
    fail_wait(abort_flag);
    return;
  }
  tc_fence_after();
  float v0[4], v1[4] = {0.f, 0.f, 0.f, 0.f};
  tmem_ld4(lane_base + 2 * kACols + b * kDCols, v0);
  if (nv > 1) tmem_ld4(lane_base + 2 * kACols + b * kDCols + 16, v1);
  tmem_ld_wait();
  {
    const float2 f = fs[blk];
    float t = v0[3] * 0.000244140625f;  // planes 4, 3, 2 scaled down, then plane 1
    t = fmaf(v0[2], 0.00390625f, t);
    t = fmaf(v0[1], 0.0625f, t);
    t += v0[0];
    acc = fmaf(d0, fmaf(t, f.x, -f.y), acc);
  }
  if (nv > 1) {
    const float2 f = fs[blk + 1];
    float t = v1[3] * 0.000244140625f;
    t = fmaf(v1[2], 0.00390625f, t);
    t = fmaf(v1[1], 0.0625f, t);
    t += v1[0];
    acc = fmaf(d1, fmaf(t, f.x, -f.y), acc);
  }
  tc_fence_before();
}

// A worker's code words and block scales of row r for slot (K quarter kq, nv
// blocks) of the tile in stage `st`: block blk's 32 bytes are 16-byte chunks
// 2 (blk % 4) and 2 (blk % 4) + 1 of box blk / 4, chunk c of box row r at
// c ^ (r % 8); a missing second block (nv = 1) reads the first one again.
__device__ __forceinline__ void load_slot(const uint8_t* st, int r, int kq, int nv, uint4 (&u)[kSlotBlocks][2],
                                          uint16_t (&dh)[kSlotBlocks]) {
  const uint16_t* scales = reinterpret_cast<const uint16_t*>(st + kTileCodeBytes);
#pragma unroll
  for (int bi = 0; bi < kSlotBlocks; ++bi) {
    const int blk = kq * kSlotBlocks + (bi < nv ? bi : 0);
    const uint8_t* rowp = st + (blk >> 2) * kBoxBytes + r * 128;
    const int c0 = 2 * (blk & 3);
    u[bi][0] = *reinterpret_cast<const uint4*>(rowp + ((c0 ^ (r & 7)) << 4));
    u[bi][1] = *reinterpret_cast<const uint4*>(rowp + (((c0 + 1) ^ (r & 7)) << 4));
    dh[bi] = scales[r * 8 + blk];
  }
}

// The e4m3 A operand of a slot's nv blocks from their code words: per word
// w & 0x03030303, w & 0x0C0C0C0C and the same masks of w >> 4 (codes 4i + c
// at bit offset 0 or 2 of byte i), into tensor-memory columns a_cols ..
__device__ __forceinline__ void unpack_slot(const uint4 (&u)[kSlotBlocks][2], int nv, uint32_t a_cols) {
#pragma unroll
  for (int bi = 0; bi < kSlotBlocks; ++bi) {
    if (bi < nv) {
      const uint32_t wd[8] = {u[bi][0].x, u[bi][0].y, u[bi][0].z, u[bi][0].w,
                              u[bi][1].x, u[bi][1].y, u[bi][1].z, u[bi][1].w};
#pragma unroll
      for (int m4 = 0; m4 < 2; ++m4) {
        uint32_t o[16];
#pragma unroll
        for (int mm = 0; mm < 4; ++mm) {
          const uint32_t w = wd[4 * m4 + mm], w4 = w >> 4;
          o[4 * mm + 0] = w & 0x03030303u;   // codes 4i + 0, bit offset 0
          o[4 * mm + 1] = w & 0x0C0C0C0Cu;   // codes 4i + 1, bit offset 2
          o[4 * mm + 2] = w4 & 0x03030303u;  // codes 4i + 2, bit offset 0
          o[4 * mm + 3] = w4 & 0x0C0C0C0Cu;  // codes 4i + 3, bit offset 2
        }
        tmem_st16(a_cols + 32 * bi + 16 * m4, o);
      }
    }
  }
}

__device__ __forceinline__ void bar_arrive(uint32_t id, uint32_t count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__global__ void __maxnreg__(168) tcs_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint8_t* tab = smem + kOffTab;
  float2* fs = reinterpret_cast<float2*>(smem + kOffFS);
  float* scratch_all = reinterpret_cast<float*>(smem + kOffScratch);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBars);
  uint64_t* full = bars;                    // [kStages] TMA -> workers
  uint64_t* empty = full + kStages;         // [kStages] workers -> TMA
  uint64_t* mma_done = empty + kStages;     // [kTeams][2] MMA commit -> the team's workers
  uint64_t* drain = mma_done + 2 * kTeams;  // [kTeams] last commit of each issuer
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + kTeams);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kStageWarps);
    }
    for (int i = 0; i < 2 * kTeams; ++i) mbar_init(&mma_done[i], 1);
    for (int i = 0; i < kTeams; ++i) mbar_init(&drain[i], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kWarpIssuer0) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (warp == kWarpIssuer0) tmem_relinquish();
  // Launched as a programmatic dependent: weights, activations and outputs
  // are touched only after the kernel before has completed.
  grid_dependency_wait();
  allow_dependent_launch();

  int64_t ib, ie;
  cta_range(p, 0, ib, ie);
  ItemCursor cur;

  if (warp == 0) {
    // ------------------------------- producer -------------------------------
    if (lane == 0) {
      const uint64_t policy = l2_policy_evict_first();
      int64_t tile = 0;
      bool ok = true;
      int32_t last_j = -1;
      for (int64_t item = ib; item < ie && ok; ++item) {
        cur.next(p, item);
        int64_t kbeg, kend;
        item_range(cur, kbeg, kend);
        if (cur.j != last_j) {
          prefetch_tmap(cur.mc);
          prefetch_tmap(cur.ms);
          last_j = cur.j;
        }
        for (int64_t k0 = kbeg; k0 < kend; k0 += F::kChunk, ++tile) {
          const int s = (int)(tile % kStages);
          const uint32_t par = (uint32_t)((tile / kStages) & 1);
          if (*abort_flag || !mbar_wait_bounded(&empty[s], par ^ 1u)) {
            fail_wait(abort_flag);
            ok = false;
            break;
          }
          uint8_t* st = stages + (size_t)s * kStageBytes;
          mbar_arrive_expect_tx(&full[s], (uint32_t)kStageBytes);
          const int32_t xc = (int32_t)(k0 / 16);  // u32 elements of the codes row
          const int32_t y0 = cur.rb * kRows;
          tma_load_2d(st, cur.mc, xc, y0, &full[s], policy);
          tma_load_2d(st + kBoxBytes, cur.mc, xc + 32, y0, &full[s], policy);
          tma_load_2d(st + kTileCodeBytes, cur.ms, (int32_t)(k0 / F::kBlock / 2), y0, &full[s], policy);
        }
      }
      // never leave with copies in flight
      for (int64_t t = tile - 1; t >= 0 && t >= tile - kStages; --t)
        (void)mbar_wait_bounded(&full[t % kStages], (uint32_t)((t / kStages) & 1));
    }
  } else if (warp < kWarpWorker0) {
    // ------------------------------ MMA issuers -------------------------------
    // Issuer h: per slot of its team, wait (named barrier) until the four
    // workers have written the A buffer, then one elected lane issues the
    // slot's MMAs and commits them to the buffer's mma_done barrier.  The
    // accumulator buffer is free by then: the workers ran the epilogue of the
    // buffer's previous slot before unpacking this one.  The whole warp walks
    // the list in uniform control flow (warp-uniform operands measured about
    // twice as fast per MMA as a loop run by lane 0 alone).  After an abort
    // the warp keeps meeting every barrier but issues nothing.
    const uint32_t h = (uint32_t)(warp - kWarpIssuer0);
    const uint32_t idesc = idesc_e4m3(128, 16);
    const uint32_t base = tmem + h * kTeamCols;
    uint32_t g = 0;
    for (int64_t item = ib; item < ie; ++item) {
      cur.next(p, item);
      int64_t kbeg, kend;
      item_range(cur, kbeg, kend);
      int ci = 0;
      for (int64_t k0 = kbeg; k0 < kend; k0 += F::kChunk, ++ci) {
        const int nb = chunk_blocks(k0, kend);
        for (int kq = 0; kq * kSlotBlocks < nb; ++kq, ++g) {
          const uint32_t b = g & 1u;
          named_barrier(kBarA0 + 2 * h + b, (kWorkers + 1) * 32);
          if (*abort_flag) continue;
          tc_fence_after();
          if (elect_one()) {
            const int nv = min(kSlotBlocks, nb - kSlotBlocks * kq);
            const uint32_t a_t = base + b * kACols;
            const uint32_t d_t = base + 2 * kACols + b * kDCols;
            const uint8_t* bt = tab + (ci * kBlocks + kq * kSlotBlocks) * kBlkTabBytes;
            for (int bi = 0; bi < nv; ++bi) {
              // K step t of block bi reads groups 2t and 2t+1: 128 bytes further
              const uint64_t bd = noswz_desc(bt + bi * kBlkTabBytes, 64, 0);
#pragma unroll
              for (int t = 0; t < 4; ++t)
                tc_mma_f8_ts(d_t + 16 * bi, a_t + 32 * bi + 8 * t, bd + (uint64_t)(8 * t), idesc, t > 0);
            }
            tc_commit(&mma_done[2 * h + b]);
          }
          __syncwarp();
        }
      }
    }
    if (elect_one()) tc_commit(&drain[h]);
    __syncwarp();
    if (lane == 0) (void)mbar_wait_bounded(&drain[h], 0);
    __syncwarp();
  } else {
    // -------------------------------- workers ---------------------------------
    const int cw = warp - kWarpWorker0;  // staging warp index
    const int h = cw >> 2;               // team: row half
    const int q = warp & 3;              // tensor-memory lane quarter
    const int r = h * 128 + q * 32 + lane;  // this thread's row of the tile
    const uint32_t lane_base = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)h * kTeamCols;
    float* scratch = scratch_all + cw * 128;
    int32_t cached_j = -1, cached_split = -1;
    uint32_t g = 0;
    int ring = 0;
    uint32_t ring_par = 0;
    for (int64_t item = ib; item < ie; ++item) {
      cur.next(p, item);
      int64_t kbeg, kend;
      item_range(cur, kbeg, kend);
      if (cur.j != cached_j || cur.split != cached_split) {
        // every MMA that read the previous table has completed: each team ran
        // the epilogue of its last slot at the end of the previous item
        named_barrier(kBarStage, kStageWarps * 32);
        stage_table(make_xsrc(p, cur.j, cur.job, XLink{-1, -1, cur.j, 1.f}), kbeg, (int)(kend - kbeg), tab, fs,
                    scratch, cw, lane);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the table is read by the tensor core
        named_barrier(kBarStage, kStageWarps * 32);
        cached_j = cur.j;
        cached_split = cur.split;
      }
      float acc = 0.f;
      // the slot unpacked last, whose epilogue is still to run
      bool pending = false;
      int p_nv = 0, p_blk = 0;  // its valid blocks and first block of the staged slice
      float p_d0 = 0.f, p_d1 = 0.f;  // its block scales of row r
      int ci = 0;
      for (int64_t k0 = kbeg; k0 < kend; k0 += F::kChunk, ++ci) {
        const int nb = chunk_blocks(k0, kend);
        const int s = ring;
        const uint32_t par = ring_par;
        if (++ring == kStages) {
          ring = 0;
          ring_par ^= 1u;
        }
        const bool have = !*abort_flag && mbar_wait_bounded(&full[s], par);
        if (!have && !*abort_flag) fail_wait(abort_flag);
        const uint8_t* st = stages + (size_t)s * kStageBytes;
        const int nq = (nb + kSlotBlocks - 1) / kSlotBlocks;
        // the code words and scales of a slot are loaded one slot ahead, so
        // their latency overlaps the previous slot's epilogue
        uint4 u[kSlotBlocks][2];
        uint16_t dh[kSlotBlocks];
        const bool live = have && !*abort_flag;
        if (live) load_slot(st, r, 0, min(kSlotBlocks, nb), u, dh);
        for (int kq = 0; kq < nq; ++kq) {
          const int nv = min(kSlotBlocks, nb - kSlotBlocks * kq);
          const uint32_t b = g & 1u;
          float d0 = 0.f, d1 = 0.f;
          if (live && !*abort_flag) {
            // A buffer b (and accumulator buffer b) are free: the epilogue of
            // their previous slot, g - 2, ran before this
            unpack_slot(u, nv, lane_base + b * kACols);
            d0 = __half2float(__ushort_as_half(dh[0]));
            d1 = __half2float(__ushort_as_half(dh[1]));
            tmem_st_wait();
            tc_fence_before();
          }
          bar_arrive(kBarA0 + 2 * h + b, (kWorkers + 1) * 32);
          if (live && kq + 1 < nq) load_slot(st, r, kq + 1, min(kSlotBlocks, nb - kSlotBlocks * (kq + 1)), u, dh);
          if (pending) epilogue(mma_done, h, g, abort_flag, lane_base, fs, p_nv, p_blk, p_d0, p_d1, acc);
          pending = true;
          p_nv = nv;
          p_blk = ci * kBlocks + kq * kSlotBlocks;
          p_d0 = d0;
          p_d1 = d1;
          ++g;
        }
        __syncwarp();
        if (lane == 0 && have) mbar_arrive(&empty[s]);
      }
      if (pending) epilogue(mma_done, h, g, abort_flag, lane_base, fs, p_nv, p_blk, p_d0, p_d1, acc);
      if (!*abort_flag) {
        const int64_t row = (int64_t)cur.rb * kRows + r;
        if (row < cur.job.n) {
          if (cur.job.splits == 1)
            cur.job.y[row] = acc;
          else
            cur.job.ws[(int64_t)cur.split * cur.job.n + row] = acc;
        }
      }
    }
  }

  // every role ends here; then the tensor memory goes back
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpIssuer0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace tcs

int launch_tcs(const Params& p, int grid, cudaStream_t st) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(tcs::tcs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tcs::kSmemBytes);
  });
  KQ_CUDA_TRY(attr);
  // a programmatic dependent of the stream's previous kernel
  KQ_CUDA_TRY(launch_dependent(tcs::tcs_kernel, dim3(grid), dim3(tcs::kThreads), tcs::kSmemBytes, st, p));
  return KQ_OK;
}

int read_tcs_status(int clear) {
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, tcs::g_tcs_status, sizeof(v)) != cudaSuccess) return -1;
  if (clear) {
    unsigned int z = 0;
    if (cudaMemcpyToSymbol(tcs::g_tcs_status, &z, sizeof(z)) != cudaSuccess) return -1;
  }
  return (int)v;
}

}  // namespace kq

