// Device-side structures shared by the weight-streaming kernels of libkq
// (kq_stream.cu: the mma.sync and FFMA consumers, the decode plans and the
// host entry points; kq_tcs.cu: the tcgen05 consumer of PQ2_0 at one
// activation row): tile geometry, the work list (jobs, items, linked-plan
// segments), the kernel parameters, the item cursor and the activation
// loaders.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {


// ---- geometry ---------------------------------------------------------------
constexpr int kConsumerWarps = 16;
// Warp roles: one producer warpgroup (warp 0 issues the copies, warps 1-3
// hold no role) gives registers to the sixteen consumer warps with
// setmaxnreg.  The launch allocates kThreads x kLaunchRegs registers (every
// instantiation compiles to exactly kLaunchRegs, checked before the first
// launch); the split below must not exceed it, or setmaxnreg.inc would wait
// for registers that never come.
constexpr int kProducerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + kProducerWarps);
constexpr int kLaunchRegs = 96;
constexpr int kProducerRegs = 32, kConsumerRegs = 112;
static_assert(32 * (kProducerWarps * kProducerRegs + kConsumerWarps * kConsumerRegs) <= kThreads * kLaunchRegs,
              "register split above the launch allocation");
constexpr int kRowsPerWarp = 8;   // Q8_0 rows per consumer warp
constexpr int kChunkBytes = 256;  // code bytes per row per tile (32 lanes x 8 B)
constexpr int kXMax = 18432;          // activation floats (or B-fragment words) staged per item (all m)
constexpr int kXMaxScale4 = 16384;    // the same for SCALE4, whose larger ring leaves less room
__host__ __device__ constexpr int xmax_of(int fmt) { return fmt == KQ_SCALE4 ? kXMaxScale4 : kXMax; }
constexpr int kScratchFloats = 128;   // per-warp scratch (one Hadamard block)

// Per-format tile geometry.  Q8_0: 128-row tiles (16 warps x 8 rows), a
// ring of 4 stages.  PQ2_0: 256-row tiles, each consumer warp owning 64 rows
// (four 16-row slabs) and a quarter of the tile's K, so every B fragment it
// loads serves four slabs; a ring of 2 stages of 68 KB.  The PQ2_0 K-part
// combine buffer shares its space with the staging scratch: the two are
// never in use at the same time (staging runs between CTA-wide barriers,
// after every warp has finished its handoffs).
// SCALE4 has the PQ2_0 geometry with 32-weight blocks: 16 fp16 scales per
// tile row and 512 weights (256 bytes) of codes.
template <int FMT>
struct Geo {
  static constexpr bool kMma = FMT != KQ_Q8_0;  // PQ2_0 and SCALE4 run on mma.sync
  static constexpr int kTileRows = kMma ? 256 : 128;
  static constexpr int kTileCodeBytes = kTileRows * kChunkBytes;
  static constexpr int kScalesPerRow = FMT == KQ_SCALE4 ? 16 : 8;  // fp16 scales per row per tile
  static constexpr int kTileScaleBytes = kTileRows * kScalesPerRow * 2;
  static constexpr int kStageBytes = kTileCodeBytes + kTileScaleBytes;
  static constexpr int kStages = kMma ? 2 : 4;
  static constexpr int kXMaxF = xmax_of(FMT);
  static constexpr int kBlkMax = kXMaxF / (FMT == KQ_SCALE4 ? 32 : 128);  // per-block side arrays (mma formats)
  static constexpr int kCombineFloats = kMma ? 4 * 3 * 32 * 8 : 0;  // 4 row groups x 3 handing warps
  static constexpr int kScratchRegion =
      kConsumerWarps * kScratchFloats > kCombineFloats ? kConsumerWarps * kScratchFloats : kCombineFloats;
  static constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + (size_t)kXMaxF * 4 + 2 * (size_t)kBlkMax * 4 +
                                       (size_t)kScratchRegion * 4 + 2 * kStages * 8 + 8 * 8 + 16;
};
constexpr int tile_rows(int fmt) { return fmt == KQ_Q8_0 ? Geo<KQ_Q8_0>::kTileRows : Geo<KQ_PQ2_0>::kTileRows; }
static_assert(Geo<KQ_SCALE4>::kSmemBytes <= 232448, "SCALE4 shared memory");
static_assert(Geo<KQ_PQ2_0>::kSmemBytes <= 232448, "PQ2_0 shared memory");

// One matrix of the work list.
struct Job {
  const float* x;  // m rows, row stride k
  float* y;        // m rows, row stride ldy (splits == 1)
  float* ws;       // [splits][m][n] partials (splits > 1)
  int64_t n, k, ldy;
  int64_t x_off, y_off;  // offsets into the packed activation / output (decode plan)
  int64_t ws_off;        // offset of the split partials in the step's workspace (decode plan)
  int64_t item_begin;    // first global item of this job
  int64_t items;         // row_blocks * splits
  int32_t row_blocks;
  int32_t splits;
  int32_t split_k;    // weights per split (multiple of the chunk)
  int32_t had_block;  // PQ2_0: Hadamard block of the rotation (128 or 1024)
  const int8_t* signs;  // PQ2_0: +-1 per position of K applied before the transform, or nullptr
  int64_t tile_base;    // linked plan: index of the job's first row block in Params::tiles
};

// Where a decode-plan job's activation comes from (linked plans).
struct XLink {
  int32_t src_job;    // -1: the packed input at x_off; else the output of job src_job
  int32_t dep_stage;  // the stage whose completion the staging waits for (-1: none)
  int32_t x_key;      // jobs with equal keys read the same activation (the transform memo)
  float alpha;        // the successor activation is alpha * output
};

// A linked plan's unit of work: chunks [c0, c1) of one row block of one job.
// The plan gives every CTA of a stage an equal share of the stage's weight
// bytes as a contiguous run of (row block, chunk) pairs, so a row block may be
// cut between CTAs (stream-K).  A cut row block has nseg > 1 segments; each
// writes its partial sums to slot `slot` of the block's partials.  Nobody
// waits for them inside the stage: a reader of the block's output adds the
// partials in slot order, and after the last stage the cut blocks' y is
// written as the same sums, so readers and y agree bit for bit.
struct Seg {
  int32_t j;       // job
  int32_t rb;      // row block
  int32_t c0, c1;  // chunk range of the weights
  int32_t u0, u1;  // chunks of the activation slice staged for it (one per CTA and activation)
  int32_t nseg;    // segments of this row block (1: the segment writes y itself)
  int32_t slot;    // this segment's place among them
  int64_t part;    // floats from ws_base to the row block's partials, [nseg][tile rows] (nseg > 1)
};

// A row block of a linked plan's job as a reader finds it.
struct TileOut {
  int64_t part;  // floats from ws_base to its partials (nseg > 1)
  int32_t nseg;  // 1: y holds the row block
  int32_t pad;
};

// A cut row block: y[y .. y + rows) = its nseg partials added in slot order.
struct CutOut {
  int64_t part;
  int64_t y;  // offset in the packed output
  int32_t nseg;
  int32_t rows;
};

struct Seg;
struct TileOut;
struct CutOut;

struct Params {
  CUtensorMap map_codes0;  // single GEMV / GEMM: maps of the one matrix
  CUtensorMap map_scales0;
  Job job0;
  const Job* jobs;          // decode plan: device table of jobs ...
  const CUtensorMap* maps;  // ... and their maps, [2 * j] codes, [2 * j + 1] scales
  const XLink* links;       // linked plan: activation sources, or nullptr (every job its own packed input)
  const float* x_base;      // packed activations (decode plan)
  float* y_base;            // packed outputs (decode plan)
  float* ws_base;           // split partials (linked plan)
  int32_t* stage_done;      // linked plan: per stage, the CTAs that have finished it; or nullptr
  const Seg* segs;          // linked plan: the segments, stage-major, CTA-major
  const TileOut* tiles;     // linked plan: every row block of every job, as its readers find it
  const CutOut* cuts;       // linked plan: the cut row blocks, whose y is written after the last stage
  const int64_t* bounds;    // item (segment) ranges of CTA c in stage s: [bounds[s (G+1) + c], bounds[s (G+1) + c + 1])
  int64_t total_items;
  int32_t nstages;          // stages of the plan (1 without links)
  int32_t n_cuts;
};

template <int FMT>
struct Fmt;
template <>
struct Fmt<KQ_Q8_0> {
  static constexpr int kBlock = 32;
  static constexpr int kCodesPerByte = 1;
  static constexpr int kChunk = kChunkBytes;  // 256 weights per tile row
  static constexpr int kGran = 8;             // weights per lane per tile row
};
template <>
struct Fmt<KQ_PQ2_0> {
  static constexpr int kBlock = 128;
  static constexpr int kCodesPerByte = 4;
  static constexpr int kChunk = kChunkBytes * 4;  // 1024 weights per tile row
  static constexpr int kGran = 32;
};
template <>
struct Fmt<KQ_SCALE4> {
  static constexpr int kBlock = 32;
  static constexpr int kCodesPerByte = 2;
  static constexpr int kChunk = kChunkBytes * 2;  // 512 weights per tile row
  static constexpr int kGran = 16;
};

__host__ __device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

// Item -> (job, row block, split).  Items of a job are split-major.
struct ItemCursor {
  int32_t j = -1;
  Job job;
  const CUtensorMap* mc = nullptr;
  const CUtensorMap* ms = nullptr;
  int32_t split = 0, rb = 0;  // the item's K split and 128-row block within the job
  int64_t last = -2;          // the item last decoded
  // Moves to `item` and decodes its (split, row block): by one step from the
  // previous item of the same job (items are split-major), else by one
  // 32-bit division.
  __device__ void next(const Params& p, int64_t item) {
    const int32_t j0 = j;
    seek(p, item);
    if (j == j0 && item == last + 1) {
      if (++rb == job.row_blocks) {
        rb = 0;
        ++split;
      }
    } else {
      const int32_t local = (int32_t)(item - job.item_begin);
      split = local / job.row_blocks;
      rb = local - split * job.row_blocks;
    }
    last = item;
  }
  // Linked plans: makes job jj the current job.
  __device__ void use(const Params& p, int32_t jj) {
    if (jj == j) return;
    j = jj;
    job = p.jobs[j];
    job.x = p.x_base + job.x_off;
    job.y = p.y_base + job.y_off;
    job.ws = p.ws_base + job.ws_off;
    mc = p.maps + 2 * j;
    ms = p.maps + 2 * j + 1;
  }
  __device__ void seek(const Params& p, int64_t item) {
    if (p.jobs == nullptr) {
      if (j < 0) {
        job = p.job0;
        mc = &p.map_codes0;
        ms = &p.map_scales0;
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
    job.ws = p.ws_base + job.ws_off;
    mc = p.maps + 2 * j;
    ms = p.maps + 2 * j + 1;
  }
};

__device__ __forceinline__ void cta_range(const Params& p, int stage, int64_t& b, int64_t& e) {
  if (p.bounds) {
    const int64_t* bs = p.bounds + (int64_t)stage * (gridDim.x + 1);
    b = bs[blockIdx.x];
    e = bs[blockIdx.x + 1];
  } else {
    b = p.total_items * blockIdx.x / gridDim.x;
    e = p.total_items * (blockIdx.x + 1) / gridDim.x;
  }
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }  // e in [-126, 127]

// The activation a job reads: a plain vector, or alpha times an earlier
// job's output (a dependent chain).
struct XSrc {
  const float* base;   // the vector
  int64_t row_stride;  // floats between activation rows (m > 1)
  int32_t vec4;        // base allows 16-byte loads
  float alpha;
  int32_t had;          // PQ2_0 rotation block (128 or 1024)
  const int8_t* signs;  // PQ2_0 sign per position of K, or nullptr
  const TileOut* tiles;  // linked source: its row blocks (a cut one is the sum of its partials), or nullptr
  const float* parts;    // linked source: the partials' base
};

// x[i..i+3] of activation row m; loads bypass L1 (the source may have been
// written by other CTAs of this launch).  TR > 0: a linked plan's source
// output in row blocks of TR rows, where a cut block is read as the sum of
// its partials in slot order (i % 4 == 0, so the four share a block);
// `known`, when given, is that block's entry, already read.
template <bool IO16 = false, int TR = 0>
__device__ __forceinline__ float4 load_x4(const XSrc& xs, int m, int64_t i, const TileOut* known = nullptr) {
  if constexpr (TR > 0) {
    if (xs.tiles) {
      const TileOut t = known ? *known : xs.tiles[i / TR];
      if (t.nseg > 1) {
        // up to eight partials loaded at once, then added in slot order
        const float* b = xs.parts + t.part + i % TR;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int q0 = 0; q0 < t.nseg; q0 += 8) {
          float4 u[8];
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q0 + q < t.nseg) u[q] = __ldcg(reinterpret_cast<const float4*>(b + (int64_t)(q0 + q) * TR));
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q0 + q < t.nseg) {
              if (q0 + q == 0) {
                v = u[q];
              } else {
                v.x += u[q].x;
                v.y += u[q].y;
                v.z += u[q].z;
                v.w += u[q].w;
              }
            }
        }
        v.x *= xs.alpha;
        v.y *= xs.alpha;
        v.z *= xs.alpha;
        v.w *= xs.alpha;
        return v;
      }
    }
  }
  if constexpr (IO16) {  // fp16 activations (the fp16 chain): four halves, exact in fp32
    const __half* h = reinterpret_cast<const __half*>(xs.base) + (int64_t)m * xs.row_stride + i;
    const uint2 u = __ldcg(reinterpret_cast<const uint2*>(h));
    const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
    const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    return make_float4(a.x, a.y, c.x, c.y);
  }
  const float* b = xs.base + (int64_t)m * xs.row_stride + i;
  float4 v;
  if (xs.vec4)
    v = __ldcg(reinterpret_cast<const float4*>(b));
  else
    v = make_float4(__ldcg(b), __ldcg(b + 1), __ldcg(b + 2), __ldcg(b + 3));
  v.x *= xs.alpha;
  v.y *= xs.alpha;
  v.z *= xs.alpha;
  v.w *= xs.alpha;
  return v;
}

// The rotation fields are read from the job table (or the single job), not
// from the cursor's copy, so that they stay out of registers in the tile loop.
__device__ __forceinline__ XSrc make_xsrc(const Params& p, int32_t j, const Job& job, const XLink& lk) {
  XSrc xs;
  const Job& jm = p.jobs ? p.jobs[j] : p.job0;
  xs.had = jm.had_block;
  xs.signs = jm.signs;
  xs.row_stride = job.k;
  xs.alpha = 1.f;
  xs.base = job.x;
  xs.tiles = nullptr;
  xs.parts = p.ws_base;
  if (lk.src_job >= 0) {  // a linked source: its output, cut row blocks as partials
    const Job& src = p.jobs[lk.src_job];
    xs.alpha = lk.alpha;
    xs.base = p.y_base + src.y_off;
    xs.tiles = p.tiles + src.tile_base;
  }
  xs.vec4 = (reinterpret_cast<uintptr_t>(xs.base) & 15u) == 0 ? 1 : 0;
  return xs;
}

// Unnormalised 128-point Walsh-Hadamard transform, natural (Sylvester) order,
// of a block held 4 consecutive elements per lane: strides 1 and 2 in
// registers, 4 .. 64 across lanes.
__device__ __forceinline__ void fwht128_lane4(float (&v)[4], int lane) {
  float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[2] = a0 - a2;
  v[1] = a1 + a3;
  v[3] = a1 - a3;
#pragma unroll
  for (int mk = 1; mk < 32; mk <<= 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float q = __shfl_xor_sync(0xffffffffu, v[i], mk);
      v[i] = (lane & mk) ? (q - v[i]) : (v[i] + q);
    }
  }
}


// Host launcher of the tcgen05 streaming kernel of PQ2_0 at one activation
// row (kq_tcs.cu): fp32 activation and output, unlinked work lists (a single
// GEMV with its K splits, or a decode plan without links).  Launched as a
// programmatic dependent of the stream's previous kernel.
int launch_tcs(const Params& p, int grid, cudaStream_t st);
// Status word of that kernel (bit s set = status s seen); -1 if it cannot be read.
int read_tcs_status(int clear);

}  // namespace kq
