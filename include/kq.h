/*
 * kq.h -- C ABI of libkq, the quantized weight-streaming GEMV library for
 * NVIDIA GB300 (sm_103a).
 *
 * What it computes.  Token decode of a large language model is bound by one
 * operation: a matrix-vector product that streams every quantized weight from
 * HBM once per token and dequantizes it inside the dot product.  Two block
 * formats are supported:
 *
 *   Q8_0   32 weights per block along K: an fp16 scale d and 32 int8 codes q,
 *          value d*q ("Kipp Architecture", section "Weight quantization";
 *          34 bytes per block, i.e. 136 bytes per 128-dim row as printed in
 *          "Kipp Benchmarks", Quantized KV cache bullet).
 *
 *   SCALE4 scale4_gs32 ("Kipp Benchmarks", section "Scale-only 4-bit
 *          (scale4_gs32)"): 32 weights per block, an fp16 scale d first and
 *          16 bytes of 4-bit codes q, value d*(q-8); d = (the block's weight
 *          of largest magnitude, with its sign) / -8, the codes quantized
 *          against the fp16-rounded d (18 bytes, 4.5 bits per weight).
 *
 *   PQ2_0  128 weights per block: an fp16 scale d and 2-bit codes
 *          q in {0,1,2}, element j in byte j/4 at bit offset 2*(j%4), value
 *          (q-1)*d, d = max|w| and q = round(w/d)+1 ("Bonsai 2 27B - ternary
 *          g128 + blockwise Hadamard", section 3.1).  The weights are stored
 *          rotated, W' = W R^T with R = H_n S / sqrt(n) applied
 *          block-diagonally along K (same page, sections 4.1-4.2): n = 128
 *          with S = I (the default), or the page's own n = 1024 with a +-1
 *          sign per position of K (S = diag(signs), one sign vector per K
 *          width).  The activation gets x' = R x (sign flip, then the
 *          transform) before the product; the PQ2_0 GEMV takes the UNROTATED
 *          x and applies R itself.
 *
 * Conventions.
 *  - Every function returns a kq_status (int); 0 is success.  On failure
 *    nothing has been written to any output and no work was enqueued;
 *    kq_last_error() gives a one-line reason (per calling thread).
 *  - Device entry points are asynchronous: they validate their arguments on
 *    the host, enqueue kernels on `stream` (a cudaStream_t passed as void*;
 *    NULL means the legacy default stream) and return.  The caller
 *    synchronises.  All pointers named d_* are device memory owned by the
 *    caller; the library never frees them.
 *  - GEMV/GEMM and decode-step calls allocate nothing.  Scratch memory they
 *    need is the caller's workspace, sized by the *_workspace_bytes queries.
 *  - Results are deterministic: the same inputs, shapes and split plan give
 *    bitwise the same output on every call and for every grid size.
 *  - Device pointers must be 16-byte aligned.  Sizes are int64_t elements.
 *
 * Device data layout of a quantized matrix (n rows, k columns, "planes"):
 *  - codes  Q8_0: int8 [n][k], row stride k bytes.
 *           PQ2_0: uint32 [n][k/16], row stride k/4 bytes; each 32-bit word
 *           (little endian) holds elements 16i..16i+15 of its row at bits 2j,
 *           which is the byte order of the block's qs[] read as words.
 *           SCALE4: bytes [n][k/2], row stride k/2; element j of a row in
 *           byte j/2 at bit offset 4 (j % 2), which is the blocks' nibble
 *           bytes concatenated (a 32-bit word holds elements 8i..8i+7).
 *  - scales fp16 [n][kq_scale_stride(fmt, k)]; entry [r][b] is the scale of
 *           block b of row r; the padding entries of each row are zero.
 */
#ifndef KQ_H
#define KQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KQ_OK = 0,
  KQ_ERR_INVALID_ARG = 1, /* NULL pointer, unknown format, negative or zero size   */
  KQ_ERR_SHAPE = 2,       /* k not a multiple of the block, n < 1, m out of range  */
  KQ_ERR_ALIGNMENT = 3,   /* a device pointer is not 16-byte aligned               */
  KQ_ERR_NONFINITE = 4,   /* NaN or Inf in the weights given to a quantizer        */
  KQ_ERR_RANGE = 5,       /* a block scale does not fit fp16 (above 65504)         */
  KQ_ERR_WORKSPACE = 6,   /* workspace NULL or smaller than required               */
  KQ_ERR_CUDA = 7,        /* a CUDA runtime call failed                            */
  KQ_ERR_TIMEOUT = 8,     /* a bounded wait inside a kernel expired                */
  KQ_ERR_UNSUPPORTED = 9  /* device or combination of arguments not supported      */
} kq_status;

/* KQ_PTQ1_0 is a storage format only ("Bonsai 2 27B", section 3.2: the
 * PQ2_0 trits and scale packed in base 3, 28 bytes per 128 weights, 1.75
 * bits per weight; the page ships it as a download option and unpacks it to
 * the PQ2_0 words at load time).  kq_prepare turns PTQ1_0 blocks into PQ2_0
 * planes; every GEMV runs on those. */
typedef enum { KQ_Q8_0 = 0, KQ_PQ2_0 = 1, KQ_PTQ1_0 = 2, KQ_SCALE4 = 3 } kq_format;

/* A quantized matrix resident in device memory (planes as described above).
 * had_block is the Hadamard block n of the fold: 128 or 1024 for PQ2_0 (k a
 * multiple of it), 0 for Q8_0.  signs (PQ2_0 only) is NULL for S = I, or k
 * int8 entries, each +1 or -1, in 16-byte-aligned device memory owned by
 * the caller (matrices of one K width share one vector on the page). */
typedef struct {
  int32_t fmt;
  int32_t had_block;
  int64_t n;
  int64_t k;
  const void* codes;
  const void* scales;
  const int8_t* signs;
} kq_qmat;

/* ---- status and layout ---------------------------------------------------- */

const char* kq_status_string(int status);
/* Reason of the last failing call on this thread ("" if none). */
const char* kq_last_error(void);
/* ABI version, bumped on incompatible change. */
int kq_version(void);

/* Weights per block: 32 (Q8_0, SCALE4) or 128 (PQ2_0, PTQ1_0); 0 for an unknown format. */
int64_t kq_block_size(int fmt);
/* Bytes of one block (34 for Q8_0 and PQ2_0, 28 for PTQ1_0, 18 for SCALE4) times the number
 * of blocks of an n x k matrix.  The plane queries below give, for PTQ1_0,
 * the PQ2_0 planes kq_prepare writes. */
int64_t kq_blocks_bytes(int fmt, int64_t n, int64_t k);
/* Row stride of the scales plane in fp16 elements: k/block rounded up to 8. */
int64_t kq_scale_stride(int fmt, int64_t k);
int64_t kq_codes_bytes(int fmt, int64_t n, int64_t k);
int64_t kq_scales_bytes(int fmt, int64_t n, int64_t k);

/* ---- host quantizers (offline weight preparation, deterministic) ----------- */

/* Q8_0 ("Kipp Architecture", "Weight quantization": 32-weight blocks, an fp16
 * scale against which the codes are quantized, value d*q).
 * Per row and 32-block: d = fp16(amax/127) (fp32 quotient, then round to
 * nearest even), q = round-half-away-from-zero(w / float(d)) clamped to
 * [-127, 127]; a block whose fp16 scale is zero gets q = 0.  Output: n*k/32
 * blocks of 34 bytes (d little endian, then 32 int8), row-major.
 * Errors: KQ_ERR_SHAPE (k % 32), KQ_ERR_NONFINITE, KQ_ERR_RANGE. */
int kq_quantize_q8_0(const float* w, int64_t n, int64_t k, void* blocks);

/* PQ2_0 ("Bonsai 2 27B", section 3.1 for the block, section 4.1 for the
 * weights being rotated before they are quantized).
 * Per row and 128-block of the ROTATED weights: d = fp16(max|w|), code =
 * round-half-away-from-zero(w / float(d)) clamped to [-1, 1], plus 1; a block
 * whose fp16 scale is zero gets code 1.  Output: n*k/128 blocks of 34 bytes.
 * Errors: KQ_ERR_SHAPE (k % 128), KQ_ERR_NONFINITE, KQ_ERR_RANGE. */
int kq_quantize_pq2_0(const float* w_rot, int64_t n, int64_t k, void* blocks);

/* SCALE4 per row and 32-block: m = the weight of largest magnitude (the
 * first on a tie), d = fp16(m / -8) (fp32 quotient, then round to nearest
 * even), q = round-half-away-from-zero(w / float(d)) + 8 clamped to
 * [0, 15]; a block whose fp16 scale is zero gets q = 8.  Output: n*k/32
 * blocks of 18 bytes (d little endian, then element j in byte 2 + j/2 at bit
 * offset 4 (j % 2)).  Errors: KQ_ERR_SHAPE (k % 32), KQ_ERR_NONFINITE,
 * KQ_ERR_RANGE. */
int kq_quantize_scale4(const float* w, int64_t n, int64_t k, void* blocks);

/* PTQ1_0 per row and 128-block of the ROTATED weights: the PQ2_0 scale and
 * trits (same rules as kq_quantize_pq2_0) packed in base 3: 24 bytes of five
 * trits, 2 bytes of four, then the fp16 scale (28 bytes).  A byte holds
 * ceil(256 v / 243), v its trits as a base-3 number with the first trit most
 * significant (a four-trit byte's fifth trit is 0).  Element e is trit e/16
 * of byte e%16 for e < 80, trit (e-80)/8 of byte 16+(e-80)%8 for e < 120,
 * trit (e-120)/2 of byte 24+(e-120)%2 above (the page's element-order table).
 * Errors: KQ_ERR_SHAPE (k % 128), KQ_ERR_NONFINITE, KQ_ERR_RANGE. */
int kq_quantize_ptq1_0(const float* w_rot, int64_t n, int64_t k, void* blocks);

/* Blockwise normalised Walsh-Hadamard transform of each row, on the host
 * (R = H_n / sqrt(n), Sylvester natural order, block-diagonal along K:
 * "Bonsai 2 27B", sections 4.1-4.2):
 * out[b*block + i] = (1/sqrt(block)) * sum_c H[i][c] in[b*block + c], with the
 * sum taken in FP64, one FP64 multiply, one rounding to fp32.  block is a
 * power of two dividing k.  in == out is allowed. */
int kq_hadamard_blockwise_host(const float* in, float* out, int64_t rows, int64_t k, int32_t block);

/* ---- device weight preparation ------------------------------------------- */

/* The device planes of a matrix ("Bonsai 2 27B", section 3.1: a block's qs
 * bytes read as little-endian words are its code words; "Kipp
 * Architecture": the 34-byte Q8_0 block).  Repack n*k/block AoS blocks
 * (device memory, as produced by the host
 * quantizers) into the codes and scales planes.  fmt = KQ_PTQ1_0 reads
 * 28-byte PTQ1_0 blocks and writes the PQ2_0 planes of the same trits and
 * scales (a lossless transcode; the matrix is then a PQ2_0 matrix). */
int kq_prepare(int fmt, const void* d_blocks, int64_t n, int64_t k, void* d_codes, void* d_scales, void* stream);

/* Quantize an n x k fp32 matrix in device memory straight into planes, with
 * the same rules and bit-identical results as the host quantizers.  On a
 * NaN, Inf or fp16 overflow the call still returns KQ_OK (it is
 * asynchronous); kq_device_status() then reports KQ_ERR_NONFINITE or
 * KQ_ERR_RANGE. */
int kq_quantize_q8_0_device(const float* d_w, int64_t n, int64_t k, void* d_codes, void* d_scales, void* stream);
int kq_quantize_pq2_0_device(const float* d_w_rot, int64_t n, int64_t k, void* d_codes, void* d_scales,
                             void* stream);
int kq_quantize_scale4_device(const float* d_w, int64_t n, int64_t k, void* d_codes, void* d_scales, void* stream);

/* Embedding lookup: d_out[t][0..k) = row d_ids[t] of the n x k table E,
 * dequantized; for a PQ2_0 table (stored rotated, R e per row, as the Bonsai
 * page's token_embd) the inverse rotation e = R^T z = S (H_n z)/sqrt(n) per
 * n-block follows, the transform first, then the sign flip (section 4.2), in
 * fp32.  d_ids int32 [count], d_out fp32 [count][k], both 16-byte aligned
 * device memory.  An id outside [0, n) yields a zero row and sets KQ_ERR_RANGE
 * in the device status word (kq_device_status).  PQ2_0 tables up to k =
 * 32768. */
int kq_embed(const kq_qmat* E, const int32_t* d_ids, int64_t count, float* d_out, void* stream);

/* Debug: write the dequantized n x k fp32 matrix (d*q or (q-1)*d, exact). */
int kq_dequantize(const kq_qmat* W, float* d_out, void* stream);

/* Blockwise normalised Walsh-Hadamard transform of each row on the device,
 * same arithmetic as kq_hadamard_blockwise_host (FP64 butterflies, one FP64
 * multiply, one rounding), bit-identical to it.  d_in == d_out is allowed. */
int kq_hadamard_blockwise(const float* d_in, float* d_out, int64_t rows, int64_t k, int32_t block, void* stream);

/* The page's rotation R = H_n S / sqrt(n) of each row, block-diagonal along
 * K (the Bonsai page, sections 4.1-4.2): out = (1/sqrt(n)) H_n (s * in) per
 * n-block, the sign flip exact, then the same FP64 butterflies, one FP64
 * multiply and one rounding as above (so the host and device versions are
 * bit-identical).  signs: k int8 entries, +1 or -1 (host memory for the
 * host version, device memory for the device one), or NULL for S = I.
 * Used offline to fold the rotation into weights (W' = W R^T: each row
 * w' = R w) before quantizing to PQ2_0.  block: a power of two dividing k,
 * up to 4096. */
int kq_rotate_blockwise_host(const float* in, float* out, int64_t rows, int64_t k, int32_t block,
                             const int8_t* signs);
int kq_rotate_blockwise(const float* d_in, float* d_out, int64_t rows, int64_t k, int32_t block,
                        const int8_t* d_signs, void* stream);

/* ---- GEMV / small-M GEMM --------------------------------------------------- */

/* Workspace bytes needed by a GEMV / GEMM call on W with m activation rows
 * (split-K partials; 0 when the call needs none). */
size_t kq_gemv_workspace_bytes(const kq_qmat* W, int64_t m);

/* y[n] = W x for a Q8_0 matrix: d_x fp32 [k], d_y fp32 [n].  The batch-1
 * product that bounds decode, every weight streamed once ("Kipp Benchmarks",
 * "Decode is weight-bandwidth-bound").  A small matrix (k <= 4096 and at
 * most 20 MB of codes) runs in one launch with no K split and needs no
 * workspace; larger ones use the streaming kernel's split plan. */
int kq_gemv_q8_0(const kq_qmat* W, const float* d_x, float* d_y, void* d_ws, size_t ws_bytes, void* stream);

/* y[n] = W x for a SCALE4 matrix: d_x fp32 [k], d_y fp32 [n]. */
int kq_gemv_scale4(const kq_qmat* W, const float* d_x, float* d_y, void* d_ws, size_t ws_bytes, void* stream);

/* y[n] = W' (R x) for a PQ2_0 matrix: d_x is the UNROTATED fp32 activation
 * [k]; the blockwise transform runs in the kernel's activation prologue (the
 * activation side of every folded matmul: "Bonsai 2 27B", section 4.2; the
 * ternary matvec of section 8.5).  With the 128-block rotation and no signs,
 * a small matrix (k <= 5376 and at most 16 MB of codes) runs in one launch
 * with no K split and needs no workspace, on the default consumer. */
int kq_gemv_pq2_0(const kq_qmat* W, const float* d_x, float* d_y, void* d_ws, size_t ws_bytes, void* stream);

/* The fp16 chain of the Bonsai page, section 4.4 (its token-identity
 * yardstick): d_x is an fp16 activation [k], d_y an fp16 output [n], any
 * matrix format.  For PQ2_0 the (sign flip and) transform runs in fp32 and
 * its result is rounded to fp16 before the product; the product accumulates
 * in fp32 and is rounded once to fp16 at the end (after the split second
 * pass, if any).  Same workspace as the fp32 GEMV of W; d_x and d_y 16-byte
 * aligned. */
int kq_gemv_f16(const kq_qmat* W, const void* d_x, void* d_y, void* d_ws, size_t ws_bytes, void* stream);

/* Batched decode / speculation: several activation rows against one weight
 * stream ("Kipp Benchmarks", tensor matmul section).
 * Y[m][n] = X[m][k] W^T (rotated per row for PQ2_0), X and Y row-major fp32,
 * 1 <= m <= 64.  From m = 5 on (m = 9 for SCALE4), when k <= 32768, this is
 * kq_gemm_tc with an automatic split: it reads the weights once at any m.
 * Below, the streaming kernel applies each weight tile to up to 4 activation
 * rows per pass.  kq_gemv_workspace_bytes(W, m) sizes the workspace of
 * either. */
int kq_gemm_small_m(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, void* d_ws, size_t ws_bytes,
                    void* stream);

/* Small-batch GEMM on the tensor cores (tcgen05), the batched path of
 * "Kipp Benchmarks" (tensor matmul section: each K block dequantized into a
 * 16-bit tile, then multiplied): Y[m][n] = X[m][k] W^T, X rotated per
 * 128-block for PQ2_0 (unrotated X in, as for kq_gemv_pq2_0).
 *  - 1 <= m <= 64, k <= 32768; X, Y row-major fp32, 16-byte aligned.
 *  - Weights enter the tensor core as exact fp16 code values, one fp32
 *    accumulator per quantization block, the block scale applied in the
 *    epilogue: q for Q8_0, (c-1) times a power of two for PQ2_0, (q-8) times
 *    a power of two for SCALE4 (a 4-bit code masked in place in an fp16 half
 *    is an exact subnormal; one fp16 subtraction applies the zero point).
 *    Each activation row enters as two fp16 rows, high and low part of
 *    x * 2^-e (e its largest exponent), so x keeps ~22 bits; fp32
 *    accumulation.  A Q8_0
 *    scale above 65504/127 (q*d not a finite fp16) sets KQ_ERR_RANGE.
 *  - splits: K splits (0 = automatic); with splits > 1 the partial sums are
 *    added in split order by a second pass (deterministic).
 *  - Workspace (kq_gemm_tc_workspace_bytes, 16-byte aligned): the fp16
 *    activation matrix (4 * round16(m) * k bytes), per-row exponents and the
 *    split partials; everything in it is written before it is read.
 *  - Errors: KQ_ERR_SHAPE (m or k out of range), KQ_ERR_WORKSPACE,
 *    KQ_ERR_ALIGNMENT, KQ_ERR_CUDA; a bounded device wait that expires sets
 *    KQ_ERR_TIMEOUT for kq_device_status. */
int kq_gemm_tc(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int32_t splits, void* d_ws,
               size_t ws_bytes, void* stream);
size_t kq_gemm_tc_workspace_bytes(const kq_qmat* W, int64_t m, int32_t splits);

/* GEMV/GEMM with an explicit split-K factor (1 = no split; 0 = automatic).
 * Splits are whole multiples of the format's tile chunk along K: 256
 * weights (Q8_0), 512 (SCALE4), 1024 (PQ2_0); the partial sums of each split
 * are added in split order by a second pass, so a given split factor always
 * gives bitwise the same result. */
int kq_gemm_splitk(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int32_t splits, void* d_ws,
                   size_t ws_bytes, void* stream);
size_t kq_gemm_splitk_workspace_bytes(const kq_qmat* W, int64_t m, int32_t splits);

/* Allocation-free variant of kq_gemm_splitk (no counterpart on the pages; an
 * addition of this library).  For callers that cannot allocate device
 * memory where they run the product (allocation-free serving loops, fixed
 * memory arenas, code that only receives device pointers): the split-K
 * partial sums go to a scratch array of kq_gemm_splitk_noalloc_max_bytes()
 * bytes (2 MiB) that the library reserves in device global memory on every
 * GPU that loads it and keeps until the process exits.  The call allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library routine).
 *  - Same arguments, results and bit-exactness as kq_gemm_splitk with the
 *    same split count; the caller still passes X and Y.
 *  - A split plan whose partials need more than the scratch is rejected with
 *    KQ_ERR_WORKSPACE before anything is enqueued.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and keeps it; make that
 *    first call before any stream capture on the device.  The kept address
 *    does not survive a device reset (cudaDeviceReset): do not call this
 *    entry point again in a process after resetting a device it was used on.
 *  - Every call on a device shares the one array and leaves its partials in
 *    it; nothing in it has to start at zero (each call writes every partial
 *    it reads).  Calls that overlap on the GPU (different streams without
 *    ordering) race on the array: order them on one stream or with events. */
int kq_gemm_splitk_noalloc(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int32_t splits, void* stream);
size_t kq_gemm_splitk_noalloc_max_bytes(void);

/* ---- decode-step driver ---------------------------------------------------- */

/* The decode step: a whole model's projection list streamed once per token
 * ("Bonsai 2 27B", sections 8.5-8.7: the per-token matvec stream and the
 * cost of dispatching it one kernel at a time).
 * A plan for streaming a whole model's projection list once per step: count
 * matrices of one format.  Creating it copies the descriptors and a
 * per-SM schedule to device memory (the only allocation the plan makes);
 * kq_decode_step then runs the whole list in one persistent kernel.
 * Activations are packed: matrix i reads x at offset sum_{j<i} k_j floats of
 * d_x_packed and writes y at offset sum_{j<i} n_j floats of d_y_packed. */
typedef struct kq_plan kq_plan;
int kq_decode_plan_create(const kq_qmat* mats, int64_t count, kq_plan** out);
/* Total packed activation / output lengths in floats, and weight bytes. */
int kq_decode_plan_sizes(const kq_plan* plan, int64_t* x_floats, int64_t* y_floats, int64_t* weight_bytes);
/* Workspace bytes of kq_decode_step (0 for a plan made by kq_decode_plan_create). */
size_t kq_decode_workspace_bytes(const kq_plan* plan);
/* One decode step: every matrix of the plan applied to its activation in one
 * launch (the page's token of matvecs, "Bonsai 2 27B", section 8.5, without
 * its per-matvec dispatches, sections 8.6-8.7).  d_x_packed / d_y_packed:
 * 16-byte-aligned device buffers of the plan's sizes; d_ws: the plan's
 * workspace (kq_decode_workspace_bytes; NULL when 0).  Asynchronous on
 * `stream`.  Errors: KQ_ERR_INVALID_ARG (NULL plan or buffers),
 * KQ_ERR_ALIGNMENT, KQ_ERR_WORKSPACE, KQ_ERR_CUDA. */
int kq_decode_step(kq_plan* plan, const float* d_x_packed, float* d_y_packed, void* d_ws, size_t ws_bytes,
                   void* stream);
/* One step with the activations and outputs in host memory: enqueues on
 * `stream` the copy of the plan's x_floats packed activations from
 * h_x_packed to the device buffer d_x_packed, the step, and the copy of the
 * y_floats outputs from d_y_packed back to h_y_packed (plain asynchronous
 * copies; the caller synchronises the stream before reading h_y_packed and
 * leaves h_x_packed unchanged until then).
 *  - When h_x_packed is page-locked host memory (cudaHostAlloc /
 *    cudaHostRegister) whose device mapping is 16-byte aligned, the kernel
 *    reads the activations through that mapping as it stages them, spread
 *    over the step instead of a copy before it; d_x_packed is then left
 *    unwritten.
 *  - A plan of one stage never reads its own outputs: when h_y_packed is
 *    such page-locked memory, the step writes the outputs there directly
 *    and d_y_packed is left unwritten (no copy back).
 *  - d_x_packed, d_y_packed: device buffers of the plan's sizes, 16-byte
 *    aligned, owned by the caller; h_x_packed may be NULL when x_floats is 0.
 *  - Errors: every argument check of kq_decode_step (and KQ_ERR_INVALID_ARG
 *    for a NULL host buffer) runs before anything is enqueued.  KQ_ERR_CUDA
 *    reports a copy or the step's launch that could not be enqueued; when
 *    the launch fails, the activation copy may already be enqueued. */
int kq_decode_step_host(kq_plan* plan, const float* h_x_packed, float* h_y_packed, float* d_x_packed,
                        float* d_y_packed, void* d_ws, size_t ws_bytes, void* stream);
void kq_decode_plan_destroy(kq_plan* plan);

/* Decode plans with the dependencies of a real decode step.  In a model's
 * decode the projections of a layer read activations produced by earlier
 * projections: q, k and v (or gate and up) read one shared input, o reads
 * what attention made of q, the FFN reads what the block made of o, the next
 * layer reads the FFN's output.  The Bonsai 2 27B page memoises one
 * transform per activation site, shared by q/k/v and by gate/up (sections
 * 4.2 and 7), and counts the cost of dispatching the dependent layer chain
 * one kernel at a time (sections 8.6-8.7).  A
 * linked plan states, per matrix, where its activation comes from and which
 * stage it belongs to; kq_decode_step then runs the whole list in one
 * cooperative persistent launch in which a matrix starts its arithmetic
 * only after the matrices it depends on have written their outputs, while
 * the weight stream keeps running ahead across stage boundaries.
 *
 * The operations between projections that are not projections (attention,
 * normalisation, activation functions, residual adds) are outside this
 * library; the plainest stand-in is kept: the activation of a dependent
 * matrix is alpha times a prefix of an earlier matrix's output. */
typedef enum {
  KQ_SRC_PACKED = 0,    /* a fresh slot of d_x_packed, in list order over the matrices with this kind */
  KQ_SRC_INPUT_OF = 1,  /* the same activation as matrix `of` (k equal): a grouped matvec */
  KQ_SRC_OUTPUT_OF = 2  /* x[i] = fp32(alpha * y_of[i]), i < k <= n_of; stage of `of` < this stage */
} kq_src_kind;

typedef struct {
  int32_t src;   /* kq_src_kind */
  int32_t stage; /* >= 0, nondecreasing along the list */
  int64_t of;    /* an earlier matrix (index < this one) for KQ_SRC_INPUT_OF / KQ_SRC_OUTPUT_OF */
  float alpha;   /* KQ_SRC_OUTPUT_OF: finite scale of the successor activation; else ignored */
  int32_t reserved; /* 0 */
} kq_link;

/* Creates a linked plan: count matrices of one format with one link each.
 *  - Every matrix writes its output to d_y_packed at offset sum_{j<i} n_j
 *    (all of them, also those read by later stages).  d_x_packed holds only
 *    the KQ_SRC_PACKED activations, in list order.
 *  - Work is balanced per stage over all SMs: each CTA gets a contiguous
 *    run of (row block, K chunk) pairs, so a row block may be cut between
 *    CTAs (row blocks are kept whole where that balances as well).  A cut
 *    row block's pieces write partial sums into the step's workspace;
 *    every reader (the dependent matrices' activation staging, and the
 *    write of y after the last stage) adds them in the same fixed order, so
 *    results are deterministic and readers see exactly the final y.
 *  - Matrices that share one activation (KQ_SRC_INPUT_OF) share its
 *    staged, transformed copy inside each CTA (the transform memo): a CTA
 *    stages the K range it needs from an activation once for all the
 *    matrices of the group that it works on.
 *  - Errors: KQ_ERR_INVALID_ARG (NULL, unknown kind, `of` not earlier,
 *    non-finite alpha, reserved != 0), KQ_ERR_SHAPE (k mismatch of a link,
 *    decreasing stage, an output read in its own or a later stage),
 *    KQ_ERR_UNSUPPORTED (mixed formats, k above the staging limit), KQ_ERR_CUDA.
 * kq_decode_workspace_bytes gives the step's workspace (stage counters and
 * the partials of cut row blocks); kq_decode_step runs it.  Steps of one plan that share a
 * workspace must be ordered (one stream). */
int kq_decode_plan_create_linked(const kq_qmat* mats, const kq_link* links, int64_t count, kq_plan** out);
/* Number of stages of a plan and of matrices with a row block cut between CTAs. */
int kq_decode_plan_stages(const kq_plan* plan, int32_t* stages, int32_t* split_matrices);

/* ---- read-only streaming control -------------------------------------------- */

/* The in-harness bandwidth ceiling of a kernel that reads each byte once:
 * streams d_src[0, bytes) from device memory exactly once through shared
 * memory, on the data path of the GEMV kernels (one persistent CTA per SM,
 * bulk asynchronous copies with an L2 evict-first hint into a ring of
 * `stages` buffers of `stage_bytes`, consumer warps reading every 16-byte
 * word back from shared memory), and XORs the XOR of all 32-bit words of the
 * range into *d_sink (zero *d_sink first to read that XOR itself).  Its
 * bandwidth is the control that GEMV bandwidths are compared with ("Bonsai 2
 * 27B" page, section 8: the practical ceiling measured by a read-only
 * streaming kernel; "Kipp Benchmarks", decode is weight-bandwidth-bound).
 *  - bytes: a positive multiple of 16.  d_src, d_sink: 16-byte aligned
 *    device memory owned by the caller.
 *  - stage_bytes: a multiple of 16 in [1024, 98304]; stages: 1..8; the ring
 *    (stages x stage_bytes plus 16 bytes of barriers per stage and 16 more)
 *    must fit 227 KB of shared memory.
 *  - Errors: KQ_ERR_INVALID_ARG, KQ_ERR_SHAPE, KQ_ERR_ALIGNMENT, KQ_ERR_CUDA;
 *    a bounded device wait that expires sets KQ_ERR_TIMEOUT for
 *    kq_device_status. */
int kq_stream_read(const void* d_src, int64_t bytes, int32_t stage_bytes, int32_t stages, uint32_t* d_sink,
                   void* stream);

/* Self-test of the library's bounded device waits (an addition of this
 * library, no counterpart on the pages).  Enqueues on `stream` one CTA whose
 * thread waits, with the same bounded wait every kernel here uses, on an
 * mbarrier phase that nothing completes; after limit_cycles SM clock cycles
 * (1 .. about 2e9, one second) the wait gives up and KQ_ERR_TIMEOUT is
 * recorded for kq_device_status, exactly as when a kernel's copy or peer
 * never arrives.  The kernel then returns: nothing faults or hangs, and the
 * GPU context stays usable.  Errors: KQ_ERR_INVALID_ARG (limit out of
 * range), KQ_ERR_CUDA (launch). */
int kq_selftest_bounded_wait(int64_t limit_cycles, void* stream);

/* ---- PQ2_0 consumer at one activation row ------------------------------------ */

/* Two consumers compute PQ2_0 products at one activation row (kq_gemv_pq2_0,
 * kq_gemm_splitk and kq_gemm_splitk_noalloc with m = 1, and kq_decode_step of
 * PQ2_0 plans without links); both give results within the same bound (the
 * weights are never rounded) and are deterministic.
 *  - KQ_PQ2_0_MMA_SYNC (the default): the streaming kernel's warp-level
 *    tensor-core consumer (mma.sync, fp16 code values in registers, the
 *    transformed activation as an fp16 high/low pair).
 *  - KQ_PQ2_0_TCGEN05: a 5th-generation tensor-core consumer (tcgen05.mma
 *    kind::f8f6f4): the codes masked into e4m3 values in tensor memory, the
 *    transformed activation as four e4m3 planes (relative error 2^-16), one
 *    MMA per 128 rows x 32 weights into per-block accumulators.  It needs
 *    fewer integer operations per code but, measured on GB300, streams the
 *    Bonsai-27B-shaped step slower than the default (its per-slot handoffs
 *    between warps dominate), so it is opt-in.
 * The setting is process-wide and applies to calls made after it returns.
 * Errors: KQ_ERR_INVALID_ARG for an unknown value. */
typedef enum { KQ_PQ2_0_MMA_SYNC = 0, KQ_PQ2_0_TCGEN05 = 1 } kq_pq2_0_consumer;
int kq_set_pq2_0_consumer(int consumer);
int kq_get_pq2_0_consumer(void);

/* ---- device status --------------------------------------------------------- */

/* binaryVersion (major*10 + minor) of the streaming kernel as loaded on the
 * current device: 103 for the sm_103a code this library is built with.  A
 * caller that records performance can refuse any other value. */
int kq_kernel_binary_version(int* version);

/* Synchronises the current device and returns the status word that kernels
 * set when a bounded wait expired (KQ_ERR_TIMEOUT) or a device quantizer met
 * a non-finite weight (KQ_ERR_NONFINITE) or an fp16 overflow (KQ_ERR_RANGE);
 * KQ_OK if none.  clear != 0 resets the word. */
int kq_device_status(int clear);

#ifdef __cplusplus
}
#endif

#endif /* KQ_H */
