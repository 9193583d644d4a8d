// Host-side helpers shared by the translation units of libkq.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include "kq.h"

namespace kq {

// Records a one-line reason for the calling thread and returns `status`.
int fail(int status, const char* fmt, ...);
// Clears the thread's last error (called on entry of every public function).
void clear_error();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Weights per block; PTQ1_0 (a storage format) has the PQ2_0 planes.
inline int64_t block_of(int fmt) {
  return (fmt == KQ_Q8_0 || fmt == KQ_SCALE4) ? 32 : ((fmt == KQ_PQ2_0 || fmt == KQ_PTQ1_0) ? 128 : 0);
}
inline int plane_format(int fmt) { return fmt == KQ_PTQ1_0 ? KQ_PQ2_0 : fmt; }
inline int64_t block_bytes(int fmt) { return fmt == KQ_PTQ1_0 ? 28 : (fmt == KQ_SCALE4 ? 18 : 34); }
inline int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }
inline int64_t scale_stride(int fmt, int64_t k) { return round_up(k / block_of(fmt), 8); }
inline int64_t code_row_bytes(int fmt, int64_t k) { return fmt == KQ_Q8_0 ? k : (fmt == KQ_SCALE4 ? k / 2 : k / 4); }

// Checks a kq_qmat descriptor (format, shape, plane pointers and alignment).
int check_qmat(const kq_qmat* W, int expect_fmt);

// The one-launch Q8_0 GEMV (kq_direct.cu): taken by the automatic choice
// (splits = 0) at one activation row, fp32 or fp16 chain, for k up to 4096
// and at most kGemvDirectMaxBytes of codes; it needs no workspace.
constexpr int64_t kGemvDirectMaxBytes = 20ll << 20;
bool gemv_direct_applies(const kq_qmat* W, int64_t m);
// d_x / d_y: fp32, or fp16 with io16 (the fp16 chain).
int gemv_direct(const kq_qmat* W, const void* d_x, void* d_y, bool io16, void* stream);

}  // namespace kq

#define KQ_CUDA_TRY(expr)                                                                           \
  do {                                                                                              \
    cudaError_t kq_err_ = (expr);                                                                   \
    if (kq_err_ != cudaSuccess)                                                                     \
      return ::kq::fail(KQ_ERR_CUDA, "%s: %s", #expr, cudaGetErrorString(kq_err_));                 \
  } while (0)
