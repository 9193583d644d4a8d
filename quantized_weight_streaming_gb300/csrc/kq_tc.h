// Host entry points of the tensor-core (tcgen05) small-batch GEMM in kq_tc.cu.
#pragma once

#include <cstddef>
#include <cstdint>

#include "kq.h"

namespace kq {

constexpr int kTcMaxM = 64;      // activation rows per call (B holds 2 x 64 fp16 rows)
constexpr int kTcMaxK = 32768;   // the activation prologue stages one fp32 row in shared memory
// kq_gemm_small_m uses the tensor cores from this many rows on: the
// streaming kernel reads the weights once per 4 rows, the tensor-core GEMM
// once at any M, so it wins from the second streaming pass on (Q8_0, PQ2_0);
// scale4's streaming passes are half as long, so from the third.
constexpr int tc_min_m(int fmt) { return fmt == KQ_SCALE4 ? 9 : 5; }

// Validates m and k for the tensor-core path (the descriptor is checked by the caller).
int tc_check(const kq_qmat* W, int64_t m);
// Workspace bytes of tc_gemm (splits 0 = automatic).
size_t tc_workspace_bytes(const kq_qmat* W, int64_t m, int splits);
// Y[m][n] = X W^T (X rotated per 128-block for PQ2_0) on the tensor cores.
int tc_gemm(const kq_qmat* W, const float* d_X, int64_t m, float* d_Y, int splits, void* d_ws, size_t ws_bytes,
            void* stream);
// Status word of the tensor-core kernels (bit s set = status s seen); -1 if it cannot be read.
int read_tc_status(int clear);

}  // namespace kq
