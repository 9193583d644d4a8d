// Host half of libkq: status strings, per-thread error text, layout queries,
// the offline host quantizers and the host blockwise Hadamard transform.
//
// Formats: Q8_0 ("Kipp Architecture", "Weight quantization": 32-weight
// blocks, fp16 d, int8 q, value d*q, quantized against the fp16-rounded
// scale) and PQ2_0 ("Bonsai 2 27B - ternary g128 + blockwise Hadamard",
// section 3.1: 128-weight 34-byte blocks, 2-bit codes at bit 2*(j%4), value
// (q-1)*d, d = max|w|, q = round(w/d)+1).  Rounding of w/d is half away from
// zero, decided on the FP64 quotient of the two floats.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <string>
#include <vector>

#include "kq_internal.h"

namespace kq {

static thread_local char g_last_error[512] = {0};

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

void clear_error() { g_last_error[0] = 0; }

int check_qmat(const kq_qmat* W, int expect_fmt) {
  if (!W) return fail(KQ_ERR_INVALID_ARG, "W is NULL");
  if (W->fmt != KQ_Q8_0 && W->fmt != KQ_PQ2_0 && W->fmt != KQ_SCALE4)
    return fail(KQ_ERR_INVALID_ARG, "unknown matrix format %d", W->fmt);
  if (expect_fmt >= 0 && W->fmt != expect_fmt)
    return fail(KQ_ERR_INVALID_ARG, "format %d given to an entry point for format %d", W->fmt, expect_fmt);
  if (W->n < 1) return fail(KQ_ERR_SHAPE, "n = %lld < 1", (long long)W->n);
  int64_t bs = block_of(W->fmt);
  if (W->k < bs || W->k % bs != 0)
    return fail(KQ_ERR_SHAPE, "k = %lld is not a positive multiple of %lld", (long long)W->k, (long long)bs);
  if (W->fmt == KQ_PQ2_0) {
    if (W->had_block != 128 && W->had_block != 1024)
      return fail(KQ_ERR_UNSUPPORTED, "had_block = %d (PQ2_0 takes 128 or 1024)", W->had_block);
    if (W->k % W->had_block != 0)
      return fail(KQ_ERR_SHAPE, "k = %lld is not a multiple of had_block = %d", (long long)W->k, W->had_block);
  } else {
    if (W->had_block != 0) return fail(KQ_ERR_UNSUPPORTED, "had_block = %d (this format takes 0)", W->had_block);
    if (W->signs) return fail(KQ_ERR_UNSUPPORTED, "signs given for a matrix without rotation");
  }
  if (!W->codes || !W->scales) return fail(KQ_ERR_INVALID_ARG, "NULL plane pointer");
  if (!aligned16(W->codes) || !aligned16(W->scales)) return fail(KQ_ERR_ALIGNMENT, "plane not 16-byte aligned");
  if (W->signs && !aligned16(W->signs)) return fail(KQ_ERR_ALIGNMENT, "signs not 16-byte aligned");
  return KQ_OK;
}

}  // namespace kq

using namespace kq;

extern "C" {

const char* kq_status_string(int s) {
  switch (s) {
    case KQ_OK: return "ok";
    case KQ_ERR_INVALID_ARG: return "invalid argument";
    case KQ_ERR_SHAPE: return "invalid shape";
    case KQ_ERR_ALIGNMENT: return "misaligned pointer";
    case KQ_ERR_NONFINITE: return "non-finite weight";
    case KQ_ERR_RANGE: return "scale out of fp16 range";
    case KQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KQ_ERR_CUDA: return "CUDA error";
    case KQ_ERR_TIMEOUT: return "bounded device wait expired";
    case KQ_ERR_UNSUPPORTED: return "unsupported";
    default: return "unknown status";
  }
}

const char* kq_last_error(void) { return g_last_error; }

int kq_version(void) { return 2; }

int64_t kq_block_size(int fmt) { return block_of(fmt); }

int64_t kq_blocks_bytes(int fmt, int64_t n, int64_t k) {
  int64_t bs = block_of(fmt);
  if (!bs || n < 0 || k < 0 || k % bs) return 0;
  return n * (k / bs) * block_bytes(fmt);
}

int64_t kq_scale_stride(int fmt, int64_t k) {
  int64_t bs = block_of(fmt);
  if (!bs || k < 0 || k % bs) return 0;
  return scale_stride(fmt, k);
}

int64_t kq_codes_bytes(int fmt, int64_t n, int64_t k) {
  int64_t bs = block_of(fmt);
  if (!bs || n < 0 || k < 0 || k % bs) return 0;
  return n * code_row_bytes(fmt, k);
}

int64_t kq_scales_bytes(int fmt, int64_t n, int64_t k) {
  int64_t bs = block_of(fmt);
  if (!bs || n < 0 || k < 0 || k % bs) return 0;
  return n * scale_stride(fmt, k) * 2;
}

// ---------------------------------------------------------------------------
// Host quantizers
// ---------------------------------------------------------------------------

static inline uint16_t half_bits_rn(float v) { return __half_as_ushort(__float2half_rn(v)); }
static inline float half_to_float(uint16_t h) { return __half2float(__ushort_as_half(h)); }

static int check_host_weights(const float* w, int64_t n, int64_t k, int64_t bs, const void* out) {
  if (!w || !out) return fail(KQ_ERR_INVALID_ARG, "NULL pointer");
  if (n < 1 || k < bs || k % bs)
    return fail(KQ_ERR_SHAPE, "n = %lld, k = %lld (k must be a positive multiple of %lld)", (long long)n,
                (long long)k, (long long)bs);
  for (int64_t i = 0; i < n * k; ++i)
    if (!std::isfinite(w[i])) return fail(KQ_ERR_NONFINITE, "weight %lld is not finite", (long long)i);
  return KQ_OK;
}

int kq_quantize_q8_0(const float* w, int64_t n, int64_t k, void* blocks) {
  clear_error();
  if (int s = check_host_weights(w, n, k, 32, blocks)) return s;
  const int64_t nb = k / 32;
  // First pass: scales only, so that a range error leaves the output untouched.
  std::vector<uint16_t> dh(static_cast<size_t>(n * nb));
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* src = w + r * k + b * 32;
      float amax = 0.f;
      for (int j = 0; j < 32; ++j) amax = std::fmax(amax, std::fabs(src[j]));
      uint16_t h = half_bits_rn(amax / 127.0f);
      if ((h & 0x7C00u) == 0x7C00u)
        return fail(KQ_ERR_RANGE, "row %lld block %lld: scale %g overflows fp16", (long long)r, (long long)b,
                    (double)(amax / 127.0f));
      dh[static_cast<size_t>(r * nb + b)] = h;
    }
  }
  uint8_t* out = static_cast<uint8_t*>(blocks);
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* src = w + r * k + b * 32;
      uint8_t* blk = out + (r * nb + b) * 34;
      uint16_t h = dh[static_cast<size_t>(r * nb + b)];
      double d = half_to_float(h);
      blk[0] = static_cast<uint8_t>(h & 0xFF);
      blk[1] = static_cast<uint8_t>(h >> 8);
      for (int j = 0; j < 32; ++j) {
        long q = 0;
        if (d != 0.0) q = std::lround(static_cast<double>(src[j]) / d);
        q = q > 127 ? 127 : (q < -127 ? -127 : q);
        blk[2 + j] = static_cast<uint8_t>(static_cast<int8_t>(q));
      }
    }
  }
  return KQ_OK;
}

int kq_quantize_pq2_0(const float* w_rot, int64_t n, int64_t k, void* blocks) {
  clear_error();
  if (int s = check_host_weights(w_rot, n, k, 128, blocks)) return s;
  const int64_t nb = k / 128;
  std::vector<uint16_t> dh(static_cast<size_t>(n * nb));
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* src = w_rot + r * k + b * 128;
      float amax = 0.f;
      for (int j = 0; j < 128; ++j) amax = std::fmax(amax, std::fabs(src[j]));
      uint16_t h = half_bits_rn(amax);
      if ((h & 0x7C00u) == 0x7C00u)
        return fail(KQ_ERR_RANGE, "row %lld block %lld: scale %g overflows fp16", (long long)r, (long long)b,
                    (double)amax);
      dh[static_cast<size_t>(r * nb + b)] = h;
    }
  }
  uint8_t* out = static_cast<uint8_t*>(blocks);
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* src = w_rot + r * k + b * 128;
      uint8_t* blk = out + (r * nb + b) * 34;
      uint16_t h = dh[static_cast<size_t>(r * nb + b)];
      double d = half_to_float(h);
      blk[0] = static_cast<uint8_t>(h & 0xFF);
      blk[1] = static_cast<uint8_t>(h >> 8);
      std::memset(blk + 2, 0, 32);
      for (int j = 0; j < 128; ++j) {
        long t = 0;
        if (d != 0.0) t = std::lround(static_cast<double>(src[j]) / d);
        t = t > 1 ? 1 : (t < -1 ? -1 : t);
        blk[2 + j / 4] |= static_cast<uint8_t>((t + 1) << (2 * (j % 4)));
      }
    }
  }
  return KQ_OK;
}

int kq_quantize_scale4(const float* w, int64_t n, int64_t k, void* blocks) {
  clear_error();
  if (int s = check_host_weights(w, n, k, 32, blocks)) return s;
  const int64_t nb = k / 32;
  // First pass: scales only, so that a range error leaves the output untouched.
  std::vector<uint16_t> dh(static_cast<size_t>(n * nb));
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* src = w + r * k + b * 32;
      float m = 0.f;  // the weight of largest magnitude, with its sign, the first on a tie
      for (int j = 0; j < 32; ++j)
        if (std::fabs(src[j]) > std::fabs(m)) m = src[j];
      uint16_t h = half_bits_rn(m / -8.0f);
      if ((h & 0x7C00u) == 0x7C00u)
        return fail(KQ_ERR_RANGE, "row %lld block %lld: scale %g overflows fp16", (long long)r, (long long)b,
                    (double)(m / -8.0f));
      dh[static_cast<size_t>(r * nb + b)] = h;
    }
  }
  uint8_t* out = static_cast<uint8_t*>(blocks);
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* src = w + r * k + b * 32;
      uint8_t* blk = out + (r * nb + b) * 18;
      const uint16_t h = dh[static_cast<size_t>(r * nb + b)];
      const double d = half_to_float(h);
      blk[0] = static_cast<uint8_t>(h & 0xFF);
      blk[1] = static_cast<uint8_t>(h >> 8);
      std::memset(blk + 2, 0, 16);
      for (int j = 0; j < 32; ++j) {
        long q = 8;
        if (d != 0.0) q = std::lround(static_cast<double>(src[j]) / d) + 8;
        q = q > 15 ? 15 : (q < 0 ? 0 : q);
        blk[2 + j / 2] |= static_cast<uint8_t>(q << (4 * (j % 2)));
      }
    }
  }
  return KQ_OK;
}

// PTQ1_0: the PQ2_0 scale and trits, then the base-3 packing.
static void ptq1_0_place(int e, int* byte, int* n) {
  if (e < 80) {
    *byte = e % 16;
    *n = e / 16;
  } else if (e < 120) {
    *byte = 16 + (e - 80) % 8;
    *n = (e - 80) / 8;
  } else {
    *byte = 24 + (e - 120) % 2;
    *n = (e - 120) / 2;
  }
}

int kq_quantize_ptq1_0(const float* w_rot, int64_t n, int64_t k, void* blocks) {
  clear_error();
  if (int s = check_host_weights(w_rot, n, k, 128, blocks)) return s;
  const int64_t nb = k / 128;
  // the scales first, so that a range error leaves the output untouched
  std::vector<uint16_t> dh(static_cast<size_t>(n * nb));
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* src = w_rot + r * k + b * 128;
      float amax = 0.f;
      for (int j = 0; j < 128; ++j) amax = std::fmax(amax, std::fabs(src[j]));
      uint16_t h = half_bits_rn(amax);
      if ((h & 0x7C00u) == 0x7C00u)
        return fail(KQ_ERR_RANGE, "row %lld block %lld: scale %g overflows fp16", (long long)r, (long long)b,
                    (double)amax);
      dh[static_cast<size_t>(r * nb + b)] = h;
    }
  }
  uint8_t* out = static_cast<uint8_t*>(blocks);
  for (int64_t r = 0; r < n; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const float* src = w_rot + r * k + b * 128;
      uint8_t* blk = out + (r * nb + b) * 28;
      const uint16_t h = dh[static_cast<size_t>(r * nb + b)];
      const double d = half_to_float(h);
      int v[26] = {0};  // each byte's trits as a base-3 number, first trit most significant
      int trits[26][5] = {};
      for (int j = 0; j < 128; ++j) {
        long t = 0;
        if (d != 0.0) t = std::lround(static_cast<double>(src[j]) / d);
        t = t > 1 ? 1 : (t < -1 ? -1 : t);
        int byte, tn;
        ptq1_0_place(j, &byte, &tn);
        trits[byte][tn] = static_cast<int>(t + 1);
      }
      for (int i = 0; i < 26; ++i) {
        for (int tn = 0; tn < 5; ++tn) v[i] = v[i] * 3 + trits[i][tn];
        blk[i] = static_cast<uint8_t>((256 * v[i] + 242) / 243);  // ceil(256 v / 243)
      }
      blk[26] = static_cast<uint8_t>(h & 0xFF);
      blk[27] = static_cast<uint8_t>(h >> 8);
    }
  }
  return KQ_OK;
}

// ---------------------------------------------------------------------------
// Host blockwise Hadamard: in-place FP64 butterflies (natural Sylvester order),
// then one FP64 multiply by 1/sqrt(block) and one rounding to fp32.
// ---------------------------------------------------------------------------

int kq_hadamard_blockwise_host(const float* in, float* out, int64_t rows, int64_t k, int32_t block) {
  return kq_rotate_blockwise_host(in, out, rows, k, block, nullptr);
}

int kq_rotate_blockwise_host(const float* in, float* out, int64_t rows, int64_t k, int32_t block,
                             const int8_t* signs) {
  clear_error();
  if (!in || !out) return fail(KQ_ERR_INVALID_ARG, "NULL pointer");
  if (block < 1 || (block & (block - 1)) != 0) return fail(KQ_ERR_SHAPE, "block %d is not a power of two", block);
  if (rows < 1 || k < block || k % block)
    return fail(KQ_ERR_SHAPE, "rows = %lld, k = %lld, block = %d", (long long)rows, (long long)k, block);
  if (signs)
    for (int64_t c = 0; c < k; ++c)
      if (signs[c] != 1 && signs[c] != -1) return fail(KQ_ERR_INVALID_ARG, "signs[%lld] = %d", (long long)c, signs[c]);
  const double scale = 1.0 / std::sqrt(static_cast<double>(block));
  std::vector<double> v(static_cast<size_t>(block));
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b0 = 0; b0 < k; b0 += block) {
      const float* src = in + r * k + b0;
      for (int32_t i = 0; i < block; ++i) v[i] = signs ? (double)signs[b0 + i] * src[i] : (double)src[i];
      for (int32_t h = 1; h < block; h <<= 1) {
        for (int32_t i = 0; i < block; i += 2 * h) {
          for (int32_t j = i; j < i + h; ++j) {
            double a = v[j], c = v[j + h];
            v[j] = a + c;
            v[j + h] = a - c;
          }
        }
      }
      float* dst = out + r * k + b0;
      for (int32_t i = 0; i < block; ++i) dst[i] = static_cast<float>(scale * v[i]);
    }
  }
  return KQ_OK;
}

// One decode step with host buffers: the copies around kq_decode_step, on
// the caller's stream (plain cudaMemcpyAsync; pinned buffers make them
// asynchronous).  Uses the plan only through its public queries.
//
// A plan of one stage only writes its outputs (no matrix reads an earlier
// one's), so when h_y is page-locked host memory the step stores them through
// h_y's device mapping as each row block finishes, and the copy back after the
// step disappears from the step's critical path.
// The device mapping of a page-locked host buffer (cudaHostAlloc or
// cudaHostRegister) if it is 16-byte aligned, else nullptr (pageable memory:
// the caller's copies serve it).
static float* mapped_device_pointer(const float* h) {
  cudaPointerAttributes pa{};
  if (cudaPointerGetAttributes(&pa, h) != cudaSuccess) {
    (void)cudaGetLastError();  // not a pointer the runtime knows
    return nullptr;
  }
  if (pa.type == cudaMemoryTypeHost && pa.devicePointer && aligned16(pa.devicePointer))
    return static_cast<float*>(pa.devicePointer);
  return nullptr;
}

int kq_decode_step_host(kq_plan* plan, const float* h_x_packed, float* h_y_packed, float* d_x_packed,
                        float* d_y_packed, void* d_ws, size_t ws_bytes, void* stream) {
  clear_error();
  if (!plan) return fail(KQ_ERR_INVALID_ARG, "NULL plan");
  int64_t xf = 0, yf = 0;
  if (int s = kq_decode_plan_sizes(plan, &xf, &yf, nullptr)) return s;
  if ((!h_x_packed && xf > 0) || !h_y_packed) return fail(KQ_ERR_INVALID_ARG, "NULL host buffer");
  if ((!d_x_packed && xf > 0) || !d_y_packed) return fail(KQ_ERR_INVALID_ARG, "NULL device buffer");
  if (!aligned16(d_x_packed) || !aligned16(d_y_packed)) return fail(KQ_ERR_ALIGNMENT, "x or y not 16-byte aligned");
  const size_t need = kq_decode_workspace_bytes(plan);
  if (need > 0 && (!d_ws || ws_bytes < need))
    return fail(KQ_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", need, d_ws ? ws_bytes : (size_t)0);
  if (need > 0 && !aligned16(d_ws)) return fail(KQ_ERR_ALIGNMENT, "workspace not 16-byte aligned");
  int32_t stages = 0;
  if (int s = kq_decode_plan_stages(plan, &stages, nullptr)) return s;
  // Page-locked host buffers with a 16-byte-aligned device mapping are read
  // (x) or written (y, one-stage plans only: no stage reads them back) by the
  // kernel itself, so no copy runs before or after it.
  float* y_direct = stages == 1 ? mapped_device_pointer(h_y_packed) : nullptr;
  const float* x_direct = xf > 0 ? mapped_device_pointer(h_x_packed) : nullptr;
  cudaStream_t st = (cudaStream_t)stream;
  if (xf > 0 && !x_direct)
    KQ_CUDA_TRY(cudaMemcpyAsync(d_x_packed, h_x_packed, (size_t)xf * sizeof(float), cudaMemcpyHostToDevice, st));
  const float* x_in = x_direct ? x_direct : d_x_packed;
  if (y_direct) return kq_decode_step(plan, x_in, y_direct, d_ws, ws_bytes, stream);
  if (int s = kq_decode_step(plan, x_in, d_y_packed, d_ws, ws_bytes, stream)) return s;
  KQ_CUDA_TRY(cudaMemcpyAsync(h_y_packed, d_y_packed, (size_t)yf * sizeof(float), cudaMemcpyDeviceToHost, st));
  return KQ_OK;
}

}  // extern "C"
