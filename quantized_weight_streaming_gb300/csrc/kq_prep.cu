// Device weight preparation of libkq: AoS block -> plane repacking, the
// device quantizers, the blockwise Walsh-Hadamard transform and the debug
// dequantizer.  None of these is on the per-token path; they prepare weights
// once ("rotate, then quantize": Bonsai 2 27B - ternary g128 + blockwise
// Hadamard, sections 3.1 and 4.2).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "kq_device.cuh"
#include "kq_internal.h"

namespace kq {

// Status word of this translation unit (KQ_ERR_* bits, see kq_device_status).
__device__ unsigned int g_prep_status = 0;

__device__ __forceinline__ void prep_flag(int status) { atomicOr(&g_prep_status, 1u << status); }

// --------------------------------------------------------------------------
// AoS 34-byte blocks -> planes.  Both formats keep the code bytes in block
// order, so the codes plane is the concatenation of the blocks' code bytes.
// --------------------------------------------------------------------------
// A block is the fp16 scale then cb code bytes (32 for Q8_0 and PQ2_0, 16 for
// SCALE4); the code bytes of a row's blocks are concatenated in the plane.
__global__ void prepare_kernel(const uint8_t* __restrict__ blocks, int64_t n, int64_t nb, int64_t sstride, int cb,
                               uint8_t* __restrict__ codes, uint16_t* __restrict__ scales) {
  int64_t total = n * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / nb, b = i % nb;
    const uint8_t* blk = blocks + i * (2 + cb);
    scales[r * sstride + b] = (uint16_t)(blk[0] | (blk[1] << 8));
    uint8_t* dst = codes + i * cb;  // row r, bytes b*cb .. (row stride nb*cb)
    for (int j = 0; j < cb; ++j) dst[j] = blk[2 + j];
  }
}

// PTQ1_0 block -> PQ2_0 planes: trit n of byte q is ((q 3^n) mod 256) * 3 / 256;
// element e sits in byte e%16 (e < 80, trit e/16), 16+(e-80)%8 (e < 120,
// trit (e-80)/8) or 24+(e-120)%2 (trit (e-120)/2); the fp16 scale is last.
// One thread per block; the trit becomes the PQ2_0 code of the same element.
__global__ void prepare_ptq1_0_kernel(const uint8_t* __restrict__ blocks, int64_t n, int64_t nb, int64_t sstride,
                                      uint8_t* __restrict__ codes, uint16_t* __restrict__ scales) {
  int64_t total = n * nb;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / nb, b = i % nb;
    const uint8_t* blk = blocks + i * 28;
    scales[r * sstride + b] = (uint16_t)(blk[26] | (blk[27] << 8));
    uint32_t words[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int e = 0; e < 128; ++e) {
      int byte, tn;
      if (e < 80) {
        byte = e % 16;
        tn = e / 16;
      } else if (e < 120) {
        byte = 16 + (e - 80) % 8;
        tn = (e - 80) / 8;
      } else {
        byte = 24 + (e - 120) % 2;
        tn = (e - 120) / 2;
      }
      const uint32_t pw[5] = {1u, 3u, 9u, 27u, 81u};
      const uint32_t trit = (((uint32_t)blk[byte] * pw[tn]) & 0xFFu) * 3u >> 8;
      words[e / 16] |= trit << (2 * (e % 16));
    }
    uint32_t* dst = reinterpret_cast<uint32_t*>(codes + i * 32);  // row r, bytes b*32 .. (row stride nb*32)
#pragma unroll
    for (int w = 0; w < 8; ++w) dst[w] = words[w];
  }
}

__global__ void zero_scale_padding_kernel(int64_t n, int64_t nb, int64_t sstride, uint16_t* __restrict__ scales) {
  int64_t pad = sstride - nb;
  int64_t total = n * pad;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x)
    scales[(i / pad) * sstride + nb + i % pad] = 0;
}

// --------------------------------------------------------------------------
// Device quantizers: one warp per block.  Same arithmetic as the host ones:
// fp32 amax (and fp32 quotient amax/127 for Q8_0), fp16 round-to-nearest-even,
// codes from the FP64 quotient w/d rounded half away from zero.
// --------------------------------------------------------------------------
__global__ void quantize_q8_0_kernel(const float* __restrict__ w, int64_t n, int64_t k, int64_t sstride,
                                     int8_t* __restrict__ codes, uint16_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = k / 32;
  const int64_t total = n * nb;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t i = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; i < total; i += warps) {
    int64_t r = i / nb, b = i % nb;
    float v = w[r * k + b * 32 + lane];
    if (!isfinite(v)) prep_flag(KQ_ERR_NONFINITE);
    float a = fabsf(v);
#pragma unroll
    for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    __half dh = __float2half_rn(a / 127.0f);
    if (__hisinf(dh)) prep_flag(KQ_ERR_RANGE);
    double d = (double)__half2float(dh);
    double q = 0.0;
    if (d != 0.0) q = fmin(127.0, fmax(-127.0, round((double)v / d)));
    codes[r * k + b * 32 + lane] = (int8_t)q;
    if (lane == 0) scales[r * sstride + b] = __half_as_ushort(dh);
  }
}

// SCALE4: lane j of the warp holds weight j of the 32-block; the signed
// weight of largest magnitude (the first on a tie) by a warp reduction on
// (magnitude, -index).
__global__ void quantize_scale4_kernel(const float* __restrict__ w, int64_t n, int64_t k, int64_t sstride,
                                       uint8_t* __restrict__ codes, uint16_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = k / 32;
  const int64_t total = n * nb;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t i = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; i < total; i += warps) {
    int64_t r = i / nb, b = i % nb;
    const float v = w[r * k + b * 32 + lane];
    if (!isfinite(v)) prep_flag(KQ_ERR_NONFINITE);
    float a = fabsf(v);
    int at = lane;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float a2 = __shfl_xor_sync(0xffffffffu, a, o);
      const int at2 = __shfl_xor_sync(0xffffffffu, at, o);
      if (a2 > a || (a2 == a && at2 < at)) {
        a = a2;
        at = at2;
      }
    }
    const float m = __shfl_sync(0xffffffffu, v, at);
    const __half dh = __float2half_rn(m / -8.0f);
    if (__hisinf(dh)) prep_flag(KQ_ERR_RANGE);
    const double d = (double)__half2float(dh);
    int q = 8;
    if (d != 0.0) q = (int)fmin(15.0, fmax(0.0, round((double)v / d) + 8.0));
    // two lanes per byte: the even lane's nibble low, the odd lane's high
    const int other = __shfl_xor_sync(0xffffffffu, q, 1);
    if (!(lane & 1)) codes[r * (k / 2) + b * 16 + lane / 2] = (uint8_t)(q | (other << 4));
    if (lane == 0) scales[r * sstride + b] = __half_as_ushort(dh);
  }
}

__global__ void quantize_pq2_0_kernel(const float* __restrict__ w, int64_t n, int64_t k, int64_t sstride,
                                      uint8_t* __restrict__ codes, uint16_t* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = k / 128;
  const int64_t total = n * nb;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t i = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; i < total; i += warps) {
    int64_t r = i / nb, b = i % nb;
    // lane l holds elements 4l..4l+3, i.e. exactly the four codes of byte l
    float4 v = *reinterpret_cast<const float4*>(w + r * k + b * 128 + 4 * lane);
    if (!isfinite(v.x) || !isfinite(v.y) || !isfinite(v.z) || !isfinite(v.w)) prep_flag(KQ_ERR_NONFINITE);
    float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 16; o; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    __half dh = __float2half_rn(a);
    if (__hisinf(dh)) prep_flag(KQ_ERR_RANGE);
    double d = (double)__half2float(dh);
    float e[4] = {v.x, v.y, v.z, v.w};
    unsigned byte = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      double t = 0.0;
      if (d != 0.0) t = fmin(1.0, fmax(-1.0, round((double)e[j] / d)));
      byte |= (unsigned)((int)t + 1) << (2 * j);
    }
    codes[r * (k / 4) + b * 32 + lane] = (uint8_t)byte;
    if (lane == 0) scales[r * sstride + b] = __half_as_ushort(dh);
  }
}

// --------------------------------------------------------------------------
// Blockwise Walsh-Hadamard transform in FP64 (natural Sylvester order), then
// one FP64 multiply by 1/sqrt(block) and one rounding to fp32.
// --------------------------------------------------------------------------

// block == 128: one warp per block, four elements per lane.
// signs (NULL: none) hold one +-1 per position of a row of k = bpr blocks;
// the flip is exact in FP64 and comes before the butterflies.
__global__ void hadamard128_f64_kernel(const float* __restrict__ in, float* __restrict__ out, int64_t nblocks,
                                       double scale, const int8_t* __restrict__ signs, int64_t bpr) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t i = (int64_t)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; i < nblocks; i += warps) {
    float4 f = *reinterpret_cast<const float4*>(in + i * 128 + 4 * lane);
    double v[4] = {f.x, f.y, f.z, f.w};
    if (signs) {
      const char4 s4 = *reinterpret_cast<const char4*>(signs + (i % bpr) * 128 + 4 * lane);
      v[0] *= (double)s4.x;
      v[1] *= (double)s4.y;
      v[2] *= (double)s4.z;
      v[3] *= (double)s4.w;
    }
    // strides 1 and 2 inside the lane
    double a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
    v[0] = a0 + a2;
    v[2] = a0 - a2;
    v[1] = a1 + a3;
    v[3] = a1 - a3;
    // strides 4 .. 64 across lanes
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        double p = __shfl_xor_sync(0xffffffffu, v[t], m);
        v[t] = (lane & m) ? (p - v[t]) : (v[t] + p);
      }
    }
    float4 o;
    o.x = (float)(scale * v[0]);
    o.y = (float)(scale * v[1]);
    o.z = (float)(scale * v[2]);
    o.w = (float)(scale * v[3]);
    *reinterpret_cast<float4*>(out + i * 128 + 4 * lane) = o;
  }
}

// Any power-of-two block up to 4096: one CTA per block, butterflies in shared memory.
__global__ void hadamard_f64_smem_kernel(const float* __restrict__ in, float* __restrict__ out, int64_t nblocks,
                                         int block, double scale, const int8_t* __restrict__ signs, int64_t bpr) {
  extern __shared__ double buf[];
  for (int64_t i = blockIdx.x; i < nblocks; i += gridDim.x) {
    const int8_t* sg = signs ? signs + (i % bpr) * block : nullptr;
    for (int j = threadIdx.x; j < block; j += blockDim.x)
      buf[j] = sg ? (double)sg[j] * (double)in[i * block + j] : (double)in[i * block + j];
    __syncthreads();
    for (int h = 1; h < block; h <<= 1) {
      for (int t = threadIdx.x; t < block / 2; t += blockDim.x) {
        int lo = (t / h) * 2 * h + (t % h);
        double a = buf[lo], c = buf[lo + h];
        buf[lo] = a + c;
        buf[lo + h] = a - c;
      }
      __syncthreads();
    }
    for (int j = threadIdx.x; j < block; j += blockDim.x) out[i * block + j] = (float)(scale * buf[j]);
    __syncthreads();
  }
}

// --------------------------------------------------------------------------
// Embedding lookup: rows of a quantized table, dequantized; a rotated PQ2_0
// table stores R e per row, so the lookup returns e = R^T z = S (H z)/sqrt(n)
// per n-block, the transform first, then the sign flip (the Bonsai page,
// section 4.2).  One CTA per token; PQ2_0 rows go through shared memory
// (k floats): each warp dequantizes and transforms 128-blocks (4 elements per
// lane), an 8-point pass joins them into 1024-blocks (H_1024 = H_8 (x)
// H_128), then the scale, the signs and the store.
// --------------------------------------------------------------------------
__global__ void embed_kernel(int fmt, const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                             int64_t n, int64_t k, int64_t sstride, const int32_t* __restrict__ ids, int64_t count,
                             int had, const int8_t* __restrict__ signs, float* __restrict__ out) {
  extern __shared__ float zrow[];  // k floats (PQ2_0)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  for (int64_t t = blockIdx.x; t < count; t += gridDim.x) {
    const int64_t id = ids[t];
    float* o = out + t * k;
    if (id < 0 || id >= n) {
      if (threadIdx.x == 0) prep_flag(KQ_ERR_RANGE);
      for (int64_t c = threadIdx.x; c < k; c += blockDim.x) o[c] = 0.f;
      continue;
    }
    const uint16_t* srow = scales + id * sstride;
    if (fmt == KQ_Q8_0) {
      const int8_t* q = reinterpret_cast<const int8_t*>(codes) + id * k;
      for (int64_t c = threadIdx.x; c < k; c += blockDim.x)
        o[c] = (float)q[c] * __half2float(__ushort_as_half(srow[c / 32]));
      continue;
    }
    if (fmt == KQ_SCALE4) {
      const uint8_t* q = codes + id * (k / 2);
      for (int64_t c = threadIdx.x; c < k; c += blockDim.x)
        o[c] = (float)((int)((q[c / 2] >> (4 * (c % 2))) & 15) - 8) * __half2float(__ushort_as_half(srow[c / 32]));
      continue;
    }
    // PQ2_0: words of 16 codes, element 16i + j at bits 2j of word i
    const uint32_t* w = reinterpret_cast<const uint32_t*>(codes + id * (k / 4));
    for (int64_t b = warp; b < k / 128; b += nwarps) {
      const float d = __half2float(__ushort_as_half(srow[b]));
      const uint32_t word = w[b * 8 + lane / 4];
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] = (float)((int)((word >> (2 * (4 * (lane & 3) + e))) & 3u) - 1) * d;
      float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
      v[0] = a0 + a2;
      v[2] = a0 - a2;
      v[1] = a1 + a3;
      v[3] = a1 - a3;
#pragma unroll
      for (int mk = 1; mk < 32; mk <<= 1) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float q = __shfl_xor_sync(0xffffffffu, v[e], mk);
          v[e] = (lane & mk) ? (q - v[e]) : (v[e] + q);
        }
      }
      *reinterpret_cast<float4*>(zrow + b * 128 + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
    }
    __syncthreads();
    if (had == 1024) {
      for (int64_t c = threadIdx.x; c < (k / 1024) * 128; c += blockDim.x) {
        float* col = zrow + (c / 128) * 1024 + (c % 128);
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
        for (int a = 0; a < 8; ++a) col[a * 128] = v[a];
      }
      __syncthreads();
    }
    const float scale = had == 1024 ? 0.03125f : 0.08838834764831845f;
    for (int64_t c = threadIdx.x; c < k; c += blockDim.x) {
      const float e = zrow[c] * scale;
      o[c] = signs ? e * (float)signs[c] : e;
    }
    __syncthreads();  // zrow is reused by the next token
  }
}

// --------------------------------------------------------------------------
// Debug dequantizer.
// --------------------------------------------------------------------------
__global__ void dequant_kernel(int fmt, const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales,
                               int64_t n, int64_t k, int64_t sstride, float* __restrict__ out) {
  const int64_t total = n * k;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    int64_t r = i / k, c = i % k;
    if (fmt == KQ_Q8_0) {
      float d = __half2float(__ushort_as_half(scales[r * sstride + c / 32]));
      out[i] = (float)(int8_t)codes[i] * d;
    } else if (fmt == KQ_SCALE4) {
      float d = __half2float(__ushort_as_half(scales[r * sstride + c / 32]));
      int q = (codes[r * (k / 2) + c / 2] >> (4 * (c % 2))) & 15;
      out[i] = (float)(q - 8) * d;
    } else {
      float d = __half2float(__ushort_as_half(scales[r * sstride + c / 128]));
      int code = (codes[r * (k / 4) + c / 4] >> (2 * (c % 4))) & 3;
      out[i] = (float)(code - 1) * d;
    }
  }
}

static int grid_for(int64_t work, int threads) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  int64_t g = (work + threads - 1) / threads;
  int64_t cap = (int64_t)sms * 8;
  return (int)(g < 1 ? 1 : (g > cap ? cap : g));
}

int read_prep_status(int clear) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_prep_status, sizeof(v));
  if (e != cudaSuccess) return -1;
  if (clear) {
    unsigned int z = 0;
    cudaMemcpyToSymbol(g_prep_status, &z, sizeof(z));
  }
  return (int)v;
}

}  // namespace kq

using namespace kq;

static int check_planes_out(int fmt, int64_t n, int64_t k, const void* codes, const void* scales) {
  int64_t bs = block_of(fmt);
  if (!bs) return fail(KQ_ERR_INVALID_ARG, "unknown format %d", fmt);
  if (n < 1 || k < bs || k % bs)
    return fail(KQ_ERR_SHAPE, "n = %lld, k = %lld (k must be a positive multiple of %lld)", (long long)n,
                (long long)k, (long long)bs);
  if (!codes || !scales) return fail(KQ_ERR_INVALID_ARG, "NULL plane pointer");
  if (!aligned16(codes) || !aligned16(scales)) return fail(KQ_ERR_ALIGNMENT, "plane not 16-byte aligned");
  return KQ_OK;
}

extern "C" {

int kq_prepare(int fmt, const void* d_blocks, int64_t n, int64_t k, void* d_codes, void* d_scales, void* stream) {
  clear_error();
  if (int s = check_planes_out(fmt, n, k, d_codes, d_scales)) return s;
  if (!d_blocks) return fail(KQ_ERR_INVALID_ARG, "NULL blocks");
  const int64_t nb = k / block_of(fmt), ss = scale_stride(plane_format(fmt), k);
  cudaStream_t st = (cudaStream_t)stream;
  if (fmt == KQ_PTQ1_0)
    prepare_ptq1_0_kernel<<<grid_for(n * nb, 256), 256, 0, st>>>((const uint8_t*)d_blocks, n, nb, ss,
                                                                 (uint8_t*)d_codes, (uint16_t*)d_scales);
  else
    prepare_kernel<<<grid_for(n * nb, 256), 256, 0, st>>>((const uint8_t*)d_blocks, n, nb, ss,
                                                          (int)(block_bytes(fmt) - 2), (uint8_t*)d_codes,
                                                          (uint16_t*)d_scales);
  KQ_CUDA_TRY(cudaGetLastError());
  if (ss > nb) {
    zero_scale_padding_kernel<<<grid_for(n * (ss - nb), 256), 256, 0, st>>>(n, nb, ss, (uint16_t*)d_scales);
    KQ_CUDA_TRY(cudaGetLastError());
  }
  return KQ_OK;
}

static int quantize_device(int fmt, const float* d_w, int64_t n, int64_t k, void* d_codes, void* d_scales,
                           void* stream) {
  clear_error();
  if (int s = check_planes_out(fmt, n, k, d_codes, d_scales)) return s;
  if (!d_w) return fail(KQ_ERR_INVALID_ARG, "NULL weights");
  if (!aligned16(d_w)) return fail(KQ_ERR_ALIGNMENT, "weights not 16-byte aligned");
  const int64_t nb = k / block_of(fmt), ss = scale_stride(fmt, k);
  cudaStream_t st = (cudaStream_t)stream;
  if (ss > nb) {
    zero_scale_padding_kernel<<<grid_for(n * (ss - nb), 256), 256, 0, st>>>(n, nb, ss, (uint16_t*)d_scales);
    KQ_CUDA_TRY(cudaGetLastError());
  }
  int grid = grid_for(n * nb * 32, 256);
  if (fmt == KQ_Q8_0)
    quantize_q8_0_kernel<<<grid, 256, 0, st>>>(d_w, n, k, ss, (int8_t*)d_codes, (uint16_t*)d_scales);
  else if (fmt == KQ_SCALE4)
    quantize_scale4_kernel<<<grid, 256, 0, st>>>(d_w, n, k, ss, (uint8_t*)d_codes, (uint16_t*)d_scales);
  else
    quantize_pq2_0_kernel<<<grid, 256, 0, st>>>(d_w, n, k, ss, (uint8_t*)d_codes, (uint16_t*)d_scales);
  KQ_CUDA_TRY(cudaGetLastError());
  return KQ_OK;
}

int kq_quantize_q8_0_device(const float* d_w, int64_t n, int64_t k, void* d_codes, void* d_scales, void* stream) {
  return quantize_device(KQ_Q8_0, d_w, n, k, d_codes, d_scales, stream);
}

int kq_quantize_pq2_0_device(const float* d_w_rot, int64_t n, int64_t k, void* d_codes, void* d_scales,
                             void* stream) {
  return quantize_device(KQ_PQ2_0, d_w_rot, n, k, d_codes, d_scales, stream);
}

int kq_quantize_scale4_device(const float* d_w, int64_t n, int64_t k, void* d_codes, void* d_scales, void* stream) {
  return quantize_device(KQ_SCALE4, d_w, n, k, d_codes, d_scales, stream);
}

int kq_dequantize(const kq_qmat* W, float* d_out, void* stream) {
  clear_error();
  if (int s = check_qmat(W, -1)) return s;
  if (!d_out) return fail(KQ_ERR_INVALID_ARG, "NULL output");
  const int64_t ss = scale_stride(W->fmt, W->k);
  dequant_kernel<<<grid_for(W->n * W->k, 256), 256, 0, (cudaStream_t)stream>>>(
      W->fmt, (const uint8_t*)W->codes, (const uint16_t*)W->scales, W->n, W->k, ss, d_out);
  KQ_CUDA_TRY(cudaGetLastError());
  return KQ_OK;
}

int kq_embed(const kq_qmat* E, const int32_t* d_ids, int64_t count, float* d_out, void* stream) {
  clear_error();
  if (int s = check_qmat(E, -1)) return s;
  if (count < 0) return fail(KQ_ERR_SHAPE, "count = %lld", (long long)count);
  if (count == 0) return KQ_OK;
  if (!d_ids || !d_out) return fail(KQ_ERR_INVALID_ARG, "NULL ids or output");
  if (!aligned16(d_ids) || !aligned16(d_out)) return fail(KQ_ERR_ALIGNMENT, "ids or output not 16-byte aligned");
  if (E->fmt == KQ_PQ2_0 && E->k > 32768)
    return fail(KQ_ERR_UNSUPPORTED, "k = %lld above the 32768 a PQ2_0 lookup transforms in shared memory",
                (long long)E->k);
  const size_t smem = E->fmt == KQ_PQ2_0 ? (size_t)E->k * sizeof(float) : 0;
  static bool attr_set = false;
  if (!attr_set) {
    KQ_CUDA_TRY(cudaFuncSetAttribute(embed_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 32768 * 4));
    attr_set = true;
  }
  int dev = 0, sms = 0;
  KQ_CUDA_TRY(cudaGetDevice(&dev));
  KQ_CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  const int grid = (int)std::min<int64_t>(count, (int64_t)sms * 8);
  embed_kernel<<<grid, 256, smem, (cudaStream_t)stream>>>(E->fmt, (const uint8_t*)E->codes, (const uint16_t*)E->scales,
                                                          E->n, E->k, scale_stride(E->fmt, E->k), d_ids, count,
                                                          E->had_block, E->signs, d_out);
  KQ_CUDA_TRY(cudaGetLastError());
  return KQ_OK;
}

int kq_hadamard_blockwise(const float* d_in, float* d_out, int64_t rows, int64_t k, int32_t block, void* stream) {
  return kq_rotate_blockwise(d_in, d_out, rows, k, block, nullptr, stream);
}

int kq_rotate_blockwise(const float* d_in, float* d_out, int64_t rows, int64_t k, int32_t block,
                        const int8_t* d_signs, void* stream) {
  clear_error();
  if (!d_in || !d_out) return fail(KQ_ERR_INVALID_ARG, "NULL pointer");
  if (d_signs && !aligned16(d_signs)) return fail(KQ_ERR_ALIGNMENT, "signs not 16-byte aligned");
  if (block < 1 || (block & (block - 1)) != 0) return fail(KQ_ERR_SHAPE, "block %d is not a power of two", block);
  if (block > 4096) return fail(KQ_ERR_UNSUPPORTED, "block %d > 4096", block);
  if (rows < 1 || k < block || k % block)
    return fail(KQ_ERR_SHAPE, "rows = %lld, k = %lld, block = %d", (long long)rows, (long long)k, block);
  const int64_t nblocks = rows * (k / block);
  const double scale = 1.0 / sqrt((double)block);
  cudaStream_t st = (cudaStream_t)stream;
  if (block == 128) {
    if (!aligned16(d_in) || !aligned16(d_out)) return fail(KQ_ERR_ALIGNMENT, "pointer not 16-byte aligned");
    hadamard128_f64_kernel<<<grid_for(nblocks * 32, 256), 256, 0, st>>>(d_in, d_out, nblocks, scale, d_signs,
                                                                        k / block);
  } else {
    int threads = block / 2 < 32 ? 32 : (block / 2 > 256 ? 256 : block / 2);
    int grid = grid_for(nblocks * threads, threads);
    hadamard_f64_smem_kernel<<<grid, threads, (size_t)block * sizeof(double), st>>>(d_in, d_out, nblocks, block,
                                                                                    scale, d_signs, k / block);
  }
  KQ_CUDA_TRY(cudaGetLastError());
  return KQ_OK;
}

}  // extern "C"
