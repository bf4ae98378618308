// msa_quant.cu — cache producers and the standalone dequantiser.
//
//  * msa_quantize_nvfp4: per 16 elements s = E4M3(amax/6), codes = E2M1(x / S)
//    ("MiniMax-M3.1-Flash serving notes", "The capacity numbers": 4-bit values plus one FP8
//    scale per 16 values). One thread per 8 elements (one 32-bit code word); the two threads
//    of a 16-element group exchange their partial amax with one shuffle.
//  * msa_quantize_fp8: E4M3 cast (queries, index queries, FP8 index cache).
//  * msa_dequant_nvfp4: the a1/a5 operand rule on its own (NVFP4 -> E4M3 bytes).
//  * msa_kv_insert: quantise new tokens straight into their cache pages ("vLLM ofrece soporte
//    en día 0 para MiniMax-M3.1-Flash", "QKV GEMM + norm + RoPE + KV inserción fusión": K, V
//    and the index key are quantised to NVFP4 and written into their caches).
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa.h"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

// Quantise 8 consecutive elements whose 16-element group partner is lane ^ 1. Returns the
// code word; *scale_out gets the group's scale byte. All 32 lanes must call it.
__device__ __forceinline__ uint32_t quantize_word(const float (&x)[8], uint32_t* scale_out) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[j]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  const float sf = __fdiv_rn(amax, 6.0f);
  const uint32_t s = cvt_e4m3x2(sf, 0.0f) & 0xFFu;
  const float S = e4m3_to_f32(s);
  uint32_t w = 0;
  if (S != 0.0f) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float r = __fdiv_rn(x[j], S);
      const uint32_t m = e2m1_code(fabsf(r));
      const uint32_t neg = (m != 0u && signbit(r)) ? 1u : 0u;
      w |= m << (4 * j);
      w |= neg << (4 * sign_slot(j) + 3);
    }
  }
  *scale_out = s;
  return w;
}

__global__ void __launch_bounds__(256) k_quantize_nvfp4(const float* __restrict__ x, int64_t rows, int32_t cols,
                                                        uint8_t* __restrict__ vals, int64_t vstride,
                                                        uint8_t* __restrict__ scales, int64_t sstride) {
  const int64_t wpr = cols / 8;
  const int64_t total = rows * wpr;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < total;
       base += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t idx = base + threadIdx.x;
    const bool active = idx < total;
    const int64_t r = active ? idx / wpr : 0;
    const int64_t w = active ? idx % wpr : 0;
    float v[8];
    if (active) {
      const float4 a = *reinterpret_cast<const float4*>(x + r * cols + 8 * w);
      const float4 b = *reinterpret_cast<const float4*>(x + r * cols + 8 * w + 4);
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = 0.0f;
    }
    uint32_t s;
    const uint32_t word = quantize_word(v, &s);
    if (active) {
      *reinterpret_cast<uint32_t*>(vals + r * vstride + 4 * w) = word;
      if ((w & 1) == 0) scales[r * sstride + w / 2] = static_cast<uint8_t>(s);
    }
  }
}

__global__ void __launch_bounds__(256) k_quantize_fp8(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ out) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < (n + 3) / 4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = 4 * i;
    if (e + 3 < n) {
      const float4 a = *reinterpret_cast<const float4*>(x + e);
      const uint32_t v = cvt_e4m3x2(a.x, a.y) | (cvt_e4m3x2(a.z, a.w) << 16);
      *reinterpret_cast<uint32_t*>(out + e) = v;
    } else {
      for (int64_t k = e; k < n; ++k) out[k] = static_cast<uint8_t>(cvt_e4m3x2(x[k], 0.0f) & 0xFFu);
    }
  }
}

// Scalar fallback for unaligned fp8 casts.
__global__ void k_quantize_fp8_scalar(const float* __restrict__ x, int64_t n, uint8_t* __restrict__ out) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    out[i] = static_cast<uint8_t>(cvt_e4m3x2(x[i], 0.0f) & 0xFFu);
}

__global__ void __launch_bounds__(256) k_dequant_nvfp4(const uint8_t* __restrict__ vals, int64_t vstride,
                                                       const uint8_t* __restrict__ scales, int64_t sstride,
                                                       int64_t rows, int32_t cols, uint8_t* __restrict__ out) {
  __shared__ uint2 lut[256];
  build_dequant_lut(lut, threadIdx.x, blockDim.x);
  __syncthreads();
  const int64_t wpr = cols / 8;
  const int64_t total = rows * wpr;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = idx / wpr, w = idx % wpr;
    uint32_t word = 0;
    const uint8_t* src = vals + r * vstride + 4 * w;
    word = static_cast<uint32_t>(src[0]) | (static_cast<uint32_t>(src[1]) << 8) |
           (static_cast<uint32_t>(src[2]) << 16) | (static_cast<uint32_t>(src[3]) << 24);
    const uint32_t s = scales[r * sstride + w / 2];
    uint32_t lo, hi;
    dq8(word, lut[s], lo, hi);
    uint8_t* dst = out + r * cols + 8 * w;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      dst[j] = static_cast<uint8_t>(lo >> (8 * j));
      dst[4 + j] = static_cast<uint8_t>(hi >> (8 * j));
    }
  }
}

// One thread per 8 elements of one 128-element row; a token owns 8 (K, V) rows plus one
// index row. Row kinds: 0..3 K of head 0..3, 4..7 V of head 0..3, 8 index key.
__global__ void __launch_bounds__(256) k_kv_insert(const float* __restrict__ k, const float* __restrict__ v,
                                                   const float* __restrict__ ik, int64_t n,
                                                   const int64_t* __restrict__ slots, uint8_t* __restrict__ kv_pages,
                                                   uint8_t* __restrict__ index_pages, int32_t index_dtype,
                                                   int32_t num_pages, uint32_t* status) {
  const int rows_per_tok = ik != nullptr ? 9 : 8;
  const int64_t total = n * rows_per_tok * 16;  // 16 words per 128-element row
  const int64_t limit = static_cast<int64_t>(num_pages) * kBS;
  for (int64_t base = static_cast<int64_t>(blockIdx.x) * blockDim.x; base < total;
       base += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t idx = base + threadIdx.x;
    const bool in_range = idx < total;
    const int64_t row = in_range ? idx / 16 : 0;
    const int w = static_cast<int>(idx % 16);
    const int64_t tok = row / rows_per_tok;
    const int kind = static_cast<int>(row % rows_per_tok);
    const int64_t slot = in_range ? slots[tok] : -1;
    const bool bad = in_range && slot >= limit;
    const bool active = in_range && slot >= 0 && !bad;
    if (bad && w == 0) set_status(status, MSA_ERR_DEVICE_FAULT);
    const float* src = nullptr;
    if (kind < 4) src = k + (tok * 4 + kind) * kD;
    else if (kind < 8) src = v + (tok * 4 + (kind - 4)) * kD;
    else src = ik + tok * kD;
    float x[8];
    if (in_range) {
      const float4 a = *reinterpret_cast<const float4*>(src + 8 * w);
      const float4 b = *reinterpret_cast<const float4*>(src + 8 * w + 4);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = 0.0f;
    }
    const int64_t page = active ? slot / kBS : 0;
    const int prow = active ? static_cast<int>(slot % kBS) : 0;
    // Every lane runs the quantiser (it exchanges amax with its neighbour lane), whatever
    // the row kind; only the stores depend on it.
    uint32_t s;
    const uint32_t word = quantize_word(x, &s);
    if (!active) continue;
    if (kind == 8 && index_dtype == MSA_INDEX_FP8) {
      const uint32_t lo = cvt_e4m3x2(x[0], x[1]) | (cvt_e4m3x2(x[2], x[3]) << 16);
      const uint32_t hi = cvt_e4m3x2(x[4], x[5]) | (cvt_e4m3x2(x[6], x[7]) << 16);
      *reinterpret_cast<uint2*>(index_pages + page * kIdxPageFp8 + prow * kD + 8 * w) = make_uint2(lo, hi);
      continue;
    }
    uint8_t* region;
    if (kind < 8) {
      const int head = kind & 3, kv = kind >> 2;
      region = kv_pages + page * kKvPage + (head * 2 + kv) * kRegion;
    } else {
      region = index_pages + page * kIdxPageNv;
    }
    *reinterpret_cast<uint32_t*>(region + prow * kRowCodes + 4 * w) = word;
    if ((w & 1) == 0) region[kScaleOff + prow * kRowScales + w / 2] = static_cast<uint8_t>(s);
  }
}

int grid_for(int64_t work, int threads) {
  int64_t blocks = (work + threads - 1) / threads;
  if (blocks < 1) blocks = 1;
  if (blocks > 152 * 64) blocks = 152 * 64;
  return static_cast<int>(blocks);
}

}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

extern "C" msa_status msa_quantize_nvfp4(const float* x, int64_t rows, int32_t cols, uint8_t* vals,
                                         int64_t vals_row_stride, uint8_t* scales, int64_t scales_row_stride,
                                         cudaStream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0) return MSA_ERR_INVALID_ARG;
  if (rows == 0) return MSA_OK;
  if (x == nullptr || vals == nullptr || scales == nullptr) return MSA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(vals, 4) || vals_row_stride % 4 != 0) return MSA_ERR_INVALID_ARG;
  if (vals_row_stride < cols / 2 || scales_row_stride < cols / 16) return MSA_ERR_INVALID_ARG;
  const int64_t work = rows * (cols / 8);
  k_quantize_nvfp4<<<grid_for(work, 256), 256, 0, stream>>>(x, rows, cols, vals, vals_row_stride, scales,
                                                              scales_row_stride);
  return launch_status();
}

extern "C" msa_status msa_quantize_fp8(const float* x, int64_t n, uint8_t* out, cudaStream_t stream) {
  if (n < 0) return MSA_ERR_INVALID_ARG;
  if (n == 0) return MSA_OK;
  if (x == nullptr || out == nullptr) return MSA_ERR_INVALID_ARG;
  if (aligned(x, 16) && aligned(out, 4)) {
    k_quantize_fp8<<<grid_for((n + 3) / 4, 256), 256, 0, stream>>>(x, n, out);
  } else {
    k_quantize_fp8_scalar<<<grid_for(n, 256), 256, 0, stream>>>(x, n, out);
  }
  return launch_status();
}

extern "C" msa_status msa_dequant_nvfp4(const uint8_t* vals, int64_t vals_row_stride, const uint8_t* scales,
                                        int64_t scales_row_stride, int64_t rows, int32_t cols, uint8_t* out,
                                        cudaStream_t stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0) return MSA_ERR_INVALID_ARG;
  if (rows == 0) return MSA_OK;
  if (vals == nullptr || scales == nullptr || out == nullptr) return MSA_ERR_INVALID_ARG;
  if (vals_row_stride < cols / 2 || scales_row_stride < cols / 16) return MSA_ERR_INVALID_ARG;
  k_dequant_nvfp4<<<grid_for(rows * (cols / 8), 256), 256, 0, stream>>>(vals, vals_row_stride, scales,
                                                                          scales_row_stride, rows, cols, out);
  return launch_status();
}

extern "C" msa_status msa_kv_insert(const float* k, const float* v, const float* ik, int64_t n,
                                    const int64_t* slots, uint8_t* kv_pages, uint8_t* index_pages,
                                    int32_t index_dtype, int32_t num_pages, uint32_t* status, cudaStream_t stream) {
  if (n < 0 || num_pages < 0) return MSA_ERR_INVALID_ARG;
  if (n == 0) return MSA_OK;
  if (k == nullptr || v == nullptr || slots == nullptr || kv_pages == nullptr) return MSA_ERR_INVALID_ARG;
  if (ik != nullptr && index_pages == nullptr) return MSA_ERR_INVALID_ARG;
  if (index_dtype != MSA_INDEX_NVFP4 && index_dtype != MSA_INDEX_FP8) return MSA_ERR_UNSUPPORTED;
  if (!aligned(k, 16) || !aligned(v, 16) || (ik != nullptr && !aligned(ik, 16)) || !aligned(slots, 8))
    return MSA_ERR_INVALID_ARG;
  if (!aligned(kv_pages, 256) || (index_pages != nullptr && !aligned(index_pages, 256))) return MSA_ERR_INVALID_ARG;
  const int64_t work = n * (ik != nullptr ? 9 : 8) * 16;
  k_kv_insert<<<grid_for(work, 256), 256, 0, stream>>>(k, v, ik, n, slots, kv_pages, index_pages, index_dtype,
                                                       num_pages, status);
  return launch_status();
}
