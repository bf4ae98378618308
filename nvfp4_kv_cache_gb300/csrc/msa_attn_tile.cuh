// msa_attn_tile.cuh — the per-block attention pieces shared by the decode and the prefill
// attention kernels: reading a staged NVFP4 K/V row, dequantising it, and the mma.sync
// attention of one token's 16 heads over the keys of one dequantised block with an online
// softmax ("vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", "MSA primer": exact attention
// over the selected blocks; "MSA 机制详解": keys after the query position are masked).
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "msa_device.cuh"

namespace msa {

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// The 64 code bytes and 8 scale bytes of key row r of a staged NVFP4 region (128-byte swizzled).
struct RawRow {
  uint4 c[4];  // c[q]: code words of dims 32 q .. 32 q + 31
  uint2 sc;    // scale bytes of dims 16 i .. 16 i + 15, i = 0..7
};

__device__ __forceinline__ void load_row(const uint8_t* rg, int r, RawRow& raw) {
  raw.sc = lds64(rg + sw128_phys(static_cast<uint32_t>(kScaleOff + r * kRowScales)));
#pragma unroll
  for (int q = 0; q < 4; ++q) raw.c[q] = lds128(rg + sw128_phys(static_cast<uint32_t>(r * kRowCodes + 16 * q)));
}

// Dims 32 q .. 32 q + 31 of a raw row as E4M3: w[i] = dims 32 q + 4 i .. +3.
__device__ __forceinline__ void dequant_quarter(const RawRow& raw, int q, const uint2* lut, uint32_t (&w)[8]) {
  const uint32_t s2 = ((q < 2) ? raw.sc.x : raw.sc.y) >> (16 * (q & 1));
  const uint2 e0 = lut[s2 & 0xFFu], e1 = lut[(s2 >> 8) & 0xFFu];
  dq8(raw.c[q].x, e0, w[0], w[1]);
  dq8(raw.c[q].y, e0, w[2], w[3]);
  dq8(raw.c[q].z, e1, w[4], w[5]);
  dq8(raw.c[q].w, e1, w[6], w[7]);
}

// Running softmax state of one token warp for its 16 heads (rows gid and gid + 8 here).
struct WarpState {
  float m[2], l[2];
  float o[16][4];  // 16 n-tiles of 8 dims: (head gid, dims 8j+2t..+1), (head gid+8, ...)
};

// Keys 32 c .. 32 c + 31 of chunks [c_lo, c_hi) of one dequantised block for the 16 heads of
// this warp's token. kt: E4M3 [key][128] (16-byte chunk x of row k at x ^ (k & 7)); vt: f16
// [key][128] (chunk x of row k at x ^ (k & 7)). Keys past p_tok are masked; chunks wholly past
// it are skipped.
__device__ __forceinline__ void attend_tile(WarpState& st, const uint32_t (&qa)[4][4], const uint8_t* kt,
                                            const uint8_t* vt, int blk_pos0, int p_tok, float scale_log2, int c_lo,
                                            int c_hi, int lane) {
  const int t = lane & 3;
  const int r8 = lane & 7, m8 = lane >> 3;
#pragma unroll 1
  for (int c = c_lo; c < c_hi; ++c) {
    const int k0 = c * 32;
    if (blk_pos0 + k0 > p_tok) break;  // every remaining key lies after the query position
    // ---- S = Q K^T for keys k0 .. k0+31 (4 n-tiles of 8 keys)
    float x[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint8_t* krow = kt + (k0 + 8 * j + r8) * kD;
      uint32_t b0[4], b1[4];
      ldmatrix_x4(b0, krow + ((m8 ^ r8) << 4));        // dims 0..63
      ldmatrix_x4(b1, krow + (((m8 + 4) ^ r8) << 4));  // dims 64..127
      mma_e4m3_zc(x[j], qa[0][0], qa[0][1], qa[0][2], qa[0][3], b0[0], b0[1]);
      mma_e4m3(x[j], qa[1][0], qa[1][1], qa[1][2], qa[1][3], b0[2], b0[3]);
      mma_e4m3(x[j], qa[2][0], qa[2][1], qa[2][2], qa[2][3], b1[0], b1[1]);
      mma_e4m3(x[j], qa[3][0], qa[3][1], qa[3][2], qa[3][3], b1[2], b1[3]);
    }
    // ---- scale, causal mask, online softmax
    const bool need_mask = blk_pos0 + k0 + 31 > p_tok;
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v = x[j][i] * scale_log2;
        if (need_mask && blk_pos0 + k0 + 8 * j + 2 * t + (i & 1) > p_tok) v = -CUDART_INF_F;
        x[j][i] = v;
      }
      mx0 = fmaxf(mx0, fmaxf(x[j][0], x[j][1]));
      mx1 = fmaxf(mx1, fmaxf(x[j][2], x[j][3]));
    }
    mx0 = quad_max(mx0);
    mx1 = quad_max(mx1);
    const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
    const float mu0 = (mn0 == -CUDART_INF_F) ? 0.f : mn0;
    const float mu1 = (mn1 == -CUDART_INF_F) ? 0.f : mn1;
    if (__any_sync(0xffffffffu, mn0 != st.m[0] || mn1 != st.m[1])) {
      const float c0 = fast_exp2(st.m[0] - mu0), c1 = fast_exp2(st.m[1] - mu1);
      st.l[0] *= c0;
      st.l[1] *= c1;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        st.o[n][0] *= c0;
        st.o[n][1] *= c0;
        st.o[n][2] *= c1;
        st.o[n][3] *= c1;
      }
      st.m[0] = mn0;
      st.m[1] = mn1;
    }
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[j][0] = fast_exp2(x[j][0] - mu0);
      x[j][1] = fast_exp2(x[j][1] - mu0);
      x[j][2] = fast_exp2(x[j][2] - mu1);
      x[j][3] = fast_exp2(x[j][3] - mu1);
      ls0 += x[j][0] + x[j][1];
      ls1 += x[j][2] + x[j][3];
    }
    st.l[0] += ls0;
    st.l[1] += ls1;
    // ---- O += P V: 2 k-steps of 16 keys, 8 pairs of 8-dim n-tiles
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t a0 = pack_f16x2(x[2 * kk][0], x[2 * kk][1]);
      const uint32_t a1 = pack_f16x2(x[2 * kk][2], x[2 * kk][3]);
      const uint32_t a2 = pack_f16x2(x[2 * kk + 1][0], x[2 * kk + 1][1]);
      const uint32_t a3 = pack_f16x2(x[2 * kk + 1][2], x[2 * kk + 1][3]);
      const int rl = k0 + 16 * kk + (m8 & 1) * 8 + r8;
      const uint8_t* vrow = vt + rl * (2 * kD);
#pragma unroll
      for (int dn = 0; dn < 8; ++dn) {
        const int chunk = 2 * dn + (m8 >> 1);
        uint32_t r[4];
        ldmatrix_x4_trans(r, vrow + ((chunk ^ r8) << 4));
        mma_f16(st.o[2 * dn], a0, a1, a2, a3, r[0], r[1]);
        mma_f16(st.o[2 * dn + 1], a0, a1, a2, a3, r[2], r[3]);
      }
    }
  }
}

}  // namespace msa
