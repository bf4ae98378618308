// msa_attn.cu — exact sparse GQA attention over the selected blocks + split merge.
//
// What it computes ("vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", "MSA primer": exact
// attention over the selected blocks only, every query head of a GQA group using its group's
// selection; "MiniMax M3 in vLLM ...", "解码执行": split work merged from partial outputs, and
// "MSA 机制详解": the partial last block and keys after the query position are masked). K and V
// are dequantised from NVFP4 to E4M3 ("NVIDIA Blackwell optimizado kernes MSA") exactly as the
// indexer does; QK^T is an FP8 MMA with fp32 accumulation; the softmax is fp32 (exp2 with the
// log2(e) folded into the scale); PV takes P rounded to f16 and V widened exactly from E4M3 to
// f16, because P rounded to E4M3 (3 mantissa bits) would cost several percent of relative
// error.
//
// GB300 design (one CTA per (sequence, group, split)):
//  * The query tokens of a sequence (1..8, speculative decoding) mostly pick the same blocks,
//    so the CTA walks the union of their selections once ("KV-block-major" reuse): each union
//    block's K and V (2 x 9,216 B, contiguous in the page) arrive with one 1-D bulk copy into a
//    double-buffered stage, are dequantised once by all 256 threads into swizzled shared memory
//    (K as E4M3 rows, V as f16 rows), and every warp whose token selected the block consumes it.
//  * Warps split as tokens x key slices (8 / q_len warps per token), each with its own online
//    softmax state; the states are merged in shared memory at the end.
//  * QK^T: mma.sync.m16n8k32.e4m3 with the 16 heads of the group on M; the K operand is one
//    8-byte shared load per lane (8-byte-slot xor swizzle: conflict-free). PV:
//    mma.sync.m16n8k16.f16 with P taken straight from the QK^T accumulators and V fragments
//    from ldmatrix.trans (16-byte-chunk xor swizzle: conflict-free).
//  * Splits of the union list raise the CTA count when B * 4 is small; partial (lse, o) pairs
//    are merged by log-sum-exp in a second kernel.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <mutex>

#include "msa.h"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

constexpr int kAttnWarps = 8;
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr int kStageBytes = 2 * kRegion;  // K region then V region of one (page, group)

struct AttnParams {
  int32_t B, T, maxb, max_q_len, num_pages, splits;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_table;
  const uint8_t* kv_pages;
  const uint8_t* q;
  const int32_t* sel;
  float scale_log2;
  uint16_t* out;
  float* part_o;
  float* part_lse;
  uint32_t* status;
};

struct AttnSmem {
  static constexpr size_t kOffStage = 0;                                  // 2 x 18,432
  static constexpr size_t kOffK = kOffStage + 2 * kStageBytes;            // 128 x 128 B
  static constexpr size_t kOffV = kOffK + kBS * kD;                       // 128 x 256 B
  static constexpr size_t kOffLut = kOffV + kBS * kD * 2;                 // 2 KB
  static constexpr size_t kOffBar = kOffLut + 256 * 8;
  static constexpr size_t kOffUblk = kOffBar + 64;                        // 128 int
  static constexpr size_t kOffUmask = kOffUblk + 4 * 128;                 // 128 u32
  static constexpr size_t kOffUphys = kOffUmask + 4 * 128;                // 128 int
  static constexpr size_t kOffVals = kOffUphys + 4 * 128;                 // 128 int
  static constexpr size_t kOffFirst = kOffVals + 4 * 128;                 // 128 u32
  static constexpr size_t kOffMisc = kOffFirst + 4 * 128;
  static constexpr size_t kBytes = kOffMisc + 64;
  // after the block loop, the stage / K / V area holds each warp's final state
  static constexpr size_t kWarpState = 16 * 4 * 2 + 16 * kD * 4;          // m, l, O[16][128]
};
static_assert(AttnSmem::kOffLut >= kAttnWarps * AttnSmem::kWarpState, "merge area too small");

__device__ __forceinline__ float quad_max(float v) {
  v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
}
__device__ __forceinline__ float quad_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v + __shfl_xor_sync(0xffffffffu, v, 2);
}

// Per-warp running softmax state for 16 heads (rows gid and gid+8 in this lane).
struct WarpState {
  float m[2], l[2];
  float o[16][4];  // 16 n-tiles of 8 dims: (head gid, dims 8j+2t..+1), (head gid+8, ...)
};

// Attend to NJ*8 keys starting at key `k0` of the staged block (K, V in shared memory).
template <int NJ>
__device__ __forceinline__ void attend_keys(WarpState& st, const uint32_t (&qa)[4][4], const uint8_t* Ks,
                                            const uint8_t* Vs, int k0, int blk_pos0, int p_tok, float scale_log2,
                                            int lane) {
  const int gid = lane >> 2, t = lane & 3;
  float x[NJ][4];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    x[j][0] = x[j][1] = x[j][2] = x[j][3] = 0.f;
    const int key = k0 + 8 * j + gid;
    const uint8_t* row = Ks + key * kD;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint2 b = lds64(row + (((4 * t + s) ^ (key & 3)) << 3));
      mma_e4m3(x[j], qa[s][0], qa[s][1], qa[s][2], qa[s][3], b.x, b.y);
    }
  }
  // scale, causal mask, row max
  const bool need_mask = blk_pos0 + k0 + 8 * NJ - 1 > p_tok;
  float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
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
  const float c0 = fast_exp2(st.m[0] - mu0), c1 = fast_exp2(st.m[1] - mu1);
  st.m[0] = mn0;
  st.m[1] = mn1;
  float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    x[j][0] = fast_exp2(x[j][0] - mu0);
    x[j][1] = fast_exp2(x[j][1] - mu0);
    x[j][2] = fast_exp2(x[j][2] - mu1);
    x[j][3] = fast_exp2(x[j][3] - mu1);
    ls0 += x[j][0] + x[j][1];
    ls1 += x[j][2] + x[j][3];
  }
  st.l[0] = st.l[0] * c0 + ls0;
  st.l[1] = st.l[1] * c1 + ls1;
#pragma unroll
  for (int n = 0; n < 16; ++n) {
    st.o[n][0] *= c0;
    st.o[n][1] *= c0;
    st.o[n][2] *= c1;
    st.o[n][3] *= c1;
  }
  // PV: 16 keys per k-step
#pragma unroll
  for (int kk = 0; kk < NJ / 2; ++kk) {
    const uint32_t a0 = pack_f16x2(x[2 * kk][0], x[2 * kk][1]);
    const uint32_t a1 = pack_f16x2(x[2 * kk][2], x[2 * kk][3]);
    const uint32_t a2 = pack_f16x2(x[2 * kk + 1][0], x[2 * kk + 1][1]);
    const uint32_t a3 = pack_f16x2(x[2 * kk + 1][2], x[2 * kk + 1][3]);
    const int mi = lane >> 3, ri = lane & 7;
    const int key = k0 + 16 * kk + (mi & 1) * 8 + ri;
    const uint8_t* vrow = Vs + key * (kD * 2);
#pragma unroll
    for (int dn = 0; dn < 8; ++dn) {
      const int chunk = 2 * dn + (mi >> 1);
      uint32_t r[4];
      ldmatrix_x4_trans(r, vrow + ((chunk ^ (key & 7)) << 4));
      mma_f16(st.o[2 * dn], a0, a1, a2, a3, r[0], r[1]);
      mma_f16(st.o[2 * dn + 1], a0, a1, a2, a3, r[2], r[3]);
    }
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1) k_attn(const AttnParams p) {
  using S = AttnSmem;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stage = smem + S::kOffStage;
  uint8_t* Ks = smem + S::kOffK;
  uint8_t* Vs = smem + S::kOffV;
  uint2* lut = reinterpret_cast<uint2*>(smem + S::kOffLut);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  int* ublk = reinterpret_cast<int*>(smem + S::kOffUblk);
  uint32_t* umask = reinterpret_cast<uint32_t*>(smem + S::kOffUmask);
  int* uphys = reinterpret_cast<int*>(smem + S::kOffUphys);
  int* vals = reinterpret_cast<int*>(smem + S::kOffVals);
  uint32_t* first = reinterpret_cast<uint32_t*>(smem + S::kOffFirst);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc);
  uint32_t* tokbad = reinterpret_cast<uint32_t*>(smem + S::kOffMisc + 4);
  int* nunion = reinterpret_cast<int*>(smem + S::kOffMisc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x % p.splits;
  const int bg = blockIdx.x / p.splits;
  const int g = bg & 3, b = bg >> 2;

  const int q0 = p.qsl[b];
  const int ql = p.qsl[b + 1] - q0;
  const int L = p.seq_lens[b];
  if (ql <= 0) return;  // padded request row
  const bool batch_ok = ql <= p.max_q_len && L >= ql && L <= p.maxb * kBS && q0 >= 0 && q0 + ql <= p.T;
  if (!batch_ok) {
    if (tid == 0 && split == 0 && g == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
    return;
  }
  const int nb = ceil_div(L, kBS);

  if (tid == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_mbar_init();
    *abort_flag = 0;
    *tokbad = 0;
  }
  build_dequant_lut(lut, tid, kAttnThreads);
  // ---- the union of the tokens' selected blocks (distinct, ascending) -----------------
  if (tid < 128) {
    const int tok = tid >> 4, slot = tid & 15;
    int v = 0x7FFFFFFF;
    if (tok < ql) {
      const int blk = p.sel[(static_cast<int64_t>(q0 + tok) * 4 + g) * kSel + slot];
      if (blk >= nb) {
        atomicOr(tokbad, 1u << tok);
        set_status(p.status, MSA_ERR_DEVICE_FAULT);
      } else if (blk >= 0) {
        v = blk;
      }
    }
    vals[tid] = v;
  }
  __syncthreads();
  if (tid < 128) {
    const int v = vals[tid];
    bool is_first = v != 0x7FFFFFFF;
    uint32_t m = 0;
    for (int j = 0; j < 128; ++j) {
      if (vals[j] == v) {
        m |= 1u << (j >> 4);
        if (j < tid) is_first = false;
      }
    }
    first[tid] = is_first ? m : 0u;
  }
  __syncthreads();
  if (tid < 128) {
    const int v = vals[tid];
    const uint32_t m = first[tid];
    if (m != 0u) {
      int rank = 0;
      for (int j = 0; j < 128; ++j) rank += (first[j] != 0u && vals[j] < v) ? 1 : 0;
      ublk[rank] = v;
      umask[rank] = m;
    }
  }
  const int U = __syncthreads_count(tid < 128 && first[tid] != 0u);
  if (tid < U) {
    const int phys = p.block_table[static_cast<int64_t>(b) * p.maxb + ublk[tid]];
    const bool ok = phys >= 0 && phys < p.num_pages;
    uphys[tid] = ok ? phys : -1;
    if (!ok) {
      atomicOr(tokbad, umask[tid]);
      set_status(p.status, MSA_ERR_DEVICE_FAULT);
    }
  }
  if (tid == 0) *nunion = U;
  __syncthreads();

  const int u0 = (U * split) / p.splits, u1 = (U * (split + 1)) / p.splits;
  const uint32_t bad = *tokbad;

  // ---- warp roles -----------------------------------------------------------------
  const int wpt = kAttnWarps / ql;  // 8, 4, 2, 2, 1, 1, 1, 1
  const int my_tok = warp / wpt;
  const int slice = warp % wpt;
  const bool active = my_tok < ql;
  const int nk = kBS / wpt;
  const int kbase = slice * nk;
  const int p_tok = L - ql + my_tok;
  const int gid = lane >> 2, t = lane & 3;

  uint32_t qa[4][4];
  WarpState st;
  st.m[0] = st.m[1] = -CUDART_INF_F;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int n = 0; n < 16; ++n) st.o[n][0] = st.o[n][1] = st.o[n][2] = st.o[n][3] = 0.f;
  if (active) {
    const uint8_t* qrow0 = p.q + (static_cast<int64_t>(q0 + my_tok) * kQHeads + g * kHPG + gid) * kD + 32 * t;
    const uint8_t* qrow1 = qrow0 + 8 * kD;
#pragma unroll
    for (int s = 0; s < 4; ++s) {
      const uint2 x0 = ldg_nc64(qrow0 + 8 * s);
      const uint2 x1 = ldg_nc64(qrow1 + 8 * s);
      qa[s][0] = x0.x;
      qa[s][2] = x0.y;
      qa[s][1] = x1.x;
      qa[s][3] = x1.y;
    }
  }

  // ---- block loop ------------------------------------------------------------------
  auto issue = [&](int u, int buf) {
    const int phys = uphys[u];
    if (phys >= 0) {
      mbar_arrive_expect_tx(&full[buf], kStageBytes);
      bulk_g2s(stage + buf * kStageBytes, p.kv_pages + static_cast<int64_t>(phys) * kKvPage + (2 * g) * kRegion,
               kStageBytes, &full[buf]);
    } else {
      mbar_arrive(&full[buf]);
    }
  };
  if (tid == 0) {
    if (u0 < u1) issue(u0, 0);
    if (u0 + 1 < u1) issue(u0 + 1, 1);
  }
  int issued_hi = min(u1, u0 + 2);  // meaningful in thread 0 only
  bool aborted = false;
  int u_stop = u1;
  for (int u = u0; u < u1; ++u) {
    const int it = u - u0, buf = it & 1;
    if (!mbar_wait_bounded(&full[buf], static_cast<uint32_t>(it >> 1) & 1u, kWaitLimitNs, abort_flag)) {
      if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
      *abort_flag = 1;
      aborted = true;
    }
    if (__syncthreads_or(aborted ? 1 : 0)) {
      aborted = true;
      u_stop = u;
      break;
    }
    const bool page_ok = uphys[u] >= 0;
    if (page_ok) {
      // dequantise K -> E4M3 rows, V -> f16 rows (row r, dims 64h .. 64h+63 per thread)
      const uint8_t* kr = stage + buf * kStageBytes;
      const uint8_t* vr = kr + kRegion;
      const int r = tid >> 1, h = tid & 1;
      {
        const uint4 c0 = *reinterpret_cast<const uint4*>(kr + r * kRowCodes + 32 * h);
        const uint4 c1 = *reinterpret_cast<const uint4*>(kr + r * kRowCodes + 32 * h + 16);
        const uint32_t sc = *reinterpret_cast<const uint32_t*>(kr + kScaleOff + r * kRowScales + 4 * h);
        const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        const int m = r & 3;
#pragma unroll
        for (int c = 0; c < 4; ++c) {  // 16-byte chunk c of this thread = words 2c, 2c+1
          const uint2 e = lut[(sc >> (8 * c)) & 0xFFu];
          uint32_t l0, h0, l1, h1;
          dq8(w[2 * c], e, l0, h0);
          dq8(w[2 * c + 1], e, l1, h1);
          const int slot = 8 * h + 2 * c;        // logical 8-byte slot of word 2c
          const int phys = slot ^ m;
          uint4 v = (m & 1) ? make_uint4(l1, h1, l0, h0) : make_uint4(l0, h0, l1, h1);
          *reinterpret_cast<uint4*>(Ks + r * kD + ((phys & ~1) << 3)) = v;
        }
      }
      {
        const uint4 c0 = *reinterpret_cast<const uint4*>(vr + r * kRowCodes + 32 * h);
        const uint4 c1 = *reinterpret_cast<const uint4*>(vr + r * kRowCodes + 32 * h + 16);
        const uint32_t sc = *reinterpret_cast<const uint32_t*>(vr + kScaleOff + r * kRowScales + 4 * h);
        const uint32_t w[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // word i = dims 64h + 8i .. +7 = f16 chunk 8h + i
          const uint2 e = lut[(sc >> (8 * (i >> 1))) & 0xFFu];
          uint32_t lo, hi;
          dq8(w[i], e, lo, hi);
          const uint4 v = make_uint4(cvt_f16x2_e4m3x2(lo), cvt_f16x2_e4m3x2(lo >> 16), cvt_f16x2_e4m3x2(hi),
                                     cvt_f16x2_e4m3x2(hi >> 16));
          const int chunk = (8 * h + i) ^ (r & 7);
          *reinterpret_cast<uint4*>(Vs + r * (2 * kD) + (chunk << 4)) = v;
        }
      }
    }
    __syncthreads();  // K, V ready; stage[buf] free
    if (tid == 0 && u + 2 < u1) {
      issue(u + 2, buf);
      issued_hi = u + 3;
    }
    if (page_ok && active && ((umask[u] >> my_tok) & 1u) && !((bad >> my_tok) & 1u)) {
      const int blk_pos0 = ublk[u] * kBS;
      if (nk == 16) {
        attend_keys<2>(st, qa, Ks, Vs, kbase, blk_pos0, p_tok, p.scale_log2, lane);
      } else {
        for (int kc = 0; kc < nk; kc += 32)
          attend_keys<4>(st, qa, Ks, Vs, kbase + kc, blk_pos0, p_tok, p.scale_log2, lane);
      }
    }
    __syncthreads();  // before the next block overwrites K, V
  }
  if (aborted && tid == 0) {
    // wait (bounded) for the copies not yet consumed, which may still be in flight into this
    // CTA's shared memory (at most the two stages from u_stop on)
    for (int u = u_stop; u < issued_hi; ++u) {
      const int it = u - u0;
      mbar_wait_bounded(&full[it & 1], static_cast<uint32_t>(it >> 1) & 1u, kWaitLimitNs, nullptr);
    }
  }
  __syncthreads();

  // ---- merge the warps of each token, write the output or the split partial ----------
  uint8_t* ws = smem;  // reuse stage / K / V
  if (active) {
    float* mw = reinterpret_cast<float*>(ws + warp * S::kWarpState);
    float* lw = mw + 16;
    float* ow = lw + 16;
    const float l0 = quad_sum(st.l[0]), l1 = quad_sum(st.l[1]);
    if (t == 0) {
      mw[gid] = st.m[0];
      mw[gid + 8] = st.m[1];
      lw[gid] = l0;
      lw[gid + 8] = l1;
    }
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      *reinterpret_cast<float2*>(ow + gid * kD + 8 * n + 2 * t) = make_float2(st.o[n][0], st.o[n][1]);
      *reinterpret_cast<float2*>(ow + (gid + 8) * kD + 8 * n + 2 * t) = make_float2(st.o[n][2], st.o[n][3]);
    }
  }
  __syncthreads();
  const int nelem = ql * kHPG * (kD / 4);  // float4 granules
  for (int e = tid; e < nelem; e += kAttnThreads) {
    const int d4 = e % (kD / 4);
    const int hh = (e / (kD / 4)) % kHPG;
    const int tok = e / (kD / 4) / kHPG;
    float M = -CUDART_INF_F;
    for (int sl = 0; sl < wpt; ++sl) {
      const float* mw = reinterpret_cast<const float*>(ws + (tok * wpt + sl) * S::kWarpState);
      M = fmaxf(M, mw[hh]);
    }
    float Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -CUDART_INF_F) {
      for (int sl = 0; sl < wpt; ++sl) {
        const float* mw = reinterpret_cast<const float*>(ws + (tok * wpt + sl) * S::kWarpState);
        const float f = fast_exp2(mw[hh] - M);
        Lsum += mw[16 + hh] * f;
        const float4 o = *reinterpret_cast<const float4*>(mw + 32 + hh * kD + 4 * d4);
        acc.x += o.x * f;
        acc.y += o.y * f;
        acc.z += o.z * f;
        acc.w += o.w * f;
      }
    }
    const bool zero = (M == -CUDART_INF_F) || Lsum <= 0.f || ((bad >> tok) & 1u);
    const float inv = zero ? 0.f : 1.0f / Lsum;
    const int64_t orow = static_cast<int64_t>(q0 + tok) * kQHeads + g * kHPG + hh;
    if (p.splits == 1) {
      const uint2 v = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
      *reinterpret_cast<uint2*>(p.out + orow * kD + 4 * d4) = v;
    } else {
      const int64_t prow = static_cast<int64_t>(split) * p.T * kQHeads + orow;
      *reinterpret_cast<float4*>(p.part_o + prow * kD + 4 * d4) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      if (d4 == 0) p.part_lse[prow] = zero ? -CUDART_INF_F : M + __log2f(Lsum);
    }
  }
}

// out[t][h] = sum_s w_s o_s / sum_s w_s with w_s = 2^(lse_s - max lse); zeros if no split has keys.
__global__ void __launch_bounds__(256) k_attn_merge(const float* __restrict__ part_o, const float* __restrict__ part_lse,
                                                    int32_t splits, int32_t T, uint16_t* __restrict__ out) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);  // (t, h)
  const int lane = threadIdx.x & 31;
  if (row >= T * kQHeads) return;
  const int64_t stride = static_cast<int64_t>(T) * kQHeads;
  float M = -CUDART_INF_F;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, part_lse[s * stride + row]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  if (M != -CUDART_INF_F) {
    for (int s = 0; s < splits; ++s) {
      const float lse = part_lse[s * stride + row];
      if (lse == -CUDART_INF_F) continue;
      const float w = fast_exp2(lse - M);
      const float4 o = *reinterpret_cast<const float4*>(part_o + (s * stride + row) * kD + 4 * lane);
      acc.x += w * o.x;
      acc.y += w * o.y;
      acc.z += w * o.z;
      acc.w += w * o.w;
      W += w;
    }
  }
  const float inv = W > 0.f ? 1.0f / W : 0.f;
  *reinterpret_cast<uint2*>(out + static_cast<int64_t>(row) * kD + 4 * lane) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

size_t attn_ws_bytes(int T, int splits) {
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(splits) * T * kQHeads;
  return msa_host::align256(rows * kD * 4) + msa_host::align256(rows * 4);
}

}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

extern "C" size_t msa_attn_workspace_size(const msa_geometry* geo, int32_t B, int32_t T, int32_t num_splits) {
  if (check_geometry(geo) != MSA_OK || B < 0 || T < 0 || num_splits < 0 || num_splits > kMaxSplits) return 0;
  const int s = num_splits > 0 ? num_splits : auto_splits(B);
  return attn_ws_bytes(T, s);
}

msa_status msa_launch_attn_merge(const float* part_o, const float* part_lse, int32_t splits, int32_t T, uint16_t* out,
                                 cudaStream_t stream) {
  const int rows = T * kQHeads;
  k_attn_merge<<<ceil_div(rows, 8), 256, 0, stream>>>(part_o, part_lse, splits, T, out);
  return launch_status();
}

extern "C" msa_status msa_sparse_attn_decode(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                             const uint8_t* q, const int32_t* sel, float softmax_scale,
                                             int32_t num_splits, void* workspace, size_t workspace_bytes,
                                             uint16_t* out, uint32_t* status, cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = check_batch(batch)) != MSA_OK) return st;
  if ((st = check_cache(cache, false, true)) != MSA_OK) return st;
  if (num_splits < 0 || num_splits > kMaxSplits) return MSA_ERR_INVALID_ARG;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (q == nullptr || sel == nullptr || out == nullptr || !aligned(q, 16) || !aligned(sel, 4) || !aligned(out, 16))
    return MSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || softmax_scale != softmax_scale) return MSA_ERR_INVALID_ARG;
  const int splits = num_splits > 0 ? num_splits : auto_splits(batch->B);
  const size_t need = attn_ws_bytes(batch->T, splits);
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned(workspace, 256))))
    return MSA_ERR_INVALID_ARG;
  AttnParams p;
  p.B = batch->B;
  p.T = batch->T;
  p.maxb = batch->max_blocks_per_seq;
  p.max_q_len = batch->max_q_len;
  p.num_pages = cache->num_pages;
  p.splits = splits;
  p.qsl = batch->query_start_loc;
  p.seq_lens = batch->seq_lens;
  p.block_table = batch->block_table;
  p.kv_pages = cache->kv_pages;
  p.q = q;
  p.sel = sel;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = out;
  p.part_o = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  p.part_lse = splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                                     align256(static_cast<size_t>(splits) * batch->T * kQHeads * kD * 4))
                          : nullptr;
  p.status = status;
  if (cudaFuncSetAttribute(k_attn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(AttnSmem::kBytes)) !=
      cudaSuccess)
    return MSA_ERR_CUDA;
  const int grid = batch->B * 4 * splits;
  k_attn<<<grid, kAttnThreads, AttnSmem::kBytes, stream>>>(p);
  if ((st = launch_status()) != MSA_OK) return st;
  if (splits > 1) return msa_launch_attn_merge(p.part_o, p.part_lse, splits, batch->T, out, stream);
  return MSA_OK;
}

// ------------------------------------------------------------------------------------------
// Allocation-free variant of msa_sparse_attn_decode.
//
// Some callers cannot allocate device memory: a host runtime whose memory is laid out once
// by a static planner and that has no allocator to hand down to this library, or code that
// runs inside another library's callback, where a cudaMalloc would synchronise the device
// and break the caller's stream ordering. For them the split partial results live in one
// file-scope device array of kNoAllocScratchBytes bytes, which every GPU that loads this
// library holds until the process exits. The caller still passes inputs and outputs.
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB
__device__ __align__(256) uint8_t g_attn_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_attn_scratch on the current device, looked up once per device (the
// name is a host-side stand-in, not a device address).
msa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr) return MSA_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return MSA_OK;
}

}  // namespace

extern "C" size_t msa_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" msa_status msa_sparse_attn_decode_noalloc(const msa_geometry* geo, const msa_batch* batch,
                                                     const msa_cache* cache, const uint8_t* q, const int32_t* sel,
                                                     float softmax_scale, int32_t num_splits, uint16_t* out,
                                                     uint32_t* status, cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = check_batch(batch)) != MSA_OK) return st;
  if ((st = check_cache(cache, false, true)) != MSA_OK) return st;
  if (num_splits < 0 || num_splits > kMaxSplits) return MSA_ERR_INVALID_ARG;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (q == nullptr || sel == nullptr || out == nullptr || !aligned(q, 16) || !aligned(sel, 4) || !aligned(out, 16))
    return MSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || softmax_scale != softmax_scale) return MSA_ERR_INVALID_ARG;
  const int splits = num_splits > 0 ? num_splits : auto_splits(batch->B);
  const size_t need = attn_ws_bytes(batch->T, splits);
  if (need > kNoAllocScratchBytes) return MSA_ERR_INVALID_ARG;  // too many tokens x splits for the array
  void* scratch = nullptr;
  if (need > 0 && (st = scratch_address(&scratch)) != MSA_OK) return st;
  AttnParams p;
  p.B = batch->B;
  p.T = batch->T;
  p.maxb = batch->max_blocks_per_seq;
  p.max_q_len = batch->max_q_len;
  p.num_pages = cache->num_pages;
  p.splits = splits;
  p.qsl = batch->query_start_loc;
  p.seq_lens = batch->seq_lens;
  p.block_table = batch->block_table;
  p.kv_pages = cache->kv_pages;
  p.q = q;
  p.sel = sel;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = out;
  p.part_o = splits > 1 ? static_cast<float*>(scratch) : nullptr;
  p.part_lse = splits > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) +
                                                     align256(static_cast<size_t>(splits) * batch->T * kQHeads * kD * 4))
                          : nullptr;
  p.status = status;
  if (cudaFuncSetAttribute(k_attn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(AttnSmem::kBytes)) !=
      cudaSuccess)
    return MSA_ERR_CUDA;
  k_attn<<<batch->B * 4 * splits, kAttnThreads, AttnSmem::kBytes, stream>>>(p);
  if ((st = launch_status()) != MSA_OK) return st;
  if (splits > 1) return msa_launch_attn_merge(p.part_o, p.part_lse, splits, batch->T, out, stream);
  return MSA_OK;
}
