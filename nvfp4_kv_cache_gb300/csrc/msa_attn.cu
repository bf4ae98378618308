// msa_attn.cu — exact sparse GQA attention over the selected blocks + split merge.
//
// What it computes ("vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", "MSA primer": exact
// attention over the selected blocks only, every query head of a GQA group using its group's
// selection; "MiniMax M3 in vLLM ...", "解码执行": split work merged from partial outputs, and
// "MSA 机制详解": the partial last block and keys after the query position are masked;
// "解码内核中的推测解码": the draft tokens of a sequence are causal among themselves). K and V
// are dequantised from NVFP4 to E4M3 ("NVIDIA Blackwell optimizado kernes MSA") exactly as the
// indexer does; QK^T is an FP8 MMA with fp32 accumulation; the softmax is fp32 (exp2 with the
// log2(e) folded into the scale); PV takes P rounded to f16 and V widened exactly from E4M3 to
// f16, because P rounded to E4M3 (3 mantissa bits) would cost several percent of relative
// error.
//
// GB300 design: two kernels, picked by the batch's max_q_len.
//
// k_attn (every sequence has one query token: plain decode): one CTA of 12 warps per
// (sequence, group, split) that walks the union of the sequence's tokens' selected blocks
// (for one token, its 16 blocks), each block once:
//  * a 3-D tensor copy per block brings the group's K and V regions (144 rows of 128 B,
//    128-byte swizzle) into a 3-deep stage ring;
//  * four dequant warps (thread = key) turn the block into a 128 x 128 E4M3 K tile and a
//    128 x 128 f16 V tile (E4M3 -> f16 is exact) in swizzled shared memory, a 3-deep ring;
//  * eight token warps: the 16 heads of one query token are the M = 16 rows of
//    mma.sync.m16n8k32.e4m3 (S = QK^T, K fragments by ldmatrix) and mma.sync.m16n8k16.f16
//    (O += PV, V fragments by ldmatrix.trans, P straight from the S accumulators), with an
//    online softmax; a token skips the blocks it did not select. A token gets
//    8 / q_len' warps (q_len' = q_len rounded up to a power of two) that split the keys of
//    each block (and, for q_len = 1, alternate blocks too); their states are merged at the end.
//    So one token's 16 blocks are dequantised once by the whole CTA and its keys spread
//    over 8 warps: short per-token latency, for batches of few tokens.
//  * Splits of the union raise the CTA count when B x 4 is small; the partial (lse, o) pairs
//    are merged by log-sum-exp in a second kernel.
// tok::k_attn_tok (multi-token sequences): one CTA per (query token, group, split), described
// where it is defined.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>
#include <mutex>

#include "msa.h"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

constexpr int kTokWarps = 4;                                // warps 0..3: 32 keys of every block each
constexpr int kDqGroups = 2;                                // dequant groups (alternate blocks) ...
constexpr int kDqWarps = 4 * kDqGroups;                     // ... of 4 warps, thread = key: warps 4..11
constexpr int kAttnThreads = 32 * (kTokWarps + kDqWarps);   // 384
constexpr int kStages = 4;                                  // NVFP4 K+V stage ring (a multiple of the groups)
constexpr int kTiles = 3;                                   // dequantised K/V tile ring
constexpr int kStageBytes = 2 * kRegion;                    // K region then V region of one (page, group)
constexpr int kKTile = kBS * kD;                            // 128 keys x 128 E4M3
constexpr int kVTile = kBS * kD * 2;                        // 128 keys x 128 f16
constexpr int kTileBytes = kKTile + kVTile;
constexpr int kBarTok = 1, kBarDq0 = 2;                     // named barriers (0 = __syncthreads; 2, 3 groups)

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
  static constexpr size_t kOffStage = 0;                                                  // 4 x 18 KB
  static constexpr size_t kOffTile = kOffStage + static_cast<size_t>(kStages) * kStageBytes;  // 3 x 48 KB
  static constexpr size_t kOffBar = kOffTile + static_cast<size_t>(kTiles) * kTileBytes;
  // barriers: st_full [kStages]; t_full, t_empty [kTiles]
  static constexpr int kBars = kStages + 2 * kTiles;
  static constexpr size_t kOffLut = kOffBar + 8 * 16;
  static constexpr size_t kOffBlk = kOffLut + 256 * 8;  // the distinct selected blocks, their pages
  static constexpr size_t kOffPhys = kOffBlk + 4 * kSel;
  static constexpr size_t kOffMisc = kOffPhys + 4 * kSel;
  static constexpr size_t kBytes = 1024 + kOffMisc + 64;  // + alignment slack
  // after the block loop the tile ring holds each token warp's final state
  static constexpr size_t kWarpState = 16 * 4 * 2 + 16 * kD * 4;  // m, l, O[16][128]
};
static_assert(AttnSmem::kBars <= 16, "barrier area");
static_assert(AttnSmem::kOffTile % 1024 == 0 && kStageBytes % 1024 == 0, "swizzled stages sit on 1024-B boundaries");
static_assert(kTiles * kTileBytes >= kTokWarps * AttnSmem::kWarpState, "merge area too small");
static_assert(kStages % kDqGroups == 0, "each stage serves one dequant group");
static_assert(AttnSmem::kBytes <= 232448, "shared memory per CTA");

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

__global__ void __launch_bounds__(kAttnThreads, 1) k_attn(const AttnParams p, const __grid_constant__ CUtensorMap tmap) {
  using S = AttnSmem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint64_t* st_full = bars;
  uint64_t* t_full = st_full + kStages;
  uint64_t* t_empty = t_full + kTiles;
  uint2* lut = reinterpret_cast<uint2*>(smem + S::kOffLut);
  int* blk = reinterpret_cast<int*>(smem + S::kOffBlk);
  int* phys = reinterpret_cast<int*>(smem + S::kOffPhys);
  int* nblk = reinterpret_cast<int*>(smem + S::kOffMisc);
  int* bad = reinterpret_cast<int*>(smem + S::kOffMisc + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x % p.splits;
  const int tg = blockIdx.x / p.splits;
  const int t = tg >> 2, g = tg & 3;
  // the sequence of token t (largest b with qsl[b] <= t)
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int q0 = p.qsl[b], ql = p.qsl[b + 1] - q0;
  const int L = p.seq_lens[b];
  if (!(t - q0 >= 0 && t - q0 < ql && ql <= p.max_q_len && L >= ql && L <= p.maxb * kBS)) {
    if (tid == 0 && split == 0 && g == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
    return;
  }
  const int nb = ceil_div(L, kBS);
  const int p_tok = L - ql + (t - q0);

  // ---- prologue --------------------------------------------------------------------------
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) mbar_init(&st_full[i], 1);
    for (int i = 0; i < kTiles; ++i) {
      mbar_init(&t_full[i], 4);  // the four warps of the group that wrote the tile
      mbar_init(&t_empty[i], kTokWarps);
    }
    fence_mbar_init();
    *abort_flag = 0;
    *bad = 0;
  }
  build_dequant_lut(lut, tid, kAttnThreads);
  // the distinct selected blocks of (t, g), in slot order, and their pages
  if (warp == 0) {
    const int v = lane < kSel ? p.sel[(static_cast<int64_t>(t) * 4 + g) * kSel + lane] : -1;
    bool keep = v >= 0 && v < nb;
    if (lane < kSel && v >= nb) {
      set_status(p.status, MSA_ERR_DEVICE_FAULT);
      atomicOr(bad, 1);
    }
    for (int j = 0; j < kSel; ++j) {  // drop repeats of an earlier slot
      const int vj = __shfl_sync(0xffffffffu, v, j);
      if (j < lane && vj == v) keep = false;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, keep && lane < kSel);
    const int pos = __popc(m & ((1u << lane) - 1u));
    if (keep && lane < kSel) {
      blk[pos] = v;
      const int ph = p.block_table[static_cast<int64_t>(b) * p.maxb + v];
      const bool ok = ph >= 0 && ph < p.num_pages;
      phys[pos] = ok ? ph : 0;
      if (!ok) {
        set_status(p.status, MSA_ERR_DEVICE_FAULT);
        atomicOr(bad, 1);
      }
    }
    if (lane == 0) *nblk = __popc(m);
  }
  __syncthreads();
  const bool is_bad = *bad != 0;
  const int nsel = is_bad ? 0 : *nblk;  // a bad entry zero-fills the (token, group): nothing to read
  const int i0 = (nsel * split) / p.splits, i1 = (nsel * (split + 1)) / p.splits;
  const int n = i1 - i0;  // blocks of this CTA: entries i0 .. i1-1

  if (warp >= kTokWarps) {
    // ---- dequant groups: group gq takes blocks gq, gq + 2, ... (stages gq, gq + 2); thread = key
    const int gq = (warp - kTokWarps) >> 2;
    const int kr = 32 * ((warp - kTokWarps) & 3) + lane;
    const bool leader = ((warp - kTokWarps) & 3) == 0 && lane == 0;
    auto issue = [&](int j) {  // the copy of entry i0 + j into stage j % kStages
      uint64_t* bar = &st_full[j % kStages];
      mbar_arrive_expect_tx(bar, kStageBytes);
      tma_load_3d(smem + S::kOffStage + static_cast<size_t>(j % kStages) * kStageBytes, &tmap, 0,
                  2 * g * (kRegion / kD), phys[i0 + j], bar);
    };
    int issued = gq, consumed = gq;  // this group's next entry to copy / to dequantise
    if (leader) {
      prefetch_tensormap(&tmap);
      for (; issued < n && issued < gq + kStages; issued += kDqGroups) issue(issued);
    }
    for (int i = gq; i < n; i += kDqGroups) {
      const int s = i % kStages, x = i % kTiles;
      bool ok = warp_wait(&st_full[s], static_cast<uint32_t>(i / kStages) & 1u, abort_flag);
      ok = ok && warp_wait(&t_empty[x], (static_cast<uint32_t>(i / kTiles) & 1u) ^ 1u, abort_flag);
      RawRow rk, rv;  // key kr's codes and scales, read out of the stage before it is released
      if (ok) {
        const uint8_t* stg = smem + S::kOffStage + static_cast<size_t>(s) * kStageBytes;
        load_row(stg, kr, rk);
        load_row(stg + kRegion, kr, rv);
      }
      // every warp of the group has read stage s (or one of them gave up: all leave together)
      if (named_barrier_or(kBarDq0 + gq, 128, !ok)) {
        if (lane == 0 && !*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
        *abort_flag = 1;
        break;
      }
      consumed = i + kDqGroups;
      if (leader && issued < n) {
        issue(issued);
        issued += kDqGroups;
      }
      uint8_t* kt = smem + S::kOffTile + static_cast<size_t>(x) * kTileBytes;
      uint8_t* vt = kt + kKTile;
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // code word group q = dims 32 q .. 32 q + 31
        uint32_t w[8];
        dequant_quarter(rk, q, lut, w);
        *reinterpret_cast<uint4*>(kt + kr * kD + (((2 * q) ^ (kr & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(kt + kr * kD + (((2 * q + 1) ^ (kr & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[8];
        dequant_quarter(rv, q, lut, w);
#pragma unroll
        for (int h = 0; h < 4; ++h) {  // f16 chunk 4 q + h = dims 32 q + 8 h .. +7
          const uint4 v = make_uint4(cvt_f16x2_e4m3x2(w[2 * h]), cvt_f16x2_e4m3x2(w[2 * h] >> 16),
                                     cvt_f16x2_e4m3x2(w[2 * h + 1]), cvt_f16x2_e4m3x2(w[2 * h + 1] >> 16));
          *reinterpret_cast<uint4*>(vt + kr * (2 * kD) + (((4 * q + h) ^ (kr & 7)) << 4)) = v;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&t_full[x]);
    }
    // copies still in flight after a give-up: wait for them before the CTA's memory goes
    if (leader)
      for (int j = consumed; j < issued; j += kDqGroups)
        if (!mbar_wait_bounded(&st_full[j % kStages], static_cast<uint32_t>(j / kStages) & 1u, kWaitLimitNs, nullptr))
          set_status(p.status, MSA_ERR_TIMEOUT);
    return;
  }

  // ---- token warps: warp w attends keys 32 w .. 32 w + 31 of every block ------------------
  const int gid = lane >> 2, tq = lane & 3;
  WarpState st;
  st.m[0] = st.m[1] = -CUDART_INF_F;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) st.o[k][0] = st.o[k][1] = st.o[k][2] = st.o[k][3] = 0.f;
  uint32_t qa[4][4];
  {
    const uint8_t* qrow0 = p.q + (static_cast<int64_t>(t) * kQHeads + g * kHPG + gid) * kD + 4 * tq;
    const uint8_t* qrow1 = qrow0 + 8 * kD;
#pragma unroll
    for (int s = 0; s < 4; ++s) {  // k-step s: dims 32 s + 4 tq (a0, a1) and 32 s + 16 + 4 tq (a2, a3)
      qa[s][0] = ldg_nc32(qrow0 + 32 * s);
      qa[s][1] = ldg_nc32(qrow1 + 32 * s);
      qa[s][2] = ldg_nc32(qrow0 + 32 * s + 16);
      qa[s][3] = ldg_nc32(qrow1 + 32 * s + 16);
    }
  }
  for (int i = 0; i < n; ++i) {
    const int x = i % kTiles;
    if (!warp_wait(&t_full[x], static_cast<uint32_t>(i / kTiles) & 1u, abort_flag)) {
      if (lane == 0) {
        if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      break;
    }
    const uint8_t* kt = smem + S::kOffTile + static_cast<size_t>(x) * kTileBytes;
    attend_tile(st, qa, kt, kt + kKTile, blk[i0 + i] * kBS, p_tok, p.scale_log2, warp, warp + 1, lane);
    __syncwarp();
    if (lane == 0) mbar_arrive(&t_empty[x]);
  }
  named_barrier(kBarTok, 32 * kTokWarps);  // every token warp is done with the tiles

  // ---- merge the token warps' states, write the output or this split's partial -----------
  uint8_t* ws = smem + S::kOffTile;
  {
    float* mw = reinterpret_cast<float*>(ws + warp * S::kWarpState);
    float* lw = mw + 16;
    float* ow = lw + 16;
    const float l0 = quad_sum(st.l[0]), l1 = quad_sum(st.l[1]);
    if (tq == 0) {
      mw[gid] = st.m[0];
      mw[gid + 8] = st.m[1];
      lw[gid] = l0;
      lw[gid + 8] = l1;
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      *reinterpret_cast<float2*>(ow + gid * kD + 8 * k + 2 * tq) = make_float2(st.o[k][0], st.o[k][1]);
      *reinterpret_cast<float2*>(ow + (gid + 8) * kD + 8 * k + 2 * tq) = make_float2(st.o[k][2], st.o[k][3]);
    }
  }
  named_barrier(kBarTok, 32 * kTokWarps);
  const bool aborted = *abort_flag != 0;
  for (int e = tid; e < kHPG * (kD / 4); e += 32 * kTokWarps) {
    const int hh = e / (kD / 4);
    const int d4 = e % (kD / 4);
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kTokWarps; ++w) M = fmaxf(M, reinterpret_cast<const float*>(ws + w * S::kWarpState)[hh]);
    float Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kTokWarps; ++w) {
        const float* mw = reinterpret_cast<const float*>(ws + w * S::kWarpState);
        const float f = fast_exp2(mw[hh] - M);
        Lsum += mw[16 + hh] * f;
        const float4 o = *reinterpret_cast<const float4*>(mw + 32 + hh * kD + 4 * d4);
        acc.x += o.x * f;
        acc.y += o.y * f;
        acc.z += o.z * f;
        acc.w += o.w * f;
      }
    }
    const bool zero = (M == -CUDART_INF_F) || Lsum <= 0.f || is_bad || aborted;
    const float inv = zero ? 0.f : 1.0f / Lsum;
    const int64_t orow = static_cast<int64_t>(t) * kQHeads + g * kHPG + hh;
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

// ------------------------------------------------------------------------------------------
// Batches of multi-token sequences (max_q_len > 1): one CTA of 8 warps per (query token, group,
// split); a warp owns whole selected blocks (16 query heads x 128 keys):
//  * its block's K and V regions (2 x 9,216 B, contiguous in the page) arrive with one 1-D
//    bulk copy (cp.async.bulk + mbarrier) into the warp's own shared-memory stage;
//  * K is dequantised register-direct into the B fragments of mma.sync.m16n8k32.e4m3 (the
//    16 heads of the group on M), 32 keys at a time, the same lane/dim mapping as the indexer;
//  * V of those 32 keys is dequantised once into a private swizzled f16 tile and read back
//    transposed with ldmatrix.trans for mma.sync.m16n8k16.f16 (P straight from the QK^T
//    accumulators);
//  * online softmax per warp; O is rescaled only when some row maximum moved; the 8 warps'
//    states are merged in shared memory at the end.
// The tokens of one sequence select mostly different blocks (the union of 8 tokens' 16
// selections is 50-80 blocks at 16K context), so sharing a block's dequant across them saves
// little, while coupling them through one tile ring costs more: here each token is its own CTA.
// The next block's copy is issued as soon as the last V chunk of the current block has been
// dequantised, so it overlaps the remaining MMAs.
namespace tok {

constexpr int kAttnWarps = 8;
constexpr int kAttnThreads = 32 * kAttnWarps;
constexpr int kStageBytes = 2 * kRegion;  // K region then V region of one (page, group)
constexpr int kChunkKeys = 32;
constexpr int kVTileBytes = kChunkKeys * kD * 2;  // 32 keys x 128 dims f16

struct TokSmem {
  static constexpr size_t kOffStage = 0;                                        // 8 x 18,432
  static constexpr size_t kOffV = kOffStage + static_cast<size_t>(kAttnWarps) * kStageBytes;  // 8 x 8,192
  static constexpr size_t kOffLut = kOffV + static_cast<size_t>(kAttnWarps) * kVTileBytes;    // 2 KB
  static constexpr size_t kOffBar = kOffLut + 256 * 8;                          // 8 mbarriers
  static constexpr size_t kOffBlk = kOffBar + 8 * kAttnWarps;                   // 16 block ids
  static constexpr size_t kOffPhys = kOffBlk + 4 * kSel;                        // 16 page ids
  static constexpr size_t kOffMisc = kOffPhys + 4 * kSel;
  static constexpr size_t kBytes = kOffMisc + 64;
  // after the block loop, the stage area holds each warp's final state
  static constexpr size_t kWarpState = 16 * 4 * 2 + 16 * kD * 4;  // m, l, O[16][128]
};
static_assert(TokSmem::kOffV >= kAttnWarps * TokSmem::kWarpState, "merge area too small");


// Dequantise keys r0 + gid + 8i (i = 0..3), dims 32t .. 32t+31, of a staged NVFP4 region into
// the f16 tile `vt` (32 rows x 256 B, 16-byte chunk c of row r stored at chunk c ^ (r & 7)).
__device__ __forceinline__ void dequant_v_chunk(const uint8_t* vr, int r0, const uint2* lut, uint8_t* vt, int lane) {
  const int gid = lane >> 2, t = lane & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int rl = gid + 8 * i;  // row inside the tile
    const int r = r0 + rl;       // row inside the block
    const uint4 c = lds128(vr + r * kRowCodes + 16 * t);
    const uint32_t sc = *reinterpret_cast<const uint16_t*>(vr + kScaleOff + r * kRowScales + 2 * t);
    const uint2 e0 = lut[sc & 0xFFu], e1 = lut[sc >> 8];
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {  // word q = dims 32t + 8q .. +7 = f16 chunk 4t + q
      uint32_t lo, hi;
      dq8(w[q], q < 2 ? e0 : e1, lo, hi);
      const uint4 v = make_uint4(cvt_f16x2_e4m3x2(lo), cvt_f16x2_e4m3x2(lo >> 16), cvt_f16x2_e4m3x2(hi),
                                 cvt_f16x2_e4m3x2(hi >> 16));
      *reinterpret_cast<uint4*>(vt + rl * (2 * kD) + (((4 * t + q) ^ (rl & 7)) << 4)) = v;
    }
  }
}

// Copy of the next block into this warp's stage: src == nullptr means a bad page id (the
// barrier phase still completes, with no bytes).
__device__ __forceinline__ void issue_stage(uint8_t* stage, const uint8_t* src, uint64_t* bar) {
  if (src != nullptr) {
    mbar_arrive_expect_tx(bar, kStageBytes);
    bulk_g2s(stage, src, kStageBytes, bar);
  } else {
    mbar_arrive(bar);
  }
}

// One block of 128 keys (K, V staged at kr, kr + kRegion) for the 16 heads of this warp.
// Once every key and value of the stage has been read, lane 0 starts the copy of the warp's
// next block (has_next; next_src as for issue_stage) into the same stage.
__device__ __forceinline__ void attend_block(WarpState& st, const uint32_t (&qa)[4][4], uint8_t* kr,
                                             const uint2* lut, uint8_t* vt, int blk_pos0, int p_tok, float scale_log2,
                                             int lane, bool has_next, const uint8_t* next_src, uint64_t* bar) {
  const int gid = lane >> 2, t = lane & 3;
  const uint8_t* vr = kr + kRegion;
  bool issued = !has_next;
#pragma unroll 1
  for (int c = 0; c < kBS / kChunkKeys; ++c) {
    const int k0 = c * kChunkKeys;
    if (blk_pos0 + k0 > p_tok) break;  // every remaining key lies after the query position
    // ---- S = Q K^T for keys k0 .. k0+31 (4 n-tiles of 8 keys)
    float x[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int key = k0 + 8 * j + gid;
      const uint4 cw = lds128(kr + key * kRowCodes + 16 * t);
      const uint32_t sc = *reinterpret_cast<const uint16_t*>(kr + kScaleOff + key * kRowScales + 2 * t);
      const uint2 e0 = lut[sc & 0xFFu], e1 = lut[sc >> 8];
      uint32_t b[4][2];
      dq8(cw.x, e0, b[0][0], b[0][1]);
      dq8(cw.y, e0, b[1][0], b[1][1]);
      dq8(cw.z, e1, b[2][0], b[2][1]);
      dq8(cw.w, e1, b[3][0], b[3][1]);
      mma_e4m3_zc(x[j], qa[0][0], qa[0][1], qa[0][2], qa[0][3], b[0][0], b[0][1]);
#pragma unroll
      for (int s = 1; s < 4; ++s) mma_e4m3(x[j], qa[s][0], qa[s][1], qa[s][2], qa[s][3], b[s][0], b[s][1]);
    }
    // ---- V of these keys -> f16 tile; after the last chunk the stage is fully read
    dequant_v_chunk(vr, k0, lut, vt, lane);
    if (!issued && (c == kBS / kChunkKeys - 1 || blk_pos0 + k0 + kChunkKeys > p_tok)) {
      __syncwarp();
      if (lane == 0) issue_stage(kr, next_src, bar);
      issued = true;
    }
    // ---- scale, causal mask, online softmax
    const bool need_mask = blk_pos0 + k0 + kChunkKeys - 1 > p_tok;
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
    __syncwarp();  // the V tile is complete
    // ---- O += P V: 2 k-steps of 16 keys, 8 pairs of 8-dim n-tiles
    const int mi = lane >> 3, ri = lane & 7;
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
      const uint32_t a0 = pack_f16x2(x[2 * kk][0], x[2 * kk][1]);
      const uint32_t a1 = pack_f16x2(x[2 * kk][2], x[2 * kk][3]);
      const uint32_t a2 = pack_f16x2(x[2 * kk + 1][0], x[2 * kk + 1][1]);
      const uint32_t a3 = pack_f16x2(x[2 * kk + 1][2], x[2 * kk + 1][3]);
      const int rl = 16 * kk + (mi & 1) * 8 + ri;
      const uint8_t* vrow = vt + rl * (2 * kD);
#pragma unroll
      for (int dn = 0; dn < 8; ++dn) {
        const int chunk = 2 * dn + (mi >> 1);
        uint32_t r[4];
        ldmatrix_x4_trans(r, vrow + ((chunk ^ (rl & 7)) << 4));
        mma_f16(st.o[2 * dn], a0, a1, a2, a3, r[0], r[1]);
        mma_f16(st.o[2 * dn + 1], a0, a1, a2, a3, r[2], r[3]);
      }
    }
    __syncwarp();  // before the next chunk overwrites the V tile
  }
  if (!issued) {  // (not reached: the first chunk always holds a valid key)
    __syncwarp();
    if (lane == 0) issue_stage(kr, next_src, bar);
  }
}

__global__ void __launch_bounds__(kAttnThreads, 1) k_attn_tok(const AttnParams p) {
  using S = TokSmem;
  extern __shared__ __align__(128) uint8_t smem[];
  uint2* lut = reinterpret_cast<uint2*>(smem + S::kOffLut);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  int* blk = reinterpret_cast<int*>(smem + S::kOffBlk);
  int* phys = reinterpret_cast<int*>(smem + S::kOffPhys);
  int* nblk = reinterpret_cast<int*>(smem + S::kOffMisc);
  int* bad = reinterpret_cast<int*>(smem + S::kOffMisc + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x % p.splits;
  const int tg = blockIdx.x / p.splits;
  const int t = tg >> 2, g = tg & 3;

  // the sequence of token t (largest b with qsl[b] <= t)
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int q0 = p.qsl[b], ql = p.qsl[b + 1] - q0;
  const int L = p.seq_lens[b];
  if (!(t - q0 < ql && ql <= p.max_q_len && L >= ql && L <= p.maxb * kBS)) {
    if (tid == 0 && split == 0 && g == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
    return;
  }
  const int nb = ceil_div(L, kBS);
  const int p_tok = L - ql + (t - q0);

  if (tid == 0) {
    for (int w = 0; w < kAttnWarps; ++w) mbar_init(&bars[w], 1);
    fence_mbar_init();
    *abort_flag = 0;
    *bad = 0;
  }
  build_dequant_lut(lut, tid, kAttnThreads);
  // ---- the distinct selected blocks of (t, g), in slot order, and their pages
  if (warp == 0) {
    const int v = lane < kSel ? p.sel[(static_cast<int64_t>(t) * 4 + g) * kSel + lane] : -1;
    bool keep = v >= 0 && v < nb;
    if (lane < kSel && v >= nb) {
      set_status(p.status, MSA_ERR_DEVICE_FAULT);
      atomicOr(bad, 1);
    }
    // drop repeats of an earlier slot
    for (int j = 0; j < kSel; ++j) {
      const int vj = __shfl_sync(0xffffffffu, v, j);
      if (j < lane && vj == v) keep = false;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, keep && lane < kSel);
    const int pos = __popc(m & ((1u << lane) - 1u));
    if (keep && lane < kSel) {
      blk[pos] = v;
      const int ph = p.block_table[static_cast<int64_t>(b) * p.maxb + v];
      const bool ok = ph >= 0 && ph < p.num_pages;
      phys[pos] = ok ? ph : -1;
      if (!ok) {
        set_status(p.status, MSA_ERR_DEVICE_FAULT);
        atomicOr(bad, 1);
      }
    }
    if (lane == 0) *nblk = __popc(m);
  }
  __syncthreads();
  const int n = *nblk;
  const bool is_bad = *bad != 0;
  const int i0 = (n * split) / p.splits, i1 = (n * (split + 1)) / p.splits;

  // ---- per-warp blocks i0 + warp, i0 + warp + 8, ...
  const int gid = lane >> 2, tq = lane & 3;
  WarpState st;
  st.m[0] = st.m[1] = -CUDART_INF_F;
  st.l[0] = st.l[1] = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) st.o[k][0] = st.o[k][1] = st.o[k][2] = st.o[k][3] = 0.f;
  uint32_t qa[4][4];
  {
    const uint8_t* qrow0 = p.q + (static_cast<int64_t>(t) * kQHeads + g * kHPG + gid) * kD + 32 * tq;
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
  uint8_t* stage = smem + S::kOffStage + static_cast<size_t>(warp) * kStageBytes;
  uint8_t* vt = smem + S::kOffV + static_cast<size_t>(warp) * kVTileBytes;
  uint64_t* bar = &bars[warp];
  auto src_of = [&](int i) -> const uint8_t* {
    const int ph = phys[i];
    return ph >= 0 ? p.kv_pages + static_cast<int64_t>(ph) * kKvPage + (2 * g) * kRegion : nullptr;
  };
  int it = 0;
  bool inflight = false;
  if (!is_bad && i0 + warp < i1) {
    if (lane == 0) issue_stage(stage, src_of(i0 + warp), bar);
    inflight = true;
  }
  for (int i = i0 + warp; !is_bad && i < i1; i += kAttnWarps, ++it) {
    if (!mbar_wait_bounded(bar, static_cast<uint32_t>(it) & 1u, kWaitLimitNs, abort_flag)) {
      if (lane == 0) {
        if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      break;  // inflight stays true: drained below
    }
    const bool has_next = i + kAttnWarps < i1;
    // the copy of the next block starts inside, once this stage has been fully read
    attend_block(st, qa, stage, lut, vt, blk[i] * kBS, p_tok, p.scale_log2, lane, has_next,
                 has_next ? src_of(i + kAttnWarps) : nullptr, bar);
    inflight = has_next;
  }
  if (inflight && lane == 0) {
    // a copy into this warp's stage may still be in flight: wait for it (bounded)
    mbar_wait_bounded(bar, static_cast<uint32_t>(it) & 1u, kWaitLimitNs, nullptr);
  }
  __syncthreads();

  // ---- merge the 8 warps' states, write the output or this split's partial --------------
  uint8_t* ws = smem;  // reuse the stages
  {
    float* mw = reinterpret_cast<float*>(ws + warp * S::kWarpState);
    float* lw = mw + 16;
    float* ow = lw + 16;
    const float l0 = quad_sum(st.l[0]), l1 = quad_sum(st.l[1]);
    if (tq == 0) {
      mw[gid] = st.m[0];
      mw[gid + 8] = st.m[1];
      lw[gid] = l0;
      lw[gid + 8] = l1;
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      *reinterpret_cast<float2*>(ow + gid * kD + 8 * k + 2 * tq) = make_float2(st.o[k][0], st.o[k][1]);
      *reinterpret_cast<float2*>(ow + (gid + 8) * kD + 8 * k + 2 * tq) = make_float2(st.o[k][2], st.o[k][3]);
    }
  }
  __syncthreads();
  for (int e = tid; e < kHPG * (kD / 4); e += kAttnThreads) {
    const int d4 = e % (kD / 4);
    const int hh = e / (kD / 4);
    float M = -CUDART_INF_F;
#pragma unroll
    for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, reinterpret_cast<const float*>(ws + w * S::kWarpState)[hh]);
    float Lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int w = 0; w < kAttnWarps; ++w) {
        const float* mw = reinterpret_cast<const float*>(ws + w * S::kWarpState);
        const float f = fast_exp2(mw[hh] - M);
        Lsum += mw[16 + hh] * f;
        const float4 o = *reinterpret_cast<const float4*>(mw + 32 + hh * kD + 4 * d4);
        acc.x += o.x * f;
        acc.y += o.y * f;
        acc.z += o.z * f;
        acc.w += o.w * f;
      }
    }
    const bool zero = (M == -CUDART_INF_F) || Lsum <= 0.f || is_bad;
    const float inv = zero ? 0.f : 1.0f / Lsum;
    const int64_t orow = static_cast<int64_t>(t) * kQHeads + g * kHPG + hh;
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

}  // namespace tok

// ------------------------------------------------------------------------------------------
// Batches of many tokens, on the 5th-generation tensor cores: one CTA of 16 warps per (query
// token, group, split). The keys of a block are the M = 128 rows of both tcgen05 MMAs, so the
// accumulators live in TMEM and the CUDA cores only dequantise and run the softmax:
//  * S^T = K Q^T: kind::f8f6f4, A = the block's 128 x 128 E4M3 K tile in TMEM (the K dequant
//    threads store their key row with tcgen05.st), B = the token's 16 x 128 E4M3 query tile
//    (K-major, 128-byte swizzle, one tensor copy), N = 16 heads, into a ring of two TMEM
//    score buffers; one warp issues these;
//  * O^T += V^T P^T: kind::f16, A = the block's V tile as f16 (E4M3 -> f16 exact) in shared
//    memory, MN-major with 128-byte swizzle, B = P^T (16 heads x 128 keys, K-major, 128-byte
//    swizzle), N = 16, into one TMEM accumulator of 128 dims x 16 heads; another warp issues
//    these (an MMA costs ~80 cycles of issue, so S and PV each get their own issuer);
//  * three groups of four warps, thread = key = TMEM lane: K dequant, V dequant, softmax. A
//    softmax thread reads its key's 16 head scores and writes P = exp2(s - m). The reference
//    maximum m of a head only moves when some score of a block exceeds it by more than 2^8 (a
//    vote of the four softmax warps), so P <= 256 in f16, the block maximum is reduced across
//    the 128 threads only then, and O^T is rescaled in TMEM only then (after the PV MMA in
//    flight has landed);
//  * the output is O^T / l, the per-head sum l reduced across the 128 threads once.
namespace tc {

constexpr int kWarpProd = 0, kWarpMmaS = 1, kWarpMmaO = 2;  // warp 3 idles
constexpr int kWarpK = 4, kWarpV = 8, kWarpSm = 12;         // groups of four warps
constexpr int kThreads = 32 * 16;
constexpr int kStages = 4;                                   // NVFP4 K+V stage ring
constexpr int kStageBytes = 2 * kRegion;                     // K region then V region of one (page, group)
constexpr int kQTile = kHPG * kD;                            // 16 heads x 128 E4M3
constexpr int kVTile = kBS * kD * 2;                         // 128 keys x 128 f16
constexpr int kPTile = kHPG * kBS * 2;                       // 16 heads x 128 keys f16
constexpr uint32_t kVLbo = 16384;                            // V tile: the two 64-dim atom columns
constexpr uint32_t kVSbo = 1024;                             //         8-key groups
constexpr float kRescaleLog2 = 8.0f;                         // m moves when a score exceeds it by this
constexpr int kBarWork = 4;                                  // named barrier of the softmax warps
// TMEM columns: K tiles [2] 0..63, S^T [2] 64..95, O^T 96..111
constexpr uint32_t kColK = 0, kColS = 64, kColO = 96;
constexpr int kTmemCols = 128;

struct Smem {
  static constexpr size_t kOffQ = 0;                                                     // 2 KB
  static constexpr size_t kOffStage = 1024 * 2;                                           // 4 x 18 KB
  static constexpr size_t kOffV = kOffStage + static_cast<size_t>(kStages) * kStageBytes;  // 2 x 32 KB
  static constexpr size_t kOffP = kOffV + 2 * static_cast<size_t>(kVTile);                // 2 x 4 KB
  static constexpr size_t kOffBar = kOffP + 2 * static_cast<size_t>(kPTile);
  // q_full; st_full, st_empty [kStages]; ka_full, ka_empty, v_full, v_empty, s_full, s_empty,
  // p_full, p_empty [2]; o_final; fin_s; fin_o
  static constexpr int kBars = 1 + 2 * kStages + 2 * 8 + 3;
  static constexpr size_t kOffLut = kOffBar + 8 * 32;
  static constexpr size_t kOffRed = kOffLut + 256 * 8;   // [2][4 warps][16] fp32
  static constexpr size_t kOffBlk = kOffRed + 2 * 4 * 16 * 4;
  static constexpr size_t kOffPhys = kOffBlk + 4 * kSel;
  static constexpr size_t kOffMisc = kOffPhys + 4 * kSel;
  static constexpr size_t kBytes = 1024 + kOffMisc + 64;  // + alignment slack
};
static_assert(Smem::kBars <= 32, "barrier area");
static_assert(Smem::kOffStage % 1024 == 0 && Smem::kOffV % 1024 == 0 && Smem::kOffP % 1024 == 0,
              "swizzled tiles sit on 1024-B boundaries");
static_assert(Smem::kBytes <= 232448, "shared memory per CTA");

// Op-reduce v[0..15] over the 32 lanes: afterwards lanes 2h and 2h + 1 hold head h's result.
template <bool kMax>
__device__ __forceinline__ float warp_reduce16(const float (&v)[16], int lane) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  float a8[8], a4[4], a2[2];
  const bool u16 = lane & 16, u8 = lane & 8, u4 = lane & 4, u2 = lane & 2;
#pragma unroll
  for (int i = 0; i < 8; ++i) {  // keep heads 8..15 in lanes with bit 4 set
    const float send = u16 ? v[i] : v[i + 8], keep = u16 ? v[i + 8] : v[i];
    a8[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float send = u8 ? a8[i] : a8[i + 4], keep = u8 ? a8[i + 4] : a8[i];
    a4[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float send = u4 ? a4[i] : a4[i + 2], keep = u4 ? a4[i + 2] : a4[i];
    a2[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
  }
  const float send = u2 ? a2[0] : a2[1], keep = u2 ? a2[1] : a2[0];
  const float a1 = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
  return op(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
}

// Op-reduce v[0..15] over the 128 worker threads into out[0..15] (the same in every thread).
// red: [4][16] fp32 shared scratch, not reused before every worker has passed the next call's
// barrier (the caller alternates two of them).
template <bool kMax>
__device__ __forceinline__ void group_reduce16(const float (&v)[16], float (&out)[16], float* red, int wq, int lane) {
  const float r = warp_reduce16<kMax>(v, lane);
  if ((lane & 1) == 0) red[wq * 16 + (lane >> 1)] = r;
  named_barrier(kBarWork, 128);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float4 x0 = *reinterpret_cast<const float4*>(red + 4 * c);
    const float4 x1 = *reinterpret_cast<const float4*>(red + 16 + 4 * c);
    const float4 x2 = *reinterpret_cast<const float4*>(red + 32 + 4 * c);
    const float4 x3 = *reinterpret_cast<const float4*>(red + 48 + 4 * c);
    if (kMax) {
      out[4 * c + 0] = fmaxf(fmaxf(x0.x, x1.x), fmaxf(x2.x, x3.x));
      out[4 * c + 1] = fmaxf(fmaxf(x0.y, x1.y), fmaxf(x2.y, x3.y));
      out[4 * c + 2] = fmaxf(fmaxf(x0.z, x1.z), fmaxf(x2.z, x3.z));
      out[4 * c + 3] = fmaxf(fmaxf(x0.w, x1.w), fmaxf(x2.w, x3.w));
    } else {
      out[4 * c + 0] = (x0.x + x1.x) + (x2.x + x3.x);
      out[4 * c + 1] = (x0.y + x1.y) + (x2.y + x3.y);
      out[4 * c + 2] = (x0.z + x1.z) + (x2.z + x3.z);
      out[4 * c + 3] = (x0.w + x1.w) + (x2.w + x3.w);
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const AttnParams p, const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map) {
  using S = Smem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint64_t* q_full = bars;
  uint64_t* st_full = bars + 1;
  uint64_t* st_empty = st_full + kStages;
  uint64_t* ka_full = st_empty + kStages;
  uint64_t* ka_empty = ka_full + 2;
  uint64_t* v_full = ka_empty + 2;
  uint64_t* v_empty = v_full + 2;
  uint64_t* s_full = v_empty + 2;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* p_empty = p_full + 2;
  uint64_t* o_final = p_empty + 2;
  uint64_t* fin_s = o_final + 1;
  uint64_t* fin_o = fin_s + 1;
  uint2* lut = reinterpret_cast<uint2*>(smem + S::kOffLut);
  float* red = reinterpret_cast<float*>(smem + S::kOffRed);
  int* blk = reinterpret_cast<int*>(smem + S::kOffBlk);
  int* phys = reinterpret_cast<int*>(smem + S::kOffPhys);
  int* nblk = reinterpret_cast<int*>(smem + S::kOffMisc);
  int* bad = reinterpret_cast<int*>(smem + S::kOffMisc + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffMisc + 12);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x % p.splits;
  const int tg = blockIdx.x / p.splits;
  const int t = tg >> 2, g = tg & 3;
  int lo = 0, hi = p.B - 1;  // the sequence of token t (largest b with qsl[b] <= t)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int q0 = p.qsl[b], ql = p.qsl[b + 1] - q0;
  const int L = p.seq_lens[b];
  if (!(t - q0 >= 0 && t - q0 < ql && ql <= p.max_q_len && L >= ql && L <= p.maxb * kBS)) {
    if (tid == 0 && split == 0 && g == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
    return;
  }
  const int nb = ceil_div(L, kBS);
  const int p_tok = L - ql + (t - q0);

  // ---- prologue --------------------------------------------------------------------------
  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&st_full[i], 1);
      mbar_init(&st_empty[i], 8);  // the K and the V dequant warps
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ka_full[i], 4);
      mbar_init(&ka_empty[i], 1);
      mbar_init(&v_full[i], 4);
      mbar_init(&v_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&p_empty[i], 1);
    }
    mbar_init(o_final, 1);
    mbar_init(fin_s, 1);
    mbar_init(fin_o, 1);
    fence_mbar_init();
    *abort_flag = 0;
    *bad = 0;
  }
  if (warp == kWarpMmaS) tmem_alloc(tmem_slot, kTmemCols);
  build_dequant_lut(lut, tid, kThreads);
  if (warp == kWarpProd) {  // the distinct selected blocks of (t, g), in slot order, and their pages
    const int v = lane < kSel ? p.sel[(static_cast<int64_t>(t) * 4 + g) * kSel + lane] : -1;
    bool keep = v >= 0 && v < nb;
    if (lane < kSel && v >= nb) {
      set_status(p.status, MSA_ERR_DEVICE_FAULT);
      atomicOr(bad, 1);
    }
    for (int j = 0; j < kSel; ++j) {
      const int vj = __shfl_sync(0xffffffffu, v, j);
      if (j < lane && vj == v) keep = false;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, keep && lane < kSel);
    const int pos = __popc(m & ((1u << lane) - 1u));
    if (keep && lane < kSel) {
      blk[pos] = v;
      const int ph = p.block_table[static_cast<int64_t>(b) * p.maxb + v];
      const bool ok = ph >= 0 && ph < p.num_pages;
      phys[pos] = ok ? ph : 0;
      if (!ok) {
        set_status(p.status, MSA_ERR_DEVICE_FAULT);
        atomicOr(bad, 1);
      }
    }
    if (lane == 0) *nblk = __popc(m);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const bool is_bad = *bad != 0;
  const int nsel = is_bad ? 0 : *nblk;
  const int i0 = (nsel * split) / p.splits, i1 = (nsel * (split + 1)) / p.splits;
  const int n = i1 - i0;  // blocks of this CTA: entries i0 .. i1-1
  bool ok = true;
  auto give_up = [&]() {
    if (lane == 0) {
      if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
      *abort_flag = 1;
    }
  };
  // a give-up stops this warp's work at once; every later wait is skipped
  auto wait_ok = [&](uint64_t* bar, uint32_t parity) {
    if (!ok) return false;
    ok = warp_wait(bar, parity, abort_flag);
    if (!ok) give_up();
    return ok;
  };

  if (warp == kWarpProd) {
    // ---- producer ------------------------------------------------------------------------
    if (lane == 0 && n > 0) {
      prefetch_tensormap(&kv_map);
      prefetch_tensormap(&q_map);
      mbar_arrive_expect_tx(q_full, kQTile);
      tma_load_2d(smem + S::kOffQ, &q_map, 0, t * kQHeads + g * kHPG, q_full, policy_evict_first());
      int issued = 0;
      for (int j = 0; j < n; ++j) {
        const int s = j % kStages;
        if (!mbar_wait(&st_empty[s], (static_cast<uint32_t>(j / kStages) & 1u) ^ 1u, abort_flag)) {
          if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&st_full[s], kStageBytes);
        tma_load_3d(smem + S::kOffStage + static_cast<size_t>(s) * kStageBytes, &kv_map, 0, 2 * g * (kRegion / kD),
                    phys[i0 + j], &st_full[s]);
        issued = j + 1;
      }
      // copies that nobody waited for (after a give-up): wait before the CTA's memory goes
      for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
        if (!mbar_wait_bounded(&st_full[j % kStages], static_cast<uint32_t>(j / kStages) & 1u, kWaitLimitNs, nullptr))
          set_status(p.status, MSA_ERR_TIMEOUT);
      if (!mbar_wait_bounded(q_full, 0u, kWaitLimitNs, nullptr)) set_status(p.status, MSA_ERR_TIMEOUT);
    }
  } else if (warp == kWarpMmaS) {
    // ---- S(j) = K(j) Q^T; the whole warp runs the loop, lane 0 issues ------------------------
    constexpr uint32_t idesc_s = idesc_e4m3_f32(128, kHPG);
    const uint64_t dq = sw128_kmajor_desc(smem_u32(smem + S::kOffQ));
    if (n > 0) wait_ok(q_full, 0u);
    for (int j = 0; ok && j < n; ++j) {
      const int x = j & 1;
      const uint32_t par = static_cast<uint32_t>(j >> 1) & 1u;
      if (!wait_ok(&ka_full[x], par) || !wait_ok(&s_empty[x], par ^ 1u)) break;
      tc_fence_after();
      if (lane == 0) {
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = 32 E4M3 per MMA: 8 TMEM columns of A, +32 B of B
          tc_mma_f8_ta(tmem + kColS + 16 * x, tmem + kColK + 32 * x + 8 * k, dq + 2 * k, idesc_s, k > 0 ? 1u : 0u);
        tc_commit(&s_full[x]);
        tc_commit(&ka_empty[x]);
      }
      __syncwarp();
    }
    if (lane == 0) {  // nothing of this warp's is in flight when TMEM is released
      tc_commit(fin_s);
      if (!mbar_wait_bounded(fin_s, 0u, kWaitLimitNs, nullptr)) set_status(p.status, MSA_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kWarpMmaO) {
    // ---- O^T += V(j)^T P(j)^T ------------------------------------------------------------------
    constexpr uint32_t idesc_o = idesc_f16_f32_amn(128, kHPG);
    for (int j = 0; ok && j < n; ++j) {
      const int x = j & 1;
      const uint32_t par = static_cast<uint32_t>(j >> 1) & 1u;
      if (!wait_ok(&v_full[x], par) || !wait_ok(&p_full[x], par)) break;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t dv = sw128_mnmajor_desc(smem_u32(smem + S::kOffV + static_cast<size_t>(x) * kVTile), kVLbo, kVSbo);
        const uint64_t dp = sw128_kmajor_desc(smem_u32(smem + S::kOffP + static_cast<size_t>(x) * kPTile));
#pragma unroll
        for (int k = 0; k < 8; ++k)  // K = 16 keys per MMA: two 8-key groups of V; 32 B (or the next atom) of P
          tc_mma_f16(tmem + kColO, dv + ((2 * kVSbo) >> 4) * k, dp + (((k >> 2) * 2048 + (k & 3) * 32) >> 4), idesc_o,
                     (j > 0 || k > 0) ? 1u : 0u);
        tc_commit(&v_empty[x]);
        tc_commit(&p_empty[x]);
      }
      __syncwarp();
    }
    if (lane == 0) {
      tc_commit(o_final);  // every PV issued has landed (the softmax warps read O^T after it)
      tc_commit(fin_o);
      if (!mbar_wait_bounded(fin_o, 0u, kWaitLimitNs, nullptr)) set_status(p.status, MSA_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= kWarpK && warp < kWarpV) {
    // ---- K dequant: thread = key kr = TMEM lane; the row goes to K tile x in TMEM ------------
    const int kr = 32 * (warp & 3) + lane;
    const uint32_t lanes = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    for (int j = 0; j < n; ++j) {
      const int s = j % kStages, x = j & 1;
      if (!wait_ok(&st_full[s], static_cast<uint32_t>(j / kStages) & 1u)) break;
      RawRow rk;
      load_row(smem + S::kOffStage + static_cast<size_t>(s) * kStageBytes, kr, rk);
      __syncwarp();
      if (lane == 0) mbar_arrive(&st_empty[s]);
      if (!wait_ok(&ka_empty[x], (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u)) break;  // S(j - 2) has landed
      uint32_t w[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t u[8];
        dequant_quarter(rk, q, lut, u);
#pragma unroll
        for (int e = 0; e < 8; ++e) w[8 * q + e] = u[e];
      }
      tc_fence_after();
      tmem_st32(tmem + lanes + kColK + 32 * x, w);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ka_full[x]);
    }
  } else if (warp >= kWarpV && warp < kWarpSm) {
    // ---- V dequant: thread = key kr; the row goes to the f16 V tile x (MN-major: K row kr) ---
    const int kr = 32 * (warp & 3) + lane;
    for (int j = 0; j < n; ++j) {
      const int s = j % kStages, x = j & 1;
      if (!wait_ok(&st_full[s], static_cast<uint32_t>(j / kStages) & 1u)) break;
      RawRow rv;
      load_row(smem + S::kOffStage + static_cast<size_t>(s) * kStageBytes + kRegion, kr, rv);
      __syncwarp();
      if (lane == 0) mbar_arrive(&st_empty[s]);
      if (!wait_ok(&v_empty[x], (static_cast<uint32_t>(j >> 1) & 1u) ^ 1u)) break;  // PV(j - 2) has landed
      uint8_t* vt = smem + S::kOffV + static_cast<size_t>(x) * kVTile + (kr >> 3) * kVSbo + (kr & 7) * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t u[8];
        dequant_quarter(rv, q, lut, u);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {  // dims 32 q + 8 hh .. +7 = chunk cc = 4 q + hh
          const int cc = 4 * q + hh;
          const uint4 v = make_uint4(cvt_f16x2_e4m3x2(u[2 * hh]), cvt_f16x2_e4m3x2(u[2 * hh] >> 16),
                                     cvt_f16x2_e4m3x2(u[2 * hh + 1]), cvt_f16x2_e4m3x2(u[2 * hh + 1] >> 16));
          *reinterpret_cast<uint4*>(vt + (cc >> 3) * kVLbo + (((cc & 7) ^ (kr & 7)) << 4)) = v;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&v_full[x]);
    }
  } else if (warp >= kWarpSm) {
    // ---- softmax: thread = key kr = TMEM lane --------------------------------------------------
    const int wq = warp & 3;
    const int kr = 32 * wq + lane;
    const uint32_t lanes = static_cast<uint32_t>(32 * wq) << 16;
    const float c = p.scale_log2;
    float m_ref[16], l[16];
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      m_ref[h] = -CUDART_INF_F;
      l[h] = 0.f;
    }
    int nred = 0;  // reductions done: alternates the two scratch buffers
    for (int j = 0; j < n; ++j) {
      const int x = j & 1;
      const uint32_t par = static_cast<uint32_t>(j >> 1) & 1u;
      float xs[16];
      if (wait_ok(&s_full[x], par)) {
        tc_fence_after();
        uint32_t r[16];
        tmem_ld16(tmem + lanes + kColS + 16 * x, r);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[x]);
        const bool valid = blk[i0 + j] * kBS + kr <= p_tok;
#pragma unroll
        for (int h = 0; h < 16; ++h) xs[h] = valid ? __uint_as_float(r[h]) * c : -CUDART_INF_F;
      } else {
#pragma unroll
        for (int h = 0; h < 16; ++h) xs[h] = -CUDART_INF_F;
      }
      bool need = false;
#pragma unroll
      for (int h = 0; h < 16; ++h) need |= xs[h] > m_ref[h] + kRescaleLog2;
      if (named_barrier_or(kBarWork, 128, need)) {  // the same answer in all four warps
        float bm[16];
        group_reduce16<true>(xs, bm, red + 64 * (nred & 1), wq, lane);
        ++nred;
        float cf[16];
        bool moved = false;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float mn = fmaxf(m_ref[h], bm[h]);
          cf[h] = (m_ref[h] == -CUDART_INF_F) ? 0.f : fast_exp2(m_ref[h] - mn);
          moved |= mn != m_ref[h];
          m_ref[h] = mn;
          l[h] *= cf[h];
        }
        // O^T *= cf once PV(j - 1) has landed (PV(j) waits for this block's P)
        if (moved && j > 0 && wait_ok(&p_empty[(j - 1) & 1], static_cast<uint32_t>((j - 1) >> 1) & 1u)) {
          tc_fence_after();
          uint32_t o[16];
          tmem_ld16(tmem + lanes + kColO, o);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 16; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * cf[h]);
          tmem_st16(tmem + lanes + kColO, o);
          tmem_wait_st();
          tc_fence_before();
        }
      }
      // P = exp2(x - m) -> P^T tile x (free once PV(j - 2) has landed): row h, key kr
      if (wait_ok(&p_empty[x], par ^ 1u)) {
        uint8_t* pt = smem + S::kOffP + static_cast<size_t>(x) * kPTile + (kr >> 6) * 2048 + (kr & 7) * 2;
        const int ch = (kr & 63) >> 3;
#pragma unroll
        for (int h = 0; h < 16; ++h) {
          const float mu = m_ref[h] == -CUDART_INF_F ? 0.f : m_ref[h];
          const float pv = fast_exp2(xs[h] - mu);
          l[h] += pv;
          *reinterpret_cast<__half*>(pt + (h >> 3) * 1024 + (h & 7) * 128 + ((ch ^ (h & 7)) << 4)) = __float2half_rn(pv);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[x]);
      }
    }
    // ---- output: lane kr = dim kr of O^T; l summed over the 128 keys' threads --------------
    float lt[16];
    group_reduce16<false>(l, lt, red + 64 * (nred & 1), wq, lane);
    uint32_t o[16];
    const bool have = n > 0 && ok && mbar_wait(o_final, 0u, abort_flag);
    if (have) {
      tc_fence_after();
      tmem_ld16(tmem + lanes + kColO, o);
      tmem_wait_ld();
    }
    const bool zero = !have || is_bad || *abort_flag != 0;
#pragma unroll
    for (int h = 0; h < 16; ++h) {
      const bool z = zero || !(lt[h] > 0.f);
      const float val = z ? 0.f : __uint_as_float(o[h]) / lt[h];
      const int64_t orow = static_cast<int64_t>(t) * kQHeads + g * kHPG + h;
      if (p.splits == 1) {
        reinterpret_cast<__nv_bfloat16*>(p.out)[orow * kD + kr] = __float2bfloat16_rn(val);
      } else {
        const int64_t prow = static_cast<int64_t>(split) * p.T * kQHeads + orow;
        p.part_o[prow * kD + kr] = val;
        if (kr == 0) p.part_lse[prow] = z ? -CUDART_INF_F : m_ref[h] + __log2f(lt[h]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMmaS) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace tc

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

// The two kernels trade latency for throughput: k_attn spreads one (token, group) over a whole
// SM (the keys of each block over four warps, the dequant over eight), so a batch of few tokens
// finishes in one short wave; tok::k_attn_tok packs a (token, group) into 8 warps that each own
// whole blocks, which uses the SM better once there are several waves of CTAs. Measured on
// GB300: T = 8 and 32 tokens run 1.4-1.9x faster on k_attn, T = 512 1.2x faster on k_attn_tok.
bool use_tok_kernel(int T) { return 4 * T > 2 * 152; }

// Splits of each (query token, group)'s blocks for the per-token kernel, from T alone: enough
// CTAs for about two per SM of a 152-SM GB300, at most 16 (one block per split).
int tok_splits(int T) {
  const int items = 4 * T;
  if (items <= 0 || items >= 304) return 1;
  const int s = (304 + items - 1) / items;
  return s > 16 ? 16 : s;
}

size_t attn_ws_bytes(int T, int splits) {
  if (splits <= 1) return 0;
  const size_t rows = static_cast<size_t>(splits) * T * kQHeads;
  return msa_host::align256(rows * kD * 4) + msa_host::align256(rows * 4);
}

// Argument checks shared by both entry points; fills everything of p but the partial buffers.
// Returns MSA_OK with p->T == 0 when there is nothing to do.
msa_status attn_setup(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache, const uint8_t* q,
                      const int32_t* sel, float softmax_scale, int32_t num_splits, uint16_t* out, uint32_t* status,
                      AttnParams* p) {
  p->T = 0;
  msa_status st = msa_host::check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = msa_host::check_batch(batch)) != MSA_OK) return st;
  if ((st = msa_host::check_cache(cache, false, true)) != MSA_OK) return st;
  if (num_splits < 0 || num_splits > kMaxSplits) return MSA_ERR_INVALID_ARG;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (q == nullptr || sel == nullptr || out == nullptr || !msa_host::aligned(q, 16) || !msa_host::aligned(sel, 4) ||
      !msa_host::aligned(out, 16))
    return MSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || softmax_scale != softmax_scale) return MSA_ERR_INVALID_ARG;
  p->B = batch->B;
  p->T = batch->T;
  p->maxb = batch->max_blocks_per_seq;
  p->max_q_len = batch->max_q_len;
  p->num_pages = cache->num_pages;
  p->splits = num_splits > 0 ? num_splits
                             : (use_tok_kernel(batch->T) ? tok_splits(batch->T) : msa_host::auto_splits(batch->T));
  p->qsl = batch->query_start_loc;
  p->seq_lens = batch->seq_lens;
  p->block_table = batch->block_table;
  p->kv_pages = cache->kv_pages;
  p->q = q;
  p->sel = sel;
  p->scale_log2 = softmax_scale * 1.4426950408889634f;
  p->out = out;
  p->part_o = nullptr;
  p->part_lse = nullptr;
  p->status = status;
  return MSA_OK;
}

// Point p's partial buffers into `ws` (attn_ws_bytes(T, splits) bytes) when splits > 1.
void attn_bind_ws(AttnParams* p, void* ws) {
  if (p->splits <= 1) return;
  p->part_o = static_cast<float*>(ws);
  p->part_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) +
                                         msa_host::align256(static_cast<size_t>(p->splits) * p->T * kQHeads * kD * 4));
}

msa_status attn_launch(const AttnParams& p, const uint8_t* kv_pages, cudaStream_t stream) {
  if (use_tok_kernel(p.T)) {
    alignas(64) CUtensorMap kv_map, q_map;
    if (!msa_host::kv_tensor_map(&kv_map, kv_pages, static_cast<uint64_t>(p.num_pages > 0 ? p.num_pages : 1)) ||
        !msa_host::rows128_tensor_map(&q_map, p.q, static_cast<uint64_t>(p.T) * kQHeads, kHPG))
      return MSA_ERR_CUDA;
    if (cudaFuncSetAttribute(tc::k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tc::Smem::kBytes)) != cudaSuccess)
      return MSA_ERR_CUDA;
    tc::k_attn_tc<<<p.T * 4 * p.splits, tc::kThreads, tc::Smem::kBytes, stream>>>(p, kv_map, q_map);
    msa_status st = msa_host::launch_status();
    if (st != MSA_OK) return st;
    if (p.splits > 1) return msa_launch_attn_merge(p.part_o, p.part_lse, p.splits, p.T, p.out, stream);
    return MSA_OK;
  }
  if (false) {
    if (cudaFuncSetAttribute(tok::k_attn_tok, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tok::TokSmem::kBytes)) != cudaSuccess)
      return MSA_ERR_CUDA;
    tok::k_attn_tok<<<p.T * 4 * p.splits, tok::kAttnThreads, tok::TokSmem::kBytes, stream>>>(p);
    msa_status st = msa_host::launch_status();
    if (st != MSA_OK) return st;
    if (p.splits > 1) return msa_launch_attn_merge(p.part_o, p.part_lse, p.splits, p.T, p.out, stream);
    return MSA_OK;
  }
  alignas(64) CUtensorMap tmap;
  if (!msa_host::kv_tensor_map(&tmap, kv_pages, static_cast<uint64_t>(p.num_pages > 0 ? p.num_pages : 1)))
    return MSA_ERR_CUDA;
  if (cudaFuncSetAttribute(k_attn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(AttnSmem::kBytes)) !=
      cudaSuccess)
    return MSA_ERR_CUDA;
  k_attn<<<p.T * 4 * p.splits, kAttnThreads, AttnSmem::kBytes, stream>>>(p, tmap);
  msa_status st = msa_host::launch_status();
  if (st != MSA_OK) return st;
  if (p.splits > 1) return msa_launch_attn_merge(p.part_o, p.part_lse, p.splits, p.T, p.out, stream);
  return MSA_OK;
}

}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

extern "C" size_t msa_attn_workspace_size(const msa_geometry* geo, int32_t B, int32_t T, int32_t num_splits) {
  if (check_geometry(geo) != MSA_OK || B < 0 || T < 0 || num_splits < 0 || num_splits > kMaxSplits) return 0;
  // room for either kernel's automatic choice (the batch's max_q_len picks the kernel)
  const int s = num_splits > 0 ? num_splits : (use_tok_kernel(T) ? tok_splits(T) : auto_splits(T));
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
  AttnParams p;
  msa_status st = attn_setup(geo, batch, cache, q, sel, softmax_scale, num_splits, out, status, &p);
  if (st != MSA_OK || p.T == 0) return st;
  const size_t need = attn_ws_bytes(p.T, p.splits);
  if (workspace_bytes < need || (need > 0 && (workspace == nullptr || !aligned(workspace, 256))))
    return MSA_ERR_INVALID_ARG;
  attn_bind_ws(&p, workspace);
  return attn_launch(p, cache->kv_pages, stream);
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
  AttnParams p;
  msa_status st = attn_setup(geo, batch, cache, q, sel, softmax_scale, num_splits, out, status, &p);
  if (st != MSA_OK || p.T == 0) return st;
  const size_t need = attn_ws_bytes(p.T, p.splits);
  if (need > kNoAllocScratchBytes) return MSA_ERR_INVALID_ARG;  // too many tokens x splits for the array
  void* scratch = nullptr;
  if (need > 0 && (st = scratch_address(&scratch)) != MSA_OK) return st;
  attn_bind_ws(&p, scratch);
  return attn_launch(p, cache->kv_pages, stream);
}
