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
// GB300 design: two kernels, picked by the number of query tokens T (each (token, group) is
// one unit of work: the token's 16 selected blocks of the group).
//
// k_attn (T <= 76): one CTA of 12 warps per (token, group, split), a whole SM on one unit:
//  * a 3-D tensor copy per block brings the group's K and V regions (144 rows of 128 B,
//    128-byte swizzle) into a 4-deep stage ring;
//  * two dequant groups of four warps (thread = key) take alternate blocks and turn each into
//    a 128 x 128 E4M3 K tile and a 128 x 128 f16 V tile (E4M3 -> f16 is exact) in swizzled
//    shared memory, a 3-deep ring;
//  * four token warps each attend 32 keys of every block: the 16 heads are the M = 16 rows of
//    mma.sync.m16n8k32.e4m3 (S = QK^T, K fragments by ldmatrix) and mma.sync.m16n8k16.f16
//    (O += PV, V fragments by ldmatrix.trans, P straight from the S accumulators), with an
//    online softmax; the four states are merged at the end.
//  * Splits of the unit's blocks raise the CTA count when T x 4 is small; the partial
//    (lse, o) pairs are merged by log-sum-exp in a second kernel.
// tc::k_attn_tc (T > 76): a persistent tcgen05 kernel, described where it is defined.
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
#include "msa_attn_tile.cuh"
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
  int32_t t0, nt;  // the tokens [t0, t0 + nt) this launch attends for (the many-token kernel)
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
// Batches of many tokens, on the 5th-generation tensor cores: a persistent CTA of 12 warps per
// SM walks units of one (query token, group, split) each. The keys of a block are the M = 128 rows of both tcgen05 MMAs, so the
// accumulators live in TMEM and the CUDA cores only dequantise and run the softmax:
//  * S^T = K Q^T: kind::f8f6f4, A = the block's 128 x 128 E4M3 K tile in TMEM (the K dequant
//    threads store their key row with tcgen05.st), B = the token's 16 x 128 E4M3 query tile
//    (K-major, 128-byte swizzle, one tensor copy), N = 16 heads, into a ring of two TMEM
//    score buffers; one warp issues these;
//  * O^T += V^T P^T: kind::f16, A = the block's V tile as f16 (E4M3 -> f16 exact) in shared
//    memory, MN-major with 128-byte swizzle, B = P^T (16 heads x 128 keys, K-major, 128-byte
//    swizzle), N = 16, into one TMEM accumulator of 128 dims x 16 heads; another warp issues
//    these (an MMA costs ~80 cycles of issue, so S and PV each get their own issuer);
//  * two groups of four warps, thread = key = TMEM lane: K and V dequant, and softmax. A
//    softmax thread reads its key's 16 head scores and writes P = exp2(s - m). The reference
//    maximum m of a head only moves when some score of a block exceeds it by more than 2^8 (a
//    vote of the four softmax warps), so P <= 256 in f16, the block maximum is reduced across
//    the 128 threads only then, and O^T is rescaled in TMEM only then (after the PV MMA in
//    flight has landed);
//  * the output is O^T / l, the per-head sum l reduced across the 128 threads once.
namespace tc {

constexpr int kWarpProd = 0, kWarpMmaS = 1, kWarpMmaO = 2;  // PV issuers: warps 2 (even blocks), 3 (odd)
constexpr int kWarpDq = 4, kWarpSm = 12;                    // two dequant groups, one softmax group
constexpr int kThreads = 32 * 16;
constexpr int kStages = 4;                                   // NVFP4 K+V stage ring
constexpr int kStageBytes = 2 * kRegion;                     // K region then V region of one (page, group)
constexpr int kQTile = kHPG * kD;                            // 16 heads x 128 E4M3
constexpr int kVTile = kBS * kD * 2;                         // 128 keys x 128 f16
constexpr int kPTile = kHPG * kBS * 2;                       // 16 heads x 128 keys f16
constexpr int kVTiles = 3;                                   // f16 V tile ring
constexpr uint32_t kVLbo = 16384;                            // V tile: the two 64-dim atom columns
constexpr uint32_t kVSbo = 1024;                             //         8-key groups
constexpr float kRescaleLog2 = 8.0f;                         // m moves when a score exceeds it by this
constexpr int kBarWork = 4;                                  // named barrier of the softmax warps
// TMEM columns: K tiles [2] 0..63, S^T [2] 64..95, O^T [2 unit parities][2 block parities] 96..159
constexpr uint32_t kColK = 0, kColS = 64, kColO = 96;
constexpr int kTmemCols = 256;

// One unit of work = one (query token, group, split); a CTA walks units c, c + G, c + 2G, ...
// The producer resolves each unit's selected blocks into a 2-deep ring of these records.
struct UnitMeta {
  int t, g, split, p_tok;  // token, group, split, the token's position
  int n, valid, bad;       // blocks of this split; 0 = batch description inconsistent; a bad entry
  int blk[kSel];           // the split's blocks (block ids), in slot order
  int phys[kSel];          // and their pages
  int pad;
};

struct Smem {
  static constexpr size_t kOffQ = 0;                                                     // 2 x 2 KB
  static constexpr size_t kOffStage = 1024 * 4;                                           // 4 x 18 KB
  static constexpr size_t kOffV = kOffStage + static_cast<size_t>(kStages) * kStageBytes;  // 3 x 32 KB
  static constexpr size_t kOffP = kOffV + kVTiles * static_cast<size_t>(kVTile);          // 2 x 4 KB
  static constexpr size_t kOffBar = kOffP + 2 * static_cast<size_t>(kPTile);
  // st_full, st_empty [kStages]; v_full, v_empty [kVTiles]; ka_full, ka_empty, s_full, s_empty,
  // p_full, p_empty, q_full, q_empty, o_final, o_free, meta_full, meta_empty [2]; fin_s; fin_o [2]
  static constexpr int kBars = 2 * kStages + 2 * kVTiles + 2 * 12 + 3;
  static constexpr size_t kOffLut = kOffBar + 8 * 48;
  static constexpr size_t kOffRed = kOffLut + 256 * 8;   // [2][4 warps][16] fp32
  static constexpr size_t kOffCf = kOffRed + 2 * 4 * 16 * 4;   // [128 softmax threads][16] fp32
  static constexpr size_t kOffMeta = kOffCf + 128 * 16 * 4;
  static constexpr size_t kOffMisc = kOffMeta + 2 * sizeof(UnitMeta);
  static constexpr size_t kBytes = 1024 + kOffMisc + 64;  // + alignment slack
};
static_assert(Smem::kBars <= 48, "barrier area");
static_assert(Smem::kOffStage % 1024 == 0 && Smem::kOffV % 1024 == 0 && Smem::kOffP % 1024 == 0,
              "swizzled tiles sit on 1024-B boundaries");
static_assert(Smem::kBytes <= 232448, "shared memory per CTA");
static_assert(Smem::kOffCf % 16 == 0, "the rescale factors are read as float4");

// O^T(os) *= cf for this thread's lane: the rare path of the lazy reference, out of line so that
// its registers do not count against the softmax loop
__device__ __noinline__ void o_rescale(uint32_t taddr, const float4* cfp) {
#pragma unroll
  for (int xx = 0; xx < 2; ++xx) {
    uint32_t o[16];
    tmem_ld16(taddr + 16 * xx, o);
    tmem_wait_ld();
#pragma unroll
    for (int h4 = 0; h4 < 4; ++h4) {
      const float4 f = cfp[h4];
      o[4 * h4 + 0] = __float_as_uint(__uint_as_float(o[4 * h4 + 0]) * f.x);
      o[4 * h4 + 1] = __float_as_uint(__uint_as_float(o[4 * h4 + 1]) * f.y);
      o[4 * h4 + 2] = __float_as_uint(__uint_as_float(o[4 * h4 + 2]) * f.z);
      o[4 * h4 + 3] = __float_as_uint(__uint_as_float(o[4 * h4 + 3]) * f.w);
    }
    tmem_st16(taddr + 16 * xx, o);
    tmem_wait_st();
  }
}

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
  uint64_t* st_full = bars;
  uint64_t* st_empty = st_full + kStages;
  uint64_t* v_full = st_empty + kStages;
  uint64_t* v_empty = v_full + kVTiles;
  uint64_t* ka_full = v_empty + kVTiles;
  uint64_t* ka_empty = ka_full + 2;
  uint64_t* s_full = ka_empty + 2;
  uint64_t* s_empty = s_full + 2;
  uint64_t* p_full = s_empty + 2;
  uint64_t* p_empty = p_full + 2;
  uint64_t* q_full = p_empty + 2;
  uint64_t* q_empty = q_full + 2;
  uint64_t* o_final = q_empty + 2;
  uint64_t* o_free = o_final + 2;
  uint64_t* meta_full = o_free + 2;
  uint64_t* meta_empty = meta_full + 2;
  uint64_t* fin_s = meta_empty + 2;
  uint64_t* fin_o = fin_s + 1;
  uint2* lut = reinterpret_cast<uint2*>(smem + S::kOffLut);
  float* red = reinterpret_cast<float*>(smem + S::kOffRed);
  UnitMeta* metas = reinterpret_cast<UnitMeta*>(smem + S::kOffMeta);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int units = p.nt * 4 * p.splits;
  constexpr int kMetaUsers = 15;  // the S and two PV issuers, two dequant groups and the softmax group

  // ---- prologue --------------------------------------------------------------------------
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&st_full[i], 1);
      mbar_init(&st_empty[i], 4);  // the dequant group of the stage's blocks
    }
    for (int i = 0; i < kVTiles; ++i) {
      mbar_init(&v_full[i], 4);
      mbar_init(&v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ka_full[i], 4);
      mbar_init(&ka_empty[i], 1);
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 4);
      mbar_init(&p_full[i], 4);
      mbar_init(&p_empty[i], 1);
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
      mbar_init(&o_final[i], 2);  // both PV issuers
      mbar_init(&o_free[i], 4);
      mbar_init(&meta_full[i], 1);
      mbar_init(&meta_empty[i], kMetaUsers);
    }
    mbar_init(fin_s, 1);
    mbar_init(fin_o, 1);
    mbar_init(fin_o + 1, 1);
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == kWarpMmaS) tmem_alloc(tmem_slot, kTmemCols);
  build_dequant_lut(lut, tid, kThreads);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
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
  // unit k of this CTA: its record (waited for) and, when done, its release
  auto meta_get = [&](int k) -> const UnitMeta* {
    if (!wait_ok(&meta_full[k & 1], static_cast<uint32_t>(k >> 1) & 1u)) return nullptr;
    return &metas[k & 1];
  };
  auto meta_put = [&](int k) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&meta_empty[k & 1]);
  };

  if (warp == kWarpProd) {
    // ---- producer: resolve each unit, then copy its query tile and its blocks -------------
    int jg = 0, nq = 0;  // blocks and query tiles issued so far (ring positions)
    if (lane == 0) {
      prefetch_tensormap(&kv_map);
      prefetch_tensormap(&q_map);
    }
    for (int k = 0, u = blockIdx.x; u < units; ++k, u += gridDim.x) {
      if (!wait_ok(&meta_empty[k & 1], (static_cast<uint32_t>(k >> 1) & 1u) ^ 1u)) break;
      UnitMeta& m = metas[k & 1];
      const int split = u % p.splits, tg = u / p.splits, t = p.t0 + (tg >> 2), g = tg & 3;
      int lo = 0, hi = p.B - 1;  // the sequence of token t (largest b with qsl[b] <= t)
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.qsl[mid] <= t) lo = mid; else hi = mid - 1;
      }
      const int b = lo;
      const int q0 = p.qsl[b], ql = p.qsl[b + 1] - q0;
      const int L = p.seq_lens[b];
      const bool valid = t - q0 >= 0 && t - q0 < ql && ql <= p.max_q_len && L >= ql && L <= p.maxb * kBS;
      if (!valid && lane == 0 && split == 0 && g == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
      const int nb = valid ? ceil_div(L, kBS) : 0;
      // the distinct selected blocks of (t, g), in slot order, and their pages
      const int v = valid && lane < kSel ? p.sel[(static_cast<int64_t>(t) * 4 + g) * kSel + lane] : -1;
      bool keep = v >= 0 && v < nb;
      const bool out_of_range = lane < kSel && v >= nb && valid;
      for (int j = 0; j < kSel; ++j) {
        const int vj = __shfl_sync(0xffffffffu, v, j);
        if (j < lane && vj == v) keep = false;
      }
      const uint32_t msk = __ballot_sync(0xffffffffu, keep && lane < kSel);
      const int pos = __popc(msk & ((1u << lane) - 1u));
      int ph = 0;
      bool bad_page = false;
      if (keep && lane < kSel) {
        ph = p.block_table[static_cast<int64_t>(b) * p.maxb + v];
        bad_page = !(ph >= 0 && ph < p.num_pages);
      }
      const bool bad = __any_sync(0xffffffffu, out_of_range || bad_page);
      if ((out_of_range || bad_page)) set_status(p.status, MSA_ERR_DEVICE_FAULT);
      const int nsel = bad ? 0 : __popc(msk);
      const int i0 = (nsel * split) / p.splits, i1 = (nsel * (split + 1)) / p.splits;
      if (keep && lane < kSel && pos >= i0 && pos < i1) {
        m.blk[pos - i0] = v;
        m.phys[pos - i0] = bad_page ? 0 : ph;
      }
      if (lane == 0) {
        m.t = t;
        m.g = g;
        m.split = split;
        m.p_tok = L - ql + (t - q0);
        m.n = i1 - i0;
        m.valid = valid ? 1 : 0;
        m.bad = bad ? 1 : 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&meta_full[k & 1]);  // release: the record is visible to the waiters
      const int n = i1 - i0;
      if (n == 0) continue;
      // the query tile of the unit (free once the S MMAs of the unit two query tiles back landed)
      if (!wait_ok(&q_empty[nq & 1], (static_cast<uint32_t>(nq >> 1) & 1u) ^ 1u)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&q_full[nq & 1], kQTile);
        tma_load_2d(smem + S::kOffQ + static_cast<size_t>(nq & 1) * kQTile, &q_map, 0, t * kQHeads + g * kHPG,
                    &q_full[nq & 1], policy_evict_first());
      }
      ++nq;
      for (int j = 0; j < n; ++j, ++jg) {
        const int s = jg % kStages;
        if (!wait_ok(&st_empty[s], (static_cast<uint32_t>(jg / kStages) & 1u) ^ 1u)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&st_full[s], kStageBytes);
          tma_load_3d(smem + S::kOffStage + static_cast<size_t>(s) * kStageBytes, &kv_map, 0,
                      2 * g * (kRegion / kD), m.phys[j], &st_full[s]);
        }
      }
      if (!ok) break;
    }
    // copies that nobody waited for (after a give-up): wait before the CTA's memory goes
    if (lane == 0) {
      for (int j = jg > kStages ? jg - kStages : 0; j < jg; ++j)
        if (!mbar_wait_bounded(&st_full[j % kStages], static_cast<uint32_t>(j / kStages) & 1u, kWaitLimitNs, nullptr))
          set_status(p.status, MSA_ERR_TIMEOUT);
      for (int j = nq > 2 ? nq - 2 : 0; j < nq; ++j)
        if (!mbar_wait_bounded(&q_full[j & 1], static_cast<uint32_t>(j >> 1) & 1u, kWaitLimitNs, nullptr))
          set_status(p.status, MSA_ERR_TIMEOUT);
    }
  } else if (warp == kWarpMmaS) {
    // ---- S(j) = K(j) Q^T; the whole warp runs the loop, lane 0 issues ------------------------
    constexpr uint32_t idesc_s = idesc_e4m3_f32(128, kHPG);
    int jg = 0, nq = 0;
    for (int k = 0, u = blockIdx.x; u < units; ++k, u += gridDim.x) {
      const UnitMeta* m = meta_get(k);
      if (m == nullptr) break;
      const int n = m->n;
      meta_put(k);
      if (n == 0) continue;
      const int qs = nq & 1;
      if (!wait_ok(&q_full[qs], static_cast<uint32_t>(nq >> 1) & 1u)) break;
      const uint64_t dq = sw128_kmajor_desc(smem_u32(smem + S::kOffQ + static_cast<size_t>(qs) * kQTile));
      for (int j = 0; j < n; ++j, ++jg) {
        const int x = jg & 1;
        const uint32_t par = static_cast<uint32_t>(jg >> 1) & 1u;
        if (!wait_ok(&ka_full[x], par) || !wait_ok(&s_empty[x], par ^ 1u)) break;
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 32 E4M3 per MMA: 8 TMEM columns of A, +32 B of B
            tc_mma_f8_ta(tmem + kColS + 16 * x, tmem + kColK + 32 * x + 8 * kk, dq + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
          tc_commit(&s_full[x]);
          tc_commit(&ka_empty[x]);
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&q_empty[qs]);  // the query tile is free once these MMAs landed
      __syncwarp();
      ++nq;
    }
    if (lane == 0) {  // nothing of this warp's is in flight when TMEM is released
      tc_commit(fin_s);
      if (!mbar_wait_bounded(fin_s, 0u, kWaitLimitNs, nullptr)) set_status(p.status, MSA_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kWarpMmaO || warp == kWarpMmaO + 1) {
    // ---- O^T(unit, x) += V(j)^T P(j)^T for the blocks j of parity x = warp - kWarpMmaO: two
    // issuers, two accumulators (an MMA costs ~80 cycles of issue; the softmax adds the two) --
    constexpr uint32_t idesc_o = idesc_f16_f32_amn(128, kHPG);
    const int x = warp - kWarpMmaO;
    int jg = 0;
    for (int k = 0, u = blockIdx.x; u < units; ++k, u += gridDim.x) {
      const UnitMeta* m = meta_get(k);
      if (m == nullptr) break;
      const int n = m->n;
      meta_put(k);
      const int os = k & 1;
      // O^T[os] was read out by the softmax warps for unit k - 2
      if (!wait_ok(&o_free[os], (static_cast<uint32_t>(k >> 1) & 1u) ^ 1u)) break;
      bool first = true;
      for (int j = 0; j < n; ++j, ++jg) {
        if ((jg & 1) != x) continue;
        const uint32_t par = static_cast<uint32_t>(jg >> 1) & 1u;
        const int y = jg % kVTiles;
        if (!wait_ok(&v_full[y], static_cast<uint32_t>(jg / kVTiles) & 1u) || !wait_ok(&p_full[x], par)) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t dv = sw128_mnmajor_desc(smem_u32(smem + S::kOffV + static_cast<size_t>(y) * kVTile), kVLbo, kVSbo);
          const uint64_t dp = sw128_kmajor_desc(smem_u32(smem + S::kOffP + static_cast<size_t>(x) * kPTile));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // K = 16 keys per MMA: two 8-key groups of V; 32 B (or the next atom) of P
            tc_mma_f16(tmem + kColO + 32 * os + 16 * x, dv + ((2 * kVSbo) >> 4) * kk,
                       dp + (((kk >> 2) * 2048 + (kk & 3) * 32) >> 4), idesc_o, (!first || kk > 0) ? 1u : 0u);
          tc_commit(&v_empty[y]);
          tc_commit(&p_empty[x]);
        }
        __syncwarp();
        first = false;
      }
      if (!ok) break;
      if (lane == 0) tc_commit(&o_final[os]);  // every PV of this issuer for the unit has landed
      __syncwarp();
    }
    if (lane == 0) {
      tc_commit(fin_o + x);
      if (!mbar_wait_bounded(fin_o + x, 0u, kWaitLimitNs, nullptr)) set_status(p.status, MSA_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= kWarpDq && warp < kWarpSm) {
    // ---- dequant, two groups taking alternate blocks: thread = key kr = TMEM lane; K row -> K
    // tile x in TMEM, V row -> f16 V tile y in shared memory (MN-major: key kr is K row kr) ---
    const int kr = 32 * (warp & 3) + lane;
    const uint32_t lanes = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    int jg = 0;  // blocks started (K side)
    auto do_k = [&](int jb) {  // K of block jb (stage jb % kStages stays held for its V)
      const int s = jb % kStages, x = jb & 1;
      if (!wait_ok(&st_full[s], static_cast<uint32_t>(jb / kStages) & 1u)) return;
      RawRow rk;
      load_row(smem + S::kOffStage + static_cast<size_t>(s) * kStageBytes, kr, rk);
      if (!wait_ok(&ka_empty[x], (static_cast<uint32_t>(jb >> 1) & 1u) ^ 1u)) return;  // S(jb - 2) has landed
      uint32_t w[32];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t uu[8];
        dequant_quarter(rk, q, lut, uu);
#pragma unroll
        for (int e = 0; e < 8; ++e) w[8 * q + e] = uu[e];
      }
      tc_fence_after();
      tmem_st32(tmem + lanes + kColK + 32 * x, w);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ka_full[x]);
    };
    auto do_v = [&](int jb) {  // V of block jb, then its stage is free
      const int s = jb % kStages, y = jb % kVTiles;
      if (!ok) return;
      RawRow rv;
      load_row(smem + S::kOffStage + static_cast<size_t>(s) * kStageBytes + kRegion, kr, rv);
      __syncwarp();
      if (lane == 0) mbar_arrive(&st_empty[s]);
      // PV(jb - kVTiles) has landed
      if (!wait_ok(&v_empty[y], (static_cast<uint32_t>(jb / kVTiles) & 1u) ^ 1u)) return;
      uint8_t* vt = smem + S::kOffV + static_cast<size_t>(y) * kVTile + (kr >> 3) * kVSbo + (kr & 7) * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t uu[8];
        dequant_quarter(rv, q, lut, uu);
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {  // dims 32 q + 8 hh .. +7 = chunk cc = 4 q + hh
          const int cc = 4 * q + hh;
          const uint4 vv = make_uint4(cvt_f16x2_e4m3x2(uu[2 * hh]), cvt_f16x2_e4m3x2(uu[2 * hh] >> 16),
                                      cvt_f16x2_e4m3x2(uu[2 * hh + 1]), cvt_f16x2_e4m3x2(uu[2 * hh + 1] >> 16));
          *reinterpret_cast<uint4*>(vt + (cc >> 3) * kVLbo + (((cc & 7) ^ (kr & 7)) << 4)) = vv;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&v_full[y]);
    };
    const int gq = (warp - kWarpDq) >> 2;  // this group's blocks: jg % 2 == gq
    for (int k = 0, u = blockIdx.x; u < units; ++k, u += gridDim.x) {
      const UnitMeta* m = meta_get(k);
      if (m == nullptr) break;
      const int n = m->n;
      meta_put(k);
      for (int j = 0; j < n && ok; ++j, ++jg) {
        if ((jg & 1) != gq) continue;
        do_k(jg);
        do_v(jg);
      }
      if (!ok) break;
    }
  } else if (warp >= kWarpSm) {
    // ---- softmax: thread = key kr = TMEM lane ----------------------------------------------
    const int wq = warp & 3;
    const int kr = 32 * wq + lane;
    const uint32_t lanes = static_cast<uint32_t>(32 * wq) << 16;
    const float c = p.scale_log2;
    int jg = 0, nred = 0;  // blocks seen; reductions done (alternates the two scratch buffers)
    for (int k = 0, u = blockIdx.x; u < units; ++k, u += gridDim.x) {
      // every softmax warp takes the same path through a unit (the named barriers need all
      // four): a warp whose wait gave up inside the unit keeps walking with its work skipped
      const UnitMeta* m = meta_get(k);
      if (named_barrier_or(kBarWork, 128, m == nullptr)) {  // one of the four gave up: all leave
        ok = false;
        give_up();
        break;
      }
      const int n = m->n;
      const int t = m->t, g = m->g, split = m->split, p_tok = m->p_tok;
      const bool valid = m->valid != 0, bad = m->bad != 0;
      const int os = k & 1;
      // m_ref starts at a large negative finite value rather than -inf, so that the exponent
      // argument s * c - m_ref is large for any real score (the vote below takes the block's
      // maximum then) and -inf for a masked key (P = 0), with no special case for the first
      // block; 2^14 keeps s * c = d + m_ref within 2^-9 of the score (fp32 at 2^14), which only
      // shifts the reference, never a P beyond the vote's bound
      constexpr float kNoRef = -16384.0f;
      float m_ref[16], l[16];
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        m_ref[h] = kNoRef;
        l[h] = 0.f;
      }
      for (int j = 0; j < n; ++j, ++jg) {
        const int x = jg & 1;
        const uint32_t par = static_cast<uint32_t>(jg >> 1) & 1u;
        float d[16];  // exponent arguments s * c - m_ref against the current reference
        if (wait_ok(&s_full[x], par)) {
          tc_fence_after();
          uint32_t r[16];
          tmem_ld16(tmem + lanes + kColS + 16 * x, r);
          tmem_wait_ld();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[x]);
          const bool kvalid = m->blk[j] * kBS + kr <= p_tok;  // keys after the query position: -inf
#pragma unroll
          for (int h = 0; h < 16; ++h) d[h] = kvalid ? fmaf(__uint_as_float(r[h]), c, -m_ref[h]) : -CUDART_INF_F;
        } else {
#pragma unroll
          for (int h = 0; h < 16; ++h) d[h] = -CUDART_INF_F;
        }
        bool need = false;
#pragma unroll
        for (int h = 0; h < 16; ++h) need |= d[h] > kRescaleLog2;
        if (named_barrier_or(kBarWork, 128, need)) {  // the same answer in all four warps
          float cf[16];  // the block maxima of s * c, then the rescale factors
#pragma unroll
          for (int h = 0; h < 16; ++h) cf[h] = d[h] + m_ref[h];
          group_reduce16<true>(cf, cf, red + 64 * (nred & 1), wq, lane);
          ++nred;
          bool moved = false;
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const float mn = fmaxf(m_ref[h], cf[h]);
            moved |= mn != m_ref[h];
            d[h] += m_ref[h] - mn;              // the same arguments against the new reference
            cf[h] = fast_exp2(m_ref[h] - mn);  // 0 when there was no reference yet
            m_ref[h] = mn;
            l[h] *= cf[h];
          }
          {  // this thread's copy of the factors (the same in all 128 threads) for the O rescale
            float4* cfp = reinterpret_cast<float4*>(smem + S::kOffCf) + 4 * kr;
#pragma unroll
            for (int h4 = 0; h4 < 4; ++h4) cfp[h4] = make_float4(cf[4 * h4], cf[4 * h4 + 1], cf[4 * h4 + 2], cf[4 * h4 + 3]);
          }
          // both accumulators *= cf once PV(jg - 1) and PV(jg - 2) have landed (PV(jg) waits for
          // this block's P); one not yet written in this unit is rescaled harmlessly: its first
          // PV of the unit overwrites it
          if (moved && j > 0 && wait_ok(&p_empty[(jg - 1) & 1], static_cast<uint32_t>((jg - 1) >> 1) & 1u) &&
              (j < 2 || wait_ok(&p_empty[jg & 1], (static_cast<uint32_t>(jg >> 1) & 1u) ^ 1u))) {
            tc_fence_after();
            o_rescale(tmem + lanes + kColO + 32 * os, reinterpret_cast<const float4*>(smem + S::kOffCf) + 4 * kr);
            tc_fence_before();
          }
        }
        // P = exp2(s c - m) -> P^T tile x (free once PV(jg - 2) has landed): row h, key kr
        if (wait_ok(&p_empty[x], par ^ 1u)) {
          uint8_t* pt = smem + S::kOffP + static_cast<size_t>(x) * kPTile + (kr >> 6) * 2048 + (kr & 7) * 2;
          const int ch = (kr & 63) >> 3;
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const float pv = fast_exp2(d[h]);
            l[h] += pv;
            *reinterpret_cast<__half*>(pt + (h >> 3) * 1024 + (h & 7) * 128 + ((ch ^ (h & 7)) << 4)) =
                __float2half_rn(pv);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[x]);
        }
      }
      // ---- the unit's output: lane kr = dim kr of O^T; l summed over the 128 keys' threads --
      float (&lt)[16] = l;  // the per-head sums, reduced in place
      group_reduce16<false>(l, lt, red + 64 * (nred & 1), wq, lane);
      ++nred;
      uint32_t o[16];
      const bool have = n > 0 && wait_ok(&o_final[os], static_cast<uint32_t>(k >> 1) & 1u);
      if (have) {  // the accumulator of the unit's first block, plus the other one if it was used
        const int x0 = (jg - n) & 1;
        tc_fence_after();
        tmem_ld16(tmem + lanes + kColO + 32 * os + 16 * x0, o);
        tmem_wait_ld();
        if (n > 1) {
          uint32_t o2[16];
          tmem_ld16(tmem + lanes + kColO + 32 * os + 16 * (x0 ^ 1), o2);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 16; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) + __uint_as_float(o2[h]));
        }
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[os]);  // O^T[os] may be overwritten
      if (valid) {
        const bool zero = !have || bad || *abort_flag != 0;
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
      meta_put(k);
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
// SM (the keys of each block over four mma.sync warps, the dequant over eight), so a batch of
// few tokens finishes in one short wave; tc::k_attn_tc runs one persistent CTA per SM over all
// the (token, group) units with the contractions on tcgen05, which keeps the SM busier once
// there are several waves of units. The many-token kernel takes more than two units per SM.
bool use_tc_kernel(int T) { return 4 * T > 2 * 152; }

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
  p->t0 = 0;
  p->nt = batch->T;
  p->maxb = batch->max_blocks_per_seq;
  p->max_q_len = batch->max_q_len;
  p->num_pages = cache->num_pages;
  p->splits = num_splits > 0 ? num_splits
                             : (use_tc_kernel(batch->T) ? 1 : msa_host::auto_splits(batch->T));
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
  if (use_tc_kernel(p.T)) {
    alignas(64) CUtensorMap kv_map, q_map;
    if (!msa_host::kv_tensor_map(&kv_map, kv_pages, static_cast<uint64_t>(p.num_pages > 0 ? p.num_pages : 1)) ||
        !msa_host::rows128_tensor_map(&q_map, p.q, static_cast<uint64_t>(p.T) * kQHeads, kHPG))
      return MSA_ERR_CUDA;
    if (cudaFuncSetAttribute(tc::k_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(tc::Smem::kBytes)) != cudaSuccess)
      return MSA_ERR_CUDA;
    const int sms = msa_host::num_sms();
    if (sms <= 0) return MSA_ERR_CUDA;
    const int units = p.nt * 4 * p.splits;
    tc::k_attn_tc<<<units < sms ? units : sms, tc::kThreads, tc::Smem::kBytes, stream>>>(p, kv_map, q_map);
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
  const int s = num_splits > 0 ? num_splits : (use_tc_kernel(T) ? 1 : auto_splits(T));
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

// The attention of the tokens [t0, t1) alone, for batches the many-token kernel takes with one
// split (the output rows of other tokens are left as they are). The host-buffer step runs the
// attention as two such launches so that the copy of the first one's output to the host
// overlaps the second.
msa_status msa_attn_token_range(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                const uint8_t* q, const int32_t* sel, float softmax_scale, uint16_t* out,
                                uint32_t* status, int32_t t0, int32_t t1, cudaStream_t stream) {
  AttnParams p;
  msa_status st = attn_setup(geo, batch, cache, q, sel, softmax_scale, 0, out, status, &p);
  if (st != MSA_OK || p.T == 0) return st;
  if (!use_tc_kernel(p.T) || p.splits != 1 || t0 < 0 || t1 > p.T || t0 >= t1) return MSA_ERR_INVALID_ARG;
  p.t0 = t0;
  p.nt = t1 - t0;
  return attn_launch(p, cache->kv_pages, stream);
}

// Where the host-buffer step splits the attention: the second launch takes the tokens of the
// persistent grid's last kTailRounds rounds of units (one unit per SM a round, four units a
// token), so the split adds no round, and the first launch's output (the larger part) copies
// to the host while the second runs; 0 = one launch (the small-batch kernel, or too few rounds).
constexpr int kTailRounds = 3;
int32_t msa_attn_split_token(int32_t T) {
  if (!use_tc_kernel(T)) return 0;
  const int sms = num_sms();
  const int per_round = sms / 4;
  if (per_round <= 0) return 0;
  const int rounds = ceil_div(T, per_round);
  return rounds < 2 * kTailRounds ? 0 : per_round * (rounds - kTailRounds);
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
