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
// Batches of many tokens, on the 5th-generation tensor cores: a persistent CTA per SM runs three
// worker warpgroups side by side, each owning whole units (one unit = one (query token, group,
// split): the token's selected blocks of the group) from start to finish, so a unit's dequant,
// softmax and output never change hands between warp groups. Per block of 128 keys, the four
// warps of a warpgroup (thread = key row):
//  * dequantise the block's K rows from NVFP4 to E4M3 straight into a TMEM tile (tcgen05.st),
//    the A operand of S^T = K Q^T (kind::f8f6f4, N = 16 heads, keys on the M = 128 rows);
//  * dequantise its V rows to E4M3 over the stage buffer the copy brought them in (in place:
//    every raw row is read before the first E4M3 row is written), the MN-major A operand of
//    O^T += V^T P^T (kind::f8f6f4, N = 32);
//  * run the softmax on S^T: P = exp2(s c - m) with m a per-head reference that only moves when
//    a score exceeds it by more than 2^8 (a vote of the four warps; the first block of a unit
//    always sets it), so P <= 256 fits E4M3; P is split into hi = E4M3(P) and lo =
//    E4M3(16 (P - hi)) (error <= 2^-8 P), stored as rows 0..15 and 16..31 of the 32 x 128 B
//    operand P^T, so one MMA per 32 keys accumulates both parts of the sum into two column
//    groups of O^T;
//  * at the unit's end, read O^T (thread = dim), add hi + lo / 16, divide by the per-head sum.
// The softmax thread takes S^T with the 16x256b TMEM load shape (four keys x four heads a
// thread), so its four keys of one head are four consecutive key positions of P^T, stored as one
// 32-bit word: the K rows go to TMEM lanes in an order that makes this hold (kappa below) and
// the V rows go to the P^T key position of their key.
// One issuer warp per warpgroup issues its MMAs and its tensor copies (a 3-deep ring of K+V
// stages of one (page, group) each, and the unit's query tile); one warp resolves units (the
// selected blocks, their pages) into a ring of records for the three warpgroups.
namespace tc {

constexpr int kWgs = 3;                               // worker warpgroups (warps 4w .. 4w + 3)
constexpr int kWarpIss = 4 * kWgs;                    // warp 12 + w: issuer of warpgroup w
constexpr int kWarpRes = kWarpIss + kWgs;             // warp 15: unit resolver, TMEM owner
constexpr int kThreads = 32 * (kWarpRes + 1);         // 512
constexpr int kStages = 3;                            // K+V stage ring of a warpgroup
constexpr int kStageBytes = 2 * kRegion;              // 18,432 (the E4M3 V tile is written over it)
constexpr int kQTile = kHPG * kD;                     // 16 heads x 128 E4M3
constexpr int kPTile = 2 * kHPG * kBS;                // P^T: 32 rows (hi, lo) x 128 keys E4M3
constexpr int kMeta = 4;                              // unit records in a warpgroup's ring
constexpr size_t kWgBytes = static_cast<size_t>(kStages) * kStageBytes + kPTile + 2 * kQTile;
constexpr int kTmemCols = 512;
constexpr uint32_t kWgCols = 128;                     // TMEM columns of a warpgroup:
constexpr uint32_t kColK = 0, kColS = 32, kColO = 64;  // K tile (32), S^T (16), O^T [2 parities] (2 x 32)
constexpr float kRescaleLog2 = 8.0f;                  // P <= 2^8 < 448, the E4M3 maximum
constexpr float kLoScale = 16.0f;                     // P^T lo rows hold kLoScale (P - hi)
constexpr uint32_t kLoScale2 = 0x4C004C00u;           // f16x2 {16, 16}
constexpr int kBarVote = 1, kBarX = 4;                // named barriers 1 + w and 4 + w of warpgroup w
static_assert(kWgBytes % 1024 == 0 && kStageBytes % 1024 == 0 && kPTile % 1024 == 0 && kQTile % 1024 == 0,
              "swizzled tiles sit on 1024-B boundaries");

// The key row of a 32-row quarter that TMEM lane `lam` (0..31) of the K tile holds:
// 8a + rotl3((b - 2a) mod 8) for lam = 8a + b. The softmax thread t reads lanes t/4 + 8i
// (i = 0..3) and stores them as P^T key positions 4 (t/4) + i; with this order both the K rows
// (thread lam reads row kappa(lam)) and the V rows (thread mu reads the row whose key position
// is mu) are read from the staged page without shared-memory bank conflicts.
__device__ __forceinline__ int kappa(int lam) {
  const int a = lam >> 3, x = ((lam & 7) - 2 * a) & 7;
  return 8 * a + (((x << 1) | (x >> 2)) & 7);
}

struct UnitMeta {
  int t, g, split, p_tok;  // token, group, split, the token's position
  int n;                   // blocks of this split (>= 1); -1 ends the warpgroup's work
  int pad[3];
  int blk[kSel];           // the split's blocks (block ids), in slot order
  int phys[kSel];          // and their pages
};

struct Smem {
  static constexpr size_t kOffWg = 0;                                             // [3] x 62 KB
  static constexpr size_t kOffBar = kOffWg + kWgs * kWgBytes;
  // per warpgroup: st_full[3], q_full[2], q_empty[2], ka_full, s_full, pv_ready, pv_done,
  // o_free[2], meta_full[4], meta_empty[4], fin
  static constexpr int kBarsPerWg = kStages + 2 + 2 + 4 + 2 + 2 * kMeta + 1;
  static constexpr size_t kOffLut = kOffBar + 8 * ((kBarsPerWg * kWgs + 1) & ~1);
  static constexpr size_t kOffRed = kOffLut + 256 * 8;              // [3][2][4 warps][16] fp32 block maxima
  static constexpr size_t kOffMref = kOffRed + kWgs * 2 * 64 * 4;   // [3][2][16] fp32 reference maxima
  static constexpr size_t kOffRedL = kOffMref + kWgs * 2 * 16 * 4;  // [3][4 warps][16] fp32 sums
  static constexpr size_t kOffMeta = kOffRedL + kWgs * 64 * 4;
  static constexpr size_t kOffQsl = kOffMeta + kWgs * kMeta * sizeof(UnitMeta);
  static constexpr size_t kOffMisc = kOffQsl + 4 * (kMaxB + 4);
  static constexpr size_t kBytes = 1024 + kOffMisc + 64;  // + alignment slack
};
static_assert(Smem::kBytes <= 232448, "shared memory per CTA");
static_assert(Smem::kOffRed % 16 == 0 && Smem::kOffMref % 16 == 0 && Smem::kOffRedL % 16 == 0, "float4 reads");

__global__ void __launch_bounds__(kThreads, 1)
    k_attn_tc(const AttnParams p, const __grid_constant__ CUtensorMap kv_map, const __grid_constant__ CUtensorMap q_map) {
  using S = Smem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint2* lut = reinterpret_cast<uint2*>(smem + S::kOffLut);
  UnitMeta* metas = reinterpret_cast<UnitMeta*>(smem + S::kOffMeta);
  int* qsl_s = reinterpret_cast<int*>(smem + S::kOffQsl);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int units = p.nt * 4 * p.splits;
  // this warp's warpgroup (workers and issuers; the resolver serves all three)
  const int w = warp < kWarpIss ? (warp >> 2) : (warp < kWarpRes ? warp - kWarpIss : 0);
  uint64_t* wbar = reinterpret_cast<uint64_t*>(smem + S::kOffBar) + S::kBarsPerWg * w;
  uint64_t* st_full = wbar;
  uint64_t* q_full = st_full + kStages;
  uint64_t* q_empty = q_full + 2;
  uint64_t* ka_full = q_empty + 2;
  uint64_t* s_full = ka_full + 1;
  uint64_t* pv_ready = s_full + 1;
  uint64_t* pv_done = pv_ready + 1;
  uint64_t* o_free = pv_done + 1;
  uint64_t* meta_full = o_free + 2;
  uint64_t* meta_empty = meta_full + kMeta;
  uint64_t* fin = meta_empty + kMeta;
  uint8_t* wgb = smem + S::kOffWg + static_cast<size_t>(w) * kWgBytes;
  uint8_t* ptile = wgb + static_cast<size_t>(kStages) * kStageBytes;
  uint8_t* qtile = ptile + kPTile;
  UnitMeta* wmeta = metas + kMeta * w;

  // ---- prologue --------------------------------------------------------------------------
  if (tid == 0) {
    for (int x = 0; x < kWgs; ++x) {
      uint64_t* b = reinterpret_cast<uint64_t*>(smem + S::kOffBar) + S::kBarsPerWg * x;
      for (int i = 0; i < kStages; ++i) mbar_init(b + i, 1);              // st_full
      for (int i = 0; i < 2; ++i) {
        mbar_init(b + kStages + i, 1);                                     // q_full
        mbar_init(b + kStages + 2 + i, 1);                                 // q_empty (commit)
      }
      mbar_init(b + kStages + 4, 4);                                       // ka_full: the 4 workers
      mbar_init(b + kStages + 5, 1);                                       // s_full (commit)
      mbar_init(b + kStages + 6, 4);                                       // pv_ready
      mbar_init(b + kStages + 7, 1);                                       // pv_done (commit)
      for (int i = 0; i < 2; ++i) mbar_init(b + kStages + 8 + i, 4);       // o_free
      for (int i = 0; i < kMeta; ++i) {
        mbar_init(b + kStages + 10 + i, 1);                                // meta_full (resolver)
        mbar_init(b + kStages + 10 + kMeta + i, 4);                        // meta_empty (workers)
      }
      mbar_init(b + kStages + 10 + 2 * kMeta, 1);                          // fin (commit)
    }
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == kWarpRes) tmem_alloc(tmem_slot, kTmemCols);
  build_dequant_lut(lut, tid, kThreads);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tw = tmem + kWgCols * static_cast<uint32_t>(w);
  bool ok = true;
  auto give_up = [&]() {
    if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
    *abort_flag = 1;
  };
  auto wait1 = [&](uint64_t* bar, uint32_t parity) {  // one thread's bounded wait
    if (!ok) return false;
    ok = mbar_wait(bar, parity, abort_flag);
    if (!ok) give_up();
    return ok;
  };
  auto waitw = [&](uint64_t* bar, uint32_t parity) {  // a whole warp's bounded wait
    if (!ok) return false;
    ok = warp_wait(bar, parity, abort_flag);
    if (!ok && lane == 0) give_up();
    return ok;
  };

  if (warp == kWarpRes) {
    // ---- resolver: the CTA's units c, c + G, ... in order, the non-empty ones dealt to the
    // warpgroups in turn; an empty unit (a bad selection or page, or a split with no blocks) has
    // its output zero-filled here, an invalid one (an inconsistent batch) is left as it is ------
    for (int i = lane; i <= p.B; i += 32) qsl_s[i] = p.qsl[i];
    __syncwarp();
    int written0 = 0, written1 = 0, written2 = 0;  // records dealt to each warpgroup
    int turn = 0;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
      const int split = u % p.splits, tg = u / p.splits, t = p.t0 + (tg >> 2), g = tg & 3;
      int lo = 0, hi = p.B - 1;  // the sequence of token t (largest b with qsl[b] <= t)
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (qsl_s[mid] <= t) lo = mid; else hi = mid - 1;
      }
      const int b = lo;
      const int q0 = qsl_s[b], ql = qsl_s[b + 1] - q0;
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
      if (out_of_range || bad_page) set_status(p.status, MSA_ERR_DEVICE_FAULT);
      const int nsel = bad ? 0 : __popc(msk);
      const int i0 = (nsel * split) / p.splits, i1 = (nsel * (split + 1)) / p.splits;
      if (i1 == i0) {
        if (valid) {  // nothing to attend: zero output (or an empty partial)
          const int64_t row0 = static_cast<int64_t>(t) * kQHeads + g * kHPG;
          if (p.splits == 1) {
            uint4* o = reinterpret_cast<uint4*>(p.out + row0 * kD);
            for (int e = lane; e < kHPG * kD / 8; e += 32) o[e] = make_uint4(0u, 0u, 0u, 0u);
          } else {
            const int64_t prow0 = static_cast<int64_t>(split) * p.T * kQHeads + row0;
            float4* o = reinterpret_cast<float4*>(p.part_o + prow0 * kD);
            for (int e = lane; e < kHPG * kD / 4; e += 32) o[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (lane < kHPG) p.part_lse[prow0 + lane] = -CUDART_INF_F;
          }
        }
        continue;
      }
      const int x = turn;
      turn = turn + 1 == kWgs ? 0 : turn + 1;
      uint64_t* xb = reinterpret_cast<uint64_t*>(smem + S::kOffBar) + S::kBarsPerWg * x;
      uint64_t* x_meta_full = xb + kStages + 10;
      uint64_t* x_meta_empty = x_meta_full + kMeta;
      const int k = x == 0 ? written0++ : (x == 1 ? written1++ : written2++);
      if (!waitw(&x_meta_empty[k % kMeta], (static_cast<uint32_t>(k / kMeta) & 1u) ^ 1u)) break;
      UnitMeta& m = metas[kMeta * x + k % kMeta];
      if (keep && lane < kSel && pos >= i0 && pos < i1) {
        m.blk[pos - i0] = v;
        m.phys[pos - i0] = ph;
      }
      if (lane == 0) {
        m.t = t;
        m.g = g;
        m.split = split;
        m.p_tok = L - ql + (t - q0);
        m.n = i1 - i0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&x_meta_full[k % kMeta]);  // release: the record is visible to the waiters
    }
    // the end of every warpgroup's list
    for (int x = 0; x < kWgs && ok; ++x) {
      uint64_t* xb = reinterpret_cast<uint64_t*>(smem + S::kOffBar) + S::kBarsPerWg * x;
      uint64_t* x_meta_full = xb + kStages + 10;
      uint64_t* x_meta_empty = x_meta_full + kMeta;
      const int k = x == 0 ? written0 : (x == 1 ? written1 : written2);
      if (!waitw(&x_meta_empty[k % kMeta], (static_cast<uint32_t>(k / kMeta) & 1u) ^ 1u)) break;
      if (lane == 0) {
        metas[kMeta * x + k % kMeta].n = -1;
        mbar_arrive(&x_meta_full[k % kMeta]);
      }
      __syncwarp();
    }
  } else if (warp >= kWarpIss) {
    // ---- issuer of warpgroup w (lane 0): S and PV MMAs, and the copies of the blocks
    // (kStages ahead of the PVs) and of each unit's query tile -------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_e4m3_f32(128, kHPG);
      constexpr uint32_t idesc_pv = idesc_e4m3_f32_amn(128, 2 * kHPG);
      prefetch_tensormap(&kv_map);
      prefetch_tensormap(&q_map);
      const uint64_t qpol = policy_evict_first();
      // copy cursor: record kt, its block jt; jg_t blocks issued. It copies a record's query tile
      // when it enters the record and may enter record kt only while the MMAs are at record
      // kt - 1 or later: the query buffer it refills was then released by record kt - 2's last
      // S, which has been issued, so the wait for it always ends.
      int kt = 0, jt = 0, jg_t = 0;
      bool t_end = false, t_in = false;
      auto copy_fill = [&](int upto, int k_mma) {  // copies of blocks jg_t .. upto - 1 (stages free)
        while (jg_t < upto && !t_end && ok) {
          if (!t_in) {
            if (kt >= k_mma + 2) return;
            if (!wait1(&meta_full[kt % kMeta], static_cast<uint32_t>(kt / kMeta) & 1u)) return;
            const UnitMeta& m = wmeta[kt % kMeta];
            if (m.n < 0) {
              t_end = true;
              return;
            }
            if (!wait1(&q_empty[kt & 1], (static_cast<uint32_t>(kt >> 1) & 1u) ^ 1u)) return;
            mbar_arrive_expect_tx(&q_full[kt & 1], kQTile);
            tma_load_2d(qtile + (kt & 1) * kQTile, &q_map, 0, m.t * kQHeads + m.g * kHPG, &q_full[kt & 1], qpol);
            t_in = true;
            jt = 0;
          }
          const UnitMeta& m = wmeta[kt % kMeta];
          const int s = jg_t % kStages;
          mbar_arrive_expect_tx(&st_full[s], kStageBytes);
          tma_load_3d(wgb + static_cast<size_t>(s) * kStageBytes, &kv_map, 0, 2 * m.g * (kRegion / kD), m.phys[jt],
                      &st_full[s]);
          ++jg_t;
          if (++jt == m.n) {
            t_in = false;
            ++kt;
          }
        }
      };
      int jg = 0;
      for (int k = 0; ok; ++k) {
        copy_fill(jg + kStages, k);  // the stages of blocks before jg + kStages are free
        if (!wait1(&meta_full[k % kMeta], static_cast<uint32_t>(k / kMeta) & 1u)) break;
        const int n = wmeta[k % kMeta].n;
        if (n < 0) break;
        const int x = k & 1;  // query buffer and O^T accumulator of the unit
        const uint64_t dq = sw128_kmajor_desc(smem_u32(qtile + x * kQTile));
        auto issue_s = [&](int jb, bool last) {  // S^T = K(jb) Q^T
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 32 E4M3 per MMA: 8 TMEM columns of A, +32 B of B
            tc_mma_f8_ta(tw + kColS, tw + kColK + 8 * kk, dq + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
          tc_commit(s_full);
          if (last) tc_commit(&q_empty[x]);  // the query tile is free once these MMAs landed
        };
        if (!wait1(&q_full[x], static_cast<uint32_t>(k >> 1) & 1u) || !wait1(ka_full, static_cast<uint32_t>(jg) & 1u))
          break;
        issue_s(jg, n == 1);
        for (int j = 0; j < n; ++j, ++jg) {
          if (j + 1 < n) {  // S of the next block as soon as its K tile is in TMEM
            if (!wait1(ka_full, static_cast<uint32_t>(jg + 1) & 1u)) break;
            issue_s(jg + 1, j + 2 == n);
          }
          // O^T[x] was read out by the workers for record k - 2
          if (j == 0 && !wait1(&o_free[x], (static_cast<uint32_t>(k >> 1) & 1u) ^ 1u)) break;
          if (!wait1(pv_ready, static_cast<uint32_t>(jg) & 1u)) break;
          tc_fence_after();
          {
            const uint32_t vaddr = smem_u32(wgb + static_cast<size_t>(jg % kStages) * kStageBytes);
            const uint64_t dp = sw128_kmajor_desc(smem_u32(ptile));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // K = 32 keys per MMA: four 8-key groups of V (4 KB), +32 B of P^T
              tc_mma_f8(tw + kColO + 32 * x, sw128_mnmajor8_desc(vaddr + 4096 * kk), dp + 2 * kk, idesc_pv,
                        (j > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(pv_done);
          // the block's stage is free once PV(jg) has landed: refill it
          if (!wait1(pv_done, static_cast<uint32_t>(jg) & 1u)) break;
          copy_fill(jg + 1 + kStages, k);
        }
      }
      // nothing of this thread's is in flight when the CTA ends: its MMAs, then its copies
      tc_commit(fin);
      if (!mbar_wait_bounded(fin, 0u, kWaitLimitNs, nullptr)) set_status(p.status, MSA_ERR_TIMEOUT);
      for (int j = jg_t > kStages ? jg_t - kStages : 0; j < jg_t; ++j)
        if (!mbar_wait_bounded(&st_full[j % kStages], static_cast<uint32_t>(j / kStages) & 1u, kWaitLimitNs, nullptr))
          set_status(p.status, MSA_ERR_TIMEOUT);
      const int nq = kt + (t_in ? 1 : 0);  // query tiles issued
      for (int j = nq > 2 ? nq - 2 : 0; j < nq; ++j)
        if (!mbar_wait_bounded(&q_full[j & 1], static_cast<uint32_t>(j >> 1) & 1u, kWaitLimitNs, nullptr))
          set_status(p.status, MSA_ERR_TIMEOUT);
    }
  } else {
    // ---- worker warp q of warpgroup w ------------------------------------------------------
    const int q = warp & 3;
    const uint32_t lanes = static_cast<uint32_t>(32 * q) << 16;
    const int key_k = 32 * q + kappa(lane);                                // K row -> TMEM lane 32 q + lane
    const int vrow = 32 * q + lane;                                        // V tile row (key position)
    const int key_v = 32 * q + kappa((lane >> 2) + 8 * (lane & 3));       // the key at that position
    const int hb = 2 * (lane & 3);  // this thread's heads: hb, hb + 1, hb + 8, hb + 9 (slot hh)
    // P^T row n = head (hi) or 16 + head (lo) sits at (n / 8) KB + (n % 8) x 128 B; this thread's
    // word (keys 32 q + 4 (lane / 4) .. + 3) is in chunk 2 q + lane / 16 of the row, swizzled by
    // n % 8 (= hb or hb + 1): two offsets, the rest are immediates
    const int pch = 2 * q + (lane >> 4), pb = 4 * ((lane >> 2) & 3);
    const uint32_t psw0 = static_cast<uint32_t>(hb * 128 + ((pch ^ hb) << 4) + pb);
    const uint32_t psw1 = static_cast<uint32_t>((hb + 1) * 128 + ((pch ^ (hb + 1)) << 4) + pb);
    const float c = p.scale_log2;
    float* redm = reinterpret_cast<float*>(smem + S::kOffRed) + w * 128;    // [2][4][16]
    float* mref = reinterpret_cast<float*>(smem + S::kOffMref) + w * 32;    // [2][16]
    float* redl = reinterpret_cast<float*>(smem + S::kOffRedL) + w * 64;    // [4][16]
    const int bar_vote = kBarVote + w, bar_x = kBarX + w;
    int jg = 0, nre = 0;  // blocks seen; rescale events (alternate the two reduction buffers)

    // K rows of block jb -> the TMEM K tile; with `finish`, the stores are waited for and the
    // tile announced here, else by k_finish() once the caller has other work in flight
    auto k_finish = [&]() {
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ka_full);
    };
    auto do_k = [&](int jb, bool finish) {
      if (!waitw(&st_full[jb % kStages], static_cast<uint32_t>(jb / kStages) & 1u)) return false;
      RawRow rk;
      load_row(wgb + static_cast<size_t>(jb % kStages) * kStageBytes, key_k, rk);
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {  // each quarter goes to TMEM while the next is dequantised
        uint32_t uu[8];
        dequant_quarter(rk, qq, lut, uu);
        tmem_st8(tw + lanes + kColK + 8 * qq, uu);
      }
      if (finish) k_finish();
      return true;
    };

    for (int k = 0;; ++k) {
      const bool got = waitw(&meta_full[k % kMeta], static_cast<uint32_t>(k / kMeta) & 1u);
      if (named_barrier_or(bar_vote, 128, !got)) break;  // one of the four gave up: all leave
      const UnitMeta& m = wmeta[k % kMeta];
      const int n = m.n;
      if (n < 0) break;
      const int t = m.t, g = m.g, split = m.split, p_tok = m.p_tok;
      const int x = k & 1;
      float m_ref[4], l[4];
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) m_ref[hh] = l[hh] = 0.f;
      do_k(jg, true);
      bool quit = false;
      for (int j = 0; j < n; ++j, ++jg) {
        uint8_t* stg = wgb + static_cast<size_t>(jg % kStages) * kStageBytes;
        RawRow rv;
        if (ok) load_row(stg + kRegion, key_v, rv);  // V raw row, read before anyone overwrites the stage
        float d[4][4];  // [key i][head slot hh]: exponent arguments s c - m_ref
        if (waitw(s_full, static_cast<uint32_t>(jg) & 1u)) {
          tc_fence_after();
          uint32_t ra[8], rb[8];
          tmem_ld16x256_x2(tw + lanes + kColS, ra);
          tmem_ld16x256_x2(tw + lanes + (16u << 16) + kColS, rb);
          tmem_wait_ld();
#pragma unroll
          for (int o = 0; o < 2; ++o)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              d[e >> 1][2 * o + (e & 1)] = fmaf(__uint_as_float(ra[4 * o + e]), c, -m_ref[2 * o + (e & 1)]);
              d[2 + (e >> 1)][2 * o + (e & 1)] = fmaf(__uint_as_float(rb[4 * o + e]), c, -m_ref[2 * o + (e & 1)]);
            }
          const int base = m.blk[j] * kBS;
          if (base + kBS - 1 > p_tok) {  // the local block: keys after the query position get P = 0
#pragma unroll
            for (int i = 0; i < 4; ++i)
              if (base + 32 * q + kappa((lane >> 2) + 8 * i) > p_tok) {
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) d[i][hh] = -CUDART_INF_F;
              }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int hh = 0; hh < 4; ++hh) d[i][hh] = -CUDART_INF_F;
        }
        bool need = j == 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) need |= d[i][hh] > kRescaleLog2;
        // every raw row of the stage has been read, every warp has its scores (the same answer in
        // all four warps)
        if (named_barrier_or(bar_vote, 128, need || !ok || *abort_flag != 0)) {
          if (named_barrier_or(bar_x, 128, !ok || *abort_flag != 0)) {  // a give-up, decided alike in all four
            quit = true;
            break;
          }
          // ---- the reference moves: block maxima of s c per head over the 128 keys
          const bool first = j == 0;
          float* rm = redm + 64 * (nre & 1);
          const float* mr_old = mref + 16 * (nre & 1);
          float* mr_new = mref + 16 * ((nre & 1) ^ 1);
          ++nre;
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
            float bm = fmaxf(fmaxf(d[0][hh], d[1][hh]), fmaxf(d[2][hh], d[3][hh])) + m_ref[hh];
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
            if (lane < 4) rm[16 * q + hb + (hh & 1) + 8 * (hh >> 1)] = bm;
          }
          named_barrier(bar_x, 128);
          // the new reference of a head: the block maximum (first block) or the larger of the two
          auto new_ref = [&](int h, float& mo, float& cf) {
            const float bx = fmaxf(fmaxf(rm[h], rm[16 + h]), fmaxf(rm[32 + h], rm[48 + h]));
            mo = first ? 0.f : mr_old[h];
            float mn = first ? bx : fmaxf(mo, bx);
            if (!(mn > -CUDART_INF_F)) mn = mo;  // no valid key in the block (cannot happen): keep it finite
            cf = first ? 0.f : fast_exp2(mo - mn);
            return mn;
          };
          bool moved = false;
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {  // this thread's own heads
            const int h = hb + (hh & 1) + 8 * (hh >> 1);
            float mo, cf;
            const float mn = new_ref(h, mo, cf);
            moved |= mn != mo;
#pragma unroll
            for (int i = 0; i < 4; ++i) d[i][hh] += m_ref[hh] - mn;
            l[hh] *= cf;
            m_ref[hh] = mn;
            if (q == 0 && lane < 4) mr_new[h] = mn;
          }
          // O^T *= cf once PV(jg - 1) has landed (this thread's lane = dim 32 q + lane), four heads
          // (their hi and lo columns) at a time; every thread of the group takes the same branch
          if (__any_sync(0xffffffffu, moved) && !first && waitw(pv_done, static_cast<uint32_t>(jg - 1) & 1u)) {
            tc_fence_after();
#pragma unroll 1
            for (int h4 = 0; h4 < 4; ++h4) {
              float cf4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float mo;
                new_ref(4 * h4 + e, mo, cf4[e]);
              }
#pragma unroll
              for (int z = 0; z < 2; ++z) {
                const uint32_t ta = tw + lanes + kColO + 32 * x + 16 * z + 4 * h4;
                uint32_t o4[4];
                tmem_ld4(ta, o4);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 4; ++e) o4[e] = __float_as_uint(__uint_as_float(o4[e]) * cf4[e]);
                tmem_st4(ta, o4);
              }
            }
            tmem_wait_st();
            tc_fence_before();
          }
        }
        // ---- K of the next block (its S MMA runs while this block's P is made); its stores are
        // waited for, and the tile announced, after this block's V rows
        const bool k_pending = j + 1 < n && do_k(jg + 1, false);
        // ---- V rows -> the E4M3 V tile over the stage: row vrow = key position, MN-major
        if (ok) {
          uint8_t* vt = stg + (vrow >> 3) * 1024 + (vrow & 7) * 128;
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            uint32_t uu[8];
            dequant_quarter(rv, qq, lut, uu);
            *reinterpret_cast<uint4*>(vt + (((2 * qq) ^ (vrow & 7)) << 4)) = make_uint4(uu[0], uu[1], uu[2], uu[3]);
            *reinterpret_cast<uint4*>(vt + (((2 * qq + 1) ^ (vrow & 7)) << 4)) = make_uint4(uu[4], uu[5], uu[6], uu[7]);
            if (qq == 3 && k_pending) k_finish();
          }
        } else if (k_pending) {
          k_finish();
        }
        // ---- P = exp2(d) -> P^T hi / lo (the tile is free once PV(jg - 1) has landed)
        if (waitw(pv_done, static_cast<uint32_t>(jg - 1) & 1u)) {
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
            float pv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pv[i] = fast_exp2(d[i][hh]);
            l[hh] += (pv[0] + pv[1]) + (pv[2] + pv[3]);
            const uint32_t h01 = cvt_e4m3x2(pv[0], pv[1]), h23 = cvt_e4m3x2(pv[2], pv[3]);
            const uint32_t r01 = sub_f16x2(pack_f16x2(pv[0], pv[1]), cvt_f16x2_e4m3x2(h01));
            const uint32_t r23 = sub_f16x2(pack_f16x2(pv[2], pv[3]), cvt_f16x2_e4m3x2(h23));
            // lo carries 16 (P - hi): |P - hi| <= P / 16, so it stays <= 448 and out of the E4M3
            // subnormals for every P that matters
            const uint32_t l01 = cvt_e4m3x2_f16x2(mul_f16x2(r01, kLoScale2)), l23 = cvt_e4m3x2_f16x2(mul_f16x2(r23, kLoScale2));
            uint8_t* pw = ptile + ((hh & 1) ? psw1 : psw0) + 1024 * (hh >> 1);
            *reinterpret_cast<uint32_t*>(pw) = h01 | (h23 << 16);
            *reinterpret_cast<uint32_t*>(pw + 2048) = l01 | (l23 << 16);
          }
        }
        fence_proxy_async_smem();  // the V tile and P^T are read by the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(pv_ready);
      }
      if (quit) break;
      // ---- the unit's output: thread = dim 32 q + lane of O^T; l summed over the 128 keys
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 4);
        l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 8);
        l[hh] += __shfl_xor_sync(0xffffffffu, l[hh], 16);
      }
      if (lane < 4) {
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) redl[16 * q + hb + (hh & 1) + 8 * (hh >> 1)] = l[hh];
      }
      const bool have = waitw(pv_done, static_cast<uint32_t>(jg - 1) & 1u);  // the last PV has landed
      uint32_t o[16];
      if (have) {  // hi + lo halves of the sum
        tc_fence_after();
        uint32_t o2[16];
        tmem_ld16(tw + lanes + kColO + 32 * x, o);
        tmem_ld16(tw + lanes + kColO + 32 * x + 16, o2);
        tmem_wait_ld();
#pragma unroll
        for (int h = 0; h < 16; ++h) o[h] = __float_as_uint(fmaf(__uint_as_float(o2[h]), 1.0f / kLoScale, __uint_as_float(o[h])));
      }
      tc_fence_before();
      named_barrier(bar_x, 128);  // every warp's sums are in redl; every warp has read O^T
      __syncwarp();
      if (lane == 0) mbar_arrive(&o_free[x]);  // O^T[x] may be overwritten
      float lt[16];
#pragma unroll
      for (int h4 = 0; h4 < 4; ++h4) {
        const float4 a0 = *reinterpret_cast<const float4*>(redl + 4 * h4);
        const float4 a1 = *reinterpret_cast<const float4*>(redl + 16 + 4 * h4);
        const float4 a2 = *reinterpret_cast<const float4*>(redl + 32 + 4 * h4);
        const float4 a3 = *reinterpret_cast<const float4*>(redl + 48 + 4 * h4);
        lt[4 * h4 + 0] = (a0.x + a1.x) + (a2.x + a3.x);
        lt[4 * h4 + 1] = (a0.y + a1.y) + (a2.y + a3.y);
        lt[4 * h4 + 2] = (a0.z + a1.z) + (a2.z + a3.z);
        lt[4 * h4 + 3] = (a0.w + a1.w) + (a2.w + a3.w);
      }
      const bool zero = !have || *abort_flag != 0;
      const int dim = 32 * q + lane;
#pragma unroll
      for (int h = 0; h < 16; ++h) {
        const bool z = zero || !(lt[h] > 0.f);
        const float val = z ? 0.f : __uint_as_float(o[h]) / lt[h];
        const int64_t orow = static_cast<int64_t>(t) * kQHeads + g * kHPG + h;
        if (p.splits == 1) {
          reinterpret_cast<__nv_bfloat16*>(p.out)[orow * kD + dim] = __float2bfloat16_rn(val);
        } else {
          const int64_t prow = static_cast<int64_t>(split) * p.T * kQHeads + orow;
          p.part_o[prow * kD + dim] = val;
        }
      }
      if (p.splits > 1 && q == 0 && lane < 4) {  // lse of this thread's four heads
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
          const int h = hb + (hh & 1) + 8 * (hh >> 1);
          float lh = 0.f;
#pragma unroll
          for (int hx = 0; hx < 16; ++hx) lh = hx == h ? lt[hx] : lh;
          const bool z = zero || !(lh > 0.f);
          const int64_t prow = static_cast<int64_t>(split) * p.T * kQHeads + static_cast<int64_t>(t) * kQHeads + g * kHPG + h;
          p.part_lse[prow] = z ? -CUDART_INF_F : m_ref[hh] + __log2f(lh);
        }
      }
      named_barrier(bar_x, 128);  // redl may be written again
      __syncwarp();
      if (lane == 0) mbar_arrive(&meta_empty[k % kMeta]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpRes) {
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
// there are several waves of units. The many-token kernel takes more than two units per SM
// (of msa_host::kTunedSms SMs: the choice depends on the arguments alone).
bool use_tc_kernel(int T) { return 4 * T > 2 * msa_host::kTunedSms; }

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
