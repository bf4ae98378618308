// msa_indexer.cu — indexer score + 128-token block max-pool of the MSA decode step.
//
// What it computes ("vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", "MSA primer"; "MiniMax
// M3 in vLLM ...", "解码索引器分数内核" and "解码内核中的推测解码"): for every query token t of every
// sequence and every GQA group g, block_scores[t][g][k] = max over the cache positions j of block
// k with j <= p_t of  index_q[t][g] . ik_fp8[j], where ik_fp8 is the NVFP4 index key dequantised
// to E4M3 ("NVIDIA Blackwell optimizado kernes MSA") — or the FP8 index key as is.
//
// GB300 design: one persistent CTA per SM; the flattened (sequence, block) page list is split
// evenly over CTAs, so ragged batches balance at page granularity. Inside a CTA the work is a
// warp-specialised pipeline; every hand-off is an mbarrier ring, so each role runs at its own
// pace and the latency of one stage hides behind the depth of the rings:
//  * producer warp: resolves 32 pages' (sequence, block, page id) at a time, the next batch's
//    block-table loads in flight while lane 0 issues one 2-D tensor copy per 128-token index
//    page into the stage ring (L2 evict-first: every byte is read once). The copy applies the
//    128-byte swizzle, so the per-row loads below are free of bank conflicts;
//  * three dequant groups of four warps take pages in turn, thread = key row = TMEM lane. An
//    NVFP4 row becomes 128 E4M3 bytes (LUT + byte-permute) stored straight into a TMEM key
//    tile (tcgen05.st): the tile never makes a round trip through shared memory. An FP8 page
//    is already the tensor core's swizzled K-major tile and stays in its stage. The groups
//    also keep each tile slot's copy of the sequence's index queries (a 32 x 128 B swizzled
//    shared tile) current;
//  * three MMA warps take pages in turn, one thread each issuing (a burst of four MMAs costs the
//    issuing thread ~450 cycles): four tcgen05.mma kind::f8f6f4 per page (M = 128 keys, N = 16 or 32
//    (token, group) columns, K = 4 x 32) into a ring of TMEM accumulators, then commits that
//    free the key tile and publish the scores;
//  * three max-pool groups of four warps (one per TMEM lane quarter) take pages in turn (a page's
//    pooling is a chain of dependent steps, so the groups overlap several pages): the 16x256b TMEM
//    load hands every thread four keys of eight columns, so a warp needs a 4-key register max
//    and a 3-step shuffle transpose-reduce. Each quarter stores its partial maxima in shared
//    memory and counts itself in; the page's last quarter combines the four and stores the block
//    scores, so no quarter ever waits for another. Keys after a query position are
//    masked on the (rare) pages that hold them.
// Every wait is bounded (MSA_ERR_TIMEOUT); no role waits on a named barrier inside its loop;
// every page id is checked (MSA_ERR_DEVICE_FAULT, the block is scored -inf); nothing traps.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "msa.h"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

constexpr int kTmemCols = 512;
// The exact-score variant (NVFP4 keys to f16 with no E4M3 re-rounding, f16 score MMA): an
// internal index kind next to MSA_INDEX_NVFP4 and MSA_INDEX_FP8.
constexpr int kIdxNvExact = 2;

// Warp roles per index kind: a producer warp, kMmaWarps MMA-issuing warps (pages in turn),
// kDqGroups dequant groups and three max-pool groups of four warps, and kDTiles TMEM
// accumulators of 32 columns. The exact (f16) keys cost twice the dequant work of the E4M3 ones,
// so that kind runs four dequant groups and two MMA warps (which have the slack) where the others
// run three of each.
template <int DT>
struct RoleCfg {
  static constexpr int kDqGroups = 3, kMmaWarps = 3, kDTiles = 9;
};
template <>
struct RoleCfg<kIdxNvExact> {
  static constexpr int kDqGroups = 4, kMmaWarps = 2, kDTiles = 6;
};
template <int DT>
struct Roles : RoleCfg<DT> {
  using C = RoleCfg<DT>;
  static constexpr int kEpGroups = 3;
  static constexpr int kWarpDq = 1 + C::kMmaWarps;           // first dequant warp
  static constexpr int kWarpEp = kWarpDq + 4 * C::kDqGroups;  // first max-pool warp
  static constexpr int kThreads = 32 * (kWarpEp + 4 * kEpGroups);
  // Partial-maximum slots of the max-pool quarters: page n uses slot n % kPartSlots. A slot is
  // written again only by page n + kPartSlots, whose MMA needed its accumulator released by all
  // four quarters at page n + kPartSlots - kDTiles, which each quarter reaches after combining
  // page n (a warp takes its pages in order): 2 * kDTiles slots are enough.
  static constexpr int kPartSlots = 2 * C::kDTiles;
  static_assert(C::kDTiles % kEpGroups == 0 && C::kDTiles % C::kMmaWarps == 0, "an accumulator serves one group");
  static_assert(kThreads <= 1024, "one CTA");
};

// Key tiles and query tiles per index kind: E4M3 keys take 32 TMEM columns a tile and the
// query tile is 32 rows x 128 E4M3; exact keys take 64 columns (f16) and the query tile is
// 32 rows x 128 f16 (two 64-element K atoms of 4 KB).
template <int DT>
struct TileCfg {
  static constexpr int kATiles = 6;        // TMEM key tiles
  static constexpr int kACols = 32;        // TMEM columns of one key tile
  static constexpr int kBTile = 32 * kD;   // bytes of one query tile
  static constexpr int kLutBytes = 256 * 8;
};
template <>
struct TileCfg<kIdxNvExact> {
  static constexpr int kATiles = 4;
  static constexpr int kACols = 64;
  static constexpr int kBTile = 32 * kD * 2;
  static constexpr int kLutBytes = 256 * 16;
};
template <int DT>
constexpr bool tiles_ok() {
  return TileCfg<DT>::kATiles % Roles<DT>::kDqGroups == 0 && TileCfg<DT>::kATiles % Roles<DT>::kMmaWarps == 0 &&
         TileCfg<DT>::kACols * TileCfg<DT>::kATiles + 32 * Roles<DT>::kDTiles <= kTmemCols;
}
static_assert(tiles_ok<MSA_INDEX_NVFP4>() && tiles_ok<MSA_INDEX_FP8>() && tiles_ok<kIdxNvExact>(),
              "a key tile serves one dequant group and one MMA warp; TMEM budget");

// Page n of a CTA lives in stage n % kStages, key tile n % kATiles and accumulator
// n % kDTiles; the ring sizes are multiples of the group counts, so every slot is used by one
// group, in page order, and nobody ever waits on an mbarrier phase two steps ahead of the one
// it last saw (parity cannot tell those apart).
template <int DT>
struct IdxCfg;
template <>
struct IdxCfg<MSA_INDEX_NVFP4> {
  static constexpr int kPage = kIdxPageNv;
  static constexpr int kStages = 18;
};
template <>
struct IdxCfg<MSA_INDEX_FP8> {
  static constexpr int kPage = kIdxPageFp8;
  static constexpr int kStages = 9;
};
template <>
struct IdxCfg<kIdxNvExact> {
  static constexpr int kPage = kIdxPageNv;
  static constexpr int kStages = 16;
};

struct IdxParams {
  int32_t B, T, maxb, max_q_len, num_pages;
  int32_t kb, ke;  // the scanned block range [kb, ke) of every sequence (a context shard)
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_table;
  const uint8_t* index_q;
  float* block_scores;
  uint32_t* status;
};

struct SlotInfo {
  int32_t b, k, valid, pad;
};

template <int DT>
struct IdxSmem {
  static constexpr int kStages = IdxCfg<DT>::kStages;
  static constexpr int kPage = IdxCfg<DT>::kPage;
  static constexpr int kATiles = TileCfg<DT>::kATiles;
  static constexpr int kBTile = TileCfg<DT>::kBTile;
  static constexpr int kDTiles = Roles<DT>::kDTiles, kPartSlots = Roles<DT>::kPartSlots;
  static_assert(kStages % Roles<DT>::kDqGroups == 0, "a stage serves one dequant group");
  // offsets from a 1024-byte aligned base (pages and query tiles are multiples of 1024 B)
  static constexpr size_t kOffStage = 0;
  static constexpr size_t kOffB = kOffStage + static_cast<size_t>(kStages) * kPage;
  static constexpr size_t kOffFull = kOffB + static_cast<size_t>(kATiles) * kBTile;
  static constexpr size_t kOffEmpty = kOffFull + 8 * kStages;
  static constexpr size_t kOffAFull = kOffEmpty + 8 * kStages;
  static constexpr size_t kOffAEmpty = kOffAFull + 8 * kATiles;
  static constexpr size_t kOffDFull = kOffAEmpty + 8 * kATiles;
  static constexpr size_t kOffDEmpty = kOffDFull + 8 * kDTiles;
  static constexpr size_t kOffInfo = kOffDEmpty + 8 * kDTiles;
  static constexpr size_t kOffAMeta = kOffInfo + sizeof(SlotInfo) * kStages;  // [kATiles] int2
  static constexpr size_t kOffBTag = kOffAMeta + 8 * kATiles;                 // [kATiles][4] int
  static constexpr size_t kOffPart = kOffBTag + 16 * kATiles;                 // [kPartSlots][4][32] fp32
  static constexpr size_t kOffCnt = kOffPart + 4 * kPartSlots * 4 * 32;       // [kPartSlots] int
  static constexpr size_t kOffLut = (kOffCnt + 4 * kPartSlots + 15) & ~static_cast<size_t>(15);  // 16-B entries
  static constexpr size_t kOffMisc = kOffLut + TileCfg<DT>::kLutBytes;
  static constexpr size_t kOffPtab = kOffMisc + 64;  // 32 x int4
  static constexpr size_t kOffWarpSum = kOffPtab + 32 * 16;
  static constexpr size_t kOffPrefix = kOffWarpSum + 4 * 32;
  static size_t bytes(int B) { return 1024 + kOffPrefix + 4 * static_cast<size_t>(B + 1); }
};
static_assert(IdxSmem<kIdxNvExact>::kOffLut % 16 == 0 && IdxSmem<kIdxNvExact>::kOffB % 1024 == 0,
              "the exact table's 16-B entries and the query atoms are aligned");

// Pages of sequence b that the indexer scans (0 for padded or invalid rows).
__device__ __forceinline__ int seq_pages(const IdxParams& p, int b, bool* bad) {
  const int q0 = p.qsl[b], q1 = p.qsl[b + 1];
  const int ql = q1 - q0;
  const int L = p.seq_lens[b];
  if (ql < 0 || ql > p.max_q_len || q0 < 0 || q1 > p.T || (ql > 0 && (L < ql || L > p.maxb * kBS))) {
    *bad = true;
    return 0;
  }
  const int nb = ql > 0 ? ceil_div(L, kBS) : 0;
  return max(0, min(p.ke, nb) - min(p.kb, nb));
}

// Sequence of global page gp: the largest b with prefix[b] <= gp.
__device__ __forceinline__ int page_seq(const int* prefix, int B, int gp) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= gp) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Dequantise key row r of a staged NVFP4 page (written by a 128-byte-swizzled copy) to 128
// E4M3 bytes straight into the TMEM key tile at taddr (this thread's lane, 32 columns: column c
// holds elements 4c .. 4c+3): each quarter of the row is stored while the next is dequantised.
// Completes at tmem_wait_st().
__device__ __forceinline__ void dequant_row_nvfp4_tmem(const uint8_t* pg, int r, const uint2* lut, uint32_t taddr) {
  const uint2 sc = lds64(pg + sw128_phys(static_cast<uint32_t>(kScaleOff + r * kRowScales)));
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 c = lds128(pg + sw128_phys(static_cast<uint32_t>(r * kRowCodes + 16 * q)));
    const uint32_t s2 = ((q < 2) ? sc.x : sc.y) >> (16 * (q & 1));
    const uint2 e0 = lut[s2 & 0xFFu], e1 = lut[(s2 >> 8) & 0xFFu];
    uint32_t w[8];
    dq8(c.x, e0, w[0], w[1]);
    dq8(c.y, e0, w[2], w[3]);
    dq8(c.z, e1, w[4], w[5]);
    dq8(c.w, e1, w[6], w[7]);
    tmem_st8(taddr + 8 * q, w);
  }
}

// Key row r of a staged NVFP4 page as exact f16 (table entries of build_exact_lut) straight into
// the TMEM key tile at taddr (this thread's lane, 64 columns: column c holds elements 2c, 2c+1):
// each 32 elements are stored while the next are dequantised. Completes at tmem_wait_st().
__device__ __forceinline__ void dequant_row_exact_tmem(const uint8_t* pg, int r, const uint4* lut, uint32_t taddr) {
  const uint2 sc2 = lds64(pg + sw128_phys(static_cast<uint32_t>(kScaleOff + r * kRowScales)));
#pragma unroll
  for (int q = 0; q < 4; ++q) {  // 32 elements: 32 q .. +31, scales 2 q and 2 q + 1 of the row
    const uint4 c = lds128(pg + sw128_phys(static_cast<uint32_t>(r * kRowCodes + 16 * q)));
    const uint32_t s2 = ((q < 2) ? sc2.x : sc2.y) >> (16 * (q & 1));
    const uint4 t0 = lut[s2 & 0xFFu], t1 = lut[(s2 >> 8) & 0xFFu];
    uint32_t w[16];
    uint32_t o[4];
    dq8_f16(c.x, t0, o);
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = o[e];
    dq8_f16(c.y, t0, o);
#pragma unroll
    for (int e = 0; e < 4; ++e) w[4 + e] = o[e];
    dq8_f16(c.z, t1, o);
#pragma unroll
    for (int e = 0; e < 4; ++e) w[8 + e] = o[e];
    dq8_f16(c.w, t1, o);
#pragma unroll
    for (int e = 0; e < 4; ++e) w[12 + e] = o[e];
    tmem_st16(taddr + 16 * q, w);
  }
}

// One step of a shuffle transpose-reduce: lanes l and l ^ k (k = lane bit) each keep half of
// their values, the lower-bit lane the first half, and take the max with the partner's copy.
template <int N>
__device__ __forceinline__ void xreduce_step(float (&v)[8], int lane, int k) {
  const bool up = (lane & k) != 0;
#pragma unroll
  for (int c = 0; c < N; ++c) {
    const float send = up ? v[c] : v[c + N];
    const float keep = up ? v[c + N] : v[c];
    v[c] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, k));
  }
}

// Wait on a warp's behalf: true when every lane saw the phase complete.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

template <int DT>
__global__ void __launch_bounds__(Roles<DT>::kThreads, 1)
    k_indexer(const IdxParams p, const __grid_constant__ CUtensorMap tmap) {
  using S = IdxSmem<DT>;
  using R = Roles<DT>;
  constexpr int kDqGroups = R::kDqGroups, kEpGroups = R::kEpGroups, kMmaWarps = R::kMmaWarps;
  constexpr int kWarpDq = R::kWarpDq, kWarpEp = R::kWarpEp, kIdxThreads = R::kThreads;
  constexpr int kDTiles = R::kDTiles, kPartSlots = R::kPartSlots;
  constexpr int kStages = S::kStages;
  constexpr int kATiles = TileCfg<DT>::kATiles, kACols = TileCfg<DT>::kACols, kBTile = TileCfg<DT>::kBTile;
  constexpr bool kExact = DT == kIdxNvExact;
  constexpr bool kNv = DT == MSA_INDEX_NVFP4 || kExact;  // NVFP4 pages, dequantised into TMEM
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = smem + S::kOffStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kOffFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + S::kOffEmpty);
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + S::kOffAFull);
  uint64_t* a_empty = reinterpret_cast<uint64_t*>(smem + S::kOffAEmpty);
  uint64_t* d_full = reinterpret_cast<uint64_t*>(smem + S::kOffDFull);
  uint64_t* d_empty = reinterpret_cast<uint64_t*>(smem + S::kOffDEmpty);
  uint64_t* mma_fin = reinterpret_cast<uint64_t*>(smem + S::kOffMisc + 16);
  SlotInfo* info = reinterpret_cast<SlotInfo*>(smem + S::kOffInfo);
  int2* ameta = reinterpret_cast<int2*>(smem + S::kOffAMeta);
  int* btag = reinterpret_cast<int*>(smem + S::kOffBTag);
  uint2* lut = reinterpret_cast<uint2*>(smem + S::kOffLut);
  uint4* lut16 = reinterpret_cast<uint4*>(smem + S::kOffLut);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc);
  int* bad_batch = reinterpret_cast<int*>(smem + S::kOffMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffMisc + 8);
  int* warp_sum = reinterpret_cast<int*>(smem + S::kOffWarpSum);
  int* prefix = reinterpret_cast<int*>(smem + S::kOffPrefix);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- prologue: barriers, TMEM, LUT, per-sequence page prefix sums ---------------------
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kNv ? 4 : 1);  // NVFP4: the dequant group's 4 warps; FP8: the page's MMAs
    }
    for (int i = 0; i < kATiles; ++i) {
      mbar_init(&a_full[i], 4);
      mbar_init(&a_empty[i], 1);  // the page's MMAs have completed (a commit)
    }
    for (int i = 0; i < kDTiles; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], 4);
    }
    for (int i = 0; i < kMmaWarps; ++i) mbar_init(&mma_fin[i], 1);
    fence_mbar_init();
    *abort_flag = 0;
    *bad_batch = 0;
  }
  if (tid < 4 * kATiles) btag[tid] = -1;
  if (tid < kPartSlots) reinterpret_cast<int*>(smem + S::kOffCnt)[tid] = 0;
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  if constexpr (kExact)
    build_exact_lut(lut16, tid, kIdxThreads);
  else if constexpr (kNv)
    build_dequant_lut(lut, tid, kIdxThreads);
  __syncthreads();  // flags initialised before anyone raises them
  {
    // prefix[b] = pages of sequences 0 .. b-1: per-thread counts, warp scans, one scan of
    // the warp totals
    const int per = ceil_div(p.B, kIdxThreads);
    const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
    int local = 0;
    bool bad = false;
    for (int b = b0; b < b1; ++b) {
      const int c = seq_pages(p, b, &bad);
      prefix[b] = c;
      local += c;
    }
    if (bad) *bad_batch = 1;
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int nw = kIdxThreads / 32;
      int v = lane < nw ? warp_sum[lane] : 0, x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += u;
      }
      if (lane < nw) warp_sum[lane] = x - v;  // exclusive
      if (lane == nw - 1) prefix[p.B] = x;
      if (lane == 0 && p.B > 0 && (p.qsl[0] != 0 || p.qsl[p.B] != p.T)) *bad_batch = 1;
    }
    __syncthreads();
    int run = warp_sum[warp] + incl - local;
    for (int b = b0; b < b1; ++b) {
      const int c = prefix[b];
      prefix[b] = run;
      run += c;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t t_a = tmem;                    // key tiles: columns kACols a .. kACols (a + 1) - 1
  const uint32_t t_d = tmem + kACols * kATiles; // accumulators
  if (blockIdx.x == 0 && tid == 0 && *bad_batch) set_status(p.status, MSA_ERR_INVALID_ARG);

  const int total = prefix[p.B];
  const int start = static_cast<int>((static_cast<int64_t>(total) * blockIdx.x) / gridDim.x);
  const int end = static_cast<int>((static_cast<int64_t>(total) * (blockIdx.x + 1)) / gridDim.x);
  const int npages = end - start;

  if (warp == 0) {
    // ---- producer ------------------------------------------------------------------------
    int4* ptab = reinterpret_cast<int4*>(smem + S::kOffPtab);
    const uint64_t policy = policy_evict_first();
    if (lane == 0) prefetch_tensormap(&tmap);
    auto resolve = [&](int n) -> int4 {  // (sequence, block, page id) of this CTA's page n
      if (n >= npages) return make_int4(0, 0, -1, 0);
      const int gp = start + n;
      const int b = page_seq(prefix, p.B, gp);
      const int k = p.kb + gp - prefix[b];
      return make_int4(b, k, p.block_table[static_cast<int64_t>(b) * p.maxb + k], 0);
    };
    int4 cur = resolve(lane);
    int issued = 0;
    bool stop = false;
    for (int base = 0; base < npages && !stop; base += 32) {
      ptab[lane] = cur;
      __syncwarp();
      cur = resolve(base + 32 + lane);  // the next batch's loads fly while lane 0 issues
      if (lane == 0) {
        const int cnt = min(32, npages - base);
        for (int u = 0; u < cnt; ++u) {
          const int n = base + u;
          const int slot = n % kStages;
          const uint32_t ph = static_cast<uint32_t>(n / kStages) & 1u;
          if (!mbar_wait(&empty[slot], ph ^ 1u, abort_flag)) {
            if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
            *abort_flag = 1;
            stop = true;
            break;
          }
          const int4 e = ptab[u];
          const bool valid = e.z >= 0 && e.z < p.num_pages;
          info[slot].b = e.x;
          info[slot].k = e.y;
          info[slot].valid = valid ? 1 : 0;
          if (valid) {
            mbar_arrive_expect_tx(&full[slot], S::kPage);
            tma_load_2d(stages + static_cast<size_t>(slot) * S::kPage, &tmap, 0, e.z * (S::kPage / kD), &full[slot],
                        policy);
          } else {
            set_status(p.status, MSA_ERR_DEVICE_FAULT);
            mbar_arrive(&full[slot]);
          }
          issued = n + 1;
        }
      }
      stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
      __syncwarp();
    }
    // Never leave while a copy into this CTA's shared memory may still be in flight: wait
    // for the last page issued into every slot (in a normal run they have all landed).
    if (lane == 0) {
      for (int n = issued > kStages ? issued - kStages : 0; n < issued; ++n)
        if (!mbar_wait_bounded(&full[n % kStages], static_cast<uint32_t>(n / kStages) & 1u, kWaitLimitNs, nullptr))
          set_status(p.status, MSA_ERR_TIMEOUT);
    }
  } else if (warp < kWarpDq) {
    // ---- MMA issue: pages mw, mw + kMmaWarps, ...; the whole warp runs the loop (its
    // indices stay warp-uniform), lane 0 issues -------------------------------------------------
    // rows >= 4 q_len of a query tile are zero
    constexpr uint32_t idesc = kExact ? idesc_f16_f32(128, 32) : idesc_e4m3_f32(128, 32);
    const int mw = warp - 1;
    uint64_t* fin = mma_fin + mw;
    int issued = 0;
    for (int n = mw; n < npages; n += kMmaWarps) {
      const int a = n % kATiles, d = n % kDTiles;
      if (!warp_wait(&a_full[a], static_cast<uint32_t>(n / kATiles) & 1u, abort_flag) ||
          !warp_wait(&d_empty[d], (static_cast<uint32_t>(n / kDTiles) & 1u) ^ 1u, abort_flag)) {
        if (lane == 0) {
          if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      const bool valid = ameta[a].x != 0;
      if (lane == 0) {
        if (valid) {
          const uint32_t b_addr = smem_u32(smem + S::kOffB) + static_cast<uint32_t>(a * kBTile);
          const uint32_t st_addr = smem_u32(stages) + static_cast<uint32_t>((n % kStages) * S::kPage);
          if constexpr (kExact) {
#pragma unroll
            for (int s = 0; s < 8; ++s)  // K = 16 f16 per MMA: 8 TMEM columns; 32 B of the query atom
              tc_mma_f16_ta(t_d + 32 * d, t_a + kACols * a + 8 * s,
                            sw128_kmajor_desc(b_addr + (s >> 2) * 4096 + 32 * (s & 3)), idesc, s > 0 ? 1u : 0u);
          } else {
#pragma unroll
            for (int s = 0; s < 4; ++s) {
              if constexpr (kNv)
                tc_mma_f8_ta(t_d + 32 * d, t_a + kACols * a + 8 * s, sw128_kmajor_desc(b_addr + 32 * s), idesc,
                             s > 0 ? 1u : 0u);
              else
                tc_mma_f8(t_d + 32 * d, sw128_kmajor_desc(st_addr + 32 * s), sw128_kmajor_desc(b_addr + 32 * s),
                          idesc, s > 0 ? 1u : 0u);
            }
          }
          tc_commit(&d_full[d]);
          tc_commit(&a_empty[a]);  // the key tile and query tile (and an FP8 stage) may be refilled
          if constexpr (!kNv) tc_commit(&empty[n % kStages]);
        } else {
          mbar_arrive(&d_full[d]);
          mbar_arrive(&a_empty[a]);
          if constexpr (!kNv) mbar_arrive(&empty[n % kStages]);
        }
      }
      __syncwarp();
      issued = n + 1;
    }
    // every MMA has completed before TMEM is released
    if (lane == 0 && issued > 0) {
      tc_commit(fin);
      if (!mbar_wait_bounded(fin, 0u, kWaitLimitNs, nullptr)) set_status(p.status, MSA_ERR_TIMEOUT);
    }
  } else if (warp < kWarpEp) {
    // ---- dequant groups: pages dq, dq + 2, ... ------------------------------------------------
    const int dq = (warp - kWarpDq) >> 2;
    const int wq = warp & 3;        // TMEM lane quarter this warp may access
    const int i = 32 * wq + lane;   // key row = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
    int cur_b = -1, q0 = 0, ncol = 0;
    for (int n = dq; n < npages; n += kDqGroups) {
      const int s = n % kStages, a = n % kATiles;
      if (!warp_wait(&full[s], static_cast<uint32_t>(n / kStages) & 1u, abort_flag)) break;
      const SlotInfo si = info[s];
      if (!warp_wait(&a_empty[a], (static_cast<uint32_t>(n / kATiles) & 1u) ^ 1u, abort_flag)) break;
      tc_fence_after();
      if constexpr (kNv && !kExact) {
        if (si.valid) dequant_row_nvfp4_tmem(stages + static_cast<size_t>(s) * S::kPage, i, lut, t_a + kACols * a + lane_base);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);  // the warp's reads of the stage are done
      }
      if (si.b != cur_b) {
        cur_b = si.b;
        q0 = p.qsl[cur_b];
        ncol = 4 * (p.qsl[cur_b + 1] - q0);
      }
      int* tag = btag + 4 * a + wq;
      if (*tag != cur_b) {
        // this warp's 8 rows of the slot's query tile: rows c < 4 * q_len, zero rows up to 32
        uint8_t* btile = smem + S::kOffB + static_cast<size_t>(a) * kBTile;
        if constexpr (kExact) {
          // f16 rows (E4M3 -> f16 is exact), two K atoms of 64 dims: 512 chunks of 8 dims
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int id = 128 * wq + 4 * lane + u;
            const int row = id >> 4, cc = id & 15;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (row < ncol) {
              const uint2 e = *reinterpret_cast<const uint2*>(p.index_q + static_cast<int64_t>(q0 * 4 + row) * kD + 8 * cc);
              v = make_uint4(cvt_f16x2_e4m3x2(e.x), cvt_f16x2_e4m3x2(e.x >> 16), cvt_f16x2_e4m3x2(e.y),
                             cvt_f16x2_e4m3x2(e.y >> 16));
            }
            *reinterpret_cast<uint4*>(btile + (cc >> 3) * 4096 + sw128_chunk_off(row, cc & 7)) = v;
          }
        } else {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int id = 64 * wq + 2 * lane + u;  // 256 chunks of 16 B
            const int row = id >> 3, c = id & 7;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (row < ncol)
              v = *reinterpret_cast<const uint4*>(p.index_q + static_cast<int64_t>(q0 * 4 + row) * kD + 16 * c);
            *reinterpret_cast<uint4*>(btile + sw128_chunk_off(row, c)) = v;
          }
        }
        fence_proxy_async_smem();  // visible to the tensor core
        __syncwarp();
        if (lane == 0) *tag = cur_b;
      }
      if constexpr (kExact) {  // the f16 row, then the stage is free
        const uint8_t* pg = stages + static_cast<size_t>(s) * S::kPage;
        if (si.valid) dequant_row_exact_tmem(pg, i, lut16, t_a + kACols * a + lane_base);
        tmem_wait_st();
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
      } else if constexpr (kNv) {
        tmem_wait_st();
      }
      tc_fence_before();
      if (wq == 0 && lane == 0) ameta[a] = make_int2(si.valid, ncol);
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[a]);
    }
  } else {
    // ---- max-pool warps: warp (ep, wq) pools TMEM lane quarter wq of pages ep, ep + 3, ...;
    // the quarter that finishes a page last (a shared counter) combines the four partial
    // maxima, so the quarters never wait for one another ----------------------------------------
    const int ep = (warp - kWarpEp) >> 2;
    const int wq = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(32 * wq) << 16;
    float* part = reinterpret_cast<float*>(smem + S::kOffPart);  // [kPartSlots][4 quarters][32]
    int* cnt = reinterpret_cast<int*>(smem + S::kOffCnt);         // [kPartSlots] quarters done
    // lane l holds the facts of the warp's page (base + l): block, first column row, columns,
    // first query position, page id valid
    int m_k = 0, m_q0 = 0, m_ncol = 0, m_p0 = 0, m_valid = 0;
    int j = 0;
    for (int n = ep; n < npages; n += kEpGroups, ++j) {
      if ((j & 31) == 0) {
        const int nn = n + kEpGroups * lane;
        if (nn < npages) {
          const int gp = start + nn;
          const int b = page_seq(prefix, p.B, gp);
          m_k = p.kb + gp - prefix[b];
          m_q0 = p.qsl[b];
          const int ql = p.qsl[b + 1] - m_q0;
          m_ncol = 4 * ql;
          m_p0 = p.seq_lens[b] - ql;
          const int phys = p.block_table[static_cast<int64_t>(b) * p.maxb + m_k];
          m_valid = phys >= 0 && phys < p.num_pages;
        }
      }
      const int src = j & 31;
      const int k = __shfl_sync(0xffffffffu, m_k, src);
      const int p0 = __shfl_sync(0xffffffffu, m_p0, src);
      const bool valid = __shfl_sync(0xffffffffu, m_valid, src) != 0;
      const int d = n % kDTiles;
      if (!warp_wait(&d_full[d], static_cast<uint32_t>(n / kDTiles) & 1u, abort_flag)) {
        if (lane == 0) {
          if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
          *abort_flag = 1;
        }
        break;
      }
      tc_fence_after();
      float pm = -CUDART_INF_F;  // this lane's column maximum over the quarter's 32 keys
      int col = 0;
      {
        uint32_t a[16], b[16];
        if (valid) {
          const uint32_t taddr = t_d + 32 * d + lane_base;
          tmem_ld16x256_x4(taddr, a);
          tmem_ld16x256_x4(taddr + (16u << 16), b);
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&d_empty[d]);  // the accumulator may be overwritten
        if (valid) {
          if ((k + 1) * kBS - 1 > p0) {  // keys after a query position are masked per column
            const int pos = k * kBS + 32 * wq + (lane >> 2);  // key of a[0]
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int c = 8 * (e >> 2) + 2 * (lane & 3) + (e & 1);
              const int row = 8 * ((e >> 1) & 1);
              const int lim = p0 + (c >> 2);
              if (pos + row > lim) a[e] = __float_as_uint(-CUDART_INF_F);
              if (pos + row + 16 > lim) b[e] = __float_as_uint(-CUDART_INF_F);
            }
          }
          float v[8];  // v[2o + e]: column 8o + 2(lane % 4) + e, max over this thread's 4 keys
#pragma unroll
          for (int o = 0; o < 4; ++o)
#pragma unroll
            for (int e = 0; e < 2; ++e)
              v[2 * o + e] = fmaxf(max3f(__uint_as_float(a[4 * o + e]), __uint_as_float(a[4 * o + 2 + e]),
                                         __uint_as_float(b[4 * o + e])),
                                   __uint_as_float(b[4 * o + 2 + e]));
          // the 8 lanes with equal lane % 4 hold the same columns: reduce over lane bits 4, 3, 2
          xreduce_step<4>(v, lane, 16);
          xreduce_step<2>(v, lane, 8);
          xreduce_step<1>(v, lane, 4);
          pm = v[0];
        }
        col = 16 * ((lane >> 4) & 1) + 8 * ((lane >> 3) & 1) + 2 * (lane & 3) + ((lane >> 2) & 1);
      }
      // partial maxima of this quarter, then the page's quarter count
      const int slot = n % kPartSlots;
      part[(slot * 4 + wq) * 32 + col] = pm;
      __threadfence_block();
      __syncwarp();
      int done = 0;
      if (lane == 0) done = atomicAdd(&cnt[slot], 1);
      done = __shfl_sync(0xffffffffu, done, 0);
      if (done == 3) {  // the last quarter: combine and store the block scores
        __threadfence_block();
        const int ncol = __shfl_sync(0xffffffffu, m_ncol, src), q0 = __shfl_sync(0xffffffffu, m_q0, src);
        if (lane < ncol) {
          const float* s4 = part + slot * 128;
          const float m = valid ? fmaxf(fmaxf(s4[lane], s4[32 + lane]), fmaxf(s4[64 + lane], s4[96 + lane]))
                                : -CUDART_INF_F;
          p.block_scores[static_cast<int64_t>(q0 * 4 + lane) * p.maxb + k] = m;
        }
        __syncwarp();
        if (lane == 0) cnt[slot] = 0;  // free for page n + kPartSlots
      }
    }
  }
  if (tid == 0 || (warp >= kWarpDq && lane == 0)) {
    if (*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int DT>
msa_status launch_indexer(const IdxParams& p, const uint8_t* pages, cudaStream_t stream) {
  // the index pool as rows of 128 B, one page per box
  CUtensorMap tmap;
  constexpr uint32_t kRows = IdxCfg<DT>::kPage / kD;
  if (!msa_host::rows128_tensor_map(&tmap, pages, static_cast<uint64_t>(p.num_pages > 0 ? p.num_pages : 1) * kRows,
                                    kRows))
    return MSA_ERR_CUDA;
  const int sms = msa_host::num_sms();
  if (sms <= 0) return MSA_ERR_CUDA;
  const size_t smem = IdxSmem<DT>::bytes(p.B);
  if (cudaFuncSetAttribute(k_indexer<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return MSA_ERR_CUDA;
  k_indexer<DT><<<sms, Roles<DT>::kThreads, smem, stream>>>(p, tmap);
  return msa_host::launch_status();
}

}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

namespace {
msa_status indexer_entry(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                         const uint8_t* index_q, int32_t block_begin, int32_t block_end, float* block_scores,
                         uint32_t* status, bool exact, cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = check_batch(batch)) != MSA_OK) return st;
  if ((st = check_cache(cache, true, false)) != MSA_OK) return st;
  if (block_begin < 0 || block_end < block_begin) return MSA_ERR_INVALID_ARG;
  if (batch->B == 0 || batch->T == 0 || block_end == block_begin) return MSA_OK;
  if (index_q == nullptr || block_scores == nullptr || !aligned(index_q, 16) || !aligned(block_scores, 4))
    return MSA_ERR_INVALID_ARG;
  if (cache->num_pages > (1 << 24)) return MSA_ERR_UNSUPPORTED;  // page rows index a 2^31-row tensor
  IdxParams p;
  p.B = batch->B;
  p.T = batch->T;
  p.maxb = batch->max_blocks_per_seq;
  p.max_q_len = batch->max_q_len;
  p.num_pages = cache->num_pages;
  p.kb = block_begin;
  p.ke = block_end;
  p.qsl = batch->query_start_loc;
  p.seq_lens = batch->seq_lens;
  p.block_table = batch->block_table;
  p.index_q = index_q;
  p.block_scores = block_scores;
  p.status = status;
  if (cache->index_dtype == MSA_INDEX_NVFP4)
    return exact ? launch_indexer<kIdxNvExact>(p, cache->index_pages, stream)
                 : launch_indexer<MSA_INDEX_NVFP4>(p, cache->index_pages, stream);
  return launch_indexer<MSA_INDEX_FP8>(p, cache->index_pages, stream);  // FP8 keys are never re-rounded
}
}  // namespace

extern "C" msa_status msa_indexer_decode_range(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                               const uint8_t* index_q, int32_t block_begin, int32_t block_end,
                                               float* block_scores, uint32_t* status, cudaStream_t stream) {
  return indexer_entry(geo, batch, cache, index_q, block_begin, block_end, block_scores, status, false, stream);
}

extern "C" msa_status msa_indexer_decode_exact(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                               const uint8_t* index_q, float* block_scores, uint32_t* status,
                                               cudaStream_t stream) {
  return indexer_entry(geo, batch, cache, index_q, 0, 0x7FFFFFFF, block_scores, status, true, stream);
}

extern "C" msa_status msa_indexer_decode(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                         const uint8_t* index_q, float* block_scores, uint32_t* status,
                                         cudaStream_t stream) {
  return msa_indexer_decode_range(geo, batch, cache, index_q, 0, 0x7FFFFFFF, block_scores, status, stream);
}
