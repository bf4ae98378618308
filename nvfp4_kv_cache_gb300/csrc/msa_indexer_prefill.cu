// msa_indexer_prefill.cu — the indexer for prompts: block scores of many query tokens per
// sequence.
//
// What it computes: the same scores as msa_indexer_decode ("MSA primer"; "MiniMax M3 in vLLM
// ...", "MiniMax 稀疏注意力后端" lists prefill indexer scoring as its own kernel and "预填充执行"
// scores the blocks of a prompt before selecting them): block_scores[t][g][k] = max over the
// cache positions j of block k with j <= p_t of index_q[t][g] . ik(j), -inf when block k holds no
// such j, ik the index key dequantised to E4M3 (NVFP4 cache) or as stored (FP8 cache).
//
// GB300 design: block-major. A prompt has thousands of index-query rows (4 a token) against the
// same pages, so each page is read and dequantised once for up to 16 tiles of 128 query rows and
// scored with tcgen05.mma kind::f8f6f4 as D = Q_tile K^T: A = the tile's 128 rows (32 tokens x 4
// groups, E4M3, one 2-D tensor copy), B = the page's 128 keys (E4M3, K-major, shared memory),
// M = 128 query rows, N = 128 keys, four MMAs of K = 32 into one of two 128-column TMEM
// accumulators. With the query rows on the TMEM lanes the max-pool is a per-thread max over 128
// columns. One persistent CTA of 16 warps per SM takes work items (sequence, page, group of 16
// tiles) in a fixed order that every warp role derives from the per-sequence prefix sums:
//  * warp 0 copies each item's page (one 2-D tensor copy, 128-byte swizzle) into a 2-deep stage
//    ring and its tiles into a 4-deep ring;
//  * warp 1 issues the MMAs and commits each accumulator, tile and key tile as it is used;
//  * warps 4..7 dequantise an NVFP4 page into a 2-deep ring of E4M3 key tiles (thread = key
//    row; an FP8 page is the key tile as copied);
//  * warps 8..11 and 12..15 are two epilogue warpgroups on alternate tiles (thread = query row):
//    keys after the row's position masked, the maximum stored.
// A tile none of whose tokens reaches the page, and every tile of an item whose page id is bad,
// skips the MMA: its epilogue stores -inf.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "msa.h"
#include "msa_attn_tile.cuh"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

constexpr int kPiThreads = 512;
constexpr int kPiWarpDq = 4;               // warps 4..7: the dequant group
constexpr int kPiWarpEp = 8;               // warps 8..15: two epilogue warpgroups
constexpr int kTileRows = 128;             // query rows (token x group) of a tile
constexpr int kTilesPerItem = 16;          // tiles scored against one copy of a page
constexpr int kPStages = 2;                // raw page stages
constexpr int kKTiles = 2;                 // dequantised key tiles (NVFP4)
constexpr int kQStages = 4;                // query tiles
constexpr int kTileBytes = kTileRows * kD; // 16 KB: a query tile, a key tile, an FP8 page
constexpr int kPiTmemCols = 256;           // two accumulators of 128 columns

struct PiParams {
  int32_t B, T, maxb, max_q_len, num_pages;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_table;
  float* block_scores;
  uint32_t* status;
};

struct PiSmem {
  static constexpr size_t kOffStage = 0;  // [2][16 KB] raw pages (an NVFP4 page uses 9 KB)
  static constexpr size_t kOffKTile = kOffStage + kPStages * kTileBytes;
  static constexpr size_t kOffQ = kOffKTile + kKTiles * kTileBytes;
  static constexpr size_t kOffBar = kOffQ + kQStages * kTileBytes;
  // stage_full, stage_empty [2]; ktile_full, ktile_empty [2]; q_full, q_empty [4]; d_full,
  // d_empty [2]; fin
  static constexpr int kBars = 4 * kPStages + 2 * kKTiles + 2 * kQStages + 4 + 1;
  static constexpr size_t kOffLut = kOffBar + 8 * kBars + 8;
  static constexpr size_t kOffMisc = kOffLut + 256 * 8;
  static constexpr size_t kOffWarpSum = kOffMisc + 64;
  static constexpr size_t kOffPrefix = kOffWarpSum + 4 * 32;
  static size_t bytes(int B) { return 1024 + kOffPrefix + 4 * static_cast<size_t>(B + 1); }
};
static_assert(PiSmem::kOffKTile % 1024 == 0 && PiSmem::kOffQ % 1024 == 0 && PiSmem::kOffBar % 8 == 0,
              "swizzled tiles on 1024-B boundaries");

// One work item: sequence b, its block k (page ph, ph_ok), tiles i0 .. i1-1 of its query rows.
struct PiItem {
  int b, k, ph, i0, i1;
  int q0, ql, L;
  bool ph_ok;
  bool active;  // the page is valid and some tile reaches it
};

// Tiles of 128 query rows and blocks of sequence b (0 for padded or inconsistent rows).
__device__ __forceinline__ int pi_seq_items(const PiParams& p, int b, bool* bad) {
  const int q0 = p.qsl[b], q1 = p.qsl[b + 1];
  const int ql = q1 - q0;
  const int L = p.seq_lens[b];
  if (ql < 0 || ql > p.max_q_len || q0 < 0 || q1 > p.T || (ql > 0 && (L < ql || L > p.maxb * kBS))) {
    *bad = true;
    return 0;
  }
  if (ql == 0) return 0;
  const int tiles = ceil_div(4 * ql, kTileRows);
  return ceil_div(L, kBS) * ceil_div(tiles, kTilesPerItem);
}

// The position of the last token a tile of sequence (q0, ql, L) holds.
__device__ __forceinline__ int pi_tile_last_pos(int q0, int ql, int L, int i) {
  const int t_last = min(ql - 1, (kTileRows * (i + 1) - 1) >> 2);  // token index within the sequence
  return L - ql + t_last;
}

__device__ __forceinline__ PiItem pi_item(const PiParams& p, const int* prefix, int x) {
  PiItem it;
  int lo = 0, hi = p.B - 1;  // the largest b with prefix[b] <= x
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= x) lo = mid; else hi = mid - 1;
  }
  it.b = lo;
  it.q0 = p.qsl[lo];
  it.ql = p.qsl[lo + 1] - it.q0;
  it.L = p.seq_lens[lo];
  const int nb = ceil_div(it.L, kBS);
  const int tiles = ceil_div(4 * it.ql, kTileRows);
  const int local = x - prefix[lo];
  const int tg = local / nb;
  it.k = local - tg * nb;
  it.i0 = tg * kTilesPerItem;
  it.i1 = min(tiles, it.i0 + kTilesPerItem);
  it.ph = p.block_table[static_cast<int64_t>(lo) * p.maxb + it.k];
  it.ph_ok = it.ph >= 0 && it.ph < p.num_pages;
  it.active = it.ph_ok && pi_tile_last_pos(it.q0, it.ql, it.L, it.i1 - 1) >= kBS * it.k;
  return it;
}

// Whether tile i of the item has its MMA (the page is valid and some token of the tile reaches it).
__device__ __forceinline__ bool pi_tile_live(const PiItem& it, int i) {
  return it.ph_ok && pi_tile_last_pos(it.q0, it.ql, it.L, i) >= kBS * it.k;
}

// Dequantise key row r of a staged NVFP4 page into the K-major E4M3 key tile kt (128-byte
// swizzle: 16-byte chunk c of row r at chunk c ^ (r % 8)).
__device__ __forceinline__ void pi_dequant_row(const uint8_t* pg, int r, const uint2* lut, uint8_t* kt) {
  RawRow raw;
  load_row(pg, r, raw);
  uint8_t* row = kt + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
  for (int qq = 0; qq < 4; ++qq) {
    uint32_t w[8];
    dequant_quarter(raw, qq, lut, w);
    *reinterpret_cast<uint4*>(row + (((2 * qq) ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(row + (((2 * qq + 1) ^ (r & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

template <int DT>
__global__ void __launch_bounds__(kPiThreads, 1)
    k_indexer_prefill(const PiParams p, const __grid_constant__ CUtensorMap page_map,
                      const __grid_constant__ CUtensorMap q_map) {
  using S = PiSmem;
  constexpr bool kNv = DT == MSA_INDEX_NVFP4;
  constexpr int kPageRows = (kNv ? kIdxPageNv : kIdxPageFp8) / 128;  // 128-byte rows of a page
  constexpr uint32_t kPageBytes = kNv ? kIdxPageNv : kIdxPageFp8;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint8_t* stages = smem + S::kOffStage;
  uint8_t* ktiles = smem + S::kOffKTile;
  uint8_t* qtiles = smem + S::kOffQ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  uint64_t* stage_full = bars;
  uint64_t* stage_empty = stage_full + kPStages;
  uint64_t* ktile_full = stage_empty + kPStages;
  uint64_t* ktile_empty = ktile_full + kKTiles;
  uint64_t* q_full = ktile_empty + kKTiles;
  uint64_t* q_empty = q_full + kQStages;
  uint64_t* d_full = q_empty + kQStages;
  uint64_t* d_empty = d_full + 2;
  uint64_t* fin = d_empty + 2;
  uint2* lut = reinterpret_cast<uint2*>(smem + S::kOffLut);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc);
  int* bad_batch = reinterpret_cast<int*>(smem + S::kOffMisc + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kOffMisc + 8);
  int* warp_sum = reinterpret_cast<int*>(smem + S::kOffWarpSum);
  int* prefix = reinterpret_cast<int*>(smem + S::kOffPrefix);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- prologue: barriers, TMEM, table, per-sequence item prefix sums ---------------------
  if (tid == 0) {
    for (int i = 0; i < kPStages; ++i) {
      mbar_init(&stage_full[i], 1);
      mbar_init(&stage_empty[i], kNv ? 4 : 1);  // NVFP4: the dequant group's warps; FP8: the item's MMAs
    }
    for (int i = 0; i < kKTiles; ++i) {
      mbar_init(&ktile_full[i], 4);
      mbar_init(&ktile_empty[i], 1);  // the item's MMAs (a commit)
    }
    for (int i = 0; i < kQStages; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);  // the epilogue warpgroup that read the tile's accumulator
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&d_full[i], 1);
      mbar_init(&d_empty[i], 4);  // the epilogue warpgroup's warps
    }
    mbar_init(fin, 1);
    fence_mbar_init();
    *abort_flag = 0;
    *bad_batch = 0;
  }
  if (warp == 1) tmem_alloc(tmem_slot, kPiTmemCols);
  if constexpr (kNv) build_dequant_lut(lut, tid, kPiThreads);
  __syncthreads();
  {
    // prefix[b] = items of sequences 0 .. b-1
    const int per = ceil_div(p.B, kPiThreads);
    const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
    int local = 0;
    bool bad = false;
    for (int b = b0; b < b1; ++b) {
      const int c = pi_seq_items(p, b, &bad);
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
      const int nw = kPiThreads / 32;
      const int v = lane < nw ? warp_sum[lane] : 0;
      int x = v;
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
  if (*bad_batch != 0) {  // an inconsistent batch: nothing is scored
    if (tid == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
    if (warp == 1) tmem_dealloc(*tmem_slot, kPiTmemCols);
    return;
  }
  const uint32_t tmem = *tmem_slot;
  const int items = p.B > 0 ? prefix[p.B] : 0;
  bool ok = true;
  auto give_up = [&]() {
    if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
    *abort_flag = 1;
  };
  auto wait1 = [&](uint64_t* bar, uint32_t parity) {
    if (!ok) return false;
    ok = mbar_wait(bar, parity, abort_flag);
    if (!ok) give_up();
    return ok;
  };
  auto waitw = [&](uint64_t* bar, uint32_t parity) {
    if (!ok) return false;
    ok = warp_wait(bar, parity, abort_flag);
    if (!ok && lane == 0) give_up();
    return ok;
  };

  if (warp == 0) {
    // ---- copies: each active item's page, then its live tiles ----------------------------
    if (lane == 0) {
      prefetch_tensormap(&page_map);
      prefetch_tensormap(&q_map);
      const uint64_t pol = policy_evict_first();
      int pc = 0, qc = 0;  // pages and tiles copied
      for (int x = blockIdx.x; x < items && ok; x += gridDim.x) {
        const PiItem it = pi_item(p, prefix, x);
        if (!it.active) continue;
        const int s = pc % kPStages;
        if (!wait1(&stage_empty[s], (static_cast<uint32_t>(pc / kPStages) & 1u) ^ 1u)) break;
        mbar_arrive_expect_tx(&stage_full[s], kPageBytes);
        tma_load_2d(stages + static_cast<size_t>(s) * kTileBytes, &page_map, 0, it.ph * kPageRows, &stage_full[s], pol);
        ++pc;
        for (int i = it.i0; i < it.i1 && ok; ++i) {
          if (!pi_tile_live(it, i)) continue;
          const int qs = qc % kQStages;
          if (!wait1(&q_empty[qs], (static_cast<uint32_t>(qc / kQStages) & 1u) ^ 1u)) break;
          mbar_arrive_expect_tx(&q_full[qs], kTileBytes);
          tma_load_2d(qtiles + static_cast<size_t>(qs) * kTileBytes, &q_map, 0, 4 * it.q0 + kTileRows * i, &q_full[qs],
                      pol);
          ++qc;
        }
      }
      // nothing of this thread's is in flight when the CTA ends
      for (int j = pc > kPStages ? pc - kPStages : 0; j < pc; ++j)
        if (!mbar_wait_bounded(&stage_full[j % kPStages], static_cast<uint32_t>(j / kPStages) & 1u, kWaitLimitNs,
                               nullptr))
          set_status(p.status, MSA_ERR_TIMEOUT);
      for (int j = qc > kQStages ? qc - kQStages : 0; j < qc; ++j)
        if (!mbar_wait_bounded(&q_full[j % kQStages], static_cast<uint32_t>(j / kQStages) & 1u, kWaitLimitNs, nullptr))
          set_status(p.status, MSA_ERR_TIMEOUT);
    }
  } else if (warp == 1) {
    // ---- MMAs: D[tile parity] = Q_tile K^T for every live tile -----------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(kTileRows, kBS);
      int mc = 0, qc = 0, gt = 0;  // active items, live tiles, all tiles seen
      int dn[2] = {0, 0};          // MMAs into each accumulator
      bool issued = false;
      for (int x = blockIdx.x; x < items && ok; x += gridDim.x) {
        const PiItem it = pi_item(p, prefix, x);
        if (!it.ph_ok && it.i0 < it.i1) set_status(p.status, MSA_ERR_DEVICE_FAULT);
        if (!it.active) {
          gt += it.i1 - it.i0;
          continue;
        }
        const int s = mc % kPStages;
        const uint8_t* kt;
        if constexpr (kNv) {
          if (!wait1(&ktile_full[s], static_cast<uint32_t>(mc / kKTiles) & 1u)) break;
          kt = ktiles + static_cast<size_t>(s) * kTileBytes;
        } else {
          if (!wait1(&stage_full[s], static_cast<uint32_t>(mc / kPStages) & 1u)) break;
          kt = stages + static_cast<size_t>(s) * kTileBytes;
        }
        const uint64_t kdesc = sw128_kmajor_desc(smem_u32(kt));
        for (int i = it.i0; i < it.i1 && ok; ++i, ++gt) {
          if (!pi_tile_live(it, i)) continue;
          const int e = gt & 1;
          const int qs = qc % kQStages;
          if (!wait1(&d_empty[e], (static_cast<uint32_t>(dn[e]) & 1u) ^ 1u)) break;
          if (!wait1(&q_full[qs], static_cast<uint32_t>(qc / kQStages) & 1u)) break;
          tc_fence_after();
          const uint64_t qdesc = sw128_kmajor_desc(smem_u32(qtiles + static_cast<size_t>(qs) * kTileBytes));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 32 E4M3 a step: +32 B in both operands
            tc_mma_f8(tmem + 128u * e, qdesc + 2 * kk, kdesc + 2 * kk, idesc, kk > 0 ? 1u : 0u);
          tc_commit(&d_full[e]);  // the epilogue frees the query tile once it has seen this
          issued = true;
          ++dn[e];
          ++qc;
        }
        // the key tile (the FP8 stage) is free once this item's MMAs have landed
        if constexpr (kNv)
          tc_commit(&ktile_empty[s]);
        else
          tc_commit(&stage_empty[s]);
        ++mc;
      }
      if (issued) {
        tc_commit(fin);
        if (!mbar_wait_bounded(fin, 0u, kWaitLimitNs, nullptr)) set_status(p.status, MSA_ERR_TIMEOUT);
      }
    }
  } else if (warp >= kPiWarpDq && warp < kPiWarpEp) {
    // ---- NVFP4 pages -> E4M3 key tiles (thread = key row) ----------------------------------
    if constexpr (kNv) {
      const int r = tid - 32 * kPiWarpDq;
      int dc = 0;
      for (int x = blockIdx.x; x < items && ok; x += gridDim.x) {
        const PiItem it = pi_item(p, prefix, x);
        if (!it.active) continue;
        const int s = dc % kPStages;
        if (!waitw(&stage_full[s], static_cast<uint32_t>(dc / kPStages) & 1u)) break;
        if (!waitw(&ktile_empty[s], (static_cast<uint32_t>(dc / kKTiles) & 1u) ^ 1u)) break;
        pi_dequant_row(stages + static_cast<size_t>(s) * kTileBytes, r, lut, ktiles + static_cast<size_t>(s) * kTileBytes);
        fence_proxy_async_smem();  // the key tile is read by the tensor core
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&stage_empty[s]);
          mbar_arrive(&ktile_full[s]);
        }
        ++dc;
      }
    }
  } else if (warp >= kPiWarpEp) {
    // ---- epilogue warpgroup e: tiles with gt % 2 == e; thread = query row of the tile -------
    const int e = (warp - kPiWarpEp) >> 2;
    const int wq = warp & 3;  // TMEM lane quarter
    const int r = 32 * wq + lane;
    const uint32_t taddr = tmem + 128u * e + (static_cast<uint32_t>(32 * wq) << 16);
    int gt = 0, dn = 0, qc = 0;  // all tiles, this warpgroup's live tiles, all live tiles
    for (int x = blockIdx.x; x < items; x += gridDim.x) {
      const PiItem it = pi_item(p, prefix, x);
      for (int i = it.i0; i < it.i1; ++i, ++gt) {
        const bool live = it.active && pi_tile_live(it, i);
        const int qs = qc % kQStages;
        qc += live ? 1 : 0;
        if ((gt & 1) != e) continue;
        const int rr = kTileRows * i + r;  // the row within the sequence's rows
        const bool mine = rr < 4 * it.ql;
        float m = -CUDART_INF_F;
        if (live) {
          const bool got = waitw(&d_full[e], static_cast<uint32_t>(dn) & 1u);
          // the tile's MMAs have landed: its query tile may be refilled
          if (wq == 0 && lane == 0) mbar_arrive(&q_empty[qs]);
          if (got) {
            tc_fence_after();
            // keys 0 .. nvis-1 of the block are at or before the row's position
            const int pos = it.L - it.ql + (rr >> 2);
            const int nvis = mine ? min(kBS, max(0, pos - kBS * it.k + 1)) : 0;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t v[32];
              tmem_ld32(taddr + 32 * c, v);
              tmem_wait_ld();
              float mc = -CUDART_INF_F;
              if (nvis >= 32 * c + 32) {
#pragma unroll
                for (int u = 0; u < 30; u += 3)
                  mc = fmaxf(mc, max3f(__uint_as_float(v[u]), __uint_as_float(v[u + 1]), __uint_as_float(v[u + 2])));
                mc = max3f(mc, __uint_as_float(v[30]), __uint_as_float(v[31]));
              } else {
#pragma unroll
                for (int u = 0; u < 32; ++u) mc = fmaxf(mc, 32 * c + u < nvis ? __uint_as_float(v[u]) : -CUDART_INF_F);
              }
              m = fmaxf(m, mc);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&d_empty[e]);
          ++dn;
        }
        if (mine) p.block_scores[(static_cast<int64_t>(4 * it.q0) + rr) * p.maxb + it.k] = m;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kPiTmemCols);
  }
}

template <int DT>
msa_status launch_indexer_prefill(const PiParams& p, const uint8_t* pages, const uint8_t* index_q,
                                  cudaStream_t stream) {
  constexpr uint32_t kPageRows = (DT == MSA_INDEX_NVFP4 ? kIdxPageNv : kIdxPageFp8) / 128;
  CUtensorMap page_map, q_map;
  if (!msa_host::rows128_tensor_map(&page_map, pages,
                                    static_cast<uint64_t>(p.num_pages > 0 ? p.num_pages : 1) * kPageRows, kPageRows))
    return MSA_ERR_CUDA;
  if (!msa_host::rows128_tensor_map(&q_map, index_q, static_cast<uint64_t>(p.T) * 4, kTileRows)) return MSA_ERR_CUDA;
  const int sms = msa_host::num_sms();
  if (sms <= 0) return MSA_ERR_CUDA;
  const size_t smem = PiSmem::bytes(p.B);
  if (cudaFuncSetAttribute(k_indexer_prefill<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess)
    return MSA_ERR_CUDA;
  k_indexer_prefill<DT><<<sms, kPiThreads, smem, stream>>>(p, page_map, q_map);
  return msa_host::launch_status();
}

}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

extern "C" msa_status msa_indexer_prefill(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                          const uint8_t* index_q, float* block_scores, uint32_t* status,
                                          cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = check_prefill_batch(batch)) != MSA_OK) return st;
  if ((st = check_cache(cache, true, false)) != MSA_OK) return st;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (cache->num_pages > (1 << 24)) return MSA_ERR_UNSUPPORTED;
  if (index_q == nullptr || block_scores == nullptr || !aligned(index_q, 16) || !aligned(block_scores, 4))
    return MSA_ERR_INVALID_ARG;
  PiParams p;
  p.B = batch->B;
  p.T = batch->T;
  p.maxb = batch->max_blocks_per_seq;
  p.max_q_len = batch->max_q_len;
  p.num_pages = cache->num_pages;
  p.qsl = batch->query_start_loc;
  p.seq_lens = batch->seq_lens;
  p.block_table = batch->block_table;
  p.block_scores = block_scores;
  p.status = status;
  return cache->index_dtype == MSA_INDEX_NVFP4
             ? launch_indexer_prefill<MSA_INDEX_NVFP4>(p, cache->index_pages, index_q, stream)
             : launch_indexer_prefill<MSA_INDEX_FP8>(p, cache->index_pages, index_q, stream);
}
