// msa_prefill.cu — the many-query (prefill) sparse attention: block-major, with a key-block ->
// query map and a log-sum-exp merge, on the fifth-generation tensor cores.
//
// What it computes: the same exact sparse GQA attention as msa_sparse_attn_decode ("vLLM ofrece
// soporte en día 0 para MiniMax-M3.1-Flash", "MSA primer": every query head of a group attends
// over its token's selected blocks; "MSA 机制详解": keys after the query position are masked),
// for any number of query tokens per sequence. The pages' prefill kernel is block-major ("MiniMax
// M3 in vLLM ...", "预填充": a block's keys are read and dequantised once for all the queries that
// selected it, through a key-block -> query map, and each query's per-block results are merged
// by log-sum-exp), and their NVFP4 attention kernel dequantises a page that several requests
// share through a common prefix once for up to 64 of them ("vLLM ofrece soporte en día 0 ...",
// "NVFP4 MSA kernel"). Both hold here because the map is keyed by the physical page:
//  1. k_map_count / k_map_alloc / k_map_fill: every valid (token, group, slot) selection (a
//     token's repeated block counts once; an out-of-range block or a bad page marks the (token,
//     group) bad) is filed under the key (physical page, group) through an open-addressing hash
//     table, so the selections of every sequence whose block table points at the same page land
//     in one row. Each row's selections are cut into chunks of at most 64;
//  2. k_prefill_tc: one persistent CTA per SM takes chunks in turn. A chunk's K and V regions are
//     copied (one 3-D tensor copy) and dequantised once, K to an E4M3 K-major tile and V to an
//     f16 tile read as the MN-major operand (E4M3 -> f16 is exact); then each tile of 8
//     selections (8 x 16 query heads = M 128) runs S = Q K^T (tcgen05.mma kind::f8f6f4, both
//     operands in shared memory, N = 128 keys), a softmax over the block's 128 keys (one thread
//     per query-head row) that writes P in f16, and O^T = V^T P^T (kind::f16, M = 128 dims,
//     N = 128 query-head rows). The (m, l) of every row and its unnormalised o go to the
//     selection's slot;
//  3. k_prefill_merge: per (token, group), the log-sum-exp merge of its up to 16 partials.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include <algorithm>

#include "msa.h"
#include "msa_attn_tile.cuh"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

constexpr int kChunk = 64;             // selections served by one dequantised (page, group) block
constexpr int kTileSel = 8;            // selections per MMA tile: 8 x 16 query heads = M 128
constexpr int kMaxT = 1 << 22;         // query tokens per call (entries pack t << 4 | slot)
constexpr uint64_t kNoKey = ~0ull;     // an empty hash slot

// Warp roles of k_prefill_tc. A warp reads the TMEM lanes 32 (warp % 4) .. + 31, so the softmax
// and epilogue groups are aligned sets of four warps.
constexpr int kWarpProd = 0;   // chunk fetch, entry lists, query-tile copies
constexpr int kWarpIss = 1;    // S = Q K^T issue (lane 0) for every tile; allocates TMEM
constexpr int kWarpPv = 2;     // two O^T = V^T P^T issuers (warps 2, 3): even and odd tiles
constexpr int kWarpSm = 4;     // two softmax warpgroups (warps 4-7, 8-11): even and odd tiles
constexpr int kWarpEp = 12;    // two epilogue warpgroups (warps 12-15, 16-19): even and odd tiles
constexpr int kWarpDq = 20;    // two dequant warps
constexpr int kDqWarps = 2;
constexpr int kThreads = 32 * (kWarpDq + kDqWarps);
constexpr int kMetaSlots = 4;
// Arrivals that release a chunk's entry list: every dequant, softmax and epilogue warp and the
// three issuers, each after its last use of it.
constexpr int kMetaUsers = kDqWarps + 8 + 8 + 3;

constexpr int kQBufs = 3;                // query tiles in flight (their copies take ~5,000 cycles)
constexpr int kKTile = kBS * kD;         // 128 keys x 128 E4M3, K-major, 128-byte swizzle
constexpr int kVTile = kBS * kD * 2;     // 128 keys x 128 f16, MN-major: two 64-dim atom columns
constexpr uint32_t kVLbo = 16384;        //   V tile: the two 64-dim atom columns
constexpr uint32_t kVSbo = 1024;         //           8-key groups
constexpr int kQTile = kTileSel * kHPG * kD;  // 128 query-head rows x 128 E4M3
constexpr int kPTile = 128 * kBS * 2;    // 128 query-head rows x 128 keys f16: two 64-key K atoms
constexpr int kPAtom = 128 * 128;        //   16 KB each
constexpr uint32_t kTmemCols = 512;      // S (2 x 128) and O^T (2 x 128), both double-buffered
constexpr uint32_t kColO = 256;
constexpr float kLazyMax = 128.0f;      // the largest row sum l a first-chunk reference may keep

struct PfParams {
  int32_t B, T, maxb, num_pages;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_table;
  const uint8_t* kv;
  const uint8_t* q;
  const int32_t* sel;
  float scale_log2;
  uint16_t* out;
  // workspace
  int32_t* hdr;        // [0] rows, [1] chunks, [2] entries, [3] chunk fetch counter
  uint64_t* hkeys;     // [H] page * 4 + group, kNoKey when free
  int32_t* hcnt;       // [H] selections of the slot's row; then its fill cursor
  int32_t* rowh;       // [T * 64] hash slot of row r (rows numbered in order of appearance)
  int32_t* ehash;      // [T * 64] hash slot of each selection, -1: none
  int2* entries;       // [T * 64] {t << 4 | slot, p_tok - 128 block}, grouped by row
  int4* chunks;        // [T * 65] {first entry, count, page, group}
  int32_t* tg_bad;     // [T * 4] the (token, group) saw a bad selection or page: zero output
  uint32_t* part_o;    // [T * 64 slots][128 dims][16 heads] unnormalised partial o, f16 pairs
  float2* part_ml;     // [T * 64 slots][16 heads] {m (log2 domain), l}; m = -inf: no partial
  uint32_t hmask;      // H - 1 (H a power of two)
  int32_t hbits;       // log2 H
  uint32_t* status;
};

// The sequence of token t (largest b with qsl[b] <= t) and whether the batch rows around it are
// consistent; p_tok = the token's position.
__device__ __forceinline__ bool token_seq(const PfParams& p, int t, int* b_out, int* p_tok, int* nb) {
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int q0 = p.qsl[lo], ql = p.qsl[lo + 1] - q0, L = p.seq_lens[lo];
  *b_out = lo;
  *p_tok = L - ql + (t - q0);
  *nb = ceil_div(L, kBS);
  return t - q0 >= 0 && t - q0 < ql && L >= ql && L <= p.maxb * kBS;
}

// The map's state for a new call: an empty hash table, zero counts and flags.
__global__ void __launch_bounds__(256) k_map_init(const PfParams p) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t x = i; x <= static_cast<int64_t>(p.hmask); x += stride) {
    p.hkeys[x] = kNoKey;
    p.hcnt[x] = 0;
  }
  for (int64_t x = i; x < static_cast<int64_t>(p.T) * 4; x += stride) p.tg_bad[x] = 0;
  if (i < 4) p.hdr[i] = 0;
}

// The kernels after k_map_init are launched as programmatic dependents of the kernel before them:
// each waits (griddepcontrol.wait) before it touches anything that kernel writes or reads.

// One thread per (token, group, slot): validate the selection, and file the first occurrence of
// each valid block under its (page, group) row (ehash = -1 marks a slot that gets no partial;
// k_map_fill gives those m = -inf, and the kernel writes every other slot's (m, l)).
__global__ void __launch_bounds__(256) k_map_count(const PfParams p) {
  grid_dependency_wait();
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(p.T) * 4 * kSel) return;
  const int t = static_cast<int>(e / (4 * kSel)), g = static_cast<int>((e / kSel) % 4), slot = static_cast<int>(e % kSel);
  p.ehash[e] = -1;
  int b, p_tok, nb;
  if (!token_seq(p, t, &b, &p_tok, &nb)) {
    set_status(p.status, MSA_ERR_INVALID_ARG);
    p.tg_bad[t * 4 + g] = 1;
    return;
  }
  const int32_t* row = p.sel + (static_cast<int64_t>(t) * 4 + g) * kSel;
  const int v = row[slot];
  if (v < 0) return;
  if (v >= nb) {
    set_status(p.status, MSA_ERR_DEVICE_FAULT);
    p.tg_bad[t * 4 + g] = 1;
    return;
  }
  for (int j = 0; j < slot; ++j)
    if (row[j] == v) return;  // a repeat of an earlier slot
  const int ph = p.block_table[static_cast<int64_t>(b) * p.maxb + v];
  if (!(ph >= 0 && ph < p.num_pages)) {
    set_status(p.status, MSA_ERR_DEVICE_FAULT);
    p.tg_bad[t * 4 + g] = 1;
    return;
  }
  // linear probing from a multiplicative hash; the table has at least twice as many slots as
  // there are selections, so a free or matching slot is always found
  const uint64_t key = static_cast<uint64_t>(ph) * 4 + static_cast<uint64_t>(g);
  uint32_t h = static_cast<uint32_t>((key * 0x9E3779B97F4A7C15ull) >> (64 - p.hbits)) & p.hmask;
  for (uint32_t probe = 0; probe <= p.hmask; ++probe) {
    // a key, once stored, never changes: a plain read that finds it saves the atomic
    if (*reinterpret_cast<volatile const uint64_t*>(p.hkeys + h) == key) break;
    const uint64_t old = atomicCAS(reinterpret_cast<unsigned long long*>(p.hkeys + h), kNoKey, key);
    if (old == kNoKey) {
      p.rowh[atomicAdd(&p.hdr[0], 1)] = static_cast<int32_t>(h);
      break;
    }
    if (old == key) break;
    h = (h + 1) & p.hmask;
  }
  atomicAdd(&p.hcnt[h], 1);
  p.ehash[e] = static_cast<int32_t>(h);
}

// One thread per row: the row's place in the entry list and its chunks, allocated with one
// atomic per warp (rows and chunks land in arbitrary order; only their grouping matters).
__global__ void __launch_bounds__(256) k_map_alloc(const PfParams p) {
  grid_dependency_wait();
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  const int nrows = p.hdr[0];
  if (r - lane >= nrows) return;  // the whole warp is past the last row
  const bool mine = r < nrows;
  const int h = mine ? p.rowh[r] : 0;
  const int c = mine ? p.hcnt[h] : 0;
  const int nch = (c + kChunk - 1) / kChunk;
  int ic = c, in = nch;  // inclusive warp scans
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ic, o), b = __shfl_up_sync(0xffffffffu, in, o);
    if (lane >= o) {
      ic += a;
      in += b;
    }
  }
  int base_e = 0, base_c = 0;
  if (lane == 31) {
    base_e = atomicAdd(&p.hdr[2], ic);
    base_c = atomicAdd(&p.hdr[1], in);
  }
  base_e = __shfl_sync(0xffffffffu, base_e, 31);
  base_c = __shfl_sync(0xffffffffu, base_c, 31);
  if (!mine) return;
  const int off = base_e + ic - c, ch0 = base_c + in - nch;
  p.hcnt[h] = off;  // the fill cursor
  const uint64_t key = p.hkeys[h];
  const int ph = static_cast<int>(key >> 2), g = static_cast<int>(key & 3);
  for (int j = 0; j < nch; ++j) p.chunks[ch0 + j] = make_int4(off + kChunk * j, min(kChunk, c - kChunk * j), ph, g);
}

// The same threads as k_map_count place their selection in its row: the token and slot, and
// the query position relative to the block's first key (the mask of the block's keys).
__global__ void __launch_bounds__(256) k_map_fill(const PfParams p) {
  grid_dependency_wait();
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(p.T) * 4 * kSel) return;
  const int h = p.ehash[e];
  if (h < 0) {  // a slot with no partial: m = -inf for the merge
    float2* ml = p.part_ml + e * kHPG;
#pragma unroll
    for (int x = 0; x < kHPG; ++x) ml[x] = make_float2(-CUDART_INF_F, 0.f);
    return;
  }
  const int t = static_cast<int>(e / (4 * kSel)), g = static_cast<int>((e / kSel) % 4), slot = static_cast<int>(e % kSel);
  int b, p_tok, nb;
  token_seq(p, t, &b, &p_tok, &nb);
  const int v = p.sel[(static_cast<int64_t>(t) * 4 + g) * kSel + slot];
  const int pos = atomicAdd(&p.hcnt[h], 1);
  p.entries[pos] = make_int2((t << 4) | slot, p_tok - v * kBS);
}

struct ChunkMeta {
  int32_t n, ph, g, pad;
  int2 e[kChunk];
};

struct Smem {
  static constexpr size_t kOffK = 0;                                            // [2] K tiles
  static constexpr size_t kOffV = kOffK + 2 * static_cast<size_t>(kKTile);      // [2] V tiles
  static constexpr size_t kOffQ = kOffV + 2 * static_cast<size_t>(kVTile);      // [kQBufs] Q tiles
  static constexpr size_t kOffP = kOffQ + kQBufs * static_cast<size_t>(kQTile); // [2] P tiles
  static constexpr size_t kOffLut = kOffP + 2 * static_cast<size_t>(kPTile);
  static constexpr size_t kOffMeta = kOffLut + 256 * 8;
  static constexpr size_t kOffBar = kOffMeta + kMetaSlots * sizeof(ChunkMeta);
  // barriers: meta full/empty, q full/empty, then two each of tile full/empty, s full/free,
  // p full/empty, o full/free, and one fin per issuer
  static constexpr int kNumBars = 2 * kMetaSlots + 2 * kQBufs + 2 * 2 * 4 + 3;
  static constexpr size_t kOffMisc = kOffBar + 8 * kNumBars;
  static constexpr size_t kBytes = 1024 + kOffMisc + 16;
};
static_assert(Smem::kOffK % 1024 == 0 && Smem::kOffV % 1024 == 0 && Smem::kOffQ % 1024 == 0 &&
                  Smem::kOffP % 1024 == 0 && kRegion % 1024 == 0,
              "swizzled tiles and copies start on 1024-B boundaries");
static_assert(Smem::kOffBar % 8 == 0 && Smem::kBytes <= 232448, "shared memory budget");

struct Bars {
  uint64_t* meta_full;
  uint64_t* meta_empty;
  uint64_t* kt_full;
  uint64_t* kt_empty;
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* s_full;
  uint64_t* s_free;
  uint64_t* p_full;
  uint64_t* p_empty;
  uint64_t* o_full;
  uint64_t* o_free;
  uint64_t* fin;
  __device__ explicit Bars(uint8_t* smem) {
    uint64_t* b = reinterpret_cast<uint64_t*>(smem + Smem::kOffBar);
    meta_full = b;
    meta_empty = b + kMetaSlots;
    b += 2 * kMetaSlots;
    q_full = b;
    q_empty = b + kQBufs;
    b += 2 * kQBufs;
    kt_full = b;
    kt_empty = b + 2;
    s_full = b + 4;
    s_free = b + 6;
    p_full = b + 8;
    p_empty = b + 10;
    o_full = b + 12;
    o_free = b + 14;
    fin = b + 16;
    static_assert(2 * kMetaSlots + 2 * kQBufs + 19 == Smem::kNumBars, "barrier area");
  }
};

__device__ __forceinline__ int ntiles_of(int n) { return (n + kTileSel - 1) / kTileSel; }

// Key row r of an NVFP4 K or V region in the cache (no swizzle: rows of 64 code bytes, then
// the 8 scale bytes of each row), read-only loads.
__device__ __forceinline__ void load_row_global(const uint8_t* region, int r, RawRow& raw) {
  const uint4* c = reinterpret_cast<const uint4*>(region + r * kRowCodes);
#pragma unroll
  for (int q = 0; q < 4; ++q) raw.c[q] = __ldg(c + q);
  raw.sc = __ldg(reinterpret_cast<const uint2*>(region + kScaleOff + r * kRowScales));
}

// Persistent: one CTA per SM takes chunks in turn (a global counter). Warp roles:
//  producer — the chunk's entry list into the meta ring, one tensor copy of its K and V regions,
//             and per tile one 2 KB tensor copy per selection of its token's 16 query heads;
//  dequant  — the K rows to an E4M3 K-major tile, the V rows to an f16 tile read as the MN-major
//             A operand of O^T (two 64-dim atom columns, 8-key groups, 128-byte swizzle);
//  issuer   — S(i) = Q K^T (M 128 heads x N 128 keys, E4M3) one tile ahead of O^T(i - 1) =
//             V^T P^T (M 128 dims x N 128 head rows x K 128 keys, f16);
//  softmax  — thread = query-head row: the row's max and sum over the block's unmasked keys, P in
//             f16, and the row's (m, l) to its slot (two warpgroups, alternate tiles);
//  epilogue — thread = dim: o of every head to its slot, f16 (two warpgroups, alternate tiles).
// Every wait is bounded (MSA_ERR_TIMEOUT, then every role leaves); nothing traps.
__global__ void __launch_bounds__(kThreads, 1)
    k_prefill_tc(const PfParams p, const __grid_constant__ CUtensorMap q_map) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const Bars bars(smem);
  ChunkMeta* meta = reinterpret_cast<ChunkMeta*>(smem + Smem::kOffMeta);
  uint2* lut = reinterpret_cast<uint2*>(smem + Smem::kOffLut);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Smem::kOffMisc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Smem::kOffMisc + 4);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int i = 0; i < kMetaSlots; ++i) {
      mbar_init(&bars.meta_full[i], 1);
      mbar_init(&bars.meta_empty[i], kMetaUsers);
    }
    for (int i = 0; i < kQBufs; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.kt_full[i], kDqWarps);
      mbar_init(&bars.kt_empty[i], 2);  // both O^T issuers, after their last MMA of the chunk
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.s_free[i], 4);  // the four warps of the tile's softmax warpgroup
      mbar_init(&bars.p_full[i], 4);
      mbar_init(&bars.p_empty[i], 1);
      mbar_init(&bars.o_full[i], 1);
      mbar_init(&bars.o_free[i], 4);  // the four warps of the tile's epilogue warpgroup
    }
    for (int i = 0; i < 3; ++i) mbar_init(&bars.fin[i], 1);
    fence_mbar_init();
    *abort_flag = 0;
  }
  {
    // Q tiles start as zeros: rows of a short tile's missing selections then hold finite values
    uint4* qz = reinterpret_cast<uint4*>(smem + Smem::kOffQ);
    for (int i = tid; i < kQBufs * kQTile / 16; i += kThreads) qz[i] = make_uint4(0u, 0u, 0u, 0u);
  }
  if (warp == kWarpIss) tmem_alloc(tmem_slot, kTmemCols);
  build_dequant_lut(lut, tid, kThreads);
  fence_proxy_async_smem();
  grid_dependency_wait();  // the map (the prologue above ran while it finished)
  const int nchunks = p.hdr[1];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // A warp's bounded wait; on a time-out the first to notice reports it and every role leaves.
  auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
    if (warp_wait(bar, parity, abort_flag)) return true;
    if (lane == 0) {
      if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
      *abort_flag = 1;
    }
    return false;
  };

  if (warp == kWarpProd) {
    // ---- producer ---------------------------------------------------------------------------
    if (lane == 0) prefetch_tensormap(&q_map);
    const uint64_t pol = policy_evict_last();  // a token's query heads serve up to 16 chunks
    int i = 0;  // query tiles issued
    // Takes the next chunk and publishes its entry list in meta slot kk % kMetaSlots: its count,
    // or -1 when no chunk is left (the slot then carries the end mark), -2 on a give-up.
    auto fetch_meta = [&](int kk) -> int {
      int c = 0;
      if (lane == 0) c = atomicAdd(&p.hdr[3], 1);
      c = __shfl_sync(0xffffffffu, c, 0);
      const int ms = kk % kMetaSlots;
      if (!wwait(&bars.meta_empty[ms], (static_cast<uint32_t>(kk / kMetaSlots) & 1u) ^ 1u)) return -2;
      ChunkMeta& m = meta[ms];
      if (c >= nchunks) {
        if (lane == 0) {
          m.n = -1;
          mbar_arrive(&bars.meta_full[ms]);
        }
        return -1;
      }
      const int4 ch = p.chunks[c];
      for (int e = lane; e < ch.y; e += 32) m.e[e] = p.entries[ch.x + e];
      if (lane == 0) {
        m.n = ch.y;
        m.ph = ch.z;
        m.g = ch.w;
      }
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        mbar_arrive(&bars.meta_full[ms]);
      }
      return ch.y;
    };
    // The entry list of chunk k + 1 is published before chunk k's query tiles are issued, so that
    // the dequant warps turn its K and V rows into tiles while chunk k's tiles run.
    int n_next = fetch_meta(0);
    for (int k = 0; n_next >= 0; ++k) {
      const int n = n_next;
      const ChunkMeta& m = meta[k % kMetaSlots];  // not refilled before chunk k + kMetaSlots
      n_next = fetch_meta(k + 1);
      if (n_next == -2) break;
      // the chunk's query tiles: 8 lanes copy one selection's 16 query rows each
      bool ok = true;
      for (int j = 0; j < ntiles_of(n); ++j, ++i) {
        const int qb = i % kQBufs;
        if (!(ok = wwait(&bars.q_empty[qb], (static_cast<uint32_t>(i / kQBufs) & 1u) ^ 1u))) break;
        const int ne = min(kTileSel, n - kTileSel * j);
        if (lane == 0) mbar_arrive_expect_tx(&bars.q_full[qb], static_cast<uint32_t>(ne) * kHPG * kD);
        __syncwarp();
        if (lane < ne) {
          const int t = m.e[kTileSel * j + lane].x >> 4;
          tma_load_2d(smem + Smem::kOffQ + static_cast<size_t>(qb) * kQTile + lane * kHPG * kD, &q_map, 0,
                      t * kQHeads + m.g * kHPG, &bars.q_full[qb], pol);
        }
      }
      if (!ok) break;
    }
    // never leave while a copy into this CTA's shared memory may still be in flight
    if (lane == 0) {
      for (int j = i > kQBufs ? i - kQBufs : 0; j < i; ++j)
        if (!mbar_wait_bounded(&bars.q_full[j % kQBufs], static_cast<uint32_t>(j / kQBufs) & 1u, kWaitLimitNs, nullptr))
          set_status(p.status, MSA_ERR_TIMEOUT);
    }
  } else if (warp == kWarpIss) {
    // ---- S = Q K^T for every tile, in order ---------------------------------------------------
    constexpr uint32_t idesc_s = idesc_e4m3_f32(128, 128);
    bool issued = false;
    int i = 0;
    for (int k = 0;; ++k) {
      const int ms = k % kMetaSlots;
      if (!wwait(&bars.meta_full[ms], static_cast<uint32_t>(k / kMetaSlots) & 1u)) break;
      const int n = meta[ms].n;
      if (n < 0) break;
      if (!wwait(&bars.kt_full[k & 1], static_cast<uint32_t>(k >> 1) & 1u)) break;
      bool ok = true;
      for (int j = 0; j < ntiles_of(n); ++j, ++i) {
        if (!(ok = wwait(&bars.q_full[i % kQBufs], static_cast<uint32_t>(i / kQBufs) & 1u))) break;
        if (!(ok = wwait(&bars.s_free[i & 1], (static_cast<uint32_t>(i >> 1) & 1u) ^ 1u))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t dq = sw128_kmajor_desc(smem_u32(smem + Smem::kOffQ + static_cast<size_t>(i % kQBufs) * kQTile));
          const uint64_t dk = sw128_kmajor_desc(smem_u32(smem + Smem::kOffK + static_cast<size_t>(k & 1) * kKTile));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 32 dims per MMA: +32 B in both operands' atoms
            tc_mma_f8(tmem + 128u * static_cast<uint32_t>(i & 1), dq + 2 * kk, dk + 2 * kk, idesc_s, kk > 0 ? 1u : 0u);
          tc_commit(&bars.s_full[i & 1]);
          tc_commit(&bars.q_empty[i % kQBufs]);
        }
        __syncwarp();
        issued = true;
      }
      if (!ok) break;
      if (lane == 0) mbar_arrive(&bars.meta_empty[ms]);
    }
    // nothing of this thread's is in flight when the CTA ends
    if (lane == 0 && issued) {
      tc_commit(&bars.fin[0]);
      if (!mbar_wait_bounded(&bars.fin[0], 0u, kWaitLimitNs, nullptr)) set_status(p.status, MSA_ERR_TIMEOUT);
    }
  } else if (warp < kWarpSm) {
    // ---- O^T = V^T P^T for the tiles of parity x ------------------------------------------------
    constexpr uint32_t idesc_o = idesc_f16_f32_amn(128, 128);
    const int x = warp - kWarpPv;
    bool issued = false;
    int i = 0;
    for (int k = 0;; ++k) {
      const int ms = k % kMetaSlots;
      if (!wwait(&bars.meta_full[ms], static_cast<uint32_t>(k / kMetaSlots) & 1u)) break;
      const int n = meta[ms].n;
      if (n < 0) break;
      bool ok = true;
      for (int j = 0; j < ntiles_of(n); ++j, ++i) {
        if ((i & 1) != x) continue;
        if (!(ok = wwait(&bars.p_full[x], static_cast<uint32_t>(i >> 1) & 1u))) break;
        if (!(ok = wwait(&bars.o_free[x], (static_cast<uint32_t>(i >> 1) & 1u) ^ 1u))) break;
        tc_fence_after();
        if (lane == 0) {
          const uint64_t dv =
              sw128_mnmajor_desc(smem_u32(smem + Smem::kOffV + static_cast<size_t>(k & 1) * kVTile), kVLbo, kVSbo);
          const uint64_t dp = sw128_kmajor_desc(smem_u32(smem + Smem::kOffP + static_cast<size_t>(x) * kPTile));
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)  // K = 16 keys per MMA: two 8-key groups of V; 32 B (or the next atom) of P
            tc_mma_f16(tmem + kColO + 128u * static_cast<uint32_t>(x), dv + ((2 * kVSbo) >> 4) * kk,
                       dp + (((kk >> 2) * kPAtom + (kk & 3) * 32) >> 4), idesc_o, kk > 0 ? 1u : 0u);
          tc_commit(&bars.o_full[x]);
          tc_commit(&bars.p_empty[x]);
        }
        __syncwarp();
        issued = true;
      }
      if (!ok) break;
      // this issuer's MMAs on the chunk's K and V tiles (if any) are done: the tiles may be refilled
      if (lane == 0) {
        tc_commit(&bars.kt_empty[k & 1]);
        mbar_arrive(&bars.meta_empty[ms]);
      }
    }
    if (lane == 0 && issued) {
      tc_commit(&bars.fin[1 + x]);
      if (!mbar_wait_bounded(&bars.fin[1 + x], 0u, kWaitLimitNs, nullptr)) set_status(p.status, MSA_ERR_TIMEOUT);
    }
  } else if (warp >= kWarpDq) {
    // ---- dequant warps: K rows to the K tile, V rows to the V tile ---------------------------------
    const int dt = tid - 32 * kWarpDq;
    for (int k = 0;; ++k) {
      const int ms = k % kMetaSlots;
      if (!wwait(&bars.meta_full[ms], static_cast<uint32_t>(k / kMetaSlots) & 1u)) break;
      const int n = meta[ms].n;
      if (n < 0) break;
      const int s = k & 1;
      if (!wwait(&bars.kt_empty[s], (static_cast<uint32_t>(k >> 1) & 1u) ^ 1u)) break;
      // the block's K and V regions straight from the cache (read once per chunk)
      const uint8_t* kreg = p.kv + static_cast<int64_t>(meta[ms].ph) * kKvPage + 2 * meta[ms].g * kRegion;
      uint8_t* kt = smem + Smem::kOffK + static_cast<size_t>(s) * kKTile;
      uint8_t* vt = smem + Smem::kOffV + static_cast<size_t>(s) * kVTile;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {  // this thread's K rows and V rows (keys) dt and dt + 64
        const int kr = dt + 64 * h;
        RawRow rk, rv;
        load_row_global(kreg, kr, rk);
        load_row_global(kreg + kRegion, kr, rv);
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
          uint32_t w[8];
          dequant_quarter(rk, qd, lut, w);
          *reinterpret_cast<uint4*>(kt + sw128_chunk_off(kr, 2 * qd)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(kt + sw128_chunk_off(kr, 2 * qd + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
        uint8_t* vrow = vt + (kr >> 3) * kVSbo + (kr & 7) * 128;
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
          uint32_t w[8];
          dequant_quarter(rv, qd, lut, w);
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {  // dims 32 qd + 8 hh .. +7 = chunk cc = 4 qd + hh
            const int cc = 4 * qd + hh;
            const uint4 v4 = make_uint4(cvt_f16x2_e4m3x2(w[2 * hh]), cvt_f16x2_e4m3x2(w[2 * hh] >> 16),
                                        cvt_f16x2_e4m3x2(w[2 * hh + 1]), cvt_f16x2_e4m3x2(w[2 * hh + 1] >> 16));
            *reinterpret_cast<uint4*>(vrow + (cc >> 3) * kVLbo + (((cc & 7) ^ (kr & 7)) << 4)) = v4;
          }
        }
      }
      fence_proxy_async_smem();  // the tiles are read by the tensor core
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars.kt_full[s]);
        mbar_arrive(&bars.meta_empty[ms]);
      }
    }
  } else if (warp < kWarpEp) {
    // ---- softmax warpgroup x (tiles i with i % 2 == x): thread = query-head row 32 q + lane ------
    const int x = (warp - kWarpSm) >> 2, qw = warp & 3;
    const int row = 32 * qw + lane, sel_in_tile = row >> 4, head = row & 15;
    const uint32_t lanes = static_cast<uint32_t>(32 * qw) << 16;
    const float c = p.scale_log2;
    int i = 0;
    for (int k = 0;; ++k) {
      const int ms = k % kMetaSlots;
      if (!wwait(&bars.meta_full[ms], static_cast<uint32_t>(k / kMetaSlots) & 1u)) break;
      const ChunkMeta& m = meta[ms];
      const int n = m.n;
      if (n < 0) break;
      bool ok = true;
      for (int j = 0; j < ntiles_of(n); ++j, ++i) {
        if ((i & 1) != x) continue;
        const int idx = kTileSel * j + sel_in_tile;
        const bool valid = idx < n;
        const int2 ent = valid ? m.e[idx] : make_int2(0, -1);
        const int rel = ent.y;  // keys after rel are masked (all of them when rel < 0)
        if (!(ok = wwait(&bars.s_full[x], static_cast<uint32_t>(i >> 1) & 1u))) break;
        tc_fence_after();
        const uint32_t ts = tmem + 128u * static_cast<uint32_t>(x) + lanes;
        const bool full = __all_sync(0xffffffffu, rel >= kBS - 1);  // no key of the warp's rows masked
        // chunk cc (keys 32 cc .. 32 cc + 31) of the row's raw scores, masked keys set to -inf
        auto load_chunk = [&](int cc, uint32_t (&r)[32]) {
          tmem_ld32(ts + 32 * cc, r);
          tmem_wait_ld();
          if (!full) {
#pragma unroll
            for (int u = 0; u < 32; ++u)
              r[u] = 32 * cc + u > rel ? __float_as_uint(-CUDART_INF_F) : r[u];
          }
        };
        auto chunk_max = [&](const uint32_t (&r)[32]) {
          float mr = -CUDART_INF_F;
#pragma unroll
          for (int u = 0; u < 32; u += 4)
            mr = fmaxf(mr, max3f(__uint_as_float(r[u]), __uint_as_float(r[u + 1]),
                                 fmaxf(__uint_as_float(r[u + 2]), __uint_as_float(r[u + 3]))));
          return mr * c;  // c > 0: the max of the scaled scores
        };
        uint8_t* pt = smem + Smem::kOffP + static_cast<size_t>(x) * kPTile;
        // P = 2^(s c - mx) of chunk cc, two keys at a time: the exponent by a packed fp32 FMA,
        // rounded to f16, the power by the f16x2 exp2 (a masked key's -inf gives 0); returns the
        // chunk's share of l, the sum of the f16 P that the PV MMA reads (in f16 over 8 keys a
        // half, then over the chunk)
        auto write_chunk = [&](int cc, const uint32_t (&r)[32], float mx) {
          const float mu = mx == -CUDART_INF_F ? 0.f : mx;
          uint32_t s8[4];
#pragma unroll
          for (int q8 = 0; q8 < 4; ++q8) {  // 8 keys: one 16-byte chunk of the row's f16 P
            uint32_t pw[4];
#pragma unroll
            for (int u2 = 0; u2 < 4; ++u2) {
              const int u = 8 * q8 + 2 * u2;
              float x0, x1;
              fma_f32x2(__uint_as_float(r[u]), __uint_as_float(r[u + 1]), c, c, -mu, -mu, x0, x1);
              pw[u2] = exp2_f16x2(pack_f16x2(x0, x1));
            }
            s8[q8] = add_f16x2(add_f16x2(pw[0], pw[1]), add_f16x2(pw[2], pw[3]));
            *reinterpret_cast<uint4*>(pt + (cc >> 1) * kPAtom + sw128_chunk_off(row, 4 * (cc & 1) + q8)) =
                make_uint4(pw[0], pw[1], pw[2], pw[3]);
          }
          return sum_f16x2(add_f16x2(add_f16x2(s8[0], s8[1]), add_f16x2(s8[2], s8[3])));
        };
        // The reference is the maximum over the first 32 keys only (key 0 is never masked in a
        // valid row), so a P may exceed 1. A row whose l stays within kLazyMax (the bound that
        // the row's own maximum gives: 128 keys of P <= 1) keeps that reference, the same bound
        // on its unnormalised o; any other row (P or a sum beyond f16, or a key far above the
        // first 32) is written again from the maximum over all its keys. The warp runs the
        // second pass if any of its rows needs it; the rows that kept their reference write the
        // same P again, so a row's result never depends on the rows it shares a tile with.
        float mx, l;
        {
          uint32_t r[32];
          load_chunk(0, r);
          mx = chunk_max(r);
          if (!(ok = wwait(&bars.p_empty[x], (static_cast<uint32_t>(i >> 1) & 1u) ^ 1u))) break;
          l = write_chunk(0, r, mx);
        }
#pragma unroll 1
        for (int cc = 1; cc < 4; ++cc) {
          uint32_t r[32];
          load_chunk(cc, r);
          l += write_chunk(cc, r, mx);
        }
        if (__any_sync(0xffffffffu, !(l <= kLazyMax))) {
          float m_all = -CUDART_INF_F;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t r[32];
            load_chunk(cc, r);
            m_all = fmaxf(m_all, chunk_max(r));
          }
          if (!(l <= kLazyMax)) mx = m_all;
          l = 0.f;
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t r[32];
            load_chunk(cc, r);
            l += write_chunk(cc, r, mx);
          }
        }
        tc_fence_before();
        fence_proxy_async_smem();  // P is read by the tensor core
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars.s_free[x]);
          mbar_arrive(&bars.p_full[x]);
        }
        if (valid) {
          const int t = ent.x >> 4, slot = ent.x & 15;
          const int64_t base = (static_cast<int64_t>(t) * 4 + m.g) * kSel + slot;
          p.part_ml[base * kHPG + head] = make_float2(l > 0.f ? mx : -CUDART_INF_F, l);
        }
      }
      if (!ok) break;
      if (lane == 0) mbar_arrive(&bars.meta_empty[ms]);
    }
  } else {
    // ---- epilogue warpgroup y (tiles i with i % 2 == y): thread = dim 32 q + lane ---------------
    const int y = (warp - kWarpEp) >> 2, qw = warp & 3;
    const int d = 32 * qw + lane;
    const uint32_t lanes = static_cast<uint32_t>(32 * qw) << 16;
    int i = 0;
    for (int k = 0;; ++k) {
      const int ms = k % kMetaSlots;
      if (!wwait(&bars.meta_full[ms], static_cast<uint32_t>(k / kMetaSlots) & 1u)) break;
      const ChunkMeta& m = meta[ms];
      const int n = m.n;
      if (n < 0) break;
      bool ok = true;
      for (int j = 0; j < ntiles_of(n); ++j, ++i) {
        if ((i & 1) != y) continue;
        if (!(ok = wwait(&bars.o_full[y], static_cast<uint32_t>(i >> 1) & 1u))) break;
        tc_fence_after();
        const uint32_t to = tmem + kColO + 128u * static_cast<uint32_t>(y) + lanes;
#pragma unroll 1
        for (int hc = 0; hc < 4; ++hc) {  // heads 32 hc .. 32 hc + 31: selections 2 hc, 2 hc + 1
          uint32_t o[32];
          tmem_ld32(to + 32 * hc, o);
          tmem_wait_ld();
          if (hc == 3) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.o_free[y]);
          }
#pragma unroll
          for (int ee = 0; ee < 2; ++ee) {
            const int idx = kTileSel * j + 2 * hc + ee;
            if (idx >= n) continue;
            const int2 ent = m.e[idx];
            const int t = ent.x >> 4, slot = ent.x & 15;
            const int64_t base = (static_cast<int64_t>(t) * 4 + m.g) * kSel + slot;
            uint32_t w[8];
#pragma unroll
            for (int u = 0; u < 8; ++u)
              w[u] = pack_f16x2(__uint_as_float(o[16 * ee + 2 * u]), __uint_as_float(o[16 * ee + 2 * u + 1]));
            uint4* dst = reinterpret_cast<uint4*>(p.part_o + (base * kD + d) * (kHPG / 2));
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      }
      if (!ok) break;
      if (lane == 0) mbar_arrive(&bars.meta_empty[ms]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpIss) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One CTA of 128 threads (thread = dim) per (token, group): out = sum_s 2^(m_s - M) o_s /
// sum_s 2^(m_s - M) l_s per head over the selection's partials; zero when the (token, group) is
// bad or has none.
__global__ void __launch_bounds__(128) k_prefill_merge(const PfParams p) {
  grid_dependency_wait();
  __shared__ float2 ml[kSel][kHPG];
  __shared__ float wt[kSel][kHPG];
  __shared__ float winv[kHPG];
  __shared__ int any[kSel];
  const int tg = blockIdx.x, t = tg >> 2, g = tg & 3, d = threadIdx.x;
  const int64_t base = static_cast<int64_t>(tg) * kSel;
  for (int x = d; x < kSel * kHPG; x += 128) ml[x / kHPG][x % kHPG] = p.part_ml[base * kHPG + x];
  __syncthreads();
  const bool bad = p.tg_bad[tg] != 0;
  if (d < kHPG) {
    float M = -CUDART_INF_F;
    for (int s = 0; s < kSel; ++s) M = fmaxf(M, ml[s][d].x);
    float W = 0.f;
    for (int s = 0; s < kSel; ++s) {
      const float w = (M == -CUDART_INF_F || ml[s][d].x == -CUDART_INF_F) ? 0.f : fast_exp2(ml[s][d].x - M);
      wt[s][d] = w;
      W += w * ml[s][d].y;
    }
    winv[d] = (W > 0.f && !bad) ? 1.0f / W : 0.f;
  } else if (d < kHPG + kSel) {
    const int s = d - kHPG;
    int a = 0;
    for (int h = 0; h < kHPG; ++h) a |= ml[s][h].x != -CUDART_INF_F;
    any[s] = a && !bad;
  }
  __syncthreads();
  float acc[kHPG];
#pragma unroll
  for (int h = 0; h < kHPG; ++h) acc[h] = 0.f;
  for (int s = 0; s < kSel; ++s) {
    if (!any[s]) continue;
    const uint4* src = reinterpret_cast<const uint4*>(p.part_o + ((base + s) * kD + d) * (kHPG / 2));
    const uint4 a = src[0], b = src[1];
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float2 o = __half22float2(*reinterpret_cast<const __half2*>(&w[u]));
      acc[2 * u] = fmaf(wt[s][2 * u], o.x, acc[2 * u]);
      acc[2 * u + 1] = fmaf(wt[s][2 * u + 1], o.y, acc[2 * u + 1]);
    }
  }
  uint16_t* dst = p.out + (static_cast<int64_t>(t) * kQHeads + g * kHPG) * kD + d;
#pragma unroll
  for (int h = 0; h < kHPG; ++h) dst[h * kD] = static_cast<uint16_t>(pack_bf16x2(acc[h] * winv[h], 0.f) & 0xFFFFu);
}

struct PfLayout {
  size_t hdr, hkeys, hcnt, rowh, ehash, entries, chunks, tg_bad, part_o, part_ml, total;
  uint32_t hslots;
  int hbits;
};

// The hash table has at least twice as many slots as there are selections (sized by the
// selections even when fewer distinct rows can exist: the keys' counters then spread over many
// cache lines, which their atomics need).
PfLayout pf_layout(int T) {
  using msa_host::align256;
  PfLayout l;
  const size_t ent = static_cast<size_t>(T) * 4 * kSel;
  l.hbits = 10;
  while ((size_t{1} << l.hbits) < 2 * ent) ++l.hbits;
  l.hslots = static_cast<uint32_t>(size_t{1} << l.hbits);
  l.hdr = 0;
  l.hkeys = l.hdr + 256;
  l.hcnt = l.hkeys + align256(static_cast<size_t>(l.hslots) * 8);
  l.rowh = l.hcnt + align256(static_cast<size_t>(l.hslots) * 4);
  l.ehash = l.rowh + align256(ent * 4);
  l.entries = l.ehash + align256(ent * 4);
  l.chunks = l.entries + align256(ent * 8);
  l.tg_bad = l.chunks + align256((ent + static_cast<size_t>(T)) * 16);
  l.part_o = l.tg_bad + align256(static_cast<size_t>(T) * 4 * 4);
  l.part_ml = l.part_o + align256(ent * kHPG * kD * 2);
  l.total = l.part_ml + align256(ent * kHPG * 8);
  return l;
}

}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

extern "C" size_t msa_prefill_workspace_size(const msa_geometry* geo, int32_t B, int32_t T, int32_t max_blocks_per_seq) {
  if (check_geometry(geo) != MSA_OK || B < 0 || T < 0 || T > kMaxT || max_blocks_per_seq < 1 ||
      max_blocks_per_seq > (1 << 20))
    return 0;
  return pf_layout(T).total;
}

extern "C" msa_status msa_prefill_attn(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                       const uint8_t* q, const int32_t* sel, float softmax_scale, void* workspace,
                                       size_t workspace_bytes, uint16_t* out, uint32_t* status, cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  // a prefill batch: any number of query tokens per sequence (max_q_len up to 2^20)
  if ((st = check_prefill_batch(batch)) != MSA_OK) return st;
  if ((st = check_cache(cache, false, true)) != MSA_OK) return st;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (q == nullptr || sel == nullptr || out == nullptr || !aligned(q, 16) || !aligned(sel, 4) || !aligned(out, 16))
    return MSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || softmax_scale != softmax_scale) return MSA_ERR_INVALID_ARG;
  const PfLayout lay = pf_layout(batch->T);
  if (workspace == nullptr || !aligned(workspace, 256) || workspace_bytes < lay.total) return MSA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  PfParams p;
  p.B = batch->B;
  p.T = batch->T;
  p.maxb = batch->max_blocks_per_seq;
  p.num_pages = cache->num_pages;
  p.qsl = batch->query_start_loc;
  p.seq_lens = batch->seq_lens;
  p.block_table = batch->block_table;
  p.kv = cache->kv_pages;
  p.q = q;
  p.sel = sel;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = out;
  p.hdr = reinterpret_cast<int32_t*>(ws + lay.hdr);
  p.hkeys = reinterpret_cast<uint64_t*>(ws + lay.hkeys);
  p.hcnt = reinterpret_cast<int32_t*>(ws + lay.hcnt);
  p.rowh = reinterpret_cast<int32_t*>(ws + lay.rowh);
  p.ehash = reinterpret_cast<int32_t*>(ws + lay.ehash);
  p.entries = reinterpret_cast<int2*>(ws + lay.entries);
  p.chunks = reinterpret_cast<int4*>(ws + lay.chunks);
  p.tg_bad = reinterpret_cast<int32_t*>(ws + lay.tg_bad);
  p.part_o = reinterpret_cast<uint32_t*>(ws + lay.part_o);
  p.part_ml = reinterpret_cast<float2*>(ws + lay.part_ml);
  p.hmask = lay.hslots - 1;
  p.hbits = lay.hbits;
  p.status = status;
  {
    const int64_t n = std::max<int64_t>(lay.hslots, static_cast<int64_t>(p.T) * 4);
    const int ib = static_cast<int>(std::min<int64_t>((n + 255) / 256, 8 * kTunedSms));
    k_map_init<<<ib, 256, 0, stream>>>(p);
  }
  const int64_t ent = static_cast<int64_t>(p.T) * 4 * kSel;
  const int eb = static_cast<int>((ent + 255) / 256);
  if (launch_after_previous(k_map_count, dim3(eb), dim3(256), 0, stream, p) != cudaSuccess ||
      launch_after_previous(k_map_alloc, dim3(eb), dim3(256), 0, stream, p) != cudaSuccess ||
      launch_after_previous(k_map_fill, dim3(eb), dim3(256), 0, stream, p) != cudaSuccess)
    return MSA_ERR_CUDA;
  if ((st = launch_status()) != MSA_OK) return st;
  alignas(64) CUtensorMap q_map;
  if (!rows128_tensor_map(&q_map, q, static_cast<uint64_t>(p.T) * kQHeads, kHPG)) return MSA_ERR_CUDA;
  if (cudaFuncSetAttribute(k_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Smem::kBytes)) !=
      cudaSuccess)
    return MSA_ERR_CUDA;
  const int sms = num_sms();
  if (sms <= 0) return MSA_ERR_CUDA;
  // never more CTAs than chunks can exist: at most T + 64 T (each row adds at most one chunk)
  const int64_t max_chunks = ent + p.T;
  const int grid = static_cast<int>(max_chunks < sms ? max_chunks : sms);
  if (launch_after_previous(k_prefill_tc, dim3(grid), dim3(kThreads), Smem::kBytes, stream, p, q_map) != cudaSuccess ||
      launch_after_previous(k_prefill_merge, dim3(static_cast<unsigned>(static_cast<int64_t>(p.T) * 4)), dim3(128), 0,
                            stream, p) != cudaSuccess)
    return MSA_ERR_CUDA;
  return launch_status();
}
