// msa_gather.cu — the K/V side of context-sharded decode: bringing the selected blocks' K/V to
// the rank that owns the query tokens.
//
// "vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", "Indexador NVFP4 DCP": the context is
// split across ranks, each rank scores its own blocks, and the selection is merged on the rank
// that owns the query; sparse attention then reads only the selected blocks, which lie on
// several ranks. This file gives the owner a local copy of exactly those blocks:
//  * msa_kv_gather_map numbers the distinct (sequence, block) pairs that any query token of the
//    sequence selected, sequence by sequence in block order, and records which groups selected
//    each; the numbering is the owner's block table into a gathered page pool;
//  * msa_kv_gather_pages copies, on a rank that holds blocks [block_begin, block_end) of every
//    sequence, the selected (page, group) K and V regions it holds into their gathered pages.
// The pool pages have the KV page layout, so the owner runs msa_sparse_attn_decode on it
// unchanged. Moving the pages between ranks is plain copies of the shards' pools (or their
// selected pages), never remote tensor copies or multicast.
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "msa.h"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

constexpr int kScanThreads = 1024;

// Mark: block sel[t][g][i] of token t's sequence b gets group bit g in masks[b][block].
__global__ void k_gather_mark(const int32_t* qsl, const int32_t* seq_lens, int32_t B, int32_t T, int32_t maxb,
                              const int32_t* sel, uint32_t* marks, uint32_t* status) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;  // (t, g, slot)
  if (e >= static_cast<int64_t>(T) * 4 * kSel) return;
  const int t = static_cast<int>(e / (4 * kSel)), g = static_cast<int>((e / kSel) & 3);
  int lo = 0, hi = B - 1;  // the sequence of token t (largest b with qsl[b] <= t)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int v = sel[e];
  if (v < 0) return;  // padding
  const int nb = ceil_div(seq_lens[lo], kBS);
  if (v >= nb || v >= maxb) {
    set_status(status, MSA_ERR_DEVICE_FAULT);
    return;
  }
  atomicOr(&marks[static_cast<int64_t>(lo) * maxb + v], 1u << g);
}

// Number: one CTA scans marks[0 .. n) in order; a marked entry gets the next gathered page
// index in map, its group mask in masks; unmarked entries get -1 / 0.
__global__ void __launch_bounds__(kScanThreads) k_gather_number(const uint32_t* marks, int64_t n, int32_t* map,
                                                                 uint8_t* masks, int32_t* num_gathered) {
  __shared__ int warp_tot[kScanThreads / 32];
  __shared__ int carry;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) carry = 0;
  __syncthreads();
  for (int64_t base = 0; base < n; base += kScanThreads) {
    const int64_t i = base + tid;
    const uint32_t mk = i < n ? marks[i] : 0u;
    const int f = mk != 0u ? 1 : 0;
    int incl = f;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
      const int v = warp_tot[lane];
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += u;
      }
      warp_tot[lane] = x - v;  // exclusive
    }
    __syncthreads();
    const int c0 = carry;
    if (i < n) {
      map[i] = f ? c0 + warp_tot[warp] + incl - 1 : -1;
      masks[i] = static_cast<uint8_t>(mk & 0xFu);
    }
    __syncthreads();
    if (tid == kScanThreads - 1) carry = c0 + warp_tot[warp] + incl;
    __syncthreads();
  }
  if (tid == 0) *num_gathered = carry;
}

// Copy: a warp per (sequence, block) entry of the shard's range; each group in the entry's mask
// has its K and V regions (18,432 B, contiguous in a page) copied with 16-byte loads and stores.
__global__ void k_gather_pages(const int32_t* block_table, const uint8_t* kv_pages, int32_t num_pages, int32_t B,
                               int32_t maxb, const int32_t* map, const uint8_t* masks, int32_t block_begin,
                               int32_t block_end, uint8_t* gathered, int32_t max_gathered, uint32_t* status) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t span = static_cast<int64_t>(block_end - block_begin);
  for (int64_t w = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
       w < static_cast<int64_t>(B) * span; w += warps) {
    const int b = static_cast<int>(w / span), blk = block_begin + static_cast<int>(w % span);
    const int64_t ent = static_cast<int64_t>(b) * maxb + blk;
    const int gp = map[ent];
    if (gp < 0) continue;
    const int page = block_table[ent];
    if (page < 0 || page >= num_pages || gp >= max_gathered) {
      if (lane == 0) set_status(status, MSA_ERR_DEVICE_FAULT);
      continue;
    }
    const uint32_t mk = masks[ent];
    for (int g = 0; g < kGroups; ++g) {
      if (!(mk & (1u << g))) continue;
      const uint4* src = reinterpret_cast<const uint4*>(kv_pages + static_cast<int64_t>(page) * kKvPage + g * 2 * kRegion);
      uint4* dst = reinterpret_cast<uint4*>(gathered + static_cast<int64_t>(gp) * kKvPage + g * 2 * kRegion);
      for (int i = lane; i < 2 * kRegion / 16; i += 32) dst[i] = src[i];
    }
  }
}

}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

extern "C" msa_status msa_kv_gather_map(const msa_geometry* geo, const msa_batch* batch, const int32_t* sel,
                                        int32_t* map, uint8_t* masks, int32_t* num_gathered, uint32_t* status,
                                        cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = check_batch(batch)) != MSA_OK) return st;
  if (map == nullptr || masks == nullptr || num_gathered == nullptr || !aligned(map, 4) || !aligned(num_gathered, 4))
    return MSA_ERR_INVALID_ARG;
  const int64_t n = static_cast<int64_t>(batch->B) * batch->max_blocks_per_seq;
  if (batch->T > 0 && (sel == nullptr || !aligned(sel, 4))) return MSA_ERR_INVALID_ARG;
  // the marks are built in map itself (as bits), then numbered in place by one ordered pass
  if (n > 0 && cudaMemsetAsync(map, 0, static_cast<size_t>(n) * 4, stream) != cudaSuccess) return MSA_ERR_CUDA;
  if (batch->B > 0 && batch->T > 0) {
    const int64_t e = static_cast<int64_t>(batch->T) * 4 * kSel;
    k_gather_mark<<<static_cast<unsigned>(ceil_div(static_cast<int>(e), 256)), 256, 0, stream>>>(
        batch->query_start_loc, batch->seq_lens, batch->B, batch->T, batch->max_blocks_per_seq, sel,
        reinterpret_cast<uint32_t*>(map), status);
    if ((st = launch_status()) != MSA_OK) return st;
  }
  k_gather_number<<<1, kScanThreads, 0, stream>>>(reinterpret_cast<const uint32_t*>(map), n, map, masks, num_gathered);
  return launch_status();
}

extern "C" msa_status msa_kv_gather_pages(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                          const int32_t* map, const uint8_t* masks, int32_t block_begin,
                                          int32_t block_end, uint8_t* gathered_kv, int32_t max_gathered,
                                          uint32_t* status, cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = check_batch(batch)) != MSA_OK) return st;
  if ((st = check_cache(cache, false, true)) != MSA_OK) return st;
  if (block_begin < 0 || block_end < block_begin || max_gathered < 0) return MSA_ERR_INVALID_ARG;
  const int32_t end = block_end < batch->max_blocks_per_seq ? block_end : batch->max_blocks_per_seq;
  if (batch->B == 0 || end <= block_begin || max_gathered == 0) return MSA_OK;
  if (map == nullptr || masks == nullptr || gathered_kv == nullptr || !aligned(map, 4) || !aligned(gathered_kv, 16))
    return MSA_ERR_INVALID_ARG;
  const int sms = num_sms();
  if (sms <= 0) return MSA_ERR_CUDA;
  k_gather_pages<<<4 * sms, 256, 0, stream>>>(batch->block_table, cache->kv_pages, cache->num_pages, batch->B,
                                              batch->max_blocks_per_seq, map, masks, block_begin, end, gathered_kv,
                                              max_gathered, status);
  return launch_status();
}

extern "C" int32_t msa_kv_gather_map_host(int32_t B, int32_t T, const int32_t* query_start_loc,
                                          const int32_t* seq_lens, int32_t max_blocks_per_seq, const int32_t* sel,
                                          int32_t* map, uint8_t* masks) {
  if (B < 0 || T < 0 || max_blocks_per_seq < 1) return -1;
  const int64_t n = static_cast<int64_t>(B) * max_blocks_per_seq;
  if (n > 0 && (query_start_loc == nullptr || seq_lens == nullptr || map == nullptr || masks == nullptr)) return -1;
  if (T > 0 && sel == nullptr) return -1;
  std::vector<uint32_t> marks(static_cast<size_t>(n), 0u);
  for (int b = 0; b < B; ++b) {
    const int nb = ceil_div(seq_lens[b], kBS);
    for (int t = query_start_loc[b]; t < query_start_loc[b + 1]; ++t)
      for (int g = 0; g < 4; ++g)
        for (int i = 0; i < kSel; ++i) {
          const int v = sel[(static_cast<int64_t>(t) * 4 + g) * kSel + i];
          if (v < 0) continue;
          if (v >= nb || v >= max_blocks_per_seq) return -1;
          marks[static_cast<size_t>(b) * max_blocks_per_seq + v] |= 1u << g;
        }
  }
  int32_t next = 0;
  for (int64_t i = 0; i < n; ++i) {
    map[i] = marks[i] ? next++ : -1;
    masks[i] = static_cast<uint8_t>(marks[i]);
  }
  return next;
}

extern "C" msa_status msa_kv_gather_pages_host(int32_t B, int32_t max_blocks_per_seq, const int32_t* block_table,
                                               const uint8_t* kv_pages, int32_t num_pages, const int32_t* map,
                                               const uint8_t* masks, int32_t block_begin, int32_t block_end,
                                               uint8_t* gathered_kv, int32_t max_gathered) {
  if (B < 0 || max_blocks_per_seq < 1 || block_begin < 0 || block_end < block_begin || num_pages < 0 ||
      max_gathered < 0)
    return MSA_ERR_INVALID_ARG;
  if (B > 0 && (block_table == nullptr || map == nullptr || masks == nullptr)) return MSA_ERR_INVALID_ARG;
  const int end = block_end < max_blocks_per_seq ? block_end : max_blocks_per_seq;
  for (int b = 0; b < B; ++b)
    for (int blk = block_begin; blk < end; ++blk) {
      const int64_t ent = static_cast<int64_t>(b) * max_blocks_per_seq + blk;
      const int gp = map[ent];
      if (gp < 0) continue;
      const int page = block_table[ent];
      if (page < 0 || page >= num_pages || gp >= max_gathered || kv_pages == nullptr || gathered_kv == nullptr)
        return MSA_ERR_DEVICE_FAULT;
      for (int g = 0; g < kGroups; ++g)
        if (masks[ent] & (1u << g)) {
          const uint8_t* src = kv_pages + static_cast<int64_t>(page) * kKvPage + g * 2 * kRegion;
          uint8_t* dst = gathered_kv + static_cast<int64_t>(gp) * kKvPage + g * 2 * kRegion;
          for (int i = 0; i < 2 * kRegion; ++i) dst[i] = src[i];
        }
    }
  return MSA_OK;
}
