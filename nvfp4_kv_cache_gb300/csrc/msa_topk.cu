// msa_topk.cu — per-(token, group) block selection of the MSA decode step.
//
// What it computes ("vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", "MSA primer": the top
// 16 blocks with the most recent one always kept; "MiniMax M3 in vLLM ...", "MSA 机制详解":
// init_blocks = 0, local_blocks = 1, a local block that also ranks in the top-k is not counted
// twice): local = p_t / 128 is slot 0, slots 1..15 are the 15 best of blocks 0 .. local-1 in
// descending score order, equal scores ordered by lower block id, -1 when fewer exist.
//
// Design: one warp per (token, group) row (a CTA per row, each warp a slice, for batches of few
// rows longer than one warp holds in registers). Each score becomes a unique 64-bit key
// (order-preserving fp32 bits << 32 | ~block id), so "descending score, then lower id" is one
// integer order and ties need no special case. Rows of up to 64 candidates are sorted in
// registers (warp bitonic network, two keys per lane). Longer rows are first filtered: the
// 15th largest of the 32 lane maxima is a lower bound of the 15th largest key, so only keys
// at or above it survive (typically a few dozen), and those are sorted. The indexer's scores
// are the only input, so GPU selection == the oracle's sort on the same scores, bit for bit.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "msa.h"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

constexpr int kKeysPerLane = 16;

__host__ __device__ inline uint64_t score_key(float s, int id) {
  uint32_t u;
  memcpy(&u, &s, 4);
  if (s != s) u = 0xFF800000u;   // NaN ranks as -inf
  if (s == 0.0f) u = 0u;         // -0 == +0
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}

__host__ __device__ inline int key_id(uint64_t key) {
  return static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(key & 0xFFFFFFFFull));
}

__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t w = __shfl_xor_sync(0xffffffffu, v, o);
    v = w > v ? w : v;
  }
  return v;
}

// Pop the 15 largest of the keys held by the warp (keys[] per lane plus `carry`); the result
// (descending) is returned in lanes 0..14, 0 where there are fewer than 15 keys.
template <int N>
__device__ __forceinline__ uint64_t warp_pop15(uint64_t (&keys)[N], uint64_t carry, int lane) {
  uint64_t best = carry;
#pragma unroll
  for (int i = 0; i < N; ++i) best = keys[i] > best ? keys[i] : best;
  uint64_t out = 0;
  for (int r = 0; r < 15; ++r) {
    const uint64_t m = warp_max_u64(best);
    if (m == 0) break;  // warp-uniform
    if (lane == r) out = m;
    if (best == m) {    // exactly one lane owns m (keys are unique)
      if (carry == m) carry = 0;
#pragma unroll
      for (int i = 0; i < N; ++i)
        if (keys[i] == m) keys[i] = 0;
      best = carry;
#pragma unroll
      for (int i = 0; i < N; ++i) best = keys[i] > best ? keys[i] : best;
    }
  }
  return out;
}

struct TopkParams {
  int32_t B, T, maxb, max_q_len;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const float* scores;
  int32_t* sel;
  uint32_t* status;
};

// Warp bitonic sort, descending, of 64 keys held two per lane (element 2*lane + r).
__device__ __forceinline__ void warp_sort64_desc(uint64_t& k0, uint64_t& k1, int lane) {
#pragma unroll
  for (int size = 2; size <= 64; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride == 1) {
        // partner inside the lane: elements 2*lane and 2*lane+1
        const bool desc = ((2 * lane) & size) == 0;
        const uint64_t hi = k0 > k1 ? k0 : k1, lo = k0 > k1 ? k1 : k0;
        k0 = desc ? hi : lo;
        k1 = desc ? lo : hi;
      } else {
        const int lstride = stride >> 1;  // partner lane
        const bool upper = (lane & lstride) != 0;
        const bool desc = ((2 * lane) & size) == 0;
        const uint64_t p0 = __shfl_xor_sync(0xffffffffu, k0, lstride);
        const uint64_t p1 = __shfl_xor_sync(0xffffffffu, k1, lstride);
        // the lower element of the pair keeps the larger key in a descending run
        const bool take_max = (desc != upper);
        k0 = take_max ? (k0 > p0 ? k0 : p0) : (k0 > p0 ? p0 : k0);
        k1 = take_max ? (k1 > p1 ? k1 : p1) : (k1 > p1 ? p1 : k1);
      }
    }
  }
}

// Warp bitonic sort, descending, of 32 keys, one per lane.
__device__ __forceinline__ uint64_t warp_sort32_desc(uint64_t k, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const uint64_t p = __shfl_xor_sync(0xffffffffu, k, stride);
      const bool upper = (lane & stride) != 0;
      const bool desc = (lane & size) == 0;
      const bool take_max = (desc != upper);
      k = take_max ? (k > p ? k : p) : (k > p ? p : k);
    }
  }
  return k;
}

constexpr int kRowsPerCta = 8;
constexpr int kSurvivors = 64;
constexpr int kRegKeys = 32;  // rows of up to 32 x 32 keys are held in registers (one load each)
// The same for rows of up to 128, 256 and 512 keys: fewer registers (more warps per SM) and no
// work on empty key slots.
constexpr int kRegKeysShort = 4;
constexpr int kCand = kSel - 1;  // candidates per (token, group) and shard: the 15 best non-local blocks

// The 15 largest of the n keys key_at(0 .. n-1) (unique; 0 = none), descending, into res[0..14]
// (0 past the end). One warp. The 15th largest of the 32 lane maxima bounds the 15th largest key
// (15 distinct elements reach it), so only keys at or above it survive (typically a few
// dozen) and those are sorted in registers; more than 64 survivors (adversarial ties across
// lanes) fall back to repeated warp argmax.
template <int KR = kRegKeys, class KeyAt>
__device__ void top15_keys(KeyAt key_at, int n, uint64_t* buf, uint64_t* res, int lane) {
  uint64_t k0 = 0, k1 = 0;
  bool sorted = false;
  if (n <= kSurvivors) {
    k0 = 2 * lane < n ? key_at(2 * lane) : 0ull;
    k1 = 2 * lane + 1 < n ? key_at(2 * lane + 1) : 0ull;
    sorted = true;
  } else if (n <= 32 * KR) {
    // the same filter with the row's keys loaded once, all loads in flight together
    uint64_t kk[KR];
#pragma unroll
    for (int j = 0; j < KR; ++j) kk[j] = 32 * j + lane < n ? key_at(32 * j + lane) : 0ull;
    uint64_t best = 0;
#pragma unroll
    for (int j = 0; j < KR; ++j) best = kk[j] > best ? kk[j] : best;
    const uint64_t tau = __shfl_sync(0xffffffffu, warp_sort32_desc(best, lane), 14);
    int count = 0;
#pragma unroll
    for (int j = 0; j < KR; ++j) {
      const bool keep = kk[j] >= tau && kk[j] != 0ull;
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      const int pos = count + __popc(m & ((1u << lane) - 1u));
      if (keep && pos < kSurvivors) buf[pos] = kk[j];
      count += __popc(m);
    }
    __syncwarp();
    if (count <= kSurvivors) {
      k0 = 2 * lane < count ? buf[2 * lane] : 0ull;
      k1 = 2 * lane + 1 < count ? buf[2 * lane + 1] : 0ull;
      sorted = true;
    }
    __syncwarp();
  } else {
    uint64_t best = 0;
    for (int i = lane; i < n; i += 32) {
      const uint64_t k = key_at(i);
      best = k > best ? k : best;
    }
    const uint64_t tau = __shfl_sync(0xffffffffu, warp_sort32_desc(best, lane), 14);
    int count = 0;
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      const uint64_t k = i < n ? key_at(i) : 0ull;
      const bool keep = k >= tau && k != 0ull;
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      const int pos = count + __popc(m & ((1u << lane) - 1u));
      if (keep && pos < kSurvivors) buf[pos] = k;
      count += __popc(m);
    }
    __syncwarp();
    if (count <= kSurvivors) {
      k0 = 2 * lane < count ? buf[2 * lane] : 0ull;
      k1 = 2 * lane + 1 < count ? buf[2 * lane + 1] : 0ull;
      sorted = true;
    }
    __syncwarp();
  }
  if (sorted) {
    warp_sort64_desc(k0, k1, lane);  // elements 2 lane, 2 lane + 1 of the sorted run
    if (2 * lane < kCand) res[2 * lane] = k0;
    if (2 * lane + 1 < kCand) res[2 * lane + 1] = k1;
  } else {
    uint64_t top = 0;  // repeated warp argmax, 16 keys per lane per pass, running top 15 carried
    for (int c0 = 0; c0 < n; c0 += 32 * kKeysPerLane) {
      uint64_t keys[kKeysPerLane];
#pragma unroll
      for (int i = 0; i < kKeysPerLane; ++i) {
        const int id = c0 + i * 32 + lane;
        keys[i] = id < n ? key_at(id) : 0ull;
      }
      top = warp_pop15(keys, lane < kCand ? top : 0ull, lane);
    }
    if (lane < kCand) res[lane] = top;
  }
  __syncwarp();
}

// Row (t, g) of the batch: its sequence, and local = p_t / 128 for a consistent row (-1 else,
// with MSA_ERR_INVALID_ARG raised).
__device__ __forceinline__ int row_local(const TopkParams& p, int t) {
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int q0 = p.qsl[lo], ql = p.qsl[lo + 1] - q0;
  const int L = p.seq_lens[lo];
  if (!(t - q0 < ql && ql <= p.max_q_len && L >= ql && L <= p.maxb * kBS)) return -1;
  return (L - ql + (t - q0)) / kBS;
}

// One warp per (token, group) row: sel = [local, the 15 best of blocks 0 .. local-1]; rows of up
// to 32 x KR keys are loaded into registers at once.
template <int KR>
__global__ void __launch_bounds__(32 * kRowsPerCta) k_topk(const TopkParams p) {
  __shared__ uint64_t buf[kRowsPerCta][kSurvivors];
  __shared__ uint64_t res[kRowsPerCta][kCand];
  grid_dependency_wait();  // the indexer's scores (this kernel may launch while it finishes)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerCta + warp;  // t * 4 + g
  if (row >= p.T * 4) return;
  int32_t* out = p.sel + static_cast<int64_t>(row) * kSel;
  const int local = row_local(p, row >> 2);
  if (local < 0) {
    if (lane == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
    if (lane < kSel) out[lane] = -1;
    return;
  }
  const float* s = p.scores + static_cast<int64_t>(row) * p.maxb;
  top15_keys<KR>([&](int i) { return score_key(s[i], i); }, local, buf[warp], res[warp], lane);
  if (lane == 0) out[0] = local;
  if (lane < kCand) out[1 + lane] = res[warp][lane] ? key_id(res[warp][lane]) : -1;
}

// The same selection for a batch of few rows, some longer than one warp holds in registers
// (32 x kRegKeys keys): a CTA per row, so that the rows spread over the SMs; each of its warps
// takes the 15 best of one slice of the row, then one warp the 15 best of the slices'
// candidates (keys are unique, so the 15 best of the union are the row's 15 best).
constexpr int kSplitWarps = 8;

__global__ void __launch_bounds__(32 * kSplitWarps) k_topk_split(const TopkParams p) {
  __shared__ uint64_t buf[kSplitWarps][kSurvivors];
  __shared__ uint64_t res[kSplitWarps][kCand];
  __shared__ uint64_t top[kCand];
  grid_dependency_wait();  // the indexer's scores (this kernel may launch while it finishes)
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x;  // t * 4 + g
  int32_t* out = p.sel + static_cast<int64_t>(row) * kSel;
  const int local = row_local(p, row >> 2);  // the same for every warp of the CTA
  if (local < 0) {
    if (warp == 0 && lane == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
    if (warp == 0 && lane < kSel) out[lane] = -1;
    return;
  }
  const float* s = p.scores + static_cast<int64_t>(row) * p.maxb;
  const int per = ceil_div(local, kSplitWarps);
  const int lo = min(local, warp * per), n = min(local, lo + per) - lo;
  top15_keys([&](int i) { return score_key(s[lo + i], lo + i); }, n, buf[warp], res[warp], lane);
  __syncthreads();
  if (warp == 0) {
    top15_keys([&](int i) { return res[i / kCand][i % kCand]; }, kSplitWarps * kCand, buf[0], top, lane);
    if (lane == 0) out[0] = local;
    if (lane < kCand) out[1 + lane] = top[lane] ? key_id(top[lane]) : -1;
  }
}

struct CandParams {
  TopkParams t;
  int32_t kb, ke;        // this shard's block range
  int32_t n_shards;      // merge: candidate lists per row
  uint64_t* cand;        // [rows][15] (candidates) or [n_shards][rows][15] (merge)
  const uint64_t* cand_in;
};

// A context shard's candidates: per row the 15 best of its non-local blocks in [kb, ke), as
// keys, descending (0 = none).
__global__ void __launch_bounds__(32 * kRowsPerCta) k_topk_cand(const CandParams c) {
  __shared__ uint64_t buf[kRowsPerCta][kSurvivors];
  __shared__ uint64_t res[kRowsPerCta][kCand];
  const TopkParams& p = c.t;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerCta + warp;
  if (row >= p.T * 4) return;
  uint64_t* out = c.cand + static_cast<int64_t>(row) * kCand;
  const int local = row_local(p, row >> 2);
  if (local < 0) {
    if (lane == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
    if (lane < kCand) out[lane] = 0ull;
    return;
  }
  const int lo = min(c.kb, local), n = max(0, min(c.ke, local) - lo);
  const float* s = p.scores + static_cast<int64_t>(row) * p.maxb;
  top15_keys([&](int i) { return score_key(s[lo + i], lo + i); }, n, buf[warp], res[warp], lane);
  if (lane < kCand) out[lane] = res[warp][lane];
}

// The owner's merge: per row the 15 best of the shards' n_shards x 15 candidates, behind local.
__global__ void __launch_bounds__(32 * kRowsPerCta) k_topk_merge(const CandParams c) {
  __shared__ uint64_t buf[kRowsPerCta][kSurvivors];
  __shared__ uint64_t res[kRowsPerCta][kCand];
  const TopkParams& p = c.t;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerCta + warp;
  if (row >= p.T * 4) return;
  int32_t* out = p.sel + static_cast<int64_t>(row) * kSel;
  const int local = row_local(p, row >> 2);
  if (local < 0) {
    if (lane == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
    if (lane < kSel) out[lane] = -1;
    return;
  }
  const int64_t rows = static_cast<int64_t>(p.T) * 4;
  const uint64_t* cin = c.cand_in + static_cast<int64_t>(row) * kCand;
  top15_keys([&](int i) { return cin[static_cast<int64_t>(i / kCand) * rows * kCand + i % kCand]; },
             c.n_shards * kCand, buf[warp], res[warp], lane);
  if (lane == 0) out[0] = local;
  if (lane < kCand) out[1 + lane] = res[warp][lane] ? key_id(res[warp][lane]) : -1;
}

// Host: the 15 largest of keys (descending, 0-padded), the same order as the kernels.
void host_top15(std::vector<uint64_t>& keys, uint64_t* out) {
  const size_t m = std::min<size_t>(kCand, keys.size());
  std::partial_sort(keys.begin(), keys.begin() + static_cast<std::ptrdiff_t>(m), keys.end(),
                    [](uint64_t a, uint64_t b) { return a > b; });
  for (int i = 0; i < kCand; ++i) out[i] = static_cast<size_t>(i) < m ? keys[i] : 0ull;
}
}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

namespace {
msa_status topk_setup(const msa_geometry* geo, const msa_batch* batch, const float* block_scores, int32_t* sel,
                      uint32_t* status, TopkParams* p, bool prefill = false);
msa_status topk_launch(const msa_batch* batch, const TopkParams& p, const float* block_scores, int32_t* sel,
                       cudaStream_t stream);
}  // namespace

extern "C" msa_status msa_topk_blocks(const msa_geometry* geo, const msa_batch* batch, const float* block_scores,
                                      int32_t* sel, uint32_t* status, cudaStream_t stream) {
  TopkParams p;
  const msa_status st = topk_setup(geo, batch, block_scores, sel, status, &p);
  if (st != MSA_OK) return st;
  return topk_launch(batch, p, block_scores, sel, stream);
}

extern "C" msa_status msa_topk_prefill(const msa_geometry* geo, const msa_batch* batch, const float* block_scores,
                                       int32_t* sel, uint32_t* status, cudaStream_t stream) {
  TopkParams p;
  const msa_status st = topk_setup(geo, batch, block_scores, sel, status, &p, true);
  if (st != MSA_OK) return st;
  return topk_launch(batch, p, block_scores, sel, stream);
}

namespace {
msa_status topk_launch(const msa_batch* batch, const TopkParams& p, const float* block_scores, int32_t* sel,
                       cudaStream_t stream) {
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (block_scores == nullptr || sel == nullptr || !aligned(block_scores, 4) || !aligned(sel, 4))
    return MSA_ERR_INVALID_ARG;
  // a warp per row (with as many keys a lane in registers as the longest possible row needs:
  // 4, 8, 16 or 32); a CTA per row when rows may be longer than a warp holds and so few that a
  // CTA each fits in one wave (two per SM of the part the choice is tuned for)
  const int rows = batch->T * 4;
  const dim3 grid(ceil_div(rows, kRowsPerCta)), block(32 * kRowsPerCta);
  const cudaError_t e =
      (batch->max_blocks_per_seq > 32 * kRegKeys && rows <= 2 * kTunedSms)
          ? launch_after_previous(k_topk_split, dim3(rows), dim3(32 * kSplitWarps), 0, stream, p)
      : batch->max_blocks_per_seq <= 32 * kRegKeysShort
          ? launch_after_previous(k_topk<kRegKeysShort>, grid, block, 0, stream, p)
      : batch->max_blocks_per_seq <= 32 * 8 ? launch_after_previous(k_topk<8>, grid, block, 0, stream, p)
      : batch->max_blocks_per_seq <= 32 * 16 ? launch_after_previous(k_topk<16>, grid, block, 0, stream, p)
                                             : launch_after_previous(k_topk<kRegKeys>, grid, block, 0, stream, p);
  if (e != cudaSuccess) return MSA_ERR_CUDA;
  return launch_status();
}

msa_status topk_setup(const msa_geometry* geo, const msa_batch* batch, const float* block_scores, int32_t* sel,
                      uint32_t* status, TopkParams* p, bool prefill) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = prefill ? check_prefill_batch(batch) : check_batch(batch)) != MSA_OK) return st;
  p->B = batch->B;
  p->T = batch->T;
  p->maxb = batch->max_blocks_per_seq;
  p->max_q_len = batch->max_q_len;
  p->qsl = batch->query_start_loc;
  p->seq_lens = batch->seq_lens;
  p->scores = block_scores;
  p->sel = sel;
  p->status = status;
  return MSA_OK;
}
}  // namespace

extern "C" msa_status msa_topk_candidates(const msa_geometry* geo, const msa_batch* batch, const float* block_scores,
                                          int32_t block_begin, int32_t block_end, uint64_t* cand, uint32_t* status,
                                          cudaStream_t stream) {
  CandParams c;
  msa_status st = topk_setup(geo, batch, block_scores, nullptr, status, &c.t);
  if (st != MSA_OK) return st;
  if (block_begin < 0 || block_end < block_begin) return MSA_ERR_INVALID_ARG;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (block_scores == nullptr || cand == nullptr || !aligned(block_scores, 4) || !aligned(cand, 8))
    return MSA_ERR_INVALID_ARG;
  c.kb = block_begin;
  c.ke = block_end;
  c.n_shards = 1;
  c.cand = cand;
  c.cand_in = nullptr;
  k_topk_cand<<<ceil_div(batch->T * 4, kRowsPerCta), 32 * kRowsPerCta, 0, stream>>>(c);
  return launch_status();
}

extern "C" msa_status msa_topk_merge(const msa_geometry* geo, const msa_batch* batch, const uint64_t* cand,
                                     int32_t n_shards, int32_t* sel, uint32_t* status, cudaStream_t stream) {
  CandParams c;
  msa_status st = topk_setup(geo, batch, nullptr, sel, status, &c.t);
  if (st != MSA_OK) return st;
  if (n_shards < 1 || n_shards > 256) return MSA_ERR_INVALID_ARG;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (cand == nullptr || sel == nullptr || !aligned(cand, 8) || !aligned(sel, 4)) return MSA_ERR_INVALID_ARG;
  c.kb = 0;
  c.ke = 0;
  c.n_shards = n_shards;
  c.cand = nullptr;
  c.cand_in = cand;
  k_topk_merge<<<ceil_div(batch->T * 4, kRowsPerCta), 32 * kRowsPerCta, 0, stream>>>(c);
  return launch_status();
}

extern "C" msa_status msa_topk_candidates_host(const float* block_scores, int64_t rows, int32_t max_blocks_per_seq,
                                               const int32_t* local, int32_t block_begin, int32_t block_end,
                                               uint64_t* cand) {
  if (rows < 0 || max_blocks_per_seq < 1 || block_begin < 0 || block_end < block_begin) return MSA_ERR_INVALID_ARG;
  if (rows > 0 && (block_scores == nullptr || local == nullptr || cand == nullptr)) return MSA_ERR_INVALID_ARG;
  std::vector<uint64_t> keys;
  for (int64_t r = 0; r < rows; ++r) {
    keys.clear();
    const int lc = local[r];
    if (lc > max_blocks_per_seq) return MSA_ERR_INVALID_ARG;
    const float* s = block_scores + r * max_blocks_per_seq;
    for (int k = block_begin; k < std::min(block_end, lc); ++k) keys.push_back(score_key(s[k], k));
    host_top15(keys, cand + r * kCand);
  }
  return MSA_OK;
}

extern "C" msa_status msa_topk_merge_host(const uint64_t* cand, int32_t n_shards, int64_t rows, const int32_t* local,
                                          int32_t* sel) {
  if (rows < 0 || n_shards < 1) return MSA_ERR_INVALID_ARG;
  if (rows > 0 && (cand == nullptr || local == nullptr || sel == nullptr)) return MSA_ERR_INVALID_ARG;
  std::vector<uint64_t> keys;
  uint64_t top[kCand];
  for (int64_t r = 0; r < rows; ++r) {
    int32_t* out = sel + r * kSel;
    if (local[r] < 0) {
      for (int i = 0; i < kSel; ++i) out[i] = -1;
      continue;
    }
    keys.clear();
    for (int sh = 0; sh < n_shards; ++sh)
      for (int i = 0; i < kCand; ++i) {
        const uint64_t k = cand[(static_cast<int64_t>(sh) * rows + r) * kCand + i];
        if (k != 0ull) keys.push_back(k);
      }
    host_top15(keys, top);
    out[0] = local[r];
    for (int i = 0; i < kCand; ++i) out[1 + i] = top[i] ? key_id(top[i]) : -1;
  }
  return MSA_OK;
}
