// msa_topk.cu — per-(token, group) block selection of the MSA decode step.
//
// What it computes ("vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", "MSA primer": the top
// 16 blocks with the most recent one always kept; "MiniMax M3 in vLLM ...", "MSA 机制详解":
// init_blocks = 0, local_blocks = 1, a local block that also ranks in the top-k is not counted
// twice): local = p_t / 128 is slot 0, slots 1..15 are the 15 best of blocks 0 .. local-1 in
// descending score order, equal scores ordered by lower block id, -1 when fewer exist.
//
// Design: one warp per (token, group) row. Each score becomes a unique 64-bit key
// (order-preserving fp32 bits << 32 | ~block id), so "descending score, then lower id" is one
// integer order and ties need no special case. Rows of up to 64 candidates are sorted in
// registers (warp bitonic network, two keys per lane). Longer rows are first filtered: the
// 15th largest of the 32 lane maxima is a lower bound of the 15th largest key, so only keys
// at or above it survive (typically a few dozen), and those are sorted. The indexer's scores
// are the only input, so GPU selection == the oracle's sort on the same scores, bit for bit.
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa.h"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

constexpr int kKeysPerLane = 16;

__device__ __forceinline__ uint64_t score_key(float s, int id) {
  uint32_t u = __float_as_uint(s);
  if (s != s) u = 0xFF800000u;   // NaN ranks as -inf
  if (s == 0.0f) u = 0u;         // -0 == +0
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<uint64_t>(ord) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - static_cast<uint32_t>(id));
}

__device__ __forceinline__ int key_id(uint64_t key) {
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

// One warp per (token, group) row. The 15 largest keys are all >= tau, the 15th largest of
// the 32 lane maxima (15 distinct elements reach it); the survivors of that filter (usually
// a few dozen) are sorted in registers. More than 64 survivors (adversarial ties across
// lanes) fall back to repeated warp argmax over the whole row.
__global__ void __launch_bounds__(32 * kRowsPerCta) k_topk(const TopkParams p) {
  __shared__ uint64_t buf[kRowsPerCta][kSurvivors];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kRowsPerCta + warp;  // t * 4 + g
  if (row >= p.T * 4) return;
  const int t = row >> 2;
  int lo = 0, hi = p.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (p.qsl[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int q0 = p.qsl[lo], ql = p.qsl[lo + 1] - q0;
  const int L = p.seq_lens[lo];
  int32_t* out = p.sel + static_cast<int64_t>(row) * kSel;
  if (!(t - q0 < ql && ql <= p.max_q_len && L >= ql && L <= p.maxb * kBS)) {
    if (lane == 0) set_status(p.status, MSA_ERR_INVALID_ARG);
    if (lane < kSel) out[lane] = -1;
    return;
  }
  const int local = (L - ql + (t - q0)) / kBS;
  const int ncand = local;
  const float* s = p.scores + static_cast<int64_t>(row) * p.maxb;
  uint64_t k0 = 0, k1 = 0;
  bool sorted = false;
  if (ncand <= kSurvivors) {
    const int i0 = 2 * lane, i1 = 2 * lane + 1;
    k0 = i0 < ncand ? score_key(s[i0], i0) : 0ull;
    k1 = i1 < ncand ? score_key(s[i1], i1) : 0ull;
    sorted = true;
  } else {
    uint64_t best = 0;
    for (int i = lane; i < ncand; i += 32) {
      const uint64_t k = score_key(s[i], i);
      best = k > best ? k : best;
    }
    const uint64_t tau = __shfl_sync(0xffffffffu, warp_sort32_desc(best, lane), 14);
    int count = 0;
    for (int base = 0; base < ncand; base += 32) {
      const int i = base + lane;
      const uint64_t k = i < ncand ? score_key(s[i], i) : 0ull;
      const bool keep = k >= tau && k != 0ull;
      const uint32_t m = __ballot_sync(0xffffffffu, keep);
      const int pos = count + __popc(m & ((1u << lane) - 1u));
      if (keep && pos < kSurvivors) buf[warp][pos] = k;
      count += __popc(m);
    }
    __syncwarp();
    if (count <= kSurvivors) {
      k0 = 2 * lane < count ? buf[warp][2 * lane] : 0ull;
      k1 = 2 * lane + 1 < count ? buf[warp][2 * lane + 1] : 0ull;
      sorted = true;
    }
  }
  if (sorted) {
    warp_sort64_desc(k0, k1, lane);
    // elements 0..14 of the sorted run: lane l holds 2l and 2l+1
    if (lane == 0) out[0] = local;
    if (2 * lane < 15) out[1 + 2 * lane] = k0 ? key_id(k0) : -1;
    if (2 * lane + 1 < 15) out[2 + 2 * lane] = k1 ? key_id(k1) : -1;
    return;
  }
  // fallback: repeated warp argmax, 16 keys per lane per pass, running top-15 carried
  uint64_t top = 0;
  for (int c0 = 0; c0 < ncand; c0 += 32 * kKeysPerLane) {
    uint64_t keys[kKeysPerLane];
#pragma unroll
    for (int i = 0; i < kKeysPerLane; ++i) {
      const int id = c0 + i * 32 + lane;
      keys[i] = id < ncand ? score_key(s[id], id) : 0ull;
    }
    top = warp_pop15(keys, lane < 15 ? top : 0ull, lane);
  }
  if (lane == 0) out[0] = local;
  if (lane < 15) out[1 + lane] = top ? key_id(top) : -1;
}

}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

extern "C" msa_status msa_topk_blocks(const msa_geometry* geo, const msa_batch* batch, const float* block_scores,
                                      int32_t* sel, uint32_t* status, cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = check_batch(batch)) != MSA_OK) return st;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (block_scores == nullptr || sel == nullptr || !aligned(block_scores, 4) || !aligned(sel, 4))
    return MSA_ERR_INVALID_ARG;
  TopkParams p;
  p.B = batch->B;
  p.T = batch->T;
  p.maxb = batch->max_blocks_per_seq;
  p.max_q_len = batch->max_q_len;
  p.qsl = batch->query_start_loc;
  p.seq_lens = batch->seq_lens;
  p.scores = block_scores;
  p.sel = sel;
  p.status = status;
  k_topk<<<ceil_div(batch->T * 4, kRowsPerCta), 32 * kRowsPerCta, 0, stream>>>(p);
  return launch_status();
}
