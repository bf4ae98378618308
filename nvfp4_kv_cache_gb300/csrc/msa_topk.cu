// msa_topk.cu — per-(token, group) block selection of the MSA decode step.
//
// What it computes ("vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", "MSA primer": the top
// 16 blocks with the most recent one always kept; "MiniMax M3 in vLLM ...", "MSA 机制详解":
// init_blocks = 0, local_blocks = 1, a local block that also ranks in the top-k is not counted
// twice): local = p_t / 128 is slot 0, slots 1..15 are the 15 best of blocks 0 .. local-1 in
// descending score order, equal scores ordered by lower block id, -1 when fewer exist.
//
// Design: one CTA (8 warps) per (token, group) row. Each score becomes a unique 64-bit key
// (order-preserving fp32 bits << 32 | ~block id), so "descending score, then lower id" is one
// integer order and ties need no special case. Each warp pops its 15 largest keys by
// repeated warp argmax over its slice (16 keys per lane per pass, the running top-15 carried
// in lanes 0..14); warp 0 then merges the 8 x 15 candidates the same way. The indexer's
// scores are the only input, so GPU selection == the oracle's sort on the same scores, bit
// for bit.
#include <cuda_runtime.h>
#include <stdint.h>

#include "msa.h"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

constexpr int kTopkWarps = 8;
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
  int32_t B, T, maxb;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const float* scores;
  int32_t* sel;
  uint32_t* status;
};

__global__ void __launch_bounds__(32 * kTopkWarps) k_topk(const TopkParams p) {
  __shared__ uint64_t cand[kTopkWarps][16];
  __shared__ int info[2];
  const int row = blockIdx.x;  // t * 4 + g
  const int t = row >> 2;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    // the sequence of token t: largest b with qsl[b] <= t
    int lo = 0, hi = p.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (p.qsl[mid] <= t) lo = mid; else hi = mid - 1;
    }
    const int q0 = p.qsl[lo], ql = p.qsl[lo + 1] - q0;
    const int L = p.seq_lens[lo];
    int local = -1, ncand = 0;
    if (t - q0 < ql && L >= ql && L <= p.maxb * kBS) {
      const int pos = L - ql + (t - q0);
      local = pos / kBS;
      ncand = local;
    } else {
      set_status(p.status, MSA_ERR_INVALID_ARG);
    }
    info[0] = local;
    info[1] = ncand;
  }
  __syncthreads();
  const int local = info[0], ncand = info[1];
  if (local < 0) {
    if (tid < kSel) p.sel[static_cast<int64_t>(row) * kSel + tid] = -1;
    return;
  }
  const float* s = p.scores + static_cast<int64_t>(row) * p.maxb;
  // slice of this warp: [w * per, min((w+1) * per, ncand)), per a multiple of 32
  const int per = ceil_div(ceil_div(ncand, kTopkWarps), 32) * 32;
  const int begin = warp * per, end = min(ncand, begin + per);
  uint64_t top = 0;
  for (int c0 = begin; c0 < end; c0 += 32 * kKeysPerLane) {
    uint64_t keys[kKeysPerLane];
#pragma unroll
    for (int i = 0; i < kKeysPerLane; ++i) {
      const int id = c0 + i * 32 + lane;
      keys[i] = id < end ? score_key(s[id], id) : 0ull;
    }
    top = warp_pop15(keys, lane < 15 ? top : 0ull, lane);
  }
  if (lane < 15) cand[warp][lane] = top;
  __syncthreads();
  if (warp == 0) {
    uint64_t keys[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = i * 32 + lane;  // 0 .. 127 over 8 x 16 slots
      const int w = idx >> 4, e = idx & 15;
      keys[i] = (w < kTopkWarps && e < 15) ? cand[w][e] : 0ull;
    }
    const uint64_t best = warp_pop15(keys, 0ull, lane);
    int32_t* out = p.sel + static_cast<int64_t>(row) * kSel;
    if (lane == 0) out[0] = local;
    if (lane < 15) out[1 + lane] = best ? key_id(best) : -1;
  }
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
  p.qsl = batch->query_start_loc;
  p.seq_lens = batch->seq_lens;
  p.scores = block_scores;
  p.sel = sel;
  p.status = status;
  k_topk<<<batch->T * 4, 32 * kTopkWarps, 0, stream>>>(p);
  return launch_status();
}
