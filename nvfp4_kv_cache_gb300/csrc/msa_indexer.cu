// msa_indexer.cu — indexer score + 128-token block max-pool of the MSA decode step.
//
// What it computes ("vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", "MSA primer"; "MiniMax
// M3 in vLLM ...", "解码索引器分数内核" and "解码内核中的推测解码"): for every query token t of every
// sequence and every GQA group g, block_scores[t][g][k] = max over the cache positions j of block
// k with j <= p_t of  index_q[t][g] . ik_fp8[j], where ik_fp8 is the NVFP4 index key dequantised
// to E4M3 ("NVIDIA Blackwell optimizado kernes MSA") — or the FP8 index key as is.
//
// GB300 design:
//  * The whole index cache is streamed once per step (9,216 B per NVFP4 page): the kernel is
//    HBM-bound. One persistent CTA per SM; the flattened (sequence, block) page list is split
//    evenly over CTAs, so ragged batches stay balanced at page granularity.
//  * Warp 0 lane 0 is the producer: one 1-D bulk async copy (cp.async.bulk, 16-B aligned,
//    whole page) per page into a ring of shared-memory stages, completion tracked by an
//    mbarrier transaction count; L2 evict-first since every byte is read once.
//  * Warps 1..8 consume whole pages (8 tiles of 16 tokens): register-direct dequant (LUT in
//    shared memory, one prmt per 4 values) straight into the A fragments of
//    mma.sync.m16n8k32.e4m3 with tokens on M and (query token, group) columns on N — so a
//    page's A fragments are reused by all N tiles — and the block max is kept in registers and
//    finished with three shuffles. No block score ever leaves the SM before it is final.
//  * The head-dim order inside an MMA is free (a dot product does not care) as long as A and B
//    use the same one: thread t of a quad owns dims 32t..32t+31 (two scale groups, 16 code
//    bytes), k-step s covers dims 32t+8s..32t+8s+7, so the dequantised bytes land in the A
//    registers in element order and the B fragment is one 8-byte load of index_q.
//  * Every wait is bounded (MSA_ERR_TIMEOUT) and every page id is checked (MSA_ERR_DEVICE_FAULT,
//    the block is scored -inf); nothing traps.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "msa.h"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

// Stage ring: consumer warp w owns slots w, w + W, ..., w + W*(D-1) and its j-th page lives
// in slot w + W*(j % D). Each slot thus serves one warp, in order, so a warp only ever waits
// for the phase right after the one it consumed itself (an mbarrier's parity cannot tell a
// phase from the one two steps earlier).
template <int DT>
struct IdxCfg;
template <>
struct IdxCfg<MSA_INDEX_NVFP4> {
  static constexpr int kPage = kIdxPageNv;
  static constexpr int kWarps = 8;  // consumer warps
  static constexpr int kDepth = 2;  // pages in flight per consumer warp
  static constexpr int kStages = kWarps * kDepth;
};
template <>
struct IdxCfg<MSA_INDEX_FP8> {
  static constexpr int kPage = kIdxPageFp8;
  static constexpr int kWarps = 6;
  static constexpr int kDepth = 2;
  static constexpr int kStages = kWarps * kDepth;
};
constexpr int kMaxIdxThreads = 32 * (8 + 1);

struct IdxParams {
  int32_t B, T, maxb, max_q_len, num_pages;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_table;
  const uint8_t* index_pages;
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
  static constexpr size_t kStageBytes = static_cast<size_t>(kStages) * kPage;
  static constexpr size_t kOffFull = kStageBytes;
  static constexpr size_t kOffEmpty = kOffFull + 8 * kStages;
  static constexpr size_t kOffInfo = kOffEmpty + 8 * kStages;
  static constexpr size_t kOffLut = kOffInfo + sizeof(SlotInfo) * kStages;
  static constexpr size_t kOffMisc = kOffLut + 256 * 8;
  static constexpr size_t kOffPrefix = kOffMisc + 64;
  static size_t bytes(int B) { return kOffPrefix + 4 * static_cast<size_t>(B + 1); }
};

// Pages of sequence b that the indexer scans (0 for padded or invalid rows).
__device__ __forceinline__ int seq_pages(const IdxParams& p, int b, bool* bad) {
  const int q0 = p.qsl[b], q1 = p.qsl[b + 1];
  const int ql = q1 - q0;
  const int L = p.seq_lens[b];
  if (ql < 0 || ql > p.max_q_len || q0 < 0 || q1 > p.T || (ql > 0 && (L < ql || L > p.maxb * kBS))) {
    *bad = true;
    return 0;
  }
  return ql > 0 ? ceil_div(L, kBS) : 0;
}

// Score one staged page for the N tiles of the current sequence and write its block scores.
// NT = number of 8-column tiles (columns = q_len * 4). MASK: the page holds rows after a query
// position (only the last page or two of a sequence), so rows are masked per column.
template <int DT, int NT, bool MASK>
__device__ __forceinline__ void score_page(const uint8_t* pg, const uint2* lut, const uint32_t (&bfrag)[4][4][2],
                                           int lane, int k, int p0, int ncol, int q0, const IdxParams& p) {
  const int gid = lane >> 2, t = lane & 3;
  float mx[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j) mx[j][0] = mx[j][1] = -CUDART_INF_F;
#pragma unroll 1
  for (int tile = 0; tile < kBS / 16; ++tile) {
    const int r0 = tile * 16 + gid, r1 = r0 + 8;
    uint32_t a[4][4];
    if constexpr (DT == MSA_INDEX_NVFP4) {
      const uint4 c0 = lds128(pg + r0 * kRowCodes + t * 16);
      const uint4 c1 = lds128(pg + r1 * kRowCodes + t * 16);
      const uint32_t s0 = *reinterpret_cast<const uint16_t*>(pg + kScaleOff + r0 * kRowScales + 2 * t);
      const uint32_t s1 = *reinterpret_cast<const uint16_t*>(pg + kScaleOff + r1 * kRowScales + 2 * t);
      const uint2 e00 = lut[s0 & 0xFFu], e01 = lut[s0 >> 8], e10 = lut[s1 & 0xFFu], e11 = lut[s1 >> 8];
      dq8(c0.x, e00, a[0][0], a[0][2]);
      dq8(c1.x, e10, a[0][1], a[0][3]);
      dq8(c0.y, e00, a[1][0], a[1][2]);
      dq8(c1.y, e10, a[1][1], a[1][3]);
      dq8(c0.z, e01, a[2][0], a[2][2]);
      dq8(c1.z, e11, a[2][1], a[2][3]);
      dq8(c0.w, e01, a[3][0], a[3][2]);
      dq8(c1.w, e11, a[3][1], a[3][3]);
    } else {
      // 32 E4M3 bytes per row and thread; the half loaded first alternates with the row
      // parity so the eight rows of a quarter-warp hit distinct banks.
      const int sw = gid & 1;
      const uint4 u0a = lds128(pg + r0 * kD + t * 32 + 16 * sw);
      const uint4 u0b = lds128(pg + r0 * kD + t * 32 + 16 * (1 - sw));
      const uint4 u1a = lds128(pg + r1 * kD + t * 32 + 16 * sw);
      const uint4 u1b = lds128(pg + r1 * kD + t * 32 + 16 * (1 - sw));
      const uint4 u0 = sw ? u0b : u0a, v0 = sw ? u0a : u0b;
      const uint4 u1 = sw ? u1b : u1a, v1 = sw ? u1a : u1b;
      a[0][0] = u0.x; a[0][2] = u0.y; a[1][0] = u0.z; a[1][2] = u0.w;
      a[2][0] = v0.x; a[2][2] = v0.y; a[3][0] = v0.z; a[3][2] = v0.w;
      a[0][1] = u1.x; a[0][3] = u1.y; a[1][1] = u1.z; a[1][3] = u1.w;
      a[2][1] = v1.x; a[2][3] = v1.y; a[3][1] = v1.z; a[3][3] = v1.w;
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      float acc[4];
      mma_e4m3_zc(acc, a[0][0], a[0][1], a[0][2], a[0][3], bfrag[j][0][0], bfrag[j][0][1]);
#pragma unroll
      for (int s = 1; s < 4; ++s) mma_e4m3(acc, a[s][0], a[s][1], a[s][2], a[s][3], bfrag[j][s][0], bfrag[j][s][1]);
      if constexpr (MASK) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = (i < 2) ? r0 : r1;
          const int col = j * 8 + 2 * t + (i & 1);
          const int pos = k * kBS + row;
          if (col >= ncol || pos > p0 + (col >> 2)) acc[i] = -CUDART_INF_F;
        }
      }
      mx[j][0] = fmaxf(mx[j][0], fmaxf(acc[0], acc[2]));
      mx[j][1] = fmaxf(mx[j][1], fmaxf(acc[1], acc[3]));
    }
  }
#pragma unroll
  for (int j = 0; j < NT; ++j) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float v = mx[j][e];
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
      const int col = j * 8 + 2 * t + e;
      if (gid == 0 && col < ncol) p.block_scores[static_cast<int64_t>(q0 * 4 + col) * p.maxb + k] = v;
    }
  }
}

template <int DT, bool MASK>
__device__ __forceinline__ void score_page_nt(int nt, const uint8_t* pg, const uint2* lut,
                                              const uint32_t (&bfrag)[4][4][2], int lane, int k, int p0, int ncol,
                                              int q0, const IdxParams& p) {
  switch (nt) {
    case 1: score_page<DT, 1, MASK>(pg, lut, bfrag, lane, k, p0, ncol, q0, p); break;
    case 2: score_page<DT, 2, MASK>(pg, lut, bfrag, lane, k, p0, ncol, q0, p); break;
    case 3: score_page<DT, 3, MASK>(pg, lut, bfrag, lane, k, p0, ncol, q0, p); break;
    default: score_page<DT, 4, MASK>(pg, lut, bfrag, lane, k, p0, ncol, q0, p); break;
  }
}

template <int DT>
__device__ __forceinline__ void score_page_any(int nt, const uint8_t* pg, const uint2* lut,
                                               const uint32_t (&bfrag)[4][4][2], int lane, int k, int p0, int ncol,
                                               int q0, const IdxParams& p) {
  if ((k + 1) * kBS - 1 > p0)  // some row lies after a query position: mask per column
    score_page_nt<DT, true>(nt, pg, lut, bfrag, lane, k, p0, ncol, q0, p);
  else
    score_page_nt<DT, false>(nt, pg, lut, bfrag, lane, k, p0, ncol, q0, p);
}

template <int DT>
__global__ void __launch_bounds__(kMaxIdxThreads, 1) k_indexer(const IdxParams p) {
  using S = IdxSmem<DT>;
  constexpr int kConsumerWarps = IdxCfg<DT>::kWarps;
  constexpr int kDepth = IdxCfg<DT>::kDepth;
  constexpr int kIdxThreads = 32 * (kConsumerWarps + 1);
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::kOffFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + S::kOffEmpty);
  SlotInfo* info = reinterpret_cast<SlotInfo*>(smem + S::kOffInfo);
  uint2* lut = reinterpret_cast<uint2*>(smem + S::kOffLut);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + S::kOffMisc);
  int* bad_batch = reinterpret_cast<int*>(smem + S::kOffMisc + 4);
  int* prefix = reinterpret_cast<int*>(smem + S::kOffPrefix);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- prologue: barriers, LUT, per-sequence page prefix sums --------------------------
  if (tid == 0) {
    for (int i = 0; i < S::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    fence_mbar_init();
    *abort_flag = 0;
    *bad_batch = 0;
  }
  if constexpr (DT == MSA_INDEX_NVFP4) build_dequant_lut(lut, tid, kIdxThreads);
  {
    // chunked scan: thread i sums sequences [i*per, (i+1)*per), thread 0 scans the partials
    const int per = ceil_div(p.B, kIdxThreads);
    int local = 0;
    bool bad = false;
    for (int b = tid * per; b < min(p.B, (tid + 1) * per); ++b) local += seq_pages(p, b, &bad);
    if (bad) *bad_batch = 1;
    __shared__ int partial[kMaxIdxThreads + 1];
    partial[tid] = local;
    __syncthreads();
    if (tid == 0) {
      int run = 0;
      for (int i = 0; i < kIdxThreads; ++i) {
        const int v = partial[i];
        partial[i] = run;
        run += v;
      }
      partial[kIdxThreads] = run;
    }
    __syncthreads();
    int run = partial[tid];
    for (int b = tid * per; b < min(p.B, (tid + 1) * per); ++b) {
      prefix[b] = run;
      bool dummy = false;
      run += seq_pages(p, b, &dummy);
    }
    if (tid == 0) prefix[p.B] = partial[kIdxThreads];
    if (p.qsl != nullptr && tid == 0 && p.B > 0 && (p.qsl[0] != 0 || p.qsl[p.B] != p.T)) *bad_batch = 1;
  }
  __syncthreads();
  if (blockIdx.x == 0 && tid == 0 && *bad_batch) set_status(p.status, MSA_ERR_INVALID_ARG);

  const int total = prefix[p.B];
  const int start = static_cast<int>((static_cast<int64_t>(total) * blockIdx.x) / gridDim.x);
  const int end = static_cast<int>((static_cast<int64_t>(total) * (blockIdx.x + 1)) / gridDim.x);
  const int npages = end - start;

  if (warp == 0) {
    // ---- producer ----------------------------------------------------------------------
    if (lane == 0 && npages > 0) {
      const uint64_t policy = policy_evict_first();
      // locate the sequence of the first page
      int lo = 0, hi = p.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= start) lo = mid; else hi = mid - 1;
      }
      int b = lo;
      int issued = 0;
      for (int n = 0; n < npages; ++n) {
        const int gp = start + n;
        while (prefix[b + 1] <= gp) ++b;
        const int k = gp - prefix[b];
        const int j = n / kConsumerWarps;  // the consumer's j-th page
        const int slot = (n % kConsumerWarps) + kConsumerWarps * (j % kDepth);
        const uint32_t ph = static_cast<uint32_t>(j / kDepth) & 1u;
        if (!mbar_wait_bounded(&empty[slot], ph ^ 1u, kWaitLimitNs, abort_flag)) {
          if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
          *abort_flag = 1;
          break;
        }
        const int phys = p.block_table[static_cast<int64_t>(b) * p.maxb + k];
        const bool valid = phys >= 0 && phys < p.num_pages;
        info[slot].b = b;
        info[slot].k = k;
        info[slot].valid = valid ? 1 : 0;
        if (valid) {
          mbar_arrive_expect_tx(&full[slot], S::kPage);
          bulk_g2s_stream(stages + static_cast<size_t>(slot) * S::kPage,
                          p.index_pages + static_cast<int64_t>(phys) * S::kPage, S::kPage, &full[slot], policy);
        } else {
          set_status(p.status, MSA_ERR_DEVICE_FAULT);
          mbar_arrive(&full[slot]);
        }
        issued = n + 1;
      }
      // Never leave while a copy into this CTA's shared memory may still be in flight: wait
      // for the last page issued into every slot (in a normal run they have all landed).
      const int first = issued > S::kStages ? issued - S::kStages : 0;
      for (int n = first; n < issued; ++n) {
        const int j = n / kConsumerWarps;
        const int slot = (n % kConsumerWarps) + kConsumerWarps * (j % kDepth);
        if (!mbar_wait_bounded(&full[slot], static_cast<uint32_t>(j / kDepth) & 1u, kWaitLimitNs, nullptr)) {
          set_status(p.status, MSA_ERR_TIMEOUT);
        }
      }
    }
    return;
  }

  // ---- consumers ---------------------------------------------------------------------
  const int cw = warp - 1;
  uint32_t bfrag[4][4][2];
  int cur_b = -1, q0 = 0, ncol = 0, nt = 0, p0 = 0;
  for (int n = cw; n < npages; n += kConsumerWarps) {
    const int j = n / kConsumerWarps;
    const int slot = cw + kConsumerWarps * (j % kDepth);
    const uint32_t ph = static_cast<uint32_t>(j / kDepth) & 1u;
    if (!mbar_wait_bounded(&full[slot], ph, kWaitLimitNs, abort_flag)) {
      if (lane == 0) {
        if (!*abort_flag) set_status(p.status, MSA_ERR_TIMEOUT);
        *abort_flag = 1;
      }
      break;
    }
    const SlotInfo si = info[slot];
    if (si.b != cur_b) {
      cur_b = si.b;
      q0 = p.qsl[cur_b];
      const int ql = p.qsl[cur_b + 1] - q0;
      p0 = p.seq_lens[cur_b] - ql;
      ncol = ql * 4;
      nt = ceil_div(ncol, 8);
      const int gid = lane >> 2, t = lane & 3;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int col = j * 8 + gid;
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          uint2 v = make_uint2(0u, 0u);
          if (col < ncol) v = ldg_nc64(p.index_q + static_cast<int64_t>(q0 * 4 + col) * kD + 32 * t + 8 * s);
          bfrag[j][s][0] = v.x;
          bfrag[j][s][1] = v.y;
        }
      }
    }
    const uint8_t* pg = stages + static_cast<size_t>(slot) * S::kPage;
    if (si.valid) {
      score_page_any<DT>(nt, pg, lut, bfrag, lane, si.k, p0, ncol, q0, p);
    } else if (lane < ncol) {
      p.block_scores[static_cast<int64_t>(q0 * 4 + lane) * p.maxb + si.k] = -CUDART_INF_F;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
}

}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

extern "C" msa_status msa_indexer_decode(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                         const uint8_t* index_q, float* block_scores, uint32_t* status,
                                         cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = check_batch(batch)) != MSA_OK) return st;
  if ((st = check_cache(cache, true, false)) != MSA_OK) return st;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (index_q == nullptr || block_scores == nullptr || !aligned(index_q, 16) || !aligned(block_scores, 4))
    return MSA_ERR_INVALID_ARG;
  const int sms = num_sms();
  if (sms <= 0) return MSA_ERR_CUDA;
  IdxParams p;
  p.B = batch->B;
  p.T = batch->T;
  p.maxb = batch->max_blocks_per_seq;
  p.max_q_len = batch->max_q_len;
  p.num_pages = cache->num_pages;
  p.qsl = batch->query_start_loc;
  p.seq_lens = batch->seq_lens;
  p.block_table = batch->block_table;
  p.index_pages = cache->index_pages;
  p.index_q = index_q;
  p.block_scores = block_scores;
  p.status = status;
  if (cache->index_dtype == MSA_INDEX_NVFP4) {
    const size_t smem = IdxSmem<MSA_INDEX_NVFP4>::bytes(p.B);
    if (cudaFuncSetAttribute(k_indexer<MSA_INDEX_NVFP4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MSA_ERR_CUDA;
    k_indexer<MSA_INDEX_NVFP4><<<sms, 32 * (IdxCfg<MSA_INDEX_NVFP4>::kWarps + 1), smem, stream>>>(p);
  } else {
    const size_t smem = IdxSmem<MSA_INDEX_FP8>::bytes(p.B);
    if (cudaFuncSetAttribute(k_indexer<MSA_INDEX_FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return MSA_ERR_CUDA;
    k_indexer<MSA_INDEX_FP8><<<sms, 32 * (IdxCfg<MSA_INDEX_FP8>::kWarps + 1), smem, stream>>>(p);
  }
  return launch_status();
}
