// msa_prefill.cu — the many-query (prefill) sparse attention: block-major, with a key -> query
// map and a log-sum-exp merge.
//
// What it computes: the same exact sparse GQA attention as msa_sparse_attn_decode ("vLLM ofrece
// soporte en día 0 para MiniMax-M3.1-Flash", "MSA primer": every query head of a group attends
// over its token's selected blocks; "MSA 机制详解": keys after the query position are masked),
// for any number of query tokens per sequence. The pages' prefill kernel is block-major ("MiniMax
// M3 in vLLM ...", "预填充": a block's keys are read and dequantised once for all the queries that
// selected it, through a key-block -> query map, and each query's per-block results are merged
// by log-sum-exp); so is this one:
//  1. k_map_count / k_map_scan / k_map_fill: the CSR map from every (sequence, group, block) to
//     the (token, slot) entries that selected it (a token's repeated block counts once; an
//     out-of-range block or a bad page marks the (token, group) bad);
//  2. k_prefill_attn: one CTA of 8 warps per (sequence, group, block) with entries: one 3-D
//     tensor copy of the block's K and V regions, the K rows dequantised to an E4M3 tile and
//     the V rows to an f16 tile (shared memory, swizzled) once, then each warp takes entries:
//     the 16 heads of the entry's token attend over the block's 128 keys (mma.sync e4m3 QK^T,
//     online softmax, mma.sync f16 PV) and the (lse, o) partial goes to the entry's slot (o
//     normalised, in f16: half the partial traffic of fp32);
//  3. k_prefill_merge: per (token, group), the log-sum-exp merge of its up to 16 partials.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "msa.h"
#include "msa_attn_tile.cuh"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

constexpr int kPfWarps = 8;
constexpr int kPfThreads = 32 * kPfWarps;
constexpr int kStage = 2 * kRegion;   // K region then V region of one (page, group)
constexpr int kKTile = kBS * kD;      // 128 keys x 128 E4M3
constexpr int kVTile = kBS * kD * 2;  // 128 keys x 128 f16
constexpr int kMaxQ = 1 << 20;        // query tokens per sequence
constexpr int kMaxT = 1 << 22;        // query tokens per call (entries pack t << 4 | slot)

struct PfParams {
  int32_t B, T, maxb, num_pages;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_table;
  const uint8_t* q;
  const int32_t* sel;
  float scale_log2;
  uint16_t* out;
  // workspace
  int32_t* count;    // [B * 4 * maxb] entries of each (sequence, group, block); then fill cursors
  int32_t* offset;   // [B * 4 * maxb + 1] exclusive prefix of count
  int32_t* entries;  // [T * 4 * 16] t << 4 | slot, grouped by (sequence, group, block)
  int32_t* tg_bad;   // [T * 4] the (token, group) saw a bad selection or page: zero output
  uint32_t* part_o;  // [T * 4 * 16 slots][16 heads][64] normalised partial outputs, f16 pairs
  float* part_lse;   // [T * 4 * 16 slots][16 heads] their log2-sum-exp (-inf: no partial)
  uint32_t* status;
};

struct PfSmem {
  static constexpr size_t kOffStage = 0;
  static constexpr size_t kOffK = kOffStage + kStage;   // 18,432 = 18 x 1024
  static constexpr size_t kOffV = kOffK + kKTile;
  static constexpr size_t kOffLut = kOffV + kVTile;
  static constexpr size_t kOffBar = kOffLut + 256 * 8;
  static constexpr size_t kOffMisc = kOffBar + 16;
  static constexpr size_t kBytes = 1024 + kOffMisc + 16;
};
static_assert(PfSmem::kOffK % 1024 == 0, "the stage is 1024-B aligned for the swizzled copy");

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

// One thread per (token, group, slot): count the first occurrence of each valid selected block.
// A partial slot starts as "none" (lse -inf); k_prefill_attn overwrites the slots it serves.
__global__ void __launch_bounds__(256) k_map_count(const PfParams p) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(p.T) * 4 * kSel) return;
  const int t = static_cast<int>(e / (4 * kSel)), g = static_cast<int>((e / kSel) % 4), slot = static_cast<int>(e % kSel);
  float* lse = p.part_lse + e * kHPG;
#pragma unroll
  for (int h = 0; h < kHPG; ++h) lse[h] = -CUDART_INF_F;
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
  atomicAdd(&p.count[(static_cast<int64_t>(b) * 4 + g) * p.maxb + v], 1);
}

// Exclusive scan of count into offset (one CTA of 1024 threads, each a contiguous run), then
// count := 0 so that k_map_fill can use it as the rows' cursors.
__global__ void __launch_bounds__(1024) k_map_scan(const PfParams p, int64_t rows) {
  __shared__ int64_t part[1024];
  const int tid = threadIdx.x;
  const int64_t per = (rows + 1023) / 1024, r0 = tid * per, r1 = rows < r0 + per ? rows : r0 + per;
  int64_t sum = 0;
  for (int64_t r = r0; r < r1; ++r) sum += p.count[r];
  part[tid] = sum;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {  // inclusive Hillis-Steele scan of the 1024 run totals
    const int64_t v = tid >= o ? part[tid - o] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int64_t run = part[tid] - sum;
  for (int64_t r = r0; r < r1; ++r) {
    const int c = p.count[r];
    p.offset[r] = static_cast<int32_t>(run);
    run += c;
    p.count[r] = 0;
  }
  if (tid == 1023) p.offset[rows] = static_cast<int32_t>(part[1023]);
}

// The same threads as k_map_count place their entry in its row.
__global__ void __launch_bounds__(256) k_map_fill(const PfParams p) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(p.T) * 4 * kSel) return;
  const int t = static_cast<int>(e / (4 * kSel)), g = static_cast<int>((e / kSel) % 4), slot = static_cast<int>(e % kSel);
  int b, p_tok, nb;
  if (!token_seq(p, t, &b, &p_tok, &nb)) return;
  const int32_t* row = p.sel + (static_cast<int64_t>(t) * 4 + g) * kSel;
  const int v = row[slot];
  if (v < 0 || v >= nb) return;
  for (int j = 0; j < slot; ++j)
    if (row[j] == v) return;
  const int ph = p.block_table[static_cast<int64_t>(b) * p.maxb + v];
  if (!(ph >= 0 && ph < p.num_pages)) return;
  const int64_t r = (static_cast<int64_t>(b) * 4 + g) * p.maxb + v;
  const int pos = atomicAdd(&p.count[r], 1);
  p.entries[p.offset[r] + pos] = (t << 4) | slot;
}

// One CTA per (sequence, group, block) row of the map.
__global__ void __launch_bounds__(kPfThreads) k_prefill_attn(const PfParams p, const __grid_constant__ CUtensorMap tmap) {
  using S = PfSmem;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  const int64_t r = blockIdx.x;
  const int e0 = p.offset[r], n = p.offset[r + 1] - e0;
  if (n == 0) return;
  const int v = static_cast<int>(r % p.maxb);
  const int g = static_cast<int>((r / p.maxb) % 4);
  const int b = static_cast<int>(r / (4 * static_cast<int64_t>(p.maxb)));
  const int ph = p.block_table[static_cast<int64_t>(b) * p.maxb + v];  // checked by k_map_count
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + S::kOffBar);
  volatile int* fail = reinterpret_cast<volatile int*>(smem + S::kOffMisc);
  uint2* lut = reinterpret_cast<uint2*>(smem + S::kOffLut);
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    *fail = 0;
    mbar_arrive_expect_tx(bar, kStage);
    tma_load_3d(smem + S::kOffStage, &tmap, 0, 2 * g * (kRegion / kD), ph, bar);
  }
  build_dequant_lut(lut, tid, kPfThreads);
  __syncthreads();
  // thread = key row: K rows (threads 0..127) -> E4M3 tile, V rows (128..255) -> f16 tile
  const bool ok_copy = mbar_wait(bar, 0u, nullptr);
  if (!ok_copy) *fail = 1;
  if (ok_copy) {
    const int kr = tid & 127;
    RawRow raw;
    if (tid < 128) {
      load_row(smem + S::kOffStage, kr, raw);
      uint8_t* kt = smem + S::kOffK;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[8];
        dequant_quarter(raw, q, lut, w);
        *reinterpret_cast<uint4*>(kt + kr * kD + (((2 * q) ^ (kr & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(kt + kr * kD + (((2 * q + 1) ^ (kr & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
      }
    } else {
      load_row(smem + S::kOffStage + kRegion, kr, raw);
      uint8_t* vt = smem + S::kOffV;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t w[8];
        dequant_quarter(raw, q, lut, w);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const uint4 x = make_uint4(cvt_f16x2_e4m3x2(w[2 * h]), cvt_f16x2_e4m3x2(w[2 * h] >> 16),
                                     cvt_f16x2_e4m3x2(w[2 * h + 1]), cvt_f16x2_e4m3x2(w[2 * h + 1] >> 16));
          *reinterpret_cast<uint4*>(vt + kr * (2 * kD) + (((4 * q + h) ^ (kr & 7)) << 4)) = x;
        }
      }
    }
  }
  __syncthreads();
  if (*fail) {
    if (tid == 0) set_status(p.status, MSA_ERR_TIMEOUT);
    return;
  }
  const int gid = lane >> 2, tq = lane & 3;
  const int q0 = p.qsl[b], ql = p.qsl[b + 1] - q0, L = p.seq_lens[b];
  for (int e = warp; e < n; e += kPfWarps) {
    const int ent = p.entries[e0 + e];
    const int t = ent >> 4, slot = ent & 15;
    const int p_tok = L - ql + (t - q0);
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
      for (int s = 0; s < 4; ++s) {
        qa[s][0] = ldg_nc32(qrow0 + 32 * s);
        qa[s][1] = ldg_nc32(qrow1 + 32 * s);
        qa[s][2] = ldg_nc32(qrow0 + 32 * s + 16);
        qa[s][3] = ldg_nc32(qrow1 + 32 * s + 16);
      }
    }
    attend_tile(st, qa, smem + S::kOffK, smem + S::kOffV, v * kBS, p_tok, p.scale_log2, 0, 4, lane);
    // the partial of (t, g, slot): o / l per head and log2(sum) + m
    const float l0 = quad_sum(st.l[0]), l1 = quad_sum(st.l[1]);
    const int64_t base = (static_cast<int64_t>(t) * 4 + g) * kSel + slot;
    uint32_t* po = p.part_o + base * kHPG * (kD / 2);  // f16 pairs: dims 2c, 2c + 1 in word c
    const float i0 = l0 > 0.f ? 1.f / l0 : 0.f, i1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      po[gid * (kD / 2) + 4 * k + tq] = pack_f16x2(st.o[k][0] * i0, st.o[k][1] * i0);
      po[(gid + 8) * (kD / 2) + 4 * k + tq] = pack_f16x2(st.o[k][2] * i1, st.o[k][3] * i1);
    }
    if (tq == 0) {
      p.part_lse[base * kHPG + gid] = l0 > 0.f ? st.m[0] + __log2f(l0) : -CUDART_INF_F;
      p.part_lse[base * kHPG + gid + 8] = l1 > 0.f ? st.m[1] + __log2f(l1) : -CUDART_INF_F;
    }
  }
}

// One warp per (token, head): out = sum_s 2^(lse_s - M) o_s / sum_s 2^(lse_s - M) over the
// token's partials; zero when the (token, group) is bad or has none.
__global__ void __launch_bounds__(256) k_prefill_merge(const PfParams p) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);  // t * 64 + h
  const int lane = threadIdx.x & 31;
  if (row >= static_cast<int64_t>(p.T) * kQHeads) return;
  const int t = static_cast<int>(row / kQHeads), h = static_cast<int>(row % kQHeads), g = h / kHPG, hh = h % kHPG;
  const int64_t base = (static_cast<int64_t>(t) * 4 + g) * kSel;
  float M = -CUDART_INF_F;
  for (int s = 0; s < kSel; ++s) M = fmaxf(M, p.part_lse[(base + s) * kHPG + hh]);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float W = 0.f;
  if (M != -CUDART_INF_F && !p.tg_bad[t * 4 + g]) {
    for (int s = 0; s < kSel; ++s) {
      const float lse = p.part_lse[(base + s) * kHPG + hh];
      if (lse == -CUDART_INF_F) continue;
      const float w = fast_exp2(lse - M);
      const uint2 ov = *reinterpret_cast<const uint2*>(p.part_o + ((base + s) * kHPG + hh) * (kD / 2) + 2 * lane);
      const float2 o01 = __half22float2(*reinterpret_cast<const __half2*>(&ov.x));
      const float2 o23 = __half22float2(*reinterpret_cast<const __half2*>(&ov.y));
      acc.x += w * o01.x;
      acc.y += w * o01.y;
      acc.z += w * o23.x;
      acc.w += w * o23.y;
      W += w;
    }
  }
  const float inv = W > 0.f ? 1.0f / W : 0.f;
  *reinterpret_cast<uint2*>(p.out + row * kD + 4 * lane) =
      make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv), pack_bf16x2(acc.z * inv, acc.w * inv));
}

struct PfLayout {
  size_t count, offset, entries, tg_bad, part_o, part_lse, total;
};

PfLayout pf_layout(int B, int T, int maxb) {
  using msa_host::align256;
  PfLayout l;
  const size_t rows = static_cast<size_t>(B) * 4 * maxb;
  const size_t ent = static_cast<size_t>(T) * 4 * kSel;
  l.count = 0;
  l.offset = l.count + align256(rows * 4);
  l.entries = l.offset + align256((rows + 1) * 4);
  l.tg_bad = l.entries + align256(ent * 4);
  l.part_o = l.tg_bad + align256(static_cast<size_t>(T) * 4 * 4);
  l.part_lse = l.part_o + align256(ent * kHPG * kD * 2);
  l.total = l.part_lse + align256(ent * kHPG * 4);
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
  return pf_layout(B, T, max_blocks_per_seq).total;
}

extern "C" msa_status msa_prefill_attn(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                       const uint8_t* q, const int32_t* sel, float softmax_scale, void* workspace,
                                       size_t workspace_bytes, uint16_t* out, uint32_t* status, cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if (batch == nullptr) return MSA_ERR_INVALID_ARG;
  // a prefill batch: any number of query tokens per sequence (max_q_len up to 2^20)
  if (batch->B < 0 || batch->T < 0 || batch->B > kMaxB || batch->T > kMaxT) return MSA_ERR_INVALID_ARG;
  if (batch->max_q_len < 1 || batch->max_q_len > kMaxQ) return MSA_ERR_INVALID_ARG;
  if (batch->max_blocks_per_seq < 1 || batch->max_blocks_per_seq > (1 << 20)) return MSA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch->B) * batch->max_blocks_per_seq * 4 > (int64_t{1} << 31) - 2) return MSA_ERR_UNSUPPORTED;
  if (batch->B > 0 && (batch->query_start_loc == nullptr || batch->seq_lens == nullptr || batch->block_table == nullptr))
    return MSA_ERR_INVALID_ARG;
  if ((st = check_cache(cache, false, true)) != MSA_OK) return st;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  if (q == nullptr || sel == nullptr || out == nullptr || !aligned(q, 16) || !aligned(sel, 4) || !aligned(out, 16))
    return MSA_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || softmax_scale != softmax_scale) return MSA_ERR_INVALID_ARG;
  const PfLayout lay = pf_layout(batch->B, batch->T, batch->max_blocks_per_seq);
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
  p.q = q;
  p.sel = sel;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  p.out = out;
  p.count = reinterpret_cast<int32_t*>(ws + lay.count);
  p.offset = reinterpret_cast<int32_t*>(ws + lay.offset);
  p.entries = reinterpret_cast<int32_t*>(ws + lay.entries);
  p.tg_bad = reinterpret_cast<int32_t*>(ws + lay.tg_bad);
  p.part_o = reinterpret_cast<uint32_t*>(ws + lay.part_o);
  p.part_lse = reinterpret_cast<float*>(ws + lay.part_lse);
  p.status = status;
  const int64_t rows = static_cast<int64_t>(p.B) * 4 * p.maxb;
  if (cudaMemsetAsync(p.count, 0, static_cast<size_t>(rows) * 4, stream) != cudaSuccess ||
      cudaMemsetAsync(p.tg_bad, 0, static_cast<size_t>(p.T) * 16, stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  const int64_t ent = static_cast<int64_t>(p.T) * 4 * kSel;
  const int eb = static_cast<int>((ent + 255) / 256);
  k_map_count<<<eb, 256, 0, stream>>>(p);
  k_map_scan<<<1, 1024, 0, stream>>>(p, rows);
  k_map_fill<<<eb, 256, 0, stream>>>(p);
  if ((st = launch_status()) != MSA_OK) return st;
  alignas(64) CUtensorMap tmap;
  if (!kv_tensor_map(&tmap, cache->kv_pages, static_cast<uint64_t>(cache->num_pages > 0 ? cache->num_pages : 1)))
    return MSA_ERR_CUDA;
  if (cudaFuncSetAttribute(k_prefill_attn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(PfSmem::kBytes)) !=
      cudaSuccess)
    return MSA_ERR_CUDA;
  if (rows > 0x7FFFFFFF) return MSA_ERR_UNSUPPORTED;
  k_prefill_attn<<<static_cast<unsigned>(rows), kPfThreads, PfSmem::kBytes, stream>>>(p, tmap);
  k_prefill_merge<<<static_cast<unsigned>((static_cast<int64_t>(p.T) * kQHeads + 7) / 8), 256, 0, stream>>>(p);
  return launch_status();
}
