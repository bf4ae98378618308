// msa_host.h — host-side helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "msa.h"

namespace msa_host {

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Status of the launches issued since the last check.
inline msa_status launch_status() {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

// Launch `kernel` so that it may start while the kernel before it on `stream` finishes
// (programmatic dependent launch): the kernel must call grid_dependency_wait() before it reads
// anything the previous kernel writes, and must not write what the previous kernel reads.
// After anything but a kernel on the stream the launch is ordered as usual.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_after_previous(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                         cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

inline msa_status check_geometry(const msa_geometry* g) {
  if (g == nullptr) return MSA_ERR_INVALID_ARG;
  if (g->num_q_heads != 64 || g->num_kv_heads != 4 || g->head_dim != 128 || g->index_dim != 128 ||
      g->block_size != 128 || g->topk != 16 || g->local_blocks != 1 || g->init_blocks != 0)
    return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

inline msa_status check_batch(const msa_batch* b) {
  if (b == nullptr) return MSA_ERR_INVALID_ARG;
  if (b->B < 0 || b->T < 0 || b->B > 4096) return MSA_ERR_INVALID_ARG;
  if (b->max_q_len < 1 || b->max_q_len > 8) return MSA_ERR_INVALID_ARG;
  if (b->max_blocks_per_seq < 1 || b->max_blocks_per_seq > (1 << 20)) return MSA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(b->T) > static_cast<int64_t>(b->B) * b->max_q_len) return MSA_ERR_INVALID_ARG;
  if (b->B > 0 && (b->query_start_loc == nullptr || b->seq_lens == nullptr || b->block_table == nullptr))
    return MSA_ERR_INVALID_ARG;
  if (!aligned(b->query_start_loc, 4) || !aligned(b->seq_lens, 4) || !aligned(b->block_table, 4))
    return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

// A prefill / many-query batch: any number of query tokens per sequence (max_q_len up to 2^20),
// up to 2^22 in all (T); the rest as check_batch.
inline msa_status check_prefill_batch(const msa_batch* b) {
  if (b == nullptr) return MSA_ERR_INVALID_ARG;
  if (b->B < 0 || b->T < 0 || b->B > 4096 || b->T > (1 << 22)) return MSA_ERR_INVALID_ARG;
  if (b->max_q_len < 1 || b->max_q_len > (1 << 20)) return MSA_ERR_INVALID_ARG;
  if (b->max_blocks_per_seq < 1 || b->max_blocks_per_seq > (1 << 20)) return MSA_ERR_INVALID_ARG;
  if (b->B > 0 && (b->query_start_loc == nullptr || b->seq_lens == nullptr || b->block_table == nullptr))
    return MSA_ERR_INVALID_ARG;
  if (!aligned(b->query_start_loc, 4) || !aligned(b->seq_lens, 4) || !aligned(b->block_table, 4))
    return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

inline msa_status check_cache(const msa_cache* c, bool need_index, bool need_kv) {
  if (c == nullptr) return MSA_ERR_INVALID_ARG;
  if (c->num_pages < 0) return MSA_ERR_INVALID_ARG;
  if (c->index_dtype != MSA_INDEX_NVFP4 && c->index_dtype != MSA_INDEX_FP8) return MSA_ERR_UNSUPPORTED;
  if (need_index && (c->index_pages == nullptr || !aligned(c->index_pages, 256))) return MSA_ERR_INVALID_ARG;
  if (need_kv && (c->kv_pages == nullptr || !aligned(c->kv_pages, 256))) return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

inline int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// The SM count the automatic choices below are tuned for: a GB300's 152. They are taken from
// the arguments alone, not from the device, so that workspace sizes are a pure function of the
// arguments; on a part with another SM count they still give correct results, only tuned for
// the wrong machine.
constexpr int kTunedSms = 152;

// Splits of each (query token, group)'s selected blocks: as many as keep the T x 4 x splits
// CTAs (one per SM) within one wave of kTunedSms SMs, at least 1, at most 16.
inline int auto_splits(int T) {
  const int items = 4 * T;
  if (items <= 0) return 1;
  const int s = kTunedSms / items;
  return s < 1 ? 1 : (s > 16 ? 16 : s);
}

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// A 2-D tensor map (CUtensorMap, 64-B aligned storage) over `rows` rows of 128 bytes at `base`
// (16-B aligned), box = `box_rows` rows, 128-byte swizzle (defined in msa_api.cu).
bool rows128_tensor_map(void* tmap64, const uint8_t* base, uint64_t rows, uint32_t box_rows);

// A 3-D tensor map over a KV page pool: (128 B, 576 rows, num_pages pages), box = the 144 rows
// of one head's K and V regions of one page, 128-byte swizzle (defined in msa_api.cu).
bool kv_tensor_map(void* tmap64, const uint8_t* base, uint64_t num_pages);

}  // namespace msa_host

// Launchers implemented in the kernel translation units.
msa_status msa_launch_attn_merge(const float* part_o, const float* part_lse, int32_t splits, int32_t T,
                                 uint16_t* out, cudaStream_t stream);

// The attention of the tokens [t0, t1) of the batch alone (msa_attn.cu): only for batches the
// many-token kernel takes with one split; MSA_ERR_INVALID_ARG otherwise.
msa_status msa_attn_token_range(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                const uint8_t* q, const int32_t* sel, float softmax_scale, uint16_t* out,
                                uint32_t* status, int32_t t0, int32_t t1, cudaStream_t stream);

// The token at which the host-buffer step splits the attention into two launches (0 = one).
int32_t msa_attn_split_token(int32_t T);
