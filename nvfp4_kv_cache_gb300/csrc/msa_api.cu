// msa_api.cu — the fused decode step, workspace sizing, device status and self-test entry
// points of the C ABI (include/msa.h).
//
// msa_decode_step runs the three stages of the MSA decode step ("vLLM ofrece soporte en día 0
// para MiniMax-M3.1-Flash", "MSA primer"; "MiniMax M3 in vLLM ...", "解码执行": score the
// candidate blocks, apply the local window, select the top blocks, run sparse GQA decode and
// merge split partial outputs) on one stream, with every intermediate in the caller's
// workspace and launch shapes that depend only on the integer arguments (CUDA-graph safe,
// "解码内核中的推测解码").
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "msa.h"
#include "msa_device.cuh"
#include "msa_host.h"

namespace msa {
namespace {

// cuTensorMapEncodeTiled, fetched from the driver once per process.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace
}  // namespace msa

namespace msa_host {
bool rows128_tensor_map(void* tmap64, const uint8_t* base, uint64_t rows, uint32_t box_rows) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = msa::tensor_map_encoder();
  if (enc == nullptr || rows == 0 || rows > (1ull << 32) || box_rows == 0 || box_rows > 256) return false;
  const cuuint64_t dims[2] = {128, rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(static_cast<CUtensorMap*>(tmap64), CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool kv_tensor_map(void* tmap64, const uint8_t* base, uint64_t num_pages) {
  const PFN_cuTensorMapEncodeTiled_v12000 enc = msa::tensor_map_encoder();
  if (enc == nullptr || num_pages == 0 || num_pages > (1ull << 31)) return false;
  constexpr uint64_t kRowsPerPage = msa::kKvPage / 128;  // 576
  const cuuint64_t dims[3] = {128, kRowsPerPage, num_pages};
  const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(msa::kKvPage)};
  const cuuint32_t box[3] = {128, 2 * msa::kRegion / 128, 1};  // the K and V regions of one head
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(static_cast<CUtensorMap*>(tmap64), CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(base), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace msa_host

namespace msa {
namespace {

__global__ void k_wait_selftest(uint32_t* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nobody ever arrives on `bar`: the bounded wait must give up and report it
    if (!mbar_wait_bounded(&bar, 0u, limit_ns, &abort_flag)) set_status(status, MSA_ERR_TIMEOUT);
  }
}

struct WsLayout {
  size_t scores, sel, attn, total;
};

WsLayout decode_layout(int B, int T, int maxb) {
  using msa_host::align256;
  WsLayout w;
  w.scores = 256;
  w.sel = w.scores + align256(static_cast<size_t>(T) * 4 * maxb * sizeof(float));
  w.attn = w.sel + align256(static_cast<size_t>(T) * 4 * kSel * sizeof(int32_t));
  msa_geometry geo = MSA_GEOMETRY_DEFAULT;
  w.total = w.attn + msa_attn_workspace_size(&geo, B, T, 0);
  return w;
}

}  // namespace
}  // namespace msa

using namespace msa;
using namespace msa_host;

extern "C" const char* msa_status_string(msa_status s) {
  switch (s) {
    case MSA_OK: return "MSA_OK";
    case MSA_ERR_INVALID_ARG: return "MSA_ERR_INVALID_ARG: bad pointer, size, alignment or batch description";
    case MSA_ERR_UNSUPPORTED: return "MSA_ERR_UNSUPPORTED: geometry or dtype not implemented";
    case MSA_ERR_CUDA: return "MSA_ERR_CUDA: a CUDA call or launch failed";
    case MSA_ERR_TIMEOUT: return "MSA_ERR_TIMEOUT: a device-side wait ran out of time";
    case MSA_ERR_DEVICE_FAULT: return "MSA_ERR_DEVICE_FAULT: page id or selected block out of range";
  }
  return "unknown msa_status";
}

extern "C" int32_t msa_abi_version(void) { return MSA_ABI_VERSION; }

extern "C" size_t msa_decode_workspace_size(const msa_geometry* geo, int32_t B, int32_t T,
                                            int32_t max_blocks_per_seq) {
  if (check_geometry(geo) != MSA_OK || B < 0 || T < 0 || max_blocks_per_seq < 1) return 0;
  return decode_layout(B, T, max_blocks_per_seq).total;
}

extern "C" msa_status msa_decode_step(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                      const uint8_t* q, const uint8_t* index_q, float softmax_scale,
                                      float* dbg_block_scores, int32_t* dbg_sel, void* workspace,
                                      size_t workspace_bytes, uint16_t* out, cudaStream_t stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = check_batch(batch)) != MSA_OK) return st;
  if ((st = check_cache(cache, true, true)) != MSA_OK) return st;
  if (workspace == nullptr || !aligned(workspace, 256)) return MSA_ERR_INVALID_ARG;
  const WsLayout w = decode_layout(batch->B, batch->T, batch->max_blocks_per_seq);
  if (workspace_bytes < w.total) return MSA_ERR_INVALID_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), stream) != cudaSuccess) return MSA_ERR_CUDA;
  if (batch->B == 0 || batch->T == 0) return MSA_OK;
  float* scores = dbg_block_scores != nullptr ? dbg_block_scores : reinterpret_cast<float*>(ws + w.scores);
  int32_t* sel = dbg_sel != nullptr ? dbg_sel : reinterpret_cast<int32_t*>(ws + w.sel);
  if ((st = msa_indexer_decode(geo, batch, cache, index_q, scores, status, stream)) != MSA_OK) return st;
  if ((st = msa_topk_blocks(geo, batch, scores, sel, status, stream)) != MSA_OK) return st;
  return msa_sparse_attn_decode(geo, batch, cache, q, sel, softmax_scale, 0, ws + w.attn, w.total - w.attn, out,
                                status, stream);
}

namespace {

// Page-locked host memory, and the address kernels reach it at (nullptr when they cannot).
bool page_locked(const void* ptr, void** device_ptr = nullptr) {
  if (device_ptr != nullptr) *device_ptr = nullptr;
  if (ptr == nullptr) return false;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();  // an unregistered pointer may leave an error behind on older runtimes
    return false;
  }
  if (a.type != cudaMemoryTypeHost) return false;
  if (device_ptr != nullptr) *device_ptr = a.devicePointer;
  return true;
}

// The CUDA events msa_decode_step_host orders its two streams with: one set per host thread
// and device, created on first use and released when the thread exits. Reusing them across
// calls is safe: a wait refers to the record enqueued before it, and a later record does not
// change what an earlier wait waits for.
struct StepEvents {
  static constexpr int kN = 5;
  static constexpr int kMaxDev = 64;
  cudaEvent_t e[kMaxDev][kN] = {};
  ~StepEvents() {
    for (auto& d : e)
      for (auto x : d)
        if (x != nullptr) cudaEventDestroy(x);
  }
  // the current device's set, or nullptr when it cannot be created
  cudaEvent_t* get() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
    cudaEvent_t* d = e[dev];
    for (int i = 0; i < kN; ++i)
      if (d[i] == nullptr && cudaEventCreateWithFlags(&d[i], cudaEventDisableTiming) != cudaSuccess) {
        d[i] = nullptr;
        return nullptr;
      }
    return d;
  }
};
thread_local StepEvents t_step_events;

}  // namespace

extern "C" msa_status msa_decode_step_host(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                                           const msa_host_step_io* host, uint8_t* q, uint8_t* index_q,
                                           float softmax_scale, void* workspace, size_t workspace_bytes,
                                           uint16_t* out, int32_t flags, cudaStream_t stream,
                                           cudaStream_t copy_stream) {
  msa_status st = check_geometry(geo);
  if (st != MSA_OK) return st;
  if ((st = check_batch(batch)) != MSA_OK) return st;
  if ((st = check_cache(cache, true, true)) != MSA_OK) return st;
  if (host == nullptr || workspace == nullptr || !aligned(workspace, 256) ||
      (flags & ~MSA_HOST_STEP_DIRECT_OUT) != 0)
    return MSA_ERR_INVALID_ARG;
  const bool direct = (flags & MSA_HOST_STEP_DIRECT_OUT) != 0;
  const WsLayout w = decode_layout(batch->B, batch->T, batch->max_blocks_per_seq);
  if (workspace_bytes < w.total) return MSA_ERR_INVALID_ARG;
  const size_t B = static_cast<size_t>(batch->B), T = static_cast<size_t>(batch->T);
  const size_t n_qsl = (B + 1) * 4, n_sl = B * 4, n_bt = B * static_cast<size_t>(batch->max_blocks_per_seq) * 4;
  const size_t n_q = T * kQHeads * kD, n_iq = T * 4 * kD, n_out = T * kQHeads * kD * 2;
  if (B > 0 && !(page_locked(host->query_start_loc) && page_locked(host->seq_lens) && page_locked(host->block_table)))
    return MSA_ERR_INVALID_ARG;
  void* out_dev_view = nullptr;  // host->out as the kernels address it (direct mode)
  if (T > 0) {
    if (!(page_locked(host->q) && page_locked(host->index_q) && page_locked(host->out, &out_dev_view) &&
          q != nullptr && index_q != nullptr))
      return MSA_ERR_INVALID_ARG;
    // direct: the kernels must reach host->out at its own address (unified addressing)
    if (direct ? out_dev_view != static_cast<void*>(host->out) : out == nullptr) return MSA_ERR_INVALID_ARG;
  }
  uint16_t* attn_out = direct ? host->out : out;
  cudaEvent_t* ev = t_step_events.get();
  if (ev == nullptr) return MSA_ERR_CUDA;
  cudaEvent_t e_start = ev[0], e_meta = ev[1], e_q = ev[2], e_a0 = ev[3], e_a1 = ev[4];
  auto cuda = [](cudaError_t e) { return e == cudaSuccess; };
  // the device buffers may still be read by work already on `stream`
  if (!cuda(cudaEventRecord(e_start, stream)) || !cuda(cudaStreamWaitEvent(copy_stream, e_start, 0)))
    return MSA_ERR_CUDA;
  // what the indexer reads, on both streams side by side (the block table on the copy stream,
  // the rest on `stream`), then q on the copy stream behind it
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  if (B > 0 &&
      (!cuda(cudaMemcpyAsync(const_cast<int32_t*>(batch->block_table), host->block_table, n_bt, h2d, copy_stream)) ||
       !cuda(cudaMemcpyAsync(const_cast<int32_t*>(batch->query_start_loc), host->query_start_loc, n_qsl, h2d,
                             stream)) ||
       !cuda(cudaMemcpyAsync(const_cast<int32_t*>(batch->seq_lens), host->seq_lens, n_sl, h2d, stream))))
    return MSA_ERR_CUDA;
  if (!cuda(cudaEventRecord(e_meta, copy_stream))) return MSA_ERR_CUDA;
  if (T > 0 && !cuda(cudaMemcpyAsync(q, host->q, n_q, h2d, copy_stream))) return MSA_ERR_CUDA;
  if (!cuda(cudaEventRecord(e_q, copy_stream))) return MSA_ERR_CUDA;
  if (T > 0 && !cuda(cudaMemcpyAsync(index_q, host->index_q, n_iq, h2d, stream))) return MSA_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint32_t* status = reinterpret_cast<uint32_t*>(ws);
  if (!cuda(cudaStreamWaitEvent(stream, e_meta, 0)) || !cuda(cudaMemsetAsync(status, 0, sizeof(uint32_t), stream)))
    return MSA_ERR_CUDA;
  if (T > 0) {
    float* scores = reinterpret_cast<float*>(ws + w.scores);
    int32_t* sel = reinterpret_cast<int32_t*>(ws + w.sel);
    if ((st = msa_indexer_decode(geo, batch, cache, index_q, scores, status, stream)) != MSA_OK) return st;
    if ((st = msa_topk_blocks(geo, batch, scores, sel, status, stream)) != MSA_OK) return st;
    if (!cuda(cudaStreamWaitEvent(stream, e_q, 0))) return MSA_ERR_CUDA;
    // direct: one launch that stores the output into host memory as it goes; else the attention
    // in two launches when the batch is large enough, the first one's rows copying back while
    // the second runs
    const int32_t ta = direct ? 0 : msa_attn_split_token(batch->T);
    if (ta > 0) {
      if ((st = msa_attn_token_range(geo, batch, cache, q, sel, softmax_scale, attn_out, status, 0, ta, stream)) !=
          MSA_OK)
        return st;
      if (!cuda(cudaEventRecord(e_a0, stream))) return MSA_ERR_CUDA;
      if ((st = msa_attn_token_range(geo, batch, cache, q, sel, softmax_scale, attn_out, status, ta, batch->T,
                                     stream)) != MSA_OK)
        return st;
    } else if ((st = msa_sparse_attn_decode(geo, batch, cache, q, sel, softmax_scale, 0, ws + w.attn,
                                            w.total - w.attn, attn_out, status, stream)) != MSA_OK) {
      return st;
    }
    if (!direct) {
      if (!cuda(cudaEventRecord(e_a1, stream))) return MSA_ERR_CUDA;
      const size_t row = static_cast<size_t>(kQHeads) * kD;  // bf16 elements of one token's output
      if (ta > 0 && (!cuda(cudaStreamWaitEvent(copy_stream, e_a0, 0)) ||
                     !cuda(cudaMemcpyAsync(host->out, out, static_cast<size_t>(ta) * row * 2, d2h, copy_stream))))
        return MSA_ERR_CUDA;
      if (!cuda(cudaStreamWaitEvent(copy_stream, e_a1, 0)) ||
          !cuda(cudaMemcpyAsync(host->out + static_cast<size_t>(ta) * row, out + static_cast<size_t>(ta) * row,
                                n_out - static_cast<size_t>(ta) * row * 2, d2h, copy_stream)))
        return MSA_ERR_CUDA;
    }
  }
  // e_start is free again (its wait is enqueued): it marks the end of the copy stream's work
  if (!cuda(cudaEventRecord(e_start, copy_stream)) || !cuda(cudaStreamWaitEvent(stream, e_start, 0)))
    return MSA_ERR_CUDA;
  return MSA_OK;
}

extern "C" msa_status msa_read_device_status(const void* workspace, cudaStream_t stream) {
  if (workspace == nullptr) return MSA_ERR_INVALID_ARG;
  uint32_t bits = 0;
  if (cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MSA_ERR_CUDA;
  const msa_status order[] = {MSA_ERR_DEVICE_FAULT, MSA_ERR_TIMEOUT, MSA_ERR_INVALID_ARG, MSA_ERR_CUDA,
                              MSA_ERR_UNSUPPORTED};
  for (msa_status s : order)
    if (bits & (1u << s)) return s;
  return MSA_OK;
}

extern "C" msa_status msa_selftest_wait_timeout(uint32_t* status, int64_t limit_ns, cudaStream_t stream) {
  if (status == nullptr || limit_ns < 0 || !aligned(status, 4)) return MSA_ERR_INVALID_ARG;
  k_wait_selftest<<<1, 32, 0, stream>>>(status, static_cast<unsigned long long>(limit_ns));
  return launch_status();
}
