/*
 * msa.h — C ABI of the MiniMax Sparse Attention (MSA) decode step over a paged NVFP4 cache,
 * for NVIDIA GB300 (sm_103a).
 *
 * The method (sources named by page title and section):
 *  - "vLLM ofrece soporte en día 0 para MiniMax-M3.1-Flash", section "MSA primer": the KV
 *    cache is split into 128-token blocks; a light indexer scores every key of the context
 *    with one index query per GQA group against one shared index-key head and max-pools the
 *    scores to one per block; main attention then runs exactly over the top 16 blocks, the
 *    most recent block always kept, so each query sees at most 2,048 keys.
 *  - same page, "NVIDIA Blackwell optimizado kernes MSA": the KV cache is NVFP4 while the
 *    queries stay FP8, so the kernels dequantise the cache to FP8 and run FP8 MMAs.
 *  - "MiniMax M3 in vLLM: Day-0 Serving for 1M-Token Multimodal Reasoning", sections
 *    "MSA 机制详解" (mechanism: init_blocks = 0, local_blocks = 1, partial last block masked,
 *    causal boundary inside a block, local block not counted twice, per-request block
 *    ranges), "解码执行" (decode: score, local window, top-k, sparse GQA, merge of split
 *    partial outputs) and "解码内核中的推测解码" (uniform decode query length, tokens flattened
 *    request-major, each mapped back to its request, sequence length, block table and causal
 *    position; shape-stable launch grids for CUDA graphs).
 *  - "MiniMax-M3.1-Flash serving notes", "The architecture, in operator terms" (64 query
 *    heads, 4 KV heads, head dim 128) and "The capacity numbers" (NVFP4 = 4-bit values plus
 *    one FP8 scale per 16 values, 4.5 bits per element).
 *
 * Conventions for every function:
 *  - Pointers named device are CUDA device pointers; structs are passed by host pointer and
 *    read during the call only. The caller allocates and owns every buffer, and the library
 *    allocates no device memory of its own. It keeps exactly two pieces of state between
 *    calls, each documented where it is declared: msa_decode_step_host keeps a few CUDA
 *    events per host thread and device, and msa_sparse_attn_decode_noalloc uses one
 *    file-scope device array shared by all its calls. Every other entry point keeps no state
 *    and is re-entrant. Buffers must not alias unless stated.
 *  - Every call is asynchronous on the given stream and never synchronises the host, except
 *    msa_read_device_status.
 *  - Problems found on the host (null pointers, sizes, alignment, unsupported geometry)
 *    return an error before anything is launched. A failed launch returns MSA_ERR_CUDA.
 *    Problems only the device can see (a page id outside the cache, an inconsistent batch
 *    description, a wait that ran out) set bits in a caller-provided device status word
 *    (bit 1 << code, see msa_status) and never trap; the affected outputs are zero-filled
 *    where stated.
 *  - Launch grids depend only on the integer arguments (B, T, max_blocks_per_seq, sizes)
 *    and on the device's SM count, never on device data, so a call can be captured in a CUDA
 *    graph and replayed with new device contents.
 *
 * Byte layouts (this library's; the pages fix none):
 *  - NVFP4 row of C elements (C % 16 == 0): C/2 code bytes and C/16 E4M3 scale bytes; scale
 *    k covers elements 16k..16k+15 with value E2M1(code) * E4M3(scale). The code bytes are
 *    little-endian 32-bit words; word w holds elements 8w..8w+7: element 8w+j keeps its three
 *    E2M1 magnitude bits at bits 4j..4j+2 and its sign bit at bit 4*s(j)+3, with
 *    s = (1, 3, 5, 7, 0, 2, 4, 6). (Every nibble still holds three magnitude bits and one
 *    sign bit; placing the signs this way lets the dequantiser produce FP8 bytes in element
 *    order with one byte-permute and one masked xor per four elements.)
 *  - Index page (NVFP4): 128 rows x 64 code bytes, then 128 rows x 8 scale bytes = 9,216 B.
 *    Index page (FP8): 128 rows x 128 E4M3 bytes = 16,384 B.
 *  - KV page: [4 KV heads][K, V][128 rows x 64 code bytes, then 128 rows x 8 scale bytes]
 *    = 73,728 B. Index and KV pages share the physical page id of the block table.
 *  - Page arrays must be 256-byte aligned. Several block-table entries may name one page.
 */
#ifndef MSA_H_
#define MSA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MSA_ABI_VERSION 1

typedef enum msa_status {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or batch description */
  MSA_ERR_UNSUPPORTED = 2,  /* a geometry or dtype this build does not implement */
  MSA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed */
  MSA_ERR_TIMEOUT = 4,      /* a device-side wait ran out of its time budget */
  MSA_ERR_DEVICE_FAULT = 5  /* the device found a page id outside [0, num_pages) or an
                               out-of-range selected block */
} msa_status;

/* Index-key cache dtypes: NVFP4 (72 B/token) or FP8 E4M3 (128 B/token, no scales). */
enum { MSA_INDEX_NVFP4 = 0, MSA_INDEX_FP8 = 1 };

/* The fixed MSA geometry of the method ("MSA primer"; "The architecture, in operator terms";
 * "MSA 机制详解"): 64 query heads, 4 KV heads, head and index dim 128, 128-token blocks,
 * 16 selected blocks of which 1 local block and 0 initial blocks. Any other value is
 * rejected with MSA_ERR_UNSUPPORTED. */
typedef struct msa_geometry {
  int32_t num_q_heads;   /* 64 */
  int32_t num_kv_heads;  /* 4 (= GQA groups; query head h belongs to group h / 16) */
  int32_t head_dim;      /* 128 */
  int32_t index_dim;     /* 128 */
  int32_t block_size;    /* 128 */
  int32_t topk;          /* 16, local block included */
  int32_t local_blocks;  /* 1 */
  int32_t init_blocks;   /* 0 */
} msa_geometry;

#define MSA_GEOMETRY_DEFAULT {64, 4, 128, 128, 128, 16, 1, 0}

/* One decode batch, query tokens flattened request-major ("解码内核中的推测解码").
 * Sequence b owns query tokens query_start_loc[b] .. query_start_loc[b+1]-1; its cache
 * holds seq_lens[b] tokens including those query tokens, and its i-th query token sits at
 * position seq_lens[b] - q_len_b + i and attends causally up to that position.
 * All pointers are device pointers (int32). A sequence with q_len 0 (a padded request row)
 * is skipped; a sequence with q_len > 0 needs seq_lens[b] >= q_len. */
typedef struct msa_batch {
  int32_t B;                       /* sequences */
  int32_t T;                       /* query tokens, = query_start_loc[B] */
  const int32_t* query_start_loc;  /* [B+1], device */
  const int32_t* seq_lens;         /* [B], device */
  const int32_t* block_table;      /* [B][max_blocks_per_seq] physical page ids, device */
  int32_t max_blocks_per_seq;      /* row stride of block_table; seq_lens[b] <= 128 * this */
  int32_t max_q_len;               /* upper bound on q_len, 1..8 */
} msa_batch;

/* The paged caches of one layer. */
typedef struct msa_cache {
  const uint8_t* kv_pages;     /* [num_pages][73,728 B], device, 256-B aligned */
  const uint8_t* index_pages;  /* [num_pages][9,216 B (NVFP4) | 16,384 B (FP8)], device */
  int32_t index_dtype;         /* MSA_INDEX_NVFP4 or MSA_INDEX_FP8 */
  int32_t num_pages;           /* valid page ids are 0 .. num_pages-1 */
} msa_cache;

const char* msa_status_string(msa_status s);
int32_t msa_abi_version(void);

/* ---------------------------------------------------------------- cache producers ---- */

/* NVFP4 quantisation ("The capacity numbers": 4-bit values plus one FP8 scale per 16).
 * For each run of 16 elements of a row: s = E4M3 round-to-nearest-even, saturating, of
 * amax/6 (fp32 division); S = E4M3 value of s; code_i = E2M1 round-to-nearest-even,
 * saturating at 6, of x_i / S (fp32 division), zero magnitudes coded +0; S == 0 gives all
 * codes 0. The amax/6 rule and the rounding modes are this library's reading (the pages
 * leave them open).
 *   x       [rows][cols] fp32, device, 16-B aligned, row stride cols; finite values
 *   cols    multiple of 16
 *   vals    device; row r's codes at vals + r * vals_row_stride (cols/2 bytes, stride % 4 == 0,
 *           4-B aligned)
 *   scales  device; row r's scales at scales + r * scales_row_stride (cols/16 bytes) */
msa_status msa_quantize_nvfp4(const float* x, int64_t rows, int32_t cols, uint8_t* vals,
                              int64_t vals_row_stride, uint8_t* scales,
                              int64_t scales_row_stride, cudaStream_t stream);

/* FP8 (E4M3) cast, round to nearest even, saturating to +-448, sign of zero kept.
 * Used for queries, index queries and the FP8 index-key cache. x, out: [n], device. */
msa_status msa_quantize_fp8(const float* x, int64_t n, uint8_t* out, cudaStream_t stream);

/* Dequantise NVFP4 rows to the FP8 operand the MMAs see ("NVIDIA Blackwell optimizado
 * kernes MSA"; the E4M3 re-rounding is the one "NVIDIA Rubin MSA optimizado" contrasts with
 * exact FP16 scores): out = E4M3_rne_sat(E2M1(code) * E4M3(scale)), sign = sign(code) xor
 * sign(scale), NaN scale -> 0x7F with that sign.
 *   vals [rows] x (cols/2) bytes at vals_row_stride, scales [rows] x (cols/16) at
 *   scales_row_stride, out [rows][cols] E4M3; all device; cols % 16 == 0. */
msa_status msa_dequant_nvfp4(const uint8_t* vals, int64_t vals_row_stride,
                             const uint8_t* scales, int64_t scales_row_stride, int64_t rows,
                             int32_t cols, uint8_t* out, cudaStream_t stream);

/* Paged cache insert: quantise n new tokens straight into their pages (the KV-insert step
 * of "QKV GEMM + norm + RoPE + KV inserción fusión", without the GEMM, norm and RoPE).
 *   k, v      [n][4][128] fp32, device, contiguous
 *   ik        [n][128] fp32, device (index keys), may be NULL to skip the index cache
 *   slots     [n] int64 device: physical page * 128 + row in page; -1 skips the token
 *   kv_pages, index_pages: the caches (index_pages may be NULL when ik is NULL)
 * Slots outside [0, num_pages * 128) set MSA_ERR_DEVICE_FAULT in *status (nullable) and
 * are skipped. Two tokens must not name the same slot. */
msa_status msa_kv_insert(const float* k, const float* v, const float* ik, int64_t n,
                         const int64_t* slots, uint8_t* kv_pages, uint8_t* index_pages,
                         int32_t index_dtype, int32_t num_pages, uint32_t* status,
                         cudaStream_t stream);

/* ---------------------------------------------------------------- the decode step ---- */

/* Indexer score and block max-pool ("MSA primer"; "解码执行").
 * block_scores[t][g][k] = max over the cache positions j of block k with j <= p_t of
 * sum_d index_q[t][g][d] * ik_fp8[j][d], where ik_fp8 is the index key dequantised to E4M3
 * as in msa_dequant_nvfp4 (the FP8 index cache is used as is) and p_t is token t's position;
 * -inf for a block with no such j. Products are exact, sums are fp32.
 *   index_q       [T][4][128] E4M3, device
 *   block_scores  [T][4][max_blocks_per_seq] fp32, device; entries k >= the sequence's
 *                 block count are not written
 *   status        device uint32, nullable: bad page ids set bit MSA_ERR_DEVICE_FAULT (the
 *                 page is then scored -inf), an inconsistent batch sets MSA_ERR_INVALID_ARG
 * Returns MSA_ERR_UNSUPPORTED when cache->num_pages exceeds 2^24 (the index pool is read as
 * one tensor of 128-byte rows). */
msa_status msa_indexer_decode(const msa_geometry* geo, const msa_batch* batch,
                              const msa_cache* cache, const uint8_t* index_q,
                              float* block_scores, uint32_t* status, cudaStream_t stream);

/* The indexer over one context shard ("Indexador NVFP4 DCP": the context is split across ranks
 * by block range): as msa_indexer_decode, but only blocks block_begin <= k < block_end of each
 * sequence are scanned and written (the others are left untouched). msa_indexer_decode is the
 * range [0, 2^31 - 1). block_begin < 0 or block_end < block_begin: MSA_ERR_INVALID_ARG. */
msa_status msa_indexer_decode_range(const msa_geometry* geo, const msa_batch* batch,
                                    const msa_cache* cache, const uint8_t* index_q,
                                    int32_t block_begin, int32_t block_end,
                                    float* block_scores, uint32_t* status, cudaStream_t stream);

/* Exact-score variant of msa_indexer_decode ("vLLM ofrece soporte en día 0 para
 * MiniMax-M3.1-Flash", "NVIDIA Rubin MSA optimizado": NVFP4 index keys converted straight to
 * FP16 and scored with an FP16 MMA, so the scores carry no E4M3 re-rounding). Same arguments,
 * layouts and results as msa_indexer_decode except that an NVFP4 index key element is taken
 * as E2M1(code) x E4M3(scale) exactly (f16 holds it exactly), the index query widened exactly
 * from E4M3 to f16, products accumulated in fp32. An FP8 index cache is scored exactly as
 * msa_indexer_decode scores it (its keys are never re-rounded). Errors as msa_indexer_decode. */
msa_status msa_indexer_decode_exact(const msa_geometry* geo, const msa_batch* batch,
                                    const msa_cache* cache, const uint8_t* index_q,
                                    float* block_scores, uint32_t* status, cudaStream_t stream);

/* Per-group block selection ("MSA primer"; "MSA 机制详解"). For token t at position p_t,
 * local = p_t / 128. sel[t][g][0] = local; sel[t][g][1..15] = the 15 highest-scoring blocks
 * among 0 .. local-1, in descending score order, equal scores ordered by lower block id
 * first (NaN ranks as -inf, -0 equals +0); -1 pads when fewer than 15 exist.
 *   block_scores  [T][4][max_blocks_per_seq] fp32, device (as written by the indexer)
 *   sel           [T][4][16] int32, device */
msa_status msa_topk_blocks(const msa_geometry* geo, const msa_batch* batch,
                           const float* block_scores, int32_t* sel, uint32_t* status,
                           cudaStream_t stream);

/* Context-sharded selection ("Indexador NVFP4 DCP": each rank keeps its own best blocks and
 * one gather brings them to the rank that owns the query; scores are per block, so the merge
 * is exact). A candidate is the 64-bit key (order-preserving bits of the fp32 score << 32 |
 * ~block id; NaN ranks as -inf, -0 as +0), so one integer order is "score descending, lower
 * block id first"; 0 = no candidate.
 *
 * msa_topk_candidates: for every (t, g) row, the 15 largest keys among blocks
 * block_begin <= k < min(block_end, local) (local = p_t / 128 is never a candidate), descending,
 * 0-padded.
 *   block_scores [T][4][max_blocks_per_seq] fp32, device (only the shard's range is read)
 *   cand         [T][4][15] uint64, device */
msa_status msa_topk_candidates(const msa_geometry* geo, const msa_batch* batch,
                               const float* block_scores, int32_t block_begin, int32_t block_end,
                               uint64_t* cand, uint32_t* status, cudaStream_t stream);

/* msa_topk_merge: sel[t][g] = [local, the 15 largest keys over the n_shards candidate lists as
 * block ids, -1 padded] -- for shards that partition blocks 0 .. local-1 this equals
 * msa_topk_blocks bit for bit.
 *   cand  [n_shards][T][4][15] uint64, device; 1 <= n_shards <= 256
 *   sel   [T][4][16] int32, device */
msa_status msa_topk_merge(const msa_geometry* geo, const msa_batch* batch, const uint64_t* cand,
                          int32_t n_shards, int32_t* sel, uint32_t* status, cudaStream_t stream);

/* Host-memory versions of the two (synchronous, no GPU): rows = T x 4, local[rows] the rows'
 * local blocks (a negative local marks a row to skip: no candidates, sel all -1). */
msa_status msa_topk_candidates_host(const float* block_scores, int64_t rows,
                                    int32_t max_blocks_per_seq, const int32_t* local,
                                    int32_t block_begin, int32_t block_end, uint64_t* cand);
msa_status msa_topk_merge_host(const uint64_t* cand, int32_t n_shards, int64_t rows,
                               const int32_t* local, int32_t* sel);

/* The K/V of the selected blocks, brought to the rank that owns the query tokens
 * ("Indexador NVFP4 DCP": each rank holds the blocks of its context range; the merged selection
 * names blocks on several ranks, and the owner's sparse attention needs their K/V locally).
 * The owner's copy is a pool of gathered pages in the KV page layout (73,728 B each) with its own
 * block table, so msa_sparse_attn_decode runs on it unchanged.
 *
 * msa_kv_gather_map: number the distinct (sequence, block) pairs that any query token of the
 * sequence selected in any group: sequence by sequence, in block order.
 *   sel           [T][4][16] int32, device (the merged selection; negative entries ignored; an
 *                 entry at or past the sequence's block count sets MSA_ERR_DEVICE_FAULT and is
 *                 ignored)
 *   map           [B][max_blocks_per_seq] int32, device, written: the gathered page of the pair,
 *                 or -1 -- the owner's block table into the gathered pool
 *   masks         [B][max_blocks_per_seq] uint8, device, written: bit g set when group g selected
 *                 the pair (only those groups' regions are gathered and read)
 *   num_gathered  [1] int32, device, written: the pool's page count */
msa_status msa_kv_gather_map(const msa_geometry* geo, const msa_batch* batch, const int32_t* sel,
                             int32_t* map, uint8_t* masks, int32_t* num_gathered, uint32_t* status,
                             cudaStream_t stream);

/* msa_kv_gather_pages: on a rank holding blocks [block_begin, block_end) of every sequence
 * (batch->block_table and cache describe that rank's own pages), copy the K and V regions of every
 * selected (sequence, block, group) it holds into page map[b][block] of gathered_kv. Ranks
 * whose ranges partition the blocks fill disjoint pages; each rank may write straight into the
 * owner's pool (one GPU) or into a pool of its own whose filled pages are then copied to the
 * owner. A page id outside the cache or a gathered page >= max_gathered sets
 * MSA_ERR_DEVICE_FAULT and is skipped.
 *   map, masks    as written by msa_kv_gather_map, device
 *   gathered_kv   [max_gathered][73,728 B], device, 16-byte aligned */
msa_status msa_kv_gather_pages(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                               const int32_t* map, const uint8_t* masks, int32_t block_begin,
                               int32_t block_end, uint8_t* gathered_kv, int32_t max_gathered,
                               uint32_t* status, cudaStream_t stream);

/* Host-memory versions of the two (synchronous, no GPU; arrays as above, in host memory).
 * msa_kv_gather_map_host returns the gathered page count, or -1 on a bad argument or a
 * selected block past its sequence. */
int32_t msa_kv_gather_map_host(int32_t B, int32_t T, const int32_t* query_start_loc,
                               const int32_t* seq_lens, int32_t max_blocks_per_seq, const int32_t* sel,
                               int32_t* map, uint8_t* masks);
msa_status msa_kv_gather_pages_host(int32_t B, int32_t max_blocks_per_seq, const int32_t* block_table,
                                    const uint8_t* kv_pages, int32_t num_pages, const int32_t* map,
                                    const uint8_t* masks, int32_t block_begin, int32_t block_end,
                                    uint8_t* gathered_kv, int32_t max_gathered);

/* Workspace bytes msa_sparse_attn_decode needs for num_splits partial results per token
 * (num_splits 0 = the automatic choice, which never exceeds 16). */
size_t msa_attn_workspace_size(const msa_geometry* geo, int32_t B, int32_t T, int32_t num_splits);

/* Exact sparse GQA attention over the selected blocks ("MSA primer": exact attention over
 * the selected blocks; "解码执行": split work merged from partial outputs). For query head h
 * of token t (group g = h / 16): the keys are the cache positions j <= p_t of the distinct
 * blocks listed in sel[t][g][0..15] (entries < 0 ignored); z_j = softmax_scale * q . k_j with
 * K dequantised to E4M3; out = sum_j softmax(z)_j v_j with V dequantised to E4M3; written
 * as bf16. QK^T runs as an FP8 MMA with fp32 accumulation; the softmax is fp32. For batches
 * of up to 76 query tokens PV runs with P in f16 and V widened exactly from E4M3 to f16; for
 * larger batches it runs as an FP8 MMA on the E4M3 V with P split into two E4M3 parts,
 * hi = E4M3(P) and lo = E4M3(16 (P - hi)), so P is carried to within 2^-8 of itself.
 *   q          [T][64][128] E4M3, device
 *   sel        [T][4][16] int32, device
 *   num_splits 0 = automatic; else 1..16 splits of each (sequence, group)'s block list,
 *              merged by log-sum-exp
 *   workspace  device, >= msa_attn_workspace_size(...) bytes (may be NULL when that is 0)
 *   out        [T][64][128] bf16 (uint16 bit patterns), device
 *   status     nullable; a selected block beyond the sequence or a bad page id sets
 *              MSA_ERR_DEVICE_FAULT and the affected tokens' outputs are zero-filled */
msa_status msa_sparse_attn_decode(const msa_geometry* geo, const msa_batch* batch,
                                  const msa_cache* cache, const uint8_t* q, const int32_t* sel,
                                  float softmax_scale, int32_t num_splits, void* workspace,
                                  size_t workspace_bytes, uint16_t* out, uint32_t* status,
                                  cudaStream_t stream);

/* Allocation-free form of msa_sparse_attn_decode (no counterpart on the pages; this is an
 * interface addition for callers that cannot allocate device memory, e.g. a host runtime
 * whose memory is planned once with no allocator to hand down, or code running inside
 * another library's callback where a cudaMalloc would synchronise the device). Same
 * arguments and results as msa_sparse_attn_decode without the workspace: the split partial
 * results go to one file-scope device array of msa_noalloc_scratch_bytes() bytes (16 MiB),
 * which every GPU that loads the library keeps until the process exits.
 *  - Needs at most splits * T * 64 * 129 * 4 bytes (rounded up to 256-B pieces); larger
 *    requests return MSA_ERR_INVALID_ARG before anything is launched (num_splits = 1 needs
 *    no scratch at all).
 *  - Calls no cudaMalloc / cudaFree. The first call on a device looks up the array's device
 *    address (cudaGetSymbolAddress) once for that device, so make that first call before any
 *    stream capture.
 *  - Every call shares the one array and it keeps the last call's contents (nothing in it
 *    needs to start at zero: each call writes every partial it reads). Calls whose kernels
 *    overlap on the GPU (other streams, other threads) race on it and must be serialised by
 *    the caller. */
msa_status msa_sparse_attn_decode_noalloc(const msa_geometry* geo, const msa_batch* batch,
                                          const msa_cache* cache, const uint8_t* q, const int32_t* sel,
                                          float softmax_scale, int32_t num_splits, uint16_t* out,
                                          uint32_t* status, cudaStream_t stream);

/* Size in bytes of the device array msa_sparse_attn_decode_noalloc uses. */
size_t msa_noalloc_scratch_bytes(void);

/* The indexer for prompts (the prefill / many-query path: "MiniMax M3 in vLLM ...",
 * "MiniMax 稀疏注意力后端" lists prefill indexer scoring as its own kernel, and "预填充执行" scores a
 * prompt's blocks before selecting them). The same scores as msa_indexer_decode (block_scores
 * [t][g][k] = max over the cache positions j <= p_t of block k of index_q[t][g] . ik(j), -inf
 * for a block with no such j; entries k >= the sequence's block count are not written) for a
 * batch of any number of query tokens per sequence (max_q_len up to 2^20, T up to 2^22, B up to
 * 4096). Each index page is read and dequantised once for up to 128 query tokens (512 index-query
 * rows) of its sequence. Arguments, layouts and errors as msa_indexer_decode. */
msa_status msa_indexer_prefill(const msa_geometry* geo, const msa_batch* batch,
                               const msa_cache* cache, const uint8_t* index_q,
                               float* block_scores, uint32_t* status, cudaStream_t stream);

/* msa_topk_blocks for a prefill batch (max_q_len up to 2^20, T up to 2^22): the same rule,
 * layouts and errors for every (token, group) row. */
msa_status msa_topk_prefill(const msa_geometry* geo, const msa_batch* batch,
                            const float* block_scores, int32_t* sel, uint32_t* status,
                            cudaStream_t stream);

/* Workspace bytes msa_prefill_attn needs: a hash table and the selection lists of the key-block
 * -> query map, and the per-(token, group, slot) partial results (4 KB of unnormalised output and
 * 128 B of (max, sum) per slot): about 300 KB a query token, a function of T alone (T up to
 * 2^22; B and max_blocks_per_seq are checked only). 0 for invalid arguments. */
size_t msa_prefill_workspace_size(const msa_geometry* geo, int32_t B, int32_t T,
                                  int32_t max_blocks_per_seq);

/* Sparse GQA attention for any number of query tokens per sequence (the prefill / many-query
 * path: "MiniMax M3 in vLLM ...", "预填充": block-major, a block's K and V read and dequantised
 * once for all the queries that selected it, per-block results merged by log-sum-exp). The map
 * is keyed by the physical page, so a page that several sequences share through a common prefix
 * is dequantised once for up to 64 of the (token, group) selections of all of them ("vLLM ofrece
 * soporte en día 0 ...", "NVFP4 MSA kernel"). Same result as msa_sparse_attn_decode for the same
 * inputs (up to summation order); the batch may hold up to 2^20 query tokens per sequence
 * (max_q_len) and 2^22 in all (T).
 *   q, sel      as for msa_sparse_attn_decode ([T][64][128] E4M3, [T][4][16] int32)
 *   workspace   device, 256-B aligned, >= msa_prefill_workspace_size(...) bytes. When the call's
 *               work has run, its first four int32 hold the map's counts: distinct (page, group)
 *               blocks selected, chunks of at most 64 selections (one K/V dequantisation each),
 *               selections served, and a chunk counter of the kernel's own
 *   out         [T][64][128] bf16, device
 *   status      nullable; an out-of-range selected block or a bad page id sets
 *               MSA_ERR_DEVICE_FAULT and zero-fills that (token, group); an inconsistent batch
 *               row sets MSA_ERR_INVALID_ARG; a device wait that gives up sets MSA_ERR_TIMEOUT
 * Host-checkable errors return before any launch. */
msa_status msa_prefill_attn(const msa_geometry* geo, const msa_batch* batch, const msa_cache* cache,
                            const uint8_t* q, const int32_t* sel, float softmax_scale,
                            void* workspace, size_t workspace_bytes, uint16_t* out,
                            uint32_t* status, cudaStream_t stream);

/* Workspace bytes msa_decode_step needs (depends only on its arguments). */
size_t msa_decode_workspace_size(const msa_geometry* geo, int32_t B, int32_t T,
                                 int32_t max_blocks_per_seq);

/* The whole decode step of one layer: indexer -> top-k -> sparse attention -> merge, all
 * on `stream`. The workspace starts with the device status word, which the call clears
 * first; read it with msa_read_device_status.
 *   q, index_q        as for msa_sparse_attn_decode / msa_indexer_decode
 *   dbg_block_scores  nullable [T][4][max_blocks_per_seq] fp32: when given, the scores are
 *                     written there instead of into the workspace
 *   dbg_sel           nullable [T][4][16] int32: likewise for the selection
 *   workspace         device, >= msa_decode_workspace_size(...) bytes, 256-B aligned
 *   out               [T][64][128] bf16, device */
msa_status msa_decode_step(const msa_geometry* geo, const msa_batch* batch,
                           const msa_cache* cache, const uint8_t* q, const uint8_t* index_q,
                           float softmax_scale, float* dbg_block_scores, int32_t* dbg_sel,
                           void* workspace, size_t workspace_bytes, uint16_t* out,
                           cudaStream_t stream);

/* The step's inputs and output in page-locked host memory (cudaHostAlloc or
 * cudaHostRegister), for msa_decode_step_host. Shapes as in msa_batch / msa_decode_step. */
typedef struct msa_host_step_io {
  const int32_t* query_start_loc; /* [B + 1] */
  const int32_t* seq_lens;        /* [B] */
  const int32_t* block_table;     /* [B][max_blocks_per_seq] */
  const uint8_t* q;               /* [T][64][128] E4M3 */
  const uint8_t* index_q;         /* [T][4][128] E4M3 */
  uint16_t* out;                  /* [T][64][128] bf16, written */
} msa_host_step_io;

/* Flags of msa_decode_step_host. */
enum { MSA_HOST_STEP_DIRECT_OUT = 1 };

/* msa_decode_step from host buffers (this library's own entry point: the pages run the step
 * on device-resident inputs): copies `host`'s inputs into the device buffers (batch's
 * three arrays, q, index_q), runs the step, and delivers the output into host->out, with the
 * copies on `copy_stream` and `stream` overlapping the kernels. The block table goes first on
 * the copy stream while the other batch arrays and the index queries go on `stream`; the
 * indexer starts on them while q is still copying.
 *   flags 0: the output is copied back from `out`; a batch that keeps the many-token attention
 *            kernel busy for six or more rounds of units runs it as two launches (the last
 *            three rounds in the second) so that the first launch's rows copy back while the
 *            second runs.
 *   flags MSA_HOST_STEP_DIRECT_OUT: the attention stores its output straight into host->out
 *            (no copy back, `out` unused and may be null); host->out must be reachable by
 *            kernels at its own address (page-locked memory under unified addressing, which
 *            cudaPointerGetAttributes reports), else MSA_ERR_INVALID_ARG.
 * Ordering: the copies wait for the work already on `stream` (the device buffers may be in
 * use there), and `stream` waits for the copy stream's last copy, so when `stream` reaches the
 * end of the call host->out holds the output. Same result as msa_decode_step on the same
 * inputs, bit for bit.
 *   batch      B, T, max_blocks_per_seq, max_q_len and the DEVICE arrays to fill
 *   host       page-locked host buffers (checked: MSA_ERR_INVALID_ARG otherwise)
 *   q, index_q DEVICE buffers to fill, as for msa_decode_step
 *   workspace  as for msa_decode_step
 *   out        DEVICE [T][64][128] bf16, the output before its copy back (flags 0)
 *   copy_stream may equal stream (no overlap then)
 * Host-checkable errors return before anything is enqueued. The call orders its streams with
 * CUDA events it creates once per host thread and device and keeps until the thread exits
 * (MSA_ERR_CUDA if it cannot create them). */
msa_status msa_decode_step_host(const msa_geometry* geo, const msa_batch* batch,
                                const msa_cache* cache, const msa_host_step_io* host,
                                uint8_t* q, uint8_t* index_q, float softmax_scale,
                                void* workspace, size_t workspace_bytes, uint16_t* out,
                                int32_t flags, cudaStream_t stream, cudaStream_t copy_stream);

/* Test and debugging helper: waits for `stream`, then returns the most severe code whose
 * bit is set in the status word at the start of `workspace` (MSA_OK when none). */
msa_status msa_read_device_status(const void* workspace, cudaStream_t stream);

/* Self-test of the bounded device waits: launches one CTA that waits on a shared-memory
 * barrier nobody arrives on, gives up after limit_ns nanoseconds of %globaltimer, sets
 * MSA_ERR_TIMEOUT in *status (device) and returns. Faults nothing. */
msa_status msa_selftest_wait_timeout(uint32_t* status, int64_t limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H_ */
