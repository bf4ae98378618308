"""Python binding of libmsa.so: the MSA decode step over a paged NVFP4 cache on GB300.

Argument marshalling only: every function forwards torch tensors' device pointers and the
current CUDA stream to the C ABI of the same name (include/msa.h), and raises MsaError on a
non-OK status. All arithmetic runs in the library's CUDA kernels. There is no fallback:
importing this package fails if libmsa.so has not been built (``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmsa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libmsa.so is not built ({LIB_PATH}); run `python -c 'import __graft_entry__ as g; g.build()'`")

_lib = ctypes.CDLL(LIB_PATH)

MSA_OK = 0
MSA_ERR_INVALID_ARG = 1
MSA_ERR_UNSUPPORTED = 2
MSA_ERR_CUDA = 3
MSA_ERR_TIMEOUT = 4
MSA_ERR_DEVICE_FAULT = 5
MSA_INDEX_NVFP4 = 0
MSA_INDEX_FP8 = 1
MSA_HOST_STEP_DIRECT_OUT = 1

HEAD_DIM = 128
GROUPS = 4
Q_HEADS = 64
BLOCK = 128
K_SEL = 16
INDEX_PAGE_BYTES = {MSA_INDEX_NVFP4: 9216, MSA_INDEX_FP8: 16384}
KV_PAGE_BYTES = 73728


class msa_geometry(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_q_heads", "num_kv_heads", "head_dim", "index_dim",
                                               "block_size", "topk", "local_blocks", "init_blocks")]


class msa_batch(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("query_start_loc", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
                ("max_blocks_per_seq", ctypes.c_int32), ("max_q_len", ctypes.c_int32)]


class msa_cache(ctypes.Structure):
    _fields_ = [("kv_pages", ctypes.c_void_p), ("index_pages", ctypes.c_void_p), ("index_dtype", ctypes.c_int32),
                ("num_pages", ctypes.c_int32)]


class msa_host_step_io(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("query_start_loc", "seq_lens", "block_table", "q", "index_q", "out")]


GEOMETRY = msa_geometry(64, 4, 128, 128, 128, 16, 1, 0)

_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t
_GP = ctypes.POINTER(msa_geometry)
_BP = ctypes.POINTER(msa_batch)
_CP = ctypes.POINTER(msa_cache)
_HP = ctypes.POINTER(msa_host_step_io)

_SIGS = {
    "msa_status_string": (ctypes.c_char_p, [_I32]),
    "msa_abi_version": (_I32, []),
    "msa_quantize_nvfp4": (_I32, [_P, _I64, _I32, _P, _I64, _P, _I64, _P]),
    "msa_quantize_fp8": (_I32, [_P, _I64, _P, _P]),
    "msa_dequant_nvfp4": (_I32, [_P, _I64, _P, _I64, _I64, _I32, _P, _P]),
    "msa_kv_insert": (_I32, [_P, _P, _P, _I64, _P, _P, _P, _I32, _I32, _P, _P]),
    "msa_indexer_decode": (_I32, [_GP, _BP, _CP, _P, _P, _P, _P]),
    "msa_topk_blocks": (_I32, [_GP, _BP, _P, _P, _P, _P]),
    "msa_indexer_decode_range": (_I32, [_GP, _BP, _CP, _P, _I32, _I32, _P, _P, _P]),
    "msa_indexer_decode_exact": (_I32, [_GP, _BP, _CP, _P, _P, _P, _P]),
    "msa_indexer_prefill": (_I32, [_GP, _BP, _CP, _P, _P, _P, _P]),
    "msa_topk_prefill": (_I32, [_GP, _BP, _P, _P, _P, _P]),
    "msa_prefill_workspace_size": (_SZ, [_GP, _I32, _I32, _I32]),
    "msa_prefill_attn": (_I32, [_GP, _BP, _CP, _P, _P, ctypes.c_float, _P, _SZ, _P, _P, _P]),
    "msa_topk_candidates": (_I32, [_GP, _BP, _P, _I32, _I32, _P, _P, _P]),
    "msa_topk_merge": (_I32, [_GP, _BP, _P, _I32, _P, _P, _P]),
    "msa_topk_candidates_host": (_I32, [_P, _I64, _I32, _P, _I32, _I32, _P]),
    "msa_topk_merge_host": (_I32, [_P, _I32, _I64, _P, _P]),
    "msa_kv_gather_map": (_I32, [_GP, _BP, _P, _P, _P, _P, _P, _P]),
    "msa_kv_gather_pages": (_I32, [_GP, _BP, _CP, _P, _P, _I32, _I32, _P, _I32, _P, _P]),
    "msa_kv_gather_map_host": (_I32, [_I32, _I32, _P, _P, _I32, _P, _P, _P]),
    "msa_kv_gather_pages_host": (_I32, [_I32, _I32, _P, _P, _I32, _P, _P, _I32, _I32, _P, _I32]),
    "msa_attn_workspace_size": (_SZ, [_GP, _I32, _I32, _I32]),
    "msa_sparse_attn_decode": (_I32, [_GP, _BP, _CP, _P, _P, ctypes.c_float, _I32, _P, _SZ, _P, _P, _P]),
    "msa_sparse_attn_decode_noalloc": (_I32, [_GP, _BP, _CP, _P, _P, ctypes.c_float, _I32, _P, _P, _P]),
    "msa_noalloc_scratch_bytes": (_SZ, []),
    "msa_decode_workspace_size": (_SZ, [_GP, _I32, _I32, _I32]),
    "msa_decode_step": (_I32, [_GP, _BP, _CP, _P, _P, ctypes.c_float, _P, _P, _P, _SZ, _P, _P]),
    "msa_decode_step_host": (_I32, [_GP, _BP, _CP, _HP, _P, _P, ctypes.c_float, _P, _SZ, _P, _I32, _P, _P]),
    "msa_read_device_status": (_I32, [_P, _P]),
    "msa_selftest_wait_timeout": (_I32, [_P, _I64, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(_lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class MsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {_lib.msa_status_string(code).decode()}")


def _check(code: int, where: str) -> None:
    if code != MSA_OK:
        raise MsaError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream] = None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, dtype, name: str) -> None:
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


# ------------------------------------------------------------------ descriptors ----------
class Batch:
    """Decode batch: device int32 tensors + the msa_batch struct (keeps the tensors alive)."""

    def __init__(self, query_start_loc: torch.Tensor, seq_lens: torch.Tensor, block_table: torch.Tensor,
                 max_q_len: int, T: Optional[int] = None):
        for n, t in (("query_start_loc", query_start_loc), ("seq_lens", seq_lens), ("block_table", block_table)):
            _need(t, torch.int32, n)
        self.query_start_loc, self.seq_lens, self.block_table = query_start_loc, seq_lens, block_table
        self.B = int(seq_lens.numel())
        self.T = int(T) if T is not None else int(query_start_loc[-1].item())
        self.max_blocks = int(block_table.shape[1]) if block_table.dim() == 2 else 1
        self.max_q_len = int(max_q_len)
        self.c = msa_batch(self.B, self.T, query_start_loc.data_ptr(), seq_lens.data_ptr(), block_table.data_ptr(),
                           self.max_blocks, self.max_q_len)


class Cache:
    """One layer's paged caches (uint8 device tensors) + the msa_cache struct."""

    def __init__(self, kv_pages: torch.Tensor, index_pages: torch.Tensor, index_dtype: int, num_pages: int):
        _need(kv_pages, torch.uint8, "kv_pages")
        _need(index_pages, torch.uint8, "index_pages")
        self.kv_pages, self.index_pages = kv_pages, index_pages
        self.index_dtype, self.num_pages = int(index_dtype), int(num_pages)
        self.c = msa_cache(kv_pages.data_ptr(), index_pages.data_ptr(), self.index_dtype, self.num_pages)

    @staticmethod
    def empty(num_pages: int, index_dtype: int, device="cuda") -> "Cache":
        kv = torch.zeros(num_pages * KV_PAGE_BYTES, dtype=torch.uint8, device=device)
        ix = torch.zeros(num_pages * INDEX_PAGE_BYTES[index_dtype], dtype=torch.uint8, device=device)
        return Cache(kv, ix, index_dtype, num_pages)


# ------------------------------------------------------------------ the C ABI ------------
def msa_abi_version() -> int:
    return int(_lib.msa_abi_version())


def msa_status_string(code: int) -> str:
    return _lib.msa_status_string(code).decode()


def msa_quantize_nvfp4(x: torch.Tensor, vals: torch.Tensor, scales: torch.Tensor,
                       vals_row_stride: Optional[int] = None, scales_row_stride: Optional[int] = None) -> None:
    _need(x, torch.float32, "x")
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    _check(_lib.msa_quantize_nvfp4(_ptr(x), rows, cols, _ptr(vals), vals_row_stride or cols // 2, _ptr(scales),
                                   scales_row_stride or cols // 16, _stream()), "msa_quantize_nvfp4")


def msa_quantize_fp8(x: torch.Tensor, out: torch.Tensor) -> None:
    _need(x, torch.float32, "x")
    _check(_lib.msa_quantize_fp8(_ptr(x), x.numel(), _ptr(out), _stream()), "msa_quantize_fp8")


def msa_dequant_nvfp4(vals: torch.Tensor, scales: torch.Tensor, out: torch.Tensor) -> None:
    cols = vals.shape[-1] * 2
    rows = vals.numel() // vals.shape[-1]
    _check(_lib.msa_dequant_nvfp4(_ptr(vals), cols // 2, _ptr(scales), cols // 16, rows, cols, _ptr(out), _stream()),
           "msa_dequant_nvfp4")


def msa_kv_insert(k: torch.Tensor, v: torch.Tensor, ik: Optional[torch.Tensor], slots: torch.Tensor, cache: Cache,
                  status: Optional[torch.Tensor] = None) -> None:
    _need(k, torch.float32, "k")
    _need(v, torch.float32, "v")
    _need(slots, torch.int64, "slots")
    n = int(slots.numel())
    _check(_lib.msa_kv_insert(_ptr(k), _ptr(v), _ptr(ik), n, _ptr(slots), _ptr(cache.kv_pages),
                              _ptr(cache.index_pages), cache.index_dtype, cache.num_pages, _ptr(status), _stream()),
           "msa_kv_insert")


def msa_indexer_decode(batch: Batch, cache: Cache, index_q: torch.Tensor, block_scores: torch.Tensor,
                       status: Optional[torch.Tensor] = None) -> None:
    _check(_lib.msa_indexer_decode(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), ctypes.byref(cache.c),
                                   _ptr(index_q), _ptr(block_scores), _ptr(status), _stream()),
           "msa_indexer_decode")


def msa_topk_blocks(batch: Batch, block_scores: torch.Tensor, sel: torch.Tensor,
                    status: Optional[torch.Tensor] = None) -> None:
    _check(_lib.msa_topk_blocks(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), _ptr(block_scores), _ptr(sel),
                                _ptr(status), _stream()), "msa_topk_blocks")


def msa_indexer_decode_range(batch: Batch, cache: Cache, index_q: torch.Tensor, block_begin: int, block_end: int,
                             block_scores: torch.Tensor, status: Optional[torch.Tensor] = None) -> None:
    """The indexer over one context shard: blocks block_begin <= k < block_end of every sequence."""
    _check(_lib.msa_indexer_decode_range(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), ctypes.byref(cache.c),
                                         _ptr(index_q), int(block_begin), int(block_end), _ptr(block_scores),
                                         _ptr(status), _stream()), "msa_indexer_decode_range")


def msa_indexer_decode_exact(batch: Batch, cache: Cache, index_q: torch.Tensor, block_scores: torch.Tensor,
                             status: Optional[torch.Tensor] = None) -> None:
    """The exact-score indexer: NVFP4 index keys as E2M1 x E4M3 exactly (f16 score MMA)."""
    _check(_lib.msa_indexer_decode_exact(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), ctypes.byref(cache.c),
                                         _ptr(index_q), _ptr(block_scores), _ptr(status), _stream()),
           "msa_indexer_decode_exact")


def msa_prefill_workspace_size(B: int, T: int, max_blocks_per_seq: int) -> int:
    return int(_lib.msa_prefill_workspace_size(ctypes.byref(GEOMETRY), B, T, max_blocks_per_seq))


def msa_indexer_prefill(batch: Batch, cache: Cache, index_q: torch.Tensor, block_scores: torch.Tensor,
                        status: Optional[torch.Tensor] = None) -> None:
    """The indexer for a prefill batch (any number of query tokens per sequence)."""
    _check(_lib.msa_indexer_prefill(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), ctypes.byref(cache.c),
                                    _ptr(index_q), _ptr(block_scores), _ptr(status), _stream()),
           "msa_indexer_prefill")


def msa_topk_prefill(batch: Batch, block_scores: torch.Tensor, sel: torch.Tensor,
                     status: Optional[torch.Tensor] = None) -> None:
    """The block selection for a prefill batch (any number of query tokens per sequence)."""
    _check(_lib.msa_topk_prefill(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), _ptr(block_scores), _ptr(sel),
                                 _ptr(status), _stream()), "msa_topk_prefill")


def msa_prefill_attn(batch: Batch, cache: Cache, q: torch.Tensor, sel: torch.Tensor, softmax_scale: float,
                     out: torch.Tensor, workspace: torch.Tensor, status: Optional[torch.Tensor] = None) -> None:
    """Block-major sparse attention for any number of query tokens per sequence."""
    _check(_lib.msa_prefill_attn(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), ctypes.byref(cache.c), _ptr(q),
                                 _ptr(sel), ctypes.c_float(softmax_scale), _ptr(workspace),
                                 ctypes.c_size_t(workspace.numel() * workspace.element_size()), _ptr(out),
                                 _ptr(status), _stream()), "msa_prefill_attn")


def msa_topk_candidates(batch: Batch, block_scores: torch.Tensor, block_begin: int, block_end: int,
                        cand: torch.Tensor, status: Optional[torch.Tensor] = None) -> None:
    """A context shard's 15 best non-local blocks per (t, g) as 64-bit keys (int64 tensor [T, 4, 15])."""
    _check(_lib.msa_topk_candidates(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), _ptr(block_scores),
                                    int(block_begin), int(block_end), _ptr(cand), _ptr(status), _stream()),
           "msa_topk_candidates")


def msa_topk_merge(batch: Batch, cand: torch.Tensor, n_shards: int, sel: torch.Tensor,
                   status: Optional[torch.Tensor] = None) -> None:
    """The owner's merge of n_shards candidate lists ([n_shards, T, 4, 15]) into sel [T, 4, 16]."""
    _check(_lib.msa_topk_merge(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), _ptr(cand), int(n_shards), _ptr(sel),
                               _ptr(status), _stream()), "msa_topk_merge")


def msa_topk_candidates_host(block_scores: np.ndarray, local: np.ndarray, block_begin: int,
                             block_end: int) -> np.ndarray:
    """Host version of msa_topk_candidates: block_scores float32 [rows, maxb], local int32 [rows]."""
    sc = np.ascontiguousarray(block_scores, dtype=np.float32)
    lc = np.ascontiguousarray(local, dtype=np.int32)
    out = np.zeros((sc.shape[0], 15), dtype=np.uint64)
    _check(_lib.msa_topk_candidates_host(sc.ctypes.data, sc.shape[0], sc.shape[1], lc.ctypes.data, int(block_begin),
                                         int(block_end), out.ctypes.data), "msa_topk_candidates_host")
    return out


def msa_topk_merge_host(cand: np.ndarray, local: np.ndarray) -> np.ndarray:
    """Host version of msa_topk_merge: cand uint64 [n_shards, rows, 15], local int32 [rows]."""
    cd = np.ascontiguousarray(cand, dtype=np.uint64)
    lc = np.ascontiguousarray(local, dtype=np.int32)
    out = np.zeros((cd.shape[1], 16), dtype=np.int32)
    _check(_lib.msa_topk_merge_host(cd.ctypes.data, cd.shape[0], cd.shape[1], lc.ctypes.data, out.ctypes.data),
           "msa_topk_merge_host")
    return out


def msa_kv_gather_map(batch: Batch, sel: torch.Tensor, map_out: torch.Tensor, masks: torch.Tensor,
                      num_gathered: torch.Tensor, status: Optional[torch.Tensor] = None) -> None:
    """map_out int32 [B, max_blocks], masks uint8 [B, max_blocks], num_gathered int32 [1] (device)."""
    _check(_lib.msa_kv_gather_map(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), _ptr(sel), _ptr(map_out),
                                  _ptr(masks), _ptr(num_gathered), _ptr(status), _stream()), "msa_kv_gather_map")


def msa_kv_gather_pages(batch: Batch, cache: Cache, map_in: torch.Tensor, masks: torch.Tensor, block_begin: int,
                        block_end: int, gathered_kv: torch.Tensor, max_gathered: int,
                        status: Optional[torch.Tensor] = None) -> None:
    """Copy the selected K/V regions this shard holds (blocks [block_begin, block_end)) into the
    gathered pool gathered_kv (uint8, max_gathered x 73,728 B, device)."""
    _check(_lib.msa_kv_gather_pages(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), ctypes.byref(cache.c), _ptr(map_in),
                                    _ptr(masks), int(block_begin), int(block_end), _ptr(gathered_kv),
                                    int(max_gathered), _ptr(status), _stream()), "msa_kv_gather_pages")


def msa_kv_gather_map_host(query_start_loc: np.ndarray, seq_lens: np.ndarray, max_blocks: int,
                           sel: np.ndarray):
    """Host version of msa_kv_gather_map: returns (map int32 [B, max_blocks], masks uint8, count)."""
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    sl_ = np.ascontiguousarray(sel, dtype=np.int32)
    B = sl.shape[0]
    mp = np.zeros((B, max_blocks), dtype=np.int32)
    mk = np.zeros((B, max_blocks), dtype=np.uint8)
    n = int(_lib.msa_kv_gather_map_host(B, int(qsl[-1]), qsl.ctypes.data, sl.ctypes.data, int(max_blocks),
                                        sl_.ctypes.data, mp.ctypes.data, mk.ctypes.data))
    if n < 0:
        raise MsaError(MSA_ERR_INVALID_ARG, "msa_kv_gather_map_host")
    return mp, mk, n


def msa_kv_gather_pages_host(block_table: np.ndarray, kv_pages: np.ndarray, num_pages: int, map_in: np.ndarray,
                             masks: np.ndarray, block_begin: int, block_end: int, gathered_kv: np.ndarray) -> None:
    """Host version of msa_kv_gather_pages (numpy arrays; gathered_kv uint8 [n, 73,728] is filled)."""
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    kv = np.ascontiguousarray(kv_pages, dtype=np.uint8)
    mp = np.ascontiguousarray(map_in, dtype=np.int32)
    mk = np.ascontiguousarray(masks, dtype=np.uint8)
    assert gathered_kv.dtype == np.uint8 and gathered_kv.flags.c_contiguous
    _check(_lib.msa_kv_gather_pages_host(bt.shape[0], bt.shape[1], bt.ctypes.data, kv.ctypes.data, int(num_pages),
                                         mp.ctypes.data, mk.ctypes.data, int(block_begin), int(block_end),
                                         gathered_kv.ctypes.data, gathered_kv.size // KV_PAGE_BYTES),
           "msa_kv_gather_pages_host")


def msa_attn_workspace_size(B: int, T: int, num_splits: int = 0) -> int:
    return int(_lib.msa_attn_workspace_size(ctypes.byref(GEOMETRY), B, T, num_splits))


def msa_sparse_attn_decode(batch: Batch, cache: Cache, q: torch.Tensor, sel: torch.Tensor, softmax_scale: float,
                           out: torch.Tensor, num_splits: int = 0, workspace: Optional[torch.Tensor] = None,
                           status: Optional[torch.Tensor] = None) -> None:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.msa_sparse_attn_decode(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), ctypes.byref(cache.c), _ptr(q),
                                       _ptr(sel), float(softmax_scale), num_splits, _ptr(workspace), ws_bytes,
                                       _ptr(out), _ptr(status), _stream()), "msa_sparse_attn_decode")


def msa_sparse_attn_decode_noalloc(batch: Batch, cache: Cache, q: torch.Tensor, sel: torch.Tensor,
                                   softmax_scale: float, out: torch.Tensor, num_splits: int = 0,
                                   status: Optional[torch.Tensor] = None) -> None:
    """msa_sparse_attn_decode for callers that cannot allocate: split partials go to the
    library's own device array (msa_noalloc_scratch_bytes() bytes); calls must not overlap."""
    _check(_lib.msa_sparse_attn_decode_noalloc(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), ctypes.byref(cache.c),
                                               _ptr(q), _ptr(sel), float(softmax_scale), num_splits, _ptr(out),
                                               _ptr(status), _stream()), "msa_sparse_attn_decode_noalloc")


def msa_noalloc_scratch_bytes() -> int:
    return int(_lib.msa_noalloc_scratch_bytes())


def msa_decode_workspace_size(B: int, T: int, max_blocks_per_seq: int) -> int:
    return int(_lib.msa_decode_workspace_size(ctypes.byref(GEOMETRY), B, T, max_blocks_per_seq))


def msa_decode_step(batch: Batch, cache: Cache, q: torch.Tensor, index_q: torch.Tensor, softmax_scale: float,
                    workspace: torch.Tensor, out: torch.Tensor, dbg_block_scores: Optional[torch.Tensor] = None,
                    dbg_sel: Optional[torch.Tensor] = None, stream: Optional[torch.cuda.Stream] = None) -> None:
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.msa_decode_step(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), ctypes.byref(cache.c), _ptr(q),
                                _ptr(index_q), float(softmax_scale), _ptr(dbg_block_scores), _ptr(dbg_sel),
                                _ptr(workspace), ws_bytes, _ptr(out), _stream(stream)), "msa_decode_step")


def msa_decode_step_host(batch: Batch, cache: Cache, host_qsl: torch.Tensor, host_seq_lens: torch.Tensor,
                         host_block_table: torch.Tensor, host_q: torch.Tensor, host_index_q: torch.Tensor,
                         host_out: torch.Tensor, q: torch.Tensor, index_q: torch.Tensor, softmax_scale: float,
                         workspace: torch.Tensor, out: Optional[torch.Tensor], copy_stream: torch.cuda.Stream,
                         direct_out: bool = False, stream: Optional[torch.cuda.Stream] = None) -> None:
    """msa_decode_step from page-locked host tensors: `batch`'s device arrays, q and index_q are
    filled from the host ones and host_out receives the output (copied back from `out`, or with
    direct_out stored there by the attention itself), the copies on copy_stream and `stream`
    overlapping the kernels (include/msa.h). host_out is complete once `stream` has passed the
    call."""
    for n, t in (("host_qsl", host_qsl), ("host_seq_lens", host_seq_lens), ("host_block_table", host_block_table),
                 ("host_q", host_q), ("host_index_q", host_index_q), ("host_out", host_out)):
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous page-locked host tensor")
    io = msa_host_step_io(host_qsl.data_ptr(), host_seq_lens.data_ptr(), host_block_table.data_ptr(),
                          host_q.data_ptr(), host_index_q.data_ptr(), host_out.data_ptr())
    ws_bytes = workspace.numel() * workspace.element_size()
    _check(_lib.msa_decode_step_host(ctypes.byref(GEOMETRY), ctypes.byref(batch.c), ctypes.byref(cache.c),
                                     ctypes.byref(io), _ptr(q), _ptr(index_q), float(softmax_scale), _ptr(workspace),
                                     ws_bytes, _ptr(out), MSA_HOST_STEP_DIRECT_OUT if direct_out else 0,
                                     _stream(stream), _stream(copy_stream)),
           "msa_decode_step_host")


def msa_read_device_status(workspace: torch.Tensor) -> int:
    return int(_lib.msa_read_device_status(_ptr(workspace), _stream()))


def msa_selftest_wait_timeout(status: torch.Tensor, limit_ns: int) -> None:
    _check(_lib.msa_selftest_wait_timeout(_ptr(status), int(limit_ns), _stream()), "msa_selftest_wait_timeout")


def status_bits(status: torch.Tensor) -> int:
    """Bits of a device status word (1 << msa_status code)."""
    return int(status.view(torch.int32)[0].item()) & 0xFFFFFFFF
