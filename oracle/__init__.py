"""Plain CPU oracle of the MSA decode step over a paged NVFP4 cache.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference leg may import this package. The product path (the CUDA library in
``nvfp4_kv_cache_gb300``) never imports, links or calls it, and the two share no code.

The arithmetic lives in ``msa_oracle.cpp`` (plain C++, fp64, one thread per (token, group)
unit); this module builds it with g++, loads it with ctypes and adds numpy-level wrappers
plus the byte layout of the cache pages, which the oracle defines independently of the
CUDA side so that tests can read GPU-written pages back into logical rows.

Sources (page title, section) are cited in ``msa_oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "msa_oracle.cpp")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle_msa.so")

# Geometry of the method ("MiniMax-M3.1-Flash serving notes", "The architecture, in operator
# terms": 64 query heads, 4 KV heads, head dim 128; "vLLM ofrece soporte en día 0 ...",
# "MSA primer": 128-token blocks, 16 selected blocks).
HEAD_DIM = 128
GROUPS = 4
HEADS_PER_GROUP = 16
Q_HEADS = GROUPS * HEADS_PER_GROUP
BLOCK = 128
K_SEL = 16

INDEX_NVFP4 = 0
INDEX_FP8 = 1
INDEX_NVFP4_EXACT = 2  # the exact-score reading of an NVFP4 index cache (no E4M3 re-rounding)

# Byte layout of one cache page (this library's choice; the pages fix none).
ROW_CODE_BYTES = HEAD_DIM // 2          # 64 B of E2M1 codes per 128-element row
ROW_SCALE_BYTES = HEAD_DIM // 16        # 8 E4M3 scales per row
REGION_BYTES = BLOCK * (ROW_CODE_BYTES + ROW_SCALE_BYTES)  # codes of 128 rows, then scales
INDEX_PAGE_BYTES = {INDEX_NVFP4: REGION_BYTES, INDEX_FP8: BLOCK * HEAD_DIM}
KV_PAGE_BYTES = GROUPS * 2 * REGION_BYTES  # [head][K, V][region]

_lib = None
_lock = threading.Lock()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle_msa.so`` (g++, no GPU needed)."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= os.path.getmtime(SRC):
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", SRC, "-o", tmp]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            i32p = ctypes.POINTER(ctypes.c_int32)
            L.orc_e4m3_decode.restype = ctypes.c_double
            L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.orc_e4m3_encode.restype = ctypes.c_uint8
            L.orc_e4m3_encode.argtypes = [ctypes.c_double]
            L.orc_e2m1_decode.restype = ctypes.c_double
            L.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
            L.orc_e2m1_encode.restype = ctypes.c_uint8
            L.orc_e2m1_encode.argtypes = [ctypes.c_float]
            L.orc_dequant_fp8.restype = ctypes.c_uint8
            L.orc_dequant_fp8.argtypes = [ctypes.c_uint8, ctypes.c_uint8]
            L.orc_quantize_fp8.argtypes = [f32p, ctypes.c_int64, u8p]
            L.orc_quantize_nvfp4.argtypes = [f32p, ctypes.c_int64, ctypes.c_int32, u8p, u8p]
            L.orc_unpack_nvfp4.argtypes = [u8p, ctypes.c_int64, ctypes.c_int32, u8p]
            L.orc_pack_nvfp4.argtypes = [u8p, ctypes.c_int64, ctypes.c_int32, u8p]
            L.orc_dequant_nvfp4.argtypes = [u8p, u8p, ctypes.c_int64, ctypes.c_int32, u8p]
            L.orc_indexer_seq.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, u8p, u8p,
                                          u8p, f64p, ctypes.c_int32, ctypes.c_int32]
            L.orc_select_row.argtypes = [f64p, ctypes.c_int32, ctypes.c_int32, i32p]
            L.orc_attention_seq.argtypes = [ctypes.c_int32, ctypes.c_int32, u8p, u8p, u8p, u8p, u8p,
                                            i32p, ctypes.c_double, f64p, f64p, ctypes.c_int32]
            L.orc_hardware_threads.restype = ctypes.c_int32
            _lib = L
    return _lib


def _p(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a), dtype=dtype)


def hardware_threads() -> int:
    return int(lib().orc_hardware_threads())


# ---------------------------------------------------------------------------- formats
def e4m3_decode(b) -> np.ndarray:
    b = _c(b, np.uint8)
    table = np.array([lib().orc_e4m3_decode(i) for i in range(256)], dtype=np.float64)
    return table[b]


def e4m3_encode(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return np.vectorize(lambda v: lib().orc_e4m3_encode(float(v)), otypes=[np.uint8])(x)


def e2m1_decode(c) -> np.ndarray:
    c = _c(c, np.uint8)
    table = np.array([lib().orc_e2m1_decode(i) for i in range(16)], dtype=np.float64)
    return table[c & 15]


def e2m1_encode(r) -> np.ndarray:
    r = np.asarray(r, dtype=np.float32)
    return np.vectorize(lambda v: lib().orc_e2m1_encode(float(v)), otypes=[np.uint8])(r)


def dequant_table() -> np.ndarray:
    """[256 scales][16 codes] -> E4M3 byte of E2M1(code) * E4M3(scale), re-rounded."""
    L = lib()
    return np.array([[L.orc_dequant_fp8(c, s) for c in range(16)] for s in range(256)], dtype=np.uint8)


def quantize_fp8(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().orc_quantize_fp8(_p(x, ctypes.c_float), x.size, _p(out, ctypes.c_uint8))
    return out


def quantize_nvfp4(x):
    """x[..., cols] fp32 -> (vals[..., cols/2], scales[..., cols/16]) in this library's layout."""
    x = _c(x, np.float32)
    cols = x.shape[-1]
    assert cols % 16 == 0
    rows = x.size // cols if cols else 0
    vals = np.empty(x.shape[:-1] + (cols // 2,), dtype=np.uint8)
    scales = np.empty(x.shape[:-1] + (cols // 16,), dtype=np.uint8)
    lib().orc_quantize_nvfp4(_p(x, ctypes.c_float), rows, cols, _p(vals, ctypes.c_uint8),
                             _p(scales, ctypes.c_uint8))
    return vals, scales


def unpack_nvfp4(vals) -> np.ndarray:
    vals = _c(vals, np.uint8)
    cols = vals.shape[-1] * 2
    rows = vals.size // vals.shape[-1]
    codes = np.empty(vals.shape[:-1] + (cols,), dtype=np.uint8)
    lib().orc_unpack_nvfp4(_p(vals, ctypes.c_uint8), rows, cols, _p(codes, ctypes.c_uint8))
    return codes


def pack_nvfp4(codes) -> np.ndarray:
    codes = _c(codes, np.uint8)
    cols = codes.shape[-1]
    rows = codes.size // cols
    vals = np.empty(codes.shape[:-1] + (cols // 2,), dtype=np.uint8)
    lib().orc_pack_nvfp4(_p(codes, ctypes.c_uint8), rows, cols, _p(vals, ctypes.c_uint8))
    return vals


def dequant_nvfp4(vals, scales) -> np.ndarray:
    """NVFP4 rows -> FP8 (E4M3) bytes of the dequantised values."""
    vals = _c(vals, np.uint8)
    scales = _c(scales, np.uint8)
    cols = vals.shape[-1] * 2
    rows = vals.size // vals.shape[-1]
    out = np.empty(vals.shape[:-1] + (cols,), dtype=np.uint8)
    lib().orc_dequant_nvfp4(_p(vals, ctypes.c_uint8), _p(scales, ctypes.c_uint8), rows, cols,
                            _p(out, ctypes.c_uint8))
    return out


# ---------------------------------------------------------------------------- method steps
def indexer_seq(L: int, q_len: int, iq, index_dtype: int, ik_vals, ik_scales=None,
                nthreads: int = 0) -> np.ndarray:
    """Block scores [q_len, 4, nb] (fp64) of one sequence from its logical index cache."""
    nb = (L + BLOCK - 1) // BLOCK
    iq = _c(iq, np.uint8).reshape(q_len, GROUPS, HEAD_DIM)
    ik_vals = _c(ik_vals, np.uint8)
    if index_dtype in (INDEX_NVFP4, INDEX_NVFP4_EXACT):
        ik_scales = _c(ik_scales, np.uint8)
        assert ik_vals.shape == (L, ROW_CODE_BYTES) and ik_scales.shape == (L, ROW_SCALE_BYTES)
    else:
        assert ik_vals.shape == (L, HEAD_DIM)
        ik_scales = np.zeros((1,), dtype=np.uint8)
    out = np.empty((q_len, GROUPS, max(nb, 1)), dtype=np.float64)
    lib().orc_indexer_seq(L, q_len, index_dtype, _p(iq, ctypes.c_uint8), _p(ik_vals, ctypes.c_uint8),
                          _p(ik_scales, ctypes.c_uint8), _p(out, ctypes.c_double), out.shape[2],
                          nthreads)
    return out[:, :, :nb]


def select_row(scores, local: int) -> np.ndarray:
    """sel[16] of one (token, group) row from its block scores (any float dtype)."""
    s = _c(scores, np.float64)
    sel = np.empty(K_SEL, dtype=np.int32)
    lib().orc_select_row(_p(s, ctypes.c_double), s.size, int(local), _p(sel, ctypes.c_int32))
    return sel


def select_seq(scores, L: int, q_len: int) -> np.ndarray:
    """sel [q_len, 4, 16] for one sequence from its block scores [q_len, 4, nb]."""
    scores = np.asarray(scores)
    out = np.empty((q_len, GROUPS, K_SEL), dtype=np.int32)
    for t in range(q_len):
        local = (L - q_len + t) // BLOCK
        for g in range(GROUPS):
            out[t, g] = select_row(scores[t, g], local)
    return out


def attention_seq(L: int, q_len: int, q, k_vals, k_scales, v_vals, v_scales, sel,
                  softmax_scale: float, nthreads: int = 0, want_lse: bool = False):
    """Sparse GQA attention of one sequence: out [q_len, 64, 128] fp64 (and lse)."""
    q = _c(q, np.uint8).reshape(q_len, Q_HEADS, HEAD_DIM)
    k_vals = _c(k_vals, np.uint8).reshape(L, GROUPS, ROW_CODE_BYTES)
    k_scales = _c(k_scales, np.uint8).reshape(L, GROUPS, ROW_SCALE_BYTES)
    v_vals = _c(v_vals, np.uint8).reshape(L, GROUPS, ROW_CODE_BYTES)
    v_scales = _c(v_scales, np.uint8).reshape(L, GROUPS, ROW_SCALE_BYTES)
    sel = _c(sel, np.int32).reshape(q_len, GROUPS, K_SEL)
    out = np.empty((q_len, Q_HEADS, HEAD_DIM), dtype=np.float64)
    lse = np.empty((q_len, Q_HEADS), dtype=np.float64)
    lib().orc_attention_seq(L, q_len, _p(q, ctypes.c_uint8), _p(k_vals, ctypes.c_uint8),
                            _p(k_scales, ctypes.c_uint8), _p(v_vals, ctypes.c_uint8),
                            _p(v_scales, ctypes.c_uint8), _p(sel, ctypes.c_int32),
                            float(softmax_scale), _p(out, ctypes.c_double), _p(lse, ctypes.c_double),
                            nthreads)
    return (out, lse) if want_lse else out


# ---------------------------------------------------------------------------- page layout
def index_row_offsets(page: int, row: int, index_dtype: int):
    """Byte offsets of (codes, scales) of token `row` of index page `page`."""
    base = page * INDEX_PAGE_BYTES[index_dtype]
    if index_dtype == INDEX_FP8:
        return base + row * HEAD_DIM, None
    return base + row * ROW_CODE_BYTES, base + BLOCK * ROW_CODE_BYTES + row * ROW_SCALE_BYTES


def kv_region_offset(page: int, head: int, kind: int) -> int:
    """Byte offset of the K (kind 0) or V (kind 1) region of `head` in KV page `page`."""
    return page * KV_PAGE_BYTES + (head * 2 + kind) * REGION_BYTES


def gather_index_rows(index_pages: np.ndarray, block_row, L: int, index_dtype: int):
    """Read a sequence's index keys out of raw page bytes into logical rows."""
    pages = np.asarray(index_pages, dtype=np.uint8).reshape(-1, INDEX_PAGE_BYTES[index_dtype])
    nb = (L + BLOCK - 1) // BLOCK
    blk = np.asarray(block_row[:nb], dtype=np.int64)
    if index_dtype == INDEX_FP8:
        rows = pages[blk].reshape(nb * BLOCK, HEAD_DIM)
        return rows[:L], None
    codes = pages[blk, : BLOCK * ROW_CODE_BYTES].reshape(nb * BLOCK, ROW_CODE_BYTES)
    scales = pages[blk, BLOCK * ROW_CODE_BYTES:].reshape(nb * BLOCK, ROW_SCALE_BYTES)
    return codes[:L], scales[:L]


def gather_kv_rows(kv_pages: np.ndarray, block_row, L: int):
    """Read a sequence's K/V out of raw page bytes: (k_vals, k_scales, v_vals, v_scales)."""
    pages = np.asarray(kv_pages, dtype=np.uint8).reshape(-1, GROUPS, 2, REGION_BYTES)
    nb = (L + BLOCK - 1) // BLOCK
    blk = np.asarray(block_row[:nb], dtype=np.int64)
    sel = pages[blk]  # [nb, 4, 2, region]
    codes = sel[..., : BLOCK * ROW_CODE_BYTES].reshape(nb, GROUPS, 2, BLOCK, ROW_CODE_BYTES)
    scales = sel[..., BLOCK * ROW_CODE_BYTES:].reshape(nb, GROUPS, 2, BLOCK, ROW_SCALE_BYTES)
    # -> [token, head, bytes]
    codes = codes.transpose(0, 3, 1, 2, 4).reshape(nb * BLOCK, GROUPS, 2, ROW_CODE_BYTES)[:L]
    scales = scales.transpose(0, 3, 1, 2, 4).reshape(nb * BLOCK, GROUPS, 2, ROW_SCALE_BYTES)[:L]
    return (np.ascontiguousarray(codes[:, :, 0]), np.ascontiguousarray(scales[:, :, 0]),
            np.ascontiguousarray(codes[:, :, 1]), np.ascontiguousarray(scales[:, :, 1]))


def scatter_index_rows(index_pages: np.ndarray, block_row, vals, scales, index_dtype: int) -> None:
    """Write logical index rows of one sequence into raw page bytes (inverse of gather)."""
    pages = index_pages.reshape(-1, INDEX_PAGE_BYTES[index_dtype])
    L = vals.shape[0]
    for j in range(L):
        pg, r = int(block_row[j // BLOCK]), j % BLOCK
        if index_dtype == INDEX_FP8:
            pages[pg, r * HEAD_DIM:(r + 1) * HEAD_DIM] = vals[j]
        else:
            pages[pg, r * ROW_CODE_BYTES:(r + 1) * ROW_CODE_BYTES] = vals[j]
            o = BLOCK * ROW_CODE_BYTES + r * ROW_SCALE_BYTES
            pages[pg, o:o + ROW_SCALE_BYTES] = scales[j]


def scatter_kv_rows(kv_pages: np.ndarray, block_row, k_vals, k_scales, v_vals, v_scales) -> None:
    pages = kv_pages.reshape(-1, GROUPS, 2, REGION_BYTES)
    L = k_vals.shape[0]
    for j in range(L):
        pg, r = int(block_row[j // BLOCK]), j % BLOCK
        for g in range(GROUPS):
            for kind, (cv, sv) in enumerate(((k_vals, k_scales), (v_vals, v_scales))):
                pages[pg, g, kind, r * ROW_CODE_BYTES:(r + 1) * ROW_CODE_BYTES] = cv[j, g]
                o = BLOCK * ROW_CODE_BYTES + r * ROW_SCALE_BYTES
                pages[pg, g, kind, o:o + ROW_SCALE_BYTES] = sv[j, g]


# ---------------------------------------------------------------------------- whole batch
def decode_batch(seq_lens, q_lens, iq, q, index_dtype, ik, kv, softmax_scale: float,
                 sel_override: Optional[list] = None, nthreads: int = 0):
    """Run indexer -> select -> attention for each sequence.

    ik[b] = (vals, scales) logical index rows; kv[b] = (k_vals, k_scales, v_vals, v_scales);
    iq[b] = [q_len, 4, 128] E4M3 bytes; q[b] = [q_len, 64, 128] E4M3 bytes.
    sel_override[b], when given, replaces the oracle's own selection (to run attention on the
    GPU's selected set). Returns per-sequence lists (scores, sel, out).
    """
    scores, sels, outs = [], [], []
    for b, (L, ql) in enumerate(zip(seq_lens, q_lens)):
        if ql == 0:
            scores.append(None); sels.append(None); outs.append(None)
            continue
        s = indexer_seq(L, ql, iq[b], index_dtype, ik[b][0], ik[b][1], nthreads)
        sel = select_seq(s, L, ql) if sel_override is None else np.asarray(sel_override[b])
        o = attention_seq(L, ql, q[b], *kv[b], sel, softmax_scale, nthreads)
        scores.append(s); sels.append(sel); outs.append(o)
    return scores, sels, outs
