"""The C-ABI library loads and exports every function include/msa.h declares; host-side
argument checks reject bad calls before anything is launched (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "msa.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(msa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__

    return ctypes.CDLL(__graft_entry__._load_builder().build())


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("msa_quantize_nvfp4", "msa_indexer_decode", "msa_topk_blocks", "msa_sparse_attn_decode",
              "msa_decode_step"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings_and_version(lib):
    lib.msa_status_string.restype = ctypes.c_char_p
    for code in range(6):
        assert lib.msa_status_string(code).startswith(b"MSA_")
    assert lib.msa_abi_version() == 1


def test_host_checks_without_gpu(lib):
    # rows < 0, cols not a multiple of 16, null pointers: rejected before any CUDA call
    f = lib.msa_quantize_nvfp4
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int64,
                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p]
    assert f(None, -1, 128, None, 64, None, 8, None) == 1
    assert f(None, 4, 100, None, 64, None, 8, None) == 1
    assert f(None, 4, 128, None, 64, None, 8, None) == 1
    assert f(None, 0, 128, None, 64, None, 8, None) == 0  # nothing to do

    class Geo(ctypes.Structure):
        _fields_ = [(n, ctypes.c_int32) for n in "abcdefgh"]

    bad = Geo(64, 8, 128, 128, 128, 16, 1, 0)  # 8 KV heads: not this method's geometry
    good = Geo(64, 4, 128, 128, 128, 16, 1, 0)
    ws = lib.msa_decode_workspace_size
    ws.restype = ctypes.c_size_t
    ws.argtypes = [ctypes.POINTER(Geo), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32]
    assert ws(ctypes.byref(bad), 4, 4, 32) == 0
    n = ws(ctypes.byref(good), 64, 512, 1024)
    # header + scores [T,4,maxb] f32 + sel [T,4,16] i32 (+ no split partials at B=64)
    assert n == 256 + 512 * 4 * 1024 * 4 + 512 * 4 * 16 * 4
    n1 = ws(ctypes.byref(good), 1, 1, 32)
    assert n1 > 256 + 1 * 4 * 32 * 4  # B=1 splits its work: partials need room
    g = lib.msa_topk_blocks
    g.argtypes = [ctypes.POINTER(Geo), ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p]
    assert g(ctypes.byref(bad), None, None, None, None, None) == 2
    assert g(ctypes.byref(good), None, None, None, None, None) == 1


def test_host_step_checks_without_gpu(lib):
    """msa_decode_step_host rejects bad geometry, a missing batch or host description and
    unknown flags before it makes any CUDA call."""

    class Geo(ctypes.Structure):
        _fields_ = [(n, ctypes.c_int32) for n in "abcdefgh"]

    class Batch(ctypes.Structure):
        _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("qsl", ctypes.c_void_p),
                    ("seq_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p), ("maxb", ctypes.c_int32),
                    ("max_q_len", ctypes.c_int32)]

    class Cache(ctypes.Structure):
        _fields_ = [("kv", ctypes.c_void_p), ("ix", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                    ("pages", ctypes.c_int32)]

    f = lib.msa_decode_step_host
    f.restype = ctypes.c_int32
    f.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                          ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p]
    bad = Geo(64, 8, 128, 128, 128, 16, 1, 0)
    good = Geo(64, 4, 128, 128, 128, 16, 1, 0)
    dummy = ctypes.c_void_p(0x1000)  # never dereferenced: the checks stop before any access
    batch = Batch(1, 1, dummy, dummy, dummy, 1, 1)
    cache = Cache(dummy, dummy, 0, 1)
    args = lambda geo, b, c, host, flags: (ctypes.byref(geo), b, c, host, None, None, 0.1, dummy, 1 << 20, None,
                                           flags, None, None)
    assert f(*args(bad, ctypes.byref(batch), ctypes.byref(cache), None, 0)) == 2          # unsupported geometry
    assert f(*args(good, None, ctypes.byref(cache), None, 0)) == 1                        # no batch
    assert f(*args(good, ctypes.byref(batch), ctypes.byref(cache), None, 0)) == 1         # no host description
    io = (ctypes.c_void_p * 6)(*([0x2000] * 6))
    assert f(*args(good, ctypes.byref(batch), ctypes.byref(cache), ctypes.byref(io), 4)) == 1  # unknown flag


def test_prefill_indexer_and_selection_checks_without_gpu(lib):
    """msa_indexer_prefill and msa_topk_prefill take prefill batches (more than 8 query tokens a
    sequence) and reject bad geometry, batches and caches before any CUDA call; an empty batch
    is a successful no-op."""

    class Geo(ctypes.Structure):
        _fields_ = [(n, ctypes.c_int32) for n in "abcdefgh"]

    class Batch(ctypes.Structure):
        _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("qsl", ctypes.c_void_p),
                    ("seq_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p), ("maxb", ctypes.c_int32),
                    ("max_q_len", ctypes.c_int32)]

    class Cache(ctypes.Structure):
        _fields_ = [("kv", ctypes.c_void_p), ("ix", ctypes.c_void_p), ("dtype", ctypes.c_int32),
                    ("pages", ctypes.c_int32)]

    ix = lib.msa_indexer_prefill
    ix.restype = ctypes.c_int32
    ix.argtypes = [ctypes.c_void_p] * 7
    tk = lib.msa_topk_prefill
    tk.restype = ctypes.c_int32
    tk.argtypes = [ctypes.c_void_p] * 6
    good = Geo(64, 4, 128, 128, 128, 16, 1, 0)
    bad = Geo(64, 4, 128, 128, 64, 16, 1, 0)  # 64-token blocks
    dummy = 0x1000  # never dereferenced: the checks stop before any access
    cache = Cache(0x10000, 0x10000, 0, 8)
    no_index = Cache(0x10000, None, 0, 8)
    empty = Batch(0, 0, dummy, dummy, dummy, 16, 1)
    long_prompt = Batch(1, 0, dummy, dummy, dummy, 16, 1 << 20)  # up to 2^20 tokens a sequence: accepted
    too_long = Batch(1, 4, dummy, dummy, dummy, 16, (1 << 20) + 1)
    too_many = Batch(1, (1 << 22) + 1, dummy, dummy, dummy, 16, 1 << 20)
    r = lambda p: ctypes.byref(p)
    assert ix(r(bad), r(empty), r(cache), None, None, None, None) == 2
    assert ix(r(good), None, r(cache), None, None, None, None) == 1
    assert ix(r(good), r(too_long), r(cache), None, None, None, None) == 1
    assert ix(r(good), r(too_many), r(cache), None, None, None, None) == 1
    assert ix(r(good), r(empty), r(no_index), None, None, None, None) == 1
    assert ix(r(good), r(empty), r(cache), None, None, None, None) == 0
    assert ix(r(good), r(long_prompt), r(cache), None, None, None, None) == 0  # T = 0: nothing to do
    assert tk(r(bad), r(empty), None, None, None, None) == 2
    assert tk(r(good), r(too_long), None, None, None, None) == 1
    assert tk(r(good), r(long_prompt), None, None, None, None) == 0
    # the decode selection keeps its own limit of 8 query tokens a sequence
    dk = lib.msa_topk_blocks
    dk.restype = ctypes.c_int32
    dk.argtypes = [ctypes.c_void_p] * 6
    assert dk(r(good), r(long_prompt), None, None, None, None) == 1
