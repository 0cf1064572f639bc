"""The C-ABI library loads, exports every declared symbol and validates arguments on the host.

CPU only: nothing here launches a kernel.  Invalid arguments are rejected
before any CUDA call, so the return codes can be checked without a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LIB = os.path.join(ROOT, "sparse_attention_fp4_02_b300", "libcsa2.so")


def _declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while")))


@pytest.fixture(scope="module")
def lib():
    return ctypes.CDLL(LIB)


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_binding_names_match_the_abi():
    import sparse_attention_fp4_02_b300 as m
    for n in ("kv_append_fp4", "indexer_full_select", "indexer_reindex_select", "sparse_attn_decode"):
        assert callable(getattr(m, n))
    assert set(m.EXPORTED) == set(_declared_functions())


def test_status_strings(lib):
    lib.csa2_status_string.restype = ctypes.c_char_p
    assert lib.csa2_status_string(0) == b"ok"
    assert b"invalid" in lib.csa2_status_string(1)


def test_workspace_sizes(lib):
    f = lib.csa2_workspace_bytes
    out = ctypes.c_size_t(0)
    args = lambda op, B, L, blk, nk, k: (op, B, ctypes.c_int64(L), blk, nk, k, ctypes.c_int64(0), 16, 128,
                                          ctypes.byref(out))
    assert f(*args(1, 32, 65536, 8, 2048, 512)) == 0 and out.value > 32 * 65536 // 8 * 12
    assert f(*args(1, 32, 65536, 3, 2048, 512)) == 1       # block must be a power of two <= 16
    assert f(*args(1, 32, 65536, 8, 2048, 4096)) == 1      # topk beyond 1024
    assert f(*args(1, 0, 65536, 8, 2048, 512)) == 1        # B < 1
    assert f(*args(1, 2000, 65536, 8, 2048, 512)) == 1     # B beyond 1024
    assert f(*args(1, 4, 100, 8, 16, 32)) == 1             # topk > n_keep_blocks
    assert f(*args(9, 4, 100, 8, 16, 8)) == 1              # unknown op


def test_entry_points_reject_null_arguments_without_a_gpu(lib):
    # every entry point validates before touching CUDA: null cache -> invalid argument
    P = ctypes.c_void_p
    assert lib.kv_append_fp4(None, None, 0, None, None, None, None, None, ctypes.c_int64(1), None, None,
                             ctypes.c_int64(0), None, None) == 1
    assert lib.indexer_full_select(None, None, None, 8, 2048, 512, ctypes.c_int64(100), None, None, None,
                                   ctypes.c_size_t(0), None, None, None) == 1
    assert lib.indexer_reindex_select(None, None, None, None, 8, 2048, 512, ctypes.c_int64(100), None, None,
                                      ctypes.c_size_t(0), None, None) == 1
    assert lib.sparse_attn_decode(None, None, None, 16, ctypes.c_int64(1), None, None, None, 512, 128,
                                  ctypes.c_float(0.088), None, None, None, ctypes.c_size_t(0), None, None) == 1
    assert lib.csa2_test_quantize_fp4(None, ctypes.c_int64(4), None, None, None) == 1
    assert lib.csa2_test_quantize_fp8(None, ctypes.c_int64(4), 100, None, None, None) == 1
    assert lib.csa2_test_index_scores(None, None, None, ctypes.c_int64(1), None, None, None, ctypes.c_size_t(0),
                                      None, None) == 1


def test_misaligned_cache_rejected_without_a_gpu(lib):
    import sparse_attention_fp4_02_b300 as m
    buf = ctypes.create_string_buffer(4096 + 64)
    base = (ctypes.addressof(buf) + 63) // 64 * 64
    desc = m.CacheDesc(base + 1, base + 1024, base + 2048, base + 3072, base, base + 8, 1, 16)
    err = ctypes.c_int32(0)
    r = lib.kv_append_fp4(ctypes.byref(desc), None, 0, None, None, None, None, None, ctypes.c_int64(1), None, None,
                          ctypes.c_int64(0), ctypes.byref(err), None)
    assert r == 1          # kv_codes not 16-byte aligned
