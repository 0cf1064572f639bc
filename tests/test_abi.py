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


def test_row_mode_workspace_sizes(lib):
    f = lib.csa2_workspace_bytes
    out = ctypes.c_size_t(0)
    args = lambda op, L, blk, nk, k, T: (op, 1, ctypes.c_int64(L), blk, nk, k, ctypes.c_int64(T), 16, 128,
                                          ctypes.byref(out))
    # verify rows: sized by rows and pool, independent of the context
    assert f(*args(4, 0, 8, 2048, 512, 160)) == 0
    v160 = out.value
    assert f(*args(4, 0, 8, 2048, 512, 320)) == 0 and out.value > v160
    assert f(*args(4, 0, 8, 2048, 512, 70000)) == 1        # more than 65,535 rows
    assert f(*args(4, 0, 8, 16, 32, 5)) == 1               # topk > n_keep_blocks
    # chunked rows: per-row tables for every row plus one group's selection workspace
    assert f(*args(5, 262144, 8, 2048, 512, 4096)) == 0
    c4096 = out.value
    assert c4096 > 1024 * 262144 * 4                       # the group's stored scores alone
    assert f(*args(5, 262144, 8, 2048, 512, 1024)) == 0 and out.value < c4096
    assert f(*args(5, 262144, 8, 2048, 512, (1 << 24) + 1)) == 1
    assert f(*args(5, 262144, 5, 2048, 512, 16)) == 1      # block not a power of two
    # every supported block size; fewer, larger blocks never need more workspace
    sizes = []
    for blk in (1, 2, 4, 8, 16):
        assert f(*args(5, 262144, blk, 2048, 512, 1024)) == 0
        sizes.append(out.value)
    assert sizes == sorted(sizes, reverse=True) and sizes[0] > sizes[-1]
    assert f(*args(5, 262144, 32, 2048, 512, 1024)) == 1   # block beyond 16


def test_row_mode_entry_points_reject_bad_arguments_without_a_gpu(lib):
    z64, zsz = ctypes.c_int64, ctypes.c_size_t
    assert lib.indexer_verify_select(None, None, None, None, None, z64(5), None, 8, 2048, 512, z64(100), None, None,
                                     zsz(0), None, None) == 1
    assert lib.indexer_chunked_select(None, None, None, None, None, z64(5), 8, 2048, 512, z64(100), None, None, None,
                                      zsz(0), None, None) == 1
    assert lib.indexer_reindex_select_static(None, None, None, None, 8, 2048, 512, z64(100), None, None, None) == 1
    assert lib.csa2_test_chunk_scores(None, None, None, None, None, z64(16), z64(100), None, None, None, zsz(0),
                                      None, None) == 1
    err = ctypes.c_int32(0)
    # no ring descriptors, or more sequences than the limit
    assert lib.swa_refill_fp8(None, 1, 4, None, None, None, z64(1), None, None, z64(1), ctypes.byref(err), None) == 1
    assert lib.swa_refill_fp8(None, 1, 5000, None, None, None, z64(1), None, None, z64(1), ctypes.byref(err),
                              None) == 1


def test_device_memo_keeps_each_devices_own_values(lib):
    """The per-device launch-fact table: values are kept per (device, site, key), the first
    stored value wins, a negative (failed) value is not kept, and concurrent first calls from
    many host threads agree on one value."""
    import threading
    f = lib.csa2_test_device_memo
    f.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int]
    f.restype = ctypes.c_int
    site = 1000                                   # a site no kernel uses
    assert f(0, site, 7, 148) == 148
    assert f(1, site, 7, 132) == 132             # another device keeps its own value
    assert f(0, site, 7, 999) == 148 and f(1, site, 7, 999) == 132
    assert f(0, site, 8, 3) == 3                 # another key on the same device
    assert f(5, site, 1, -1) == -1 and f(5, site, 1, 4) == 4      # a failure is retried
    got = []
    def worker(v):
        got.append(f(9, site, 42, v))
    ts = [threading.Thread(target=worker, args=(v,)) for v in range(1, 33)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert len(set(got)) == 1 and f(9, site, 42, 0) == got[0]
