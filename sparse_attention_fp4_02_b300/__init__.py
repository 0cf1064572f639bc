"""CSA2 decode over an FP4 global KV cache on B300 (sm_103a).

Thin Python binding of ``libcsa2.so`` (declared in ``include/csa2.h``).  The
functions here only marshal arguments: every step of the path runs in the
library's CUDA kernels.  PyTorch provides device memory and streams.  If the
library has not been built, importing this package raises: there is no CPU
fallback.

Entry points (same names as the C ABI): ``kv_append_fp4``, ``swa_refill_fp8``,
``indexer_full_select``, ``indexer_reindex_select``, ``indexer_reindex_select_static``,
``indexer_verify_select``, ``indexer_chunked_select``, ``sparse_attn_decode``, plus
``workspace_bytes`` and the ``Cache`` / ``SwaRing`` containers that own the device
tensors of the layouts the header documents.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# CSA2_LIB selects another build of the library (same ABI); default: the in-tree build
LIB_PATH = os.environ.get("CSA2_LIB") or os.path.join(_HERE, "libcsa2.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python sparse_attention_fp4_02_b300/build.py`")
_lib = ctypes.CDLL(LIB_PATH)

OK, ERR_INVALID_ARG, ERR_WORKSPACE, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE_TIMEOUT = range(6)
DEVERR_SEQ, DEVERR_POS, DEVERR_LEN, DEVERR_INDEX, DEVERR_POOL, DEVERR_TIMEOUT = 1, 2, 4, 8, 16, 32
OP_FULL_SELECT, OP_REINDEX_SELECT, OP_ATTN_DECODE, OP_VERIFY_SELECT, OP_CHUNKED_SELECT = 1, 2, 3, 4, 5
D, D_IDX, H_IDX = 128, 64, 8
MAX_SWA_LAYERS = 32


class CacheDesc(ctypes.Structure):
    _fields_ = [("kv_codes", ctypes.c_void_p), ("kv_scales", ctypes.c_void_p), ("ik_codes", ctypes.c_void_p),
                ("ik_scale", ctypes.c_void_p), ("seq_base", ctypes.c_void_p), ("seq_len", ctypes.c_void_p),
                ("B", ctypes.c_int32), ("T_cap", ctypes.c_int64)]


class SwaDesc(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("ring", ctypes.c_int32)]


class ProfileDesc(ctypes.Structure):
    _fields_ = [("start", ctypes.c_void_p), ("stop", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I32, _I64, _F32, _SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t


def _sig(name, args):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = ctypes.c_int
    return f


_lib.csa2_status_string.argtypes = [ctypes.c_int]
_lib.csa2_status_string.restype = ctypes.c_char_p
_ws_bytes = _sig("csa2_workspace_bytes", [ctypes.c_int, _I32, _I64, _I32, _I32, _I32, _I64, _I32, _I32,
                                          ctypes.POINTER(_SZ)])
_append = _sig("kv_append_fp4", [_P, _P, _I32, _P, _P, _P, _P, _P, _I64, _P, _P, _I64, _P, _P])
_refill = _sig("swa_refill_fp8", [_P, _I32, _I32, _P, _P, _P, _I64, _P, _P, _I64, _P, _P])
_full = _sig("indexer_full_select", [_P, _P, _P, _I32, _I32, _I32, _I64, _P, _P, _P, _SZ, _P, _P, _P])
_reindex = _sig("indexer_reindex_select", [_P, _P, _P, _P, _I32, _I32, _I32, _I64, _P, _P, _SZ, _P, _P])
_reindex_static = _sig("indexer_reindex_select_static", [_P, _P, _P, _P, _I32, _I32, _I32, _I64, _P, _P, _P])
_chunked = _sig("indexer_chunked_select", [_P, _P, _P, _P, _P, _I64, _I32, _I32, _I32, _I64, _P, _P, _P, _SZ, _P,
                                           _P])
_verify = _sig("indexer_verify_select", [_P, _P, _P, _P, _P, _I64, _P, _I32, _I32, _I32, _I64, _P, _P, _SZ, _P,
                                         _P])
_attn = _sig("sparse_attn_decode", [_P, _P, _P, _I32, _I64, _P, _P, _P, _I32, _I32, _F32, _P, _P, _P, _SZ,
                                    _P, _P])
_t_fp4 = _sig("csa2_test_quantize_fp4", [_P, _I64, _P, _P, _P])
_t_fp8 = _sig("csa2_test_quantize_fp8", [_P, _I64, _I32, _P, _P, _P])
_t_scores = _sig("csa2_test_index_scores", [_P, _P, _P, _I64, _P, _P, _P, _SZ, _P, _P])
_t_cscores = _sig("csa2_test_chunk_scores", [_P, _P, _P, _P, _P, _I64, _I64, _P, _P, _P, _SZ, _P, _P])
_t_memo = _sig("csa2_test_device_memo", [_I32, _I32, _I64, _I32])

EXPORTED = ("csa2_status_string", "csa2_workspace_bytes", "kv_append_fp4", "swa_refill_fp8", "indexer_full_select",
            "indexer_reindex_select", "indexer_reindex_select_static", "indexer_verify_select",
            "indexer_chunked_select", "sparse_attn_decode", "csa2_test_quantize_fp4", "csa2_test_quantize_fp8",
            "csa2_test_index_scores", "csa2_test_chunk_scores", "csa2_test_device_memo")


class Csa2Error(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


def status_string(status: int) -> str:
    return _lib.csa2_status_string(status).decode()


def _check(status: int, where: str):
    if status != OK:
        raise Csa2Error(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


class Cache:
    """Device tensors of one shared global cache (layouts as in csa2.h)."""

    def __init__(self, T_cap: int, B: int, device="cuda"):
        self.T_cap, self.B = int(T_cap), int(B)
        u8 = dict(dtype=torch.uint8, device=device)
        self.kv_codes = torch.empty((self.T_cap, D // 2), **u8)
        self.kv_scales = torch.empty((self.T_cap, D // 16), **u8)
        self.ik_codes = torch.empty((self.T_cap, D_IDX), **u8)
        self.ik_scale = torch.empty((self.T_cap,), dtype=torch.float32, device=device)
        self.seq_base = torch.zeros((self.B,), dtype=torch.int64, device=device)
        self.seq_len = torch.zeros((self.B,), dtype=torch.int32, device=device)

    def desc(self) -> CacheDesc:
        return CacheDesc(self.kv_codes.data_ptr(), self.kv_scales.data_ptr(), self.ik_codes.data_ptr(),
                         self.ik_scale.data_ptr(), self.seq_base.data_ptr(), self.seq_len.data_ptr(),
                         self.B, self.T_cap)


class SwaRing:
    """One layer's FP8 sliding-window ring: codes [B][ring][128] u8, scale [B][ring] f32."""

    def __init__(self, B: int, ring: int, device="cuda"):
        self.ring = int(ring)
        self.codes = torch.zeros((B, self.ring, D), dtype=torch.uint8, device=device)
        self.scale = torch.zeros((B, self.ring), dtype=torch.float32, device=device)

    def desc(self) -> SwaDesc:
        return SwaDesc(self.codes.data_ptr(), self.scale.data_ptr(), self.ring)


def workspace_bytes(op: int, B=1, max_len=0, block=8, n_keep_blocks=2048, topk=512, T=0, H=16, window=128) -> int:
    out = _SZ(0)
    _check(_ws_bytes(op, B, max_len, block, n_keep_blocks, topk, T, H, window, ctypes.byref(out)),
           "csa2_workspace_bytes")
    return int(out.value)


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """Caller-owned workspace (torch allocations are 256-byte aligned)."""
    return torch.empty((max(int(nbytes), 256),), dtype=torch.uint8, device=device)


def kv_append_fp4(cache: Cache, swa_layers, kv_new, ik_new, swa_new, rope_cos, rope_sin, seq_id, pos, d_err,
                  stream=None):
    n = int(seq_id.shape[0])
    layers = list(swa_layers or [])
    arr = (SwaDesc * max(1, len(layers)))(*[s.desc() for s in layers]) if layers else None
    _check(_append(ctypes.byref(cache.desc()), arr, len(layers), _ptr(kv_new), _ptr(ik_new), _ptr(swa_new),
                   _ptr(rope_cos), _ptr(rope_sin), int(rope_cos.shape[0]), _ptr(seq_id), _ptr(pos), n,
                   _ptr(d_err), _stream(stream)), "kv_append_fp4")


def swa_refill_fp8(swa_layers, B, swa_new, rope_cos, rope_sin, seq_id, pos, d_err, stream=None):
    """Re-append replayed window KV into every layer's FP8 ring (the global cache is not touched)."""
    layers = list(swa_layers)
    arr = (SwaDesc * len(layers))(*[s.desc() for s in layers])
    _check(_refill(arr, len(layers), int(B), _ptr(swa_new), _ptr(rope_cos), _ptr(rope_sin), int(rope_cos.shape[0]),
                   _ptr(seq_id), _ptr(pos), int(seq_id.shape[0]), _ptr(d_err), _stream(stream)), "swa_refill_fp8")


def indexer_full_select(cache: Cache, q_idx, w, block, n_keep_blocks, topk, max_len, pool_blocks, topk_idx, ws,
                        d_err, prof=None, stream=None):
    pd = None
    if prof is not None:
        pd = ctypes.byref(ProfileDesc(prof[0].cuda_event, prof[1].cuda_event))
    _check(_full(ctypes.byref(cache.desc()), _ptr(q_idx), _ptr(w), block, n_keep_blocks, topk, int(max_len),
                 _ptr(pool_blocks), _ptr(topk_idx), _ptr(ws), ws.numel(), _ptr(d_err), pd, _stream(stream)),
           "indexer_full_select")


def indexer_reindex_select(cache: Cache, q_idx, w, pool_blocks, block, n_keep_blocks, topk, max_len, topk_idx, ws,
                           d_err, stream=None):
    _check(_reindex(ctypes.byref(cache.desc()), _ptr(q_idx), _ptr(w), _ptr(pool_blocks), block, n_keep_blocks,
                    topk, int(max_len), _ptr(topk_idx), _ptr(ws), ws.numel(), _ptr(d_err), _stream(stream)),
           "indexer_reindex_select")


def indexer_reindex_select_static(cache: Cache, q_idx, w, pool_blocks, block, n_keep_blocks, topk, max_len,
                                  topk_idx, d_err, stream=None):
    """indexer_reindex_select without a workspace (scratch is a static array in the library)."""
    _check(_reindex_static(ctypes.byref(cache.desc()), _ptr(q_idx), _ptr(w), _ptr(pool_blocks), block,
                           n_keep_blocks, topk, int(max_len), _ptr(topk_idx), _ptr(d_err), _stream(stream)),
           "indexer_reindex_select_static")


def indexer_chunked_select(cache: Cache, q_idx, w, q_seq, q_pos, block, n_keep_blocks, topk, max_len, pool_blocks,
                           topk_idx, ws, d_err, stream=None):
    """Per query row: the Full selection over its session's positions up to its own."""
    _check(_chunked(ctypes.byref(cache.desc()), _ptr(q_idx), _ptr(w), _ptr(q_seq), _ptr(q_pos), int(q_seq.shape[0]),
                    block, n_keep_blocks, topk, int(max_len), _ptr(pool_blocks), _ptr(topk_idx), _ptr(ws), ws.numel(),
                    _ptr(d_err), _stream(stream)), "indexer_chunked_select")


def indexer_verify_select(cache: Cache, q_idx, w, q_seq, q_pos, pool_blocks, block, n_keep_blocks, topk, max_len,
                          topk_idx, ws, d_err, stream=None):
    """Per query row (session q_seq, position q_pos): top-k over the session's pool, causally limited."""
    _check(_verify(ctypes.byref(cache.desc()), _ptr(q_idx), _ptr(w), _ptr(q_seq), _ptr(q_pos), int(q_seq.shape[0]),
                   _ptr(pool_blocks), block, n_keep_blocks, topk, int(max_len), _ptr(topk_idx), _ptr(ws), ws.numel(),
                   _ptr(d_err), _stream(stream)), "indexer_verify_select")


def sparse_attn_decode(cache: Cache, swa: SwaRing, q, q_seq, q_pos, topk_idx, window, softmax_scale, out, lse, ws,
                       d_err, stream=None):
    T, H = int(q.shape[0]), int(q.shape[1])
    topk = int(topk_idx.shape[1]) if topk_idx is not None else 0
    _check(_attn(ctypes.byref(cache.desc()), ctypes.byref(swa.desc()), _ptr(q), H, T, _ptr(q_seq), _ptr(q_pos),
                 _ptr(topk_idx), topk, int(window), float(softmax_scale), _ptr(out), _ptr(lse), _ptr(ws),
                 ws.numel(), _ptr(d_err), _stream(stream)), "sparse_attn_decode")


# ---- test-only exports -------------------------------------------------------------

def test_quantize_fp4(x, codes, scales, stream=None):
    _check(_t_fp4(_ptr(x), int(x.shape[0]), _ptr(codes), _ptr(scales), _stream(stream)), "csa2_test_quantize_fp4")


def test_quantize_fp8(x, codes, scale, stream=None):
    _check(_t_fp8(_ptr(x), int(x.shape[0]), int(x.shape[1]), _ptr(codes), _ptr(scale), _stream(stream)),
           "csa2_test_quantize_fp8")


def test_chunk_scores(cache: Cache, q_idx, w, q_seq, q_pos, max_len, sigma, bound, ws, d_err, stream=None):
    _check(_t_cscores(ctypes.byref(cache.desc()), _ptr(q_idx), _ptr(w), _ptr(q_seq), _ptr(q_pos), int(q_seq.shape[0]),
                      int(max_len), _ptr(sigma), _ptr(bound), _ptr(ws), ws.numel(), _ptr(d_err), _stream(stream)),
           "csa2_test_chunk_scores")


def test_index_scores(cache: Cache, q_idx, w, max_len, sigma, bound, ws, d_err, stream=None):
    _check(_t_scores(ctypes.byref(cache.desc()), _ptr(q_idx), _ptr(w), int(max_len), _ptr(sigma), _ptr(bound),
                     _ptr(ws), ws.numel(), _ptr(d_err), _stream(stream)), "csa2_test_index_scores")


def raw_lib() -> ctypes.CDLL:
    """The loaded library (for ABI-level tests)."""
    return _lib
