"""Shared helpers of the GPU parity tests (comparison rules, tensor plumbing)."""
from __future__ import annotations

import numpy as np
import torch

try:  # the library must load on a GPU machine; CPU-only runs deselect the GPU tests
    import sparse_attention_fp4_02_b300 as csa2
except ImportError:
    if torch.cuda.is_available():
        raise
    csa2 = None

REL_TIE = 1e-6      # a boundary swap is allowed only between scores this close (relative)
ATTN_TOL = 2e-3     # per (row, head): max|o - r| / max|r|


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return t if dtype is None else t.to(dtype)


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def check_index_set(gpu_ids, oracle_ids, score_of, what="indices"):
    """Sets must match; a swapped pair is allowed only if the oracle's scores are within 1e-6 relative.

    Returns the number of swapped pairs (0 when identical).
    """
    g = np.asarray(gpu_ids)
    o = np.asarray(oracle_ids)
    gv = g[g >= 0]
    ov = o[o >= 0]
    assert np.all(np.diff(gv) > 0), f"{what}: GPU output not strictly ascending"
    assert np.all(g[len(gv):] == -1) and np.all(g[:len(gv)] >= 0), f"{what}: padding not at the end"
    assert len(gv) == len(ov), f"{what}: {len(gv)} selected, oracle {len(ov)}"
    only_g = np.setdiff1d(gv, ov)
    only_o = np.setdiff1d(ov, gv)
    for p in only_g:
        for q in only_o:
            a, b = score_of(int(p)), score_of(int(q))
            assert abs(a - b) <= REL_TIE * max(a, b), f"{what}: swap {p} ({a}) vs {q} ({b}) beyond tolerance"
    return len(only_g)


def attn_rel_err(out: np.ndarray, ref: np.ndarray) -> float:
    """max over (row, head) of max|o - r| / max|r| (arrays [..., H, D])."""
    num = np.abs(out - ref).max(axis=-1)
    den = np.abs(ref).max(axis=-1)
    den = np.where(den == 0, 1.0, den)
    return float((num / den).max())
