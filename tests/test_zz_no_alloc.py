"""indexer_reindex_select_static (no workspace, static scratch in the library) against
indexer_reindex_select on the same inputs.  Index outputs are integers, so they must be
identical.  Two calls in a row with different queries check that the scratch the first
call leaves behind does not leak into the second.  Collected last on purpose: it must
pass both alone in a fresh process and after every other test."""
import numpy as np
import pytest
import torch

from tests.gpu_util import csa2, dev, dev_bf16, host
from tests.test_gpu_indexer import fill, queries, run_full, run_reindex

pytestmark = pytest.mark.gpu

BLOCK, N_KEEP, TOPK = 8, 2048, 512


def _static(cache, q, w, pool, max_len):
    top = torch.full((cache.B, TOPK), -7, dtype=torch.int32, device="cuda")
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    csa2.indexer_reindex_select_static(cache, dev_bf16(q), dev(w), dev(pool), BLOCK, N_KEEP, TOPK, max_len, top,
                                       d_err)
    torch.cuda.synchronize()
    assert int(d_err.item()) == 0
    return host(top)


def test_static_scratch_matches_the_workspace_entry_on_two_calls_in_a_row():
    lengths = [40000, 1500, 70000, 9]
    cache, _ = fill(lengths, seed=3)
    max_len = max(lengths)
    q0, w0 = queries(len(lengths), layer=0, seed=3)
    pool, _ = run_full(cache, q0, w0, BLOCK, N_KEEP, TOPK, max_len)
    for layer in (1, 2):
        q, w = queries(len(lengths), layer=layer, seed=3)
        want = run_reindex(cache, q, w, pool, BLOCK, N_KEEP, TOPK, max_len)
        got = _static(cache, q, w, pool, max_len)
        np.testing.assert_array_equal(got, want)


def test_static_scratch_rejects_calls_beyond_its_size():
    cache = csa2.Cache(16, 64)
    q = torch.zeros((64, 8, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((64, 8), dtype=torch.float32, device="cuda")
    pool = torch.zeros((64, 4096), dtype=torch.int32, device="cuda")
    top = torch.zeros((64, 512), dtype=torch.int32, device="cuda")
    d_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(csa2.Csa2Error) as e:      # 64 x 4096 x 16 positions need ~17 MB of scratch
        csa2.indexer_reindex_select_static(cache, q, w, pool, 16, 4096, 512, 16, top, d_err)
    assert e.value.status == csa2.ERR_WORKSPACE
