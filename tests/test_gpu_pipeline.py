"""The serving pipeline (runner.StepPipeline): steps fed from pinned host buffers through
two alternating sets of device buffers, with the copies on their own streams, give the
same outputs as plain steps of the runner (the decode step is deterministic)."""
import numpy as np
import pytest
import torch

from sparse_attention_fp4_02_b300.runner import DecodeRunner, StepPipeline
from synth.workloads import DecodeWorkload, decoder_schedule

pytestmark = pytest.mark.gpu


def _workload(drafts):
    lengths = np.array([3000, 777, 5000, 64], dtype=np.int64)
    return DecodeWorkload(f"pipe_d{drafts}", lengths, schedule=decoder_schedule(8), drafts=drafts,
                          ring=256 if drafts > 1 else 128)


@pytest.mark.parametrize("drafts", [1, 3])
def test_pipeline_matches_plain_steps(drafts):
    r = DecodeRunner(_workload(drafts))
    r.build_cache()
    r.step()
    torch.cuda.synchronize()
    r.check_device_errors()
    ref_out, ref_lse = r.out.cpu().clone(), r.lse.cpu().clone()

    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    h_in = {"kv_new": pin(r.h_kv_new.view(np.int16)), "ik_new": pin(r.h_ik_new.view(np.int16)),
            "swa_new": pin(r.h_swa_new.view(np.int16)), "q": pin(r.h_q.view(np.int16))}
    for l in r.idx_layers:
        h_in[f"qidx{l}"] = pin(r.h_qidx[l].view(np.int16))
        h_in[f"w{l}"] = pin(r.h_w[l])
    if r.D > 1:
        for l in r.full_layers:
            h_in[f"qidx_last{l}"] = pin(r.h_qidx[l][r.D - 1::r.D].view(np.int16))
            h_in[f"w_last{l}"] = pin(r.h_w[l][r.D - 1::r.D])
    assert set(h_in) | {"out", "lse"} == set(r.step_buffers())
    pipe = StepPipeline(r)
    # the alternate set starts as garbage: the pipeline must fill it from the host before use
    for name, t in pipe.sets[1].items():
        t.zero_()
    outs = []
    pipe.begin()
    for _ in range(5):
        h_out = {"out": torch.full(r.out.shape, float("nan")).pin_memory(),
                 "lse": torch.full(r.lse.shape, float("nan")).pin_memory()}
        pipe.step(h_in, h_out)
        outs.append(h_out)
    pipe.end()
    torch.cuda.synchronize()
    r.check_device_errors()
    for h_out in outs:
        assert torch.equal(h_out["out"], ref_out)
        assert torch.equal(h_out["lse"], ref_lse)
