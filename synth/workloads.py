"""Workload shapes of the CSA2 decode path (sizes and layer schedules only).

The decoder layer schedule follows origotech.dev's deep dive, section
"Compressed Sparse Attention 2": one group of (1 Full + 3 Reuse) followed by
four groups of (1 Reindex + 3 Reuse), top-k 512, a 128-token sliding window,
and a Full layer that keeps 2,048 blocks of 8 positions.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import ragged_lengths

FULL, REINDEX, REUSE = "full", "reindex", "reuse"


def decoder_schedule(n_layers: int = 20) -> list:
    """(1 Full + 3 Reuse) then repeated (1 Reindex + 3 Reuse)."""
    sched = []
    for layer in range(n_layers):
        if layer % 4 == 0:
            sched.append(FULL if layer == 0 else REINDEX)
        else:
            sched.append(REUSE)
    return sched


@dataclass
class DecodeWorkload:
    name: str
    lengths: np.ndarray            # context length of each sequence, including this step's token
    schedule: list = field(default_factory=lambda: [FULL])
    H: int = 16                    # attention query heads
    topk: int = 512
    n_keep: int = 2048             # blocks kept by the Full layer
    block: int = 8
    window: int = 128
    ring: int = 128                # SWA ring slots per sequence and layer
    seed: int = 0
    drafts: int = 1                # query rows per sequence: the last `drafts` positions, all appended this step

    @property
    def B(self) -> int:
        return int(self.lengths.shape[0])

    @property
    def n_layers(self) -> int:
        return len(self.schedule)


@dataclass
class ChunkedWorkload:
    name: str
    cache_len: int                 # tokens in the FP4 cache of the single sequence
    n_query: int                   # consecutive query positions ending at cache_len - 1
    H: int = 64
    topk: int = 512
    window: int = 128
    ring: int = 8192               # SWA ring large enough to hold every query's window
    seed: int = 0


def verify_workload():
    """Speculative verification: 32 sessions of 65,536 tokens whose last 5 positions are drafted
    tokens, each verified by its own query row through the 20-layer schedule (origotech.dev deep
    dive, section "아키텍처는 어떻게 KV 캐시를 줄이나": the DSpark drafter proposes 5 positions at
    once).  The ring holds window + 4 positions so that the earliest draft row still sees its
    whole window."""
    return DecodeWorkload("verify_b32_ctx65536_d5_20layer", np.full(32, 65536, dtype=np.int64),
                          schedule=decoder_schedule(20), drafts=5, ring=256)


def config(i: int):
    """The five measured configurations (seed 0)."""
    if i == 0:
        return DecodeWorkload("full_layer_b1_ctx4096", np.array([4096], dtype=np.int64))
    if i == 1:
        return DecodeWorkload("decode_b32_ctx65536_full+3reuse",
                              np.full(32, 65536, dtype=np.int64),
                              schedule=[FULL, REUSE, REUSE, REUSE])
    if i == 2:
        return DecodeWorkload("decode_b4_ctx1048576_20layer",
                              np.full(4, 1048576, dtype=np.int64),
                              schedule=decoder_schedule(20))
    if i == 3:
        return ChunkedWorkload("chunked_q4096_h64_cache262144", cache_len=262144, n_query=4096)
    if i == 4:
        return DecodeWorkload("ragged_b64_ctx4k-1m_20layer",
                              ragged_lengths(0, 64), schedule=decoder_schedule(20))
    raise ValueError(f"no config {i}")
