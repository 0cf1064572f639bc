"""Decoder layer-pattern runner over the C ABI.

A decode step of the CSA2 decoder (origotech.dev deep dive, subsection
"Compressed Sparse Attention 2(CSA2)"): the new token's KV is quantised and
appended, the first Full layer's indexer scores every cached position and
keeps a 2,048-block pool plus its top-512, every Reindex layer rescores the
pool with its own indexer queries, every Reuse layer passes the indices on,
and every layer runs sparse attention over its indices plus its own
128-token FP8 window.

With ``drafts`` > 1 the step verifies speculative drafts (origotech.dev deep
dive, section "아키텍처는 어떻게 KV 캐시를 줄이나", the DSpark item): the last
``drafts`` positions of each session are appended together and each gets its
own query row.  The Full layer keeps one pool per session, scored with the
queries of the session's last row (whose causal context is the whole session);
every row of every indexer layer then takes its top-k from that shared pool,
limited to positions up to its own.

All compute happens in libcsa2.so; this module allocates device memory with
torch, fills caches from seeded synthetic inputs and sequences the calls
(optionally captured into one CUDA graph).
"""
from __future__ import annotations

import math

import numpy as np
import torch

import synth
from synth.workloads import FULL, REINDEX, REUSE, DecodeWorkload

from . import (Cache, SwaRing, OP_ATTN_DECODE, OP_CHUNKED_SELECT, OP_FULL_SELECT, OP_VERIFY_SELECT,
               alloc_workspace, indexer_chunked_select, indexer_full_select, indexer_reindex_select,
               indexer_verify_select, kv_append_fp4, sparse_attn_decode, workspace_bytes)


def _to_dev(a: np.ndarray, dtype, device):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device=device, dtype=dtype)


def _bf16_dev(bits: np.ndarray, device):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


class DecodeRunner:
    """Caches, per-step inputs and outputs of one decode workload on one GPU."""

    def __init__(self, wl: DecodeWorkload, device="cuda", rope_len: int | None = None):
        self.wl = wl
        self.device = device
        B = wl.B
        self.D = int(wl.drafts)
        self.T = B * self.D
        assert self.D >= 1 and wl.ring >= wl.window + self.D - 1, "ring must hold every draft row's window"
        L = wl.lengths.astype(np.int64)
        self.lengths = L
        self.max_len = int(L.max())
        base = np.zeros(B, dtype=np.int64)
        base[1:] = np.cumsum(((L + 15) // 16) * 16)[:-1]
        self.seq_base_np = base
        self.T_cap = int(base[-1] + ((L[-1] + 15) // 16) * 16)
        self.cache = Cache(self.T_cap, B, device)
        self.cache.seq_base.copy_(torch.from_numpy(base))
        self.cache.seq_len.copy_(torch.from_numpy(L.astype(np.int32)))
        self.swa = [SwaRing(B, wl.ring, device) for _ in range(wl.n_layers)]
        cos, sin = synth.rope_table(rope_len or self.max_len)
        self.rope_cos = torch.from_numpy(cos).to(device)
        self.rope_sin = torch.from_numpy(sin).to(device)
        self.d_err = torch.zeros(1, dtype=torch.int32, device=device)
        self.kv_outliers = synth.outlier_channels(wl.seed, synth.Stream.KV_OUTLIER)
        self.swa_outliers = synth.outlier_channels(wl.seed, synth.Stream.SWA_OUTLIER)
        self._make_step_inputs()
        self._make_outputs()

    # ------------------------------------------------------------------ inputs
    def _make_step_inputs(self):
        wl, dev, B, D, T = self.wl, self.device, self.wl.B, self.D, self.T
        s = wl.seed
        # query row r = b * D + j is position L_b - D + j of sequence b
        seq = np.repeat(np.arange(B), D)
        newpos = np.repeat(self.lengths, D) - D + np.tile(np.arange(D), B)
        rows_new = synth.row_id(seq, newpos)
        self.h_kv_new = synth.normals_bf16(s, synth.Stream.KV, 0, rows_new, 128, self.kv_outliers)
        self.h_ik_new = synth.normals_bf16(s, synth.Stream.IK, 0, rows_new, 64)
        self.h_swa_new = np.stack([synth.normals_bf16(s, synth.Stream.SWA, l, rows_new, 128, self.swa_outliers)
                                   for l in range(wl.n_layers)])
        self.h_seq_id = seq.astype(np.int32)
        self.h_pos = newpos.astype(np.int64)
        self.h_q = np.stack([synth.normals_bf16(s, synth.Stream.Q, l,
                                                synth.row_id(np.repeat(np.arange(T), wl.H), np.tile(np.arange(wl.H), T)),
                                                128).reshape(T, wl.H, 128) for l in range(wl.n_layers)])
        self.idx_layers = [l for l, m in enumerate(wl.schedule) if m in (FULL, REINDEX)]
        self.h_qidx = {l: synth.normals_bf16(s, synth.Stream.QIDX, l,
                                             synth.row_id(np.repeat(np.arange(T), 8), np.tile(np.arange(8), T)),
                                             64).reshape(T, 8, 64) for l in self.idx_layers}
        self.h_w = {l: np.stack([synth.head_weights(s, l, r) for r in range(T)]) for l in self.idx_layers}
        # device copies
        self.kv_new = _bf16_dev(self.h_kv_new, dev)
        self.ik_new = _bf16_dev(self.h_ik_new, dev)
        self.swa_new = _bf16_dev(self.h_swa_new, dev)
        self.seq_id = _to_dev(self.h_seq_id, torch.int32, dev)
        self.pos = _to_dev(self.h_pos, torch.int64, dev)
        self.q = _bf16_dev(self.h_q, dev)
        self.qidx = {l: _bf16_dev(v, dev) for l, v in self.h_qidx.items()}
        self.w = {l: _to_dev(v, torch.float32, dev) for l, v in self.h_w.items()}
        # the Full layer's pool is scored with each session's last row: a step input of its own
        self.full_layers = [l for l in self.idx_layers if wl.schedule[l] == FULL]
        self.qidx_last = {l: self.qidx[l][D - 1::D].contiguous() if D > 1 else self.qidx[l] for l in self.full_layers}
        self.w_last = {l: self.w[l][D - 1::D].contiguous() if D > 1 else self.w[l] for l in self.full_layers}

    def _make_outputs(self):
        wl, dev, B, T = self.wl, self.device, self.wl.B, self.T
        self.pool = torch.full((B, wl.n_keep), -1, dtype=torch.int32, device=dev)
        self.topk = {l: torch.full((T, wl.topk), -1, dtype=torch.int32, device=dev) for l in self.idx_layers}
        self.topk_full = {l: (torch.full((B, wl.topk), -1, dtype=torch.int32, device=dev) if self.D > 1
                              else self.topk[l]) for l in self.full_layers}
        self.out = torch.zeros((wl.n_layers, T, wl.H, 128), dtype=torch.float32, device=dev)
        self.lse = torch.zeros((wl.n_layers, T, wl.H), dtype=torch.float32, device=dev)
        self.ws_idx = alloc_workspace(workspace_bytes(OP_FULL_SELECT, B, self.max_len, wl.block, wl.n_keep, wl.topk),
                                      dev)
        self.ws_ver = (alloc_workspace(workspace_bytes(OP_VERIFY_SELECT, block=wl.block, n_keep_blocks=wl.n_keep,
                                                       topk=wl.topk, T=T), dev) if self.D > 1 else None)
        self.ws_attn = alloc_workspace(workspace_bytes(OP_ATTN_DECODE, T=T, H=wl.H, topk=wl.topk, window=wl.window),
                                       dev)
        self.tau = 1.0 / math.sqrt(128.0)

    def layer_topk(self, layer: int):
        """The index buffer layer ``layer`` attends over (Reuse layers share the previous one)."""
        src = max(l for l in self.idx_layers if l <= layer)
        return self.topk[src]

    # ------------------------------------------------------------------ cache build
    def build_cache(self, chunk: int = 1 << 18):
        """Append positions 0..L-D-1 of every sequence (the step appends the last D) and the window rows."""
        wl, dev, s = self.wl, self.device, self.wl.seed
        for b in range(wl.B):
            n_old = int(self.lengths[b]) - self.D
            for lo in range(0, n_old, chunk):
                hi = min(n_old, lo + chunk)
                pos = np.arange(lo, hi, dtype=np.int64)
                rows = synth.row_id(b, pos)
                kv = _bf16_dev(synth.normals_bf16(s, synth.Stream.KV, 0, rows, 128, self.kv_outliers), dev)
                ik = _bf16_dev(synth.normals_bf16(s, synth.Stream.IK, 0, rows, 64), dev)
                sid = torch.full((hi - lo,), b, dtype=torch.int32, device=dev)
                kv_append_fp4(self.cache, None, kv, ik, None, self.rope_cos, self.rope_sin, sid,
                              torch.from_numpy(pos).to(dev), self.d_err)
            # window rows before the new token, every layer
            lo = max(0, n_old - (wl.window - 1))
            if n_old > lo:
                pos = np.arange(lo, n_old, dtype=np.int64)
                rows = synth.row_id(b, pos)
                kv = _bf16_dev(synth.normals_bf16(s, synth.Stream.KV, 0, rows, 128, self.kv_outliers), dev)
                sw = _bf16_dev(np.stack([synth.normals_bf16(s, synth.Stream.SWA, l, rows, 128, self.swa_outliers)
                                         for l in range(wl.n_layers)]), dev)
                sid = torch.full((n_old - lo,), b, dtype=torch.int32, device=dev)
                kv_append_fp4(self.cache, self.swa, kv, None, sw, self.rope_cos, self.rope_sin, sid,
                              torch.from_numpy(pos).to(dev), self.d_err)
        torch.cuda.synchronize()

    # ------------------------------------------------------------------ the step
    def step(self, prof=None, mark=None):
        """One decode (or draft-verification) step through every layer of the schedule.

        ``mark``, if given, is called with the entry point's name after each call (the benchmark
        records a timing event there for its per-call breakdown)."""
        wl = self.wl
        mark = mark or (lambda name: None)
        kv_append_fp4(self.cache, self.swa, self.kv_new, self.ik_new, self.swa_new, self.rope_cos, self.rope_sin,
                      self.seq_id, self.pos, self.d_err)
        mark("kv_append_fp4")
        for l, mode in enumerate(wl.schedule):
            if mode == FULL:
                indexer_full_select(self.cache, self.qidx_last[l], self.w_last[l], wl.block, wl.n_keep, wl.topk,
                                    self.max_len, self.pool, self.topk_full[l], self.ws_idx, self.d_err, prof=prof)
                mark("indexer_full_select")
            if self.D > 1 and mode in (FULL, REINDEX):
                indexer_verify_select(self.cache, self.qidx[l], self.w[l], self.seq_id, self.pos, self.pool,
                                      wl.block, wl.n_keep, wl.topk, self.max_len, self.topk[l], self.ws_ver,
                                      self.d_err)
                mark("indexer_verify_select")
            elif mode == REINDEX:
                indexer_reindex_select(self.cache, self.qidx[l], self.w[l], self.pool, wl.block, wl.n_keep, wl.topk,
                                       self.max_len, self.topk[l], self.ws_idx, self.d_err)
                mark("indexer_reindex_select")
            sparse_attn_decode(self.cache, self.swa[l], self.q[l], self.seq_id, self.pos, self.layer_topk(l),
                               wl.window, self.tau, self.out[l], self.lse[l], self.ws_attn, self.d_err)
            mark("sparse_attn_decode")

    def step_bytes(self) -> dict:
        """Algorithmic bytes of one step by part: the unique bytes the method must read and write
        (the scan's 68 B per cached position, a Reindex layer's 68 B per pool position, an
        attention row's gathered FP4 rows, window rows, indices, queries and outputs, the
        append's inputs and cache rows); implementation scratch is not counted."""
        wl, L = self.wl, self.lengths
        n_re = sum(1 for m in wl.schedule if m == REINDEX)
        rows_per_seq = self.D
        attn_row = (np.minimum(L, wl.topk) * 72 + np.minimum(L, wl.window) * 132 + 4 * wl.topk
                    + 2 * wl.H * 128 + 4 * wl.H * 128 + 4 * wl.H)
        layers = wl.n_layers
        tok_read = 2 * 128 + 2 * 64 + layers * 2 * 128 + 2 * 32 * 4
        tok_write = 72 + 68 + layers * 132
        return {
            "scan": int(68 * L.sum()),
            "reindex": int(68 * np.minimum(L, wl.n_keep * wl.block).sum() * n_re * rows_per_seq),
            "attention": int(attn_row.sum() * layers * rows_per_seq),
            "append": int((tok_read + tok_write) * self.T),
        }
    def check_device_errors(self):
        v = int(self.d_err.item())
        if v:
            raise RuntimeError(f"device error bits 0x{v:x}")

    def step_buffers(self) -> dict:
        """The step's own device inputs and outputs by name: the tensors a step reads and writes
        besides the cache, the SWA rings and the selection scratch."""
        b = {"kv_new": self.kv_new, "ik_new": self.ik_new, "swa_new": self.swa_new, "q": self.q,
             "out": self.out, "lse": self.lse}
        for l in self.idx_layers:
            b[f"qidx{l}"] = self.qidx[l]
            b[f"w{l}"] = self.w[l]
        if self.D > 1:
            for l in self.full_layers:
                b[f"qidx_last{l}"] = self.qidx_last[l]
                b[f"w_last{l}"] = self.w_last[l]
        return b

    def use_buffers(self, b: dict):
        """Make later steps (and captures) read and write the given set of step buffers."""
        self.kv_new, self.ik_new, self.swa_new, self.q = b["kv_new"], b["ik_new"], b["swa_new"], b["q"]
        self.out, self.lse = b["out"], b["lse"]
        for l in self.idx_layers:
            self.qidx[l] = b[f"qidx{l}"]
            self.w[l] = b[f"w{l}"]
        for l in self.full_layers:
            self.qidx_last[l] = b[f"qidx_last{l}"] if self.D > 1 else self.qidx[l]
            self.w_last[l] = b[f"w_last{l}"] if self.D > 1 else self.w[l]

    def capture(self, prof=None):
        """Capture one step into a CUDA graph; returns the graph (replay with .replay())."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self.step(prof)           # warm-up outside capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step(prof)
        return g


class ChunkedRunner:
    """The chunked-query workload: many consecutive query rows of one sequence, each with
    its own causal top-k plus a causal window, attended in one sparse_attn_decode call.
    ``select()`` computes those top-k lists with the chunked-query indexer (every row's Full
    selection over the positions up to its own); ``use_indexer=False`` keeps seeded causal
    lists instead."""

    def __init__(self, wl, device="cuda", chunk: int = 1 << 17, use_indexer: bool = True):
        from synth.workloads import ChunkedWorkload
        assert isinstance(wl, ChunkedWorkload)
        self.wl, self.device = wl, device
        L, s = int(wl.cache_len), wl.seed
        self.cache = Cache(((L + 15) // 16) * 16, 1, device)
        self.cache.seq_base.zero_()
        self.cache.seq_len.fill_(L)
        self.swa = SwaRing(1, wl.ring, device)
        cos, sin = synth.rope_table(L + 1)
        self.rope_cos, self.rope_sin = _to_dev(cos, torch.float32, device), _to_dev(sin, torch.float32, device)
        self.d_err = torch.zeros(1, dtype=torch.int32, device=device)
        oc = synth.outlier_channels(s, synth.Stream.KV_OUTLIER)
        soc = synth.outlier_channels(s, synth.Stream.SWA_OUTLIER)
        for lo in range(0, L, chunk):
            hi = min(L, lo + chunk)
            pos = np.arange(lo, hi, dtype=np.int64)
            rows = synth.row_id(0, pos)
            kv = _bf16_dev(synth.normals_bf16(s, synth.Stream.KV, 0, rows, 128, oc), device)
            ik = _bf16_dev(synth.normals_bf16(s, synth.Stream.IK, 0, rows, 64), device)
            sid = torch.zeros(hi - lo, dtype=torch.int32, device=device)
            kv_append_fp4(self.cache, None, kv, ik, None, self.rope_cos, self.rope_sin, sid,
                          torch.from_numpy(pos).to(device), self.d_err)
        # window rows of every query: positions [first query - window + 1, L)
        lo = max(0, L - wl.n_query - wl.window + 1)
        pos = np.arange(lo, L, dtype=np.int64)
        rows = synth.row_id(0, pos)
        kv = _bf16_dev(synth.normals_bf16(s, synth.Stream.KV, 0, rows, 128, oc), device)
        sw = _bf16_dev(synth.normals_bf16(s, synth.Stream.SWA, 0, rows, 128, soc)[None], device)
        kv_append_fp4(self.cache, [self.swa], kv, None, sw, self.rope_cos, self.rope_sin,
                      torch.zeros(L - lo, dtype=torch.int32, device=device), torch.from_numpy(pos).to(device),
                      self.d_err)
        q_pos = np.arange(L - wl.n_query, L, dtype=np.int64)
        self.q_pos = torch.from_numpy(q_pos).to(device)
        self.q_seq = torch.zeros(wl.n_query, dtype=torch.int32, device=device)
        self.topk = torch.from_numpy(synth.causal_topk(s, q_pos, wl.topk)).to(device)
        # the indexer's inputs and outputs: each row's queries and weights, pool and top-k
        T = wl.n_query
        self.qidx = _bf16_dev(np.stack([synth.normals_bf16(s, synth.Stream.QIDX, 0, synth.row_id(r, np.arange(8)), 64)
                                        for r in range(T)]), device)
        self.w = _to_dev(np.stack([synth.head_weights(s, 0, r) for r in range(T)]), torch.float32, device)
        self.block, self.n_keep = 8, 2048
        self.pool = torch.full((T, self.n_keep), -1, dtype=torch.int32, device=device)
        self.ws_idx = alloc_workspace(workspace_bytes(OP_CHUNKED_SELECT, max_len=L, block=self.block,
                                                      n_keep_blocks=self.n_keep, topk=wl.topk, T=T), device)
        self.positions = int(np.sum(q_pos + 1))          # (row, position) pairs the indexer scores
        q = synth.normals_bf16(s, synth.Stream.Q, 0, np.arange(wl.n_query * wl.H), 128)
        self.q = _bf16_dev(q.reshape(wl.n_query, wl.H, 128), device)
        self.out = torch.empty((wl.n_query, wl.H, 128), dtype=torch.float32, device=device)
        self.lse = torch.empty((wl.n_query, wl.H), dtype=torch.float32, device=device)
        self.ws = alloc_workspace(0, device)
        self.tau = 1.0 / math.sqrt(128.0)
        if use_indexer:
            self.select()
        torch.cuda.synchronize()

    def select(self):
        """The chunked-query indexer: pool and top-k of every row into self.pool / self.topk."""
        wl = self.wl
        indexer_chunked_select(self.cache, self.qidx, self.w, self.q_seq, self.q_pos, self.block, self.n_keep, wl.topk,
                               wl.cache_len, self.pool, self.topk, self.ws_idx, self.d_err)

    def select_flops(self) -> float:
        """Indexer flops of one select(): 8 heads x 64 dims x 2 per (row, position <= row)."""
        return 1024.0 * self.positions

    def step(self):
        sparse_attn_decode(self.cache, self.swa, self.q, self.q_seq, self.q_pos, self.topk, self.wl.window,
                           self.tau, self.out, self.lse, self.ws, self.d_err)

    def flops(self) -> float:
        """Dense-equivalent flops of one call: S = Q K^T and O = P V over topk + window rows."""
        wl = self.wl
        return 4.0 * wl.n_query * wl.H * (wl.topk + wl.window) * 128

    def bytes(self) -> int:
        """Algorithmic bytes of one call: the unique bytes it must move, i.e. every distinct
        gathered FP4 row (72 B) and window row (132 B) once, the index lists, the bf16 queries
        and the float32 outputs and lse (rows shared by several queries are counted once)."""
        wl = self.wl
        idx = self.topk.cpu().numpy()
        uniq_rows = np.unique(idx[idx >= 0]).shape[0]
        q_pos = self.q_pos.cpu().numpy()              # consecutive positions: one run of window rows
        uniq_win = int(q_pos.max() - max(0, q_pos.min() - wl.window + 1) + 1)
        T, H = wl.n_query, wl.H
        return int(uniq_rows * 72 + uniq_win * 132 + T * wl.topk * 4 + T * H * 128 * 2 + T * H * 128 * 4 + T * H * 4)

    def check_device_errors(self):
        v = int(self.d_err.item())
        if v:
            raise RuntimeError(f"device error bits 0x{v:x}")


class StepPipeline:
    """Decode steps served from host memory: every step's inputs are copied in from pinned
    host buffers and its outputs copied back, on copy streams of their own, so that the
    copies overlap the neighbouring steps' compute.  Two sets of device inputs and outputs
    alternate, each with its own captured step graph: step k's inputs go into set k % 2
    once step k - 2 has finished with it, step k computes once its inputs are in and step
    k - 2's outputs have been read back, and step k's outputs are read back while step k + 1
    computes.  The steps themselves run in order on the current stream (they share the
    cache and the selection scratch)."""

    def __init__(self, runner: DecodeRunner):
        self.r = runner
        base = runner.step_buffers()
        alt = {k: v.clone() for k, v in base.items()}
        self.sets = [base, alt]
        self.graphs = []
        for b in self.sets:
            runner.use_buffers(b)
            self.graphs.append(runner.capture())
        runner.use_buffers(base)
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.done = [torch.cuda.Event() for _ in range(2)]
        self.out_done = [torch.cuda.Event() for _ in range(2)]
        self.k = 0

    def begin(self):
        """Order the copy streams after the work already on the current stream."""
        cur = torch.cuda.current_stream()
        self.s_in.wait_stream(cur)
        self.s_out.wait_stream(cur)

    def step(self, h_in: dict, h_out: dict):
        """Enqueue one step: h_in maps input names (see DecodeRunner.step_buffers) to pinned
        host tensors, h_out maps "out" / "lse" to pinned host tensors that receive them."""
        x = self.k & 1
        dev = self.sets[x]
        cur = torch.cuda.current_stream()
        with torch.cuda.stream(self.s_in):
            self.s_in.wait_event(self.done[x])          # step k - 2 has read this set's inputs
            for name, h in h_in.items():
                d = dev[name]
                (d.view(torch.int16) if d.dtype == torch.bfloat16 else d).copy_(h, non_blocking=True)
            self.in_ready[x].record(self.s_in)
        cur.wait_event(self.in_ready[x])
        cur.wait_event(self.out_done[x])                # step k - 2's outputs have been read back
        self.graphs[x].replay()
        self.done[x].record(cur)
        with torch.cuda.stream(self.s_out):
            self.s_out.wait_event(self.done[x])
            for name, h in h_out.items():
                h.copy_(dev[name], non_blocking=True)
            self.out_done[x].record(self.s_out)
        self.k += 1

    def end(self):
        """Order the current stream after every copy back issued so far."""
        torch.cuda.current_stream().wait_stream(self.s_out)
