"""Round driver: engine plan -> one device step -> commit, with a per-step record.

Marshalling only.  The packing and the page pool live in the C++ engine
(ms_engine_*), the arithmetic in ms_kv_append_rope and ms_mixed_step_attention.
Each round follows "Chunked Prefill 的 Token 预算" (zwjcode.cn), section 08:
schedule, run the step, then commit the request progress; the record of each
step (prefill tokens, decode tokens, step latency) is the section 12 timeline.
"""
from __future__ import annotations

import time

from . import Engine, StepGraph, attention_workspace_size, mixed_step, read_status
from .step import MetaStager


class RoundDriver:
    """Drives an Engine over caller-owned K/V page pools [num_pages, H_kv, 16, D] (bf16).

    ``step(q, k, v)`` takes the new tokens' activations (device bf16, at least
    ``num_tokens`` rows: q [T, H_q, D], k and v [T, H_kv, D]) in the planned
    row order, writes the attention output into ``out`` and returns the
    round's record.  Every step is synchronised, as a serving loop that reads
    its sampled tokens would be.

    With ``graph_buckets`` (ascending token counts) every step replays a
    captured CUDA graph of its bucket (StepGraph) instead of launching the
    kernels one by one; ``max_row_pages`` then bounds every request's pages.
    The record adds the bucket and the pad tokens.
    """

    def __init__(self, engine: Engine, k_cache, v_cache, cos, sin, H_q: int, H_kv: int, D: int,
                 scale: float | None = None, stream=None, graph_buckets=None, max_row_pages: int = 0):
        import torch
        self.engine = engine
        self.graph = None
        self.k_cache, self.v_cache = k_cache, v_cache
        self.cos, self.sin = cos, sin
        self.H_q, self.H_kv, self.D = H_q, H_kv, D
        self.scale = scale
        self.device = k_cache.device
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        budget = engine.token_budget
        num_pages = int(k_cache.shape[0])
        # upper bounds: a row holds at least one token (and a step at most 8192 rows);
        # the rows' contexts fit in the pool
        max_rows = min(max(budget, 1), 8192)
        self.round = 0
        self.ev0 = torch.cuda.Event(enable_timing=True)
        self.ev1 = torch.cuda.Event(enable_timing=True)
        if graph_buckets:
            if stream is None:  # the legacy default stream cannot be captured
                self.stream = torch.cuda.Stream(self.device)
            self.graph = StepGraph(k_cache, v_cache, cos, sin, H_q, max_rows, max_row_pages, graph_buckets,
                                   self.stream, scale)
            self.q_rot, self.out = self.graph.q_rot, self.graph.out
            return
        self.stager = MetaStager(max_rows, max(budget, 1), 64 * max_rows, self.device)  # grows on demand
        ws = attention_workspace_size(max_rows, max(budget, 1), num_pages * 16, H_q, H_kv, D)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=self.device)
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.q_rot = torch.empty((max(budget, 1), H_q, D), dtype=torch.bfloat16, device=self.device)
        self.out = torch.empty_like(self.q_rot)

    def step(self, q, k, v) -> dict:
        import torch
        t0 = time.perf_counter()
        meta = self.engine.plan()
        T = meta["num_tokens"]
        rec = {"round": self.round, "rows": meta["num_rows"], "decode_tokens": meta["num_decodes"],
               "prefill_tokens": T - meta["num_decodes"], "unused_tokens": meta["unused_tokens"],
               "deferred_decodes": meta["num_deferred"], "row_request_id": meta["row_request_id"],
               "cu_seqlens_q": meta["cu_seqlens_q"], "meta": meta}
        if T > 0 and self.graph is not None:
            g = self.graph
            t_plan = time.perf_counter()
            self.stream.wait_stream(torch.cuda.current_stream(self.device))
            with torch.cuda.stream(self.stream):
                for src, dst in ((q, g.q), (k, g.k), (v, g.v)):
                    if src.data_ptr() != dst.data_ptr():
                        dst[:T].copy_(src[:T])
            self.ev0.record(self.stream)
            rec["bucket"] = g.run(meta)
            rec["pad_tokens"] = rec["bucket"] - T
            self.ev1.record(self.stream)
            st = g.read_status()
            if st:
                raise RuntimeError(f"device status {st} in round {self.round}")
            rec["device_ms"] = self.ev0.elapsed_time(self.ev1)
        elif T > 0:
            batch = self.stager.stage(meta, self.stream)
            t_plan = time.perf_counter()
            self.ev0.record(self.stream)
            mixed_step(q[:T], k[:T], v[:T], batch.positions, batch.slot_mapping, self.cos, self.sin, self.k_cache,
                       self.v_cache, self.q_rot[:T], batch.cu_seqlens_q, batch.q_start_pos, batch.context_lens,
                       batch.block_tables, batch.context_total, self.out[:T], self.workspace,
                       dev_status=self.status, scale=self.scale, stream=self.stream)
            self.ev1.record(self.stream)
            self.stream.synchronize()
            st = read_status(self.status, self.stream) | read_status(self.workspace, self.stream)
            if st:
                raise RuntimeError(f"device status {st} in round {self.round}")
            rec["device_ms"] = self.ev0.elapsed_time(self.ev1)
        else:
            t_plan = time.perf_counter()
            rec["device_ms"] = 0.0
        t_dev = time.perf_counter()
        rec["finished"] = self.engine.commit()
        t_end = time.perf_counter()
        rec["host_ms"] = ((t_plan - t0) + (t_end - t_dev)) * 1e3
        rec["wall_ms"] = (t_end - t0) * 1e3
        self.round += 1
        return rec
