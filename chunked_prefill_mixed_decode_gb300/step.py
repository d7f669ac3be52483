"""One mixed step end to end through the C ABI: host metadata -> device, append, attention.

Marshalling only (torch for device memory and streams): the packing runs in
ms_build_batch_metadata, the arithmetic in ms_kv_append_rope and
ms_mixed_step_attention.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import (attention_workspace_size, build_batch_metadata, kv_append_rope, mixed_step_attention,
               rope_table)

META_KEYS = ("cu_seqlens_q", "q_start_pos", "context_lens", "positions", "slot_mapping", "block_tables")


@dataclasses.dataclass
class DeviceBatch:
    """Device copies of one step's metadata plus the host-side sizes the calls need."""
    cu_seqlens_q: object
    q_start_pos: object
    context_lens: object
    positions: object
    slot_mapping: object
    block_tables: object
    num_rows: int
    num_tokens: int
    num_decodes: int
    context_total: int
    host: dict

    @property
    def h2d_bytes(self) -> int:
        return sum(int(self.host[k].nbytes) for k in META_KEYS)


def to_device(meta: dict, device, non_blocking: bool = False) -> DeviceBatch:
    import torch
    t = {}
    for k in META_KEYS:
        a = np.ascontiguousarray(meta[k], dtype=np.int32)
        if a.size == 0:
            a = np.zeros(1, dtype=np.int32)  # keep a valid device pointer for empty arrays
        src = torch.from_numpy(a)
        if non_blocking:
            src = src.pin_memory()
        t[k] = src.to(device, non_blocking=non_blocking)
    bt = t["block_tables"]
    S = int(meta["num_rows"])
    stride = int(meta["bt_stride"])
    t["block_tables"] = bt.view(max(S, 1), max(stride, 1)) if S > 0 and stride > 0 else bt.view(1, 1)
    return DeviceBatch(t["cu_seqlens_q"], t["q_start_pos"], t["context_lens"], t["positions"], t["slot_mapping"],
                       t["block_tables"], S, int(meta["num_tokens"]), int(meta["num_decodes"]),
                       int(np.asarray(meta["context_lens"], dtype=np.int64).sum()), meta)


def schedule(states, block_tables, token_budget, max_chunk=0) -> dict:
    return build_batch_metadata(states, block_tables, token_budget, max_chunk)


def rope_tables_device(max_pos: int, D: int, device, base: float = 10000.0):
    import torch
    cos, sin = rope_table(max_pos, D, base)
    return torch.from_numpy(cos).to(device), torch.from_numpy(sin).to(device)


def workspace_for(batch: DeviceBatch, H_q: int, H_kv: int, D: int, device):
    import torch
    n = attention_workspace_size(max(batch.num_rows, 1), max(batch.num_tokens, 1), batch.context_total, H_q, H_kv,
                                 D)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def run_step(q, k, v, batch: DeviceBatch, cos, sin, k_cache, v_cache, out, workspace, q_rot=None,
             dev_status=None, scale=None, stream=None):
    """kv_append_rope then mixed_step_attention on one stream; returns q_rot."""
    if q_rot is None:
        q_rot = q
    T = batch.num_tokens
    kv_append_rope(q[:T], k[:T], v[:T], batch.positions, batch.slot_mapping, cos, sin, k_cache, v_cache,
                   q_rot=q_rot[:T], dev_status=dev_status, stream=stream)
    mixed_step_attention(q_rot[:T], k_cache, v_cache, batch.cu_seqlens_q, batch.q_start_pos, batch.context_lens,
                         batch.block_tables, batch.context_total, out[:T], workspace, scale=scale, stream=stream)
    return q_rot
