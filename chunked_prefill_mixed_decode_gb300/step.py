"""One mixed step end to end through the C ABI: host metadata -> device, append, attention.

Marshalling only (torch for device memory and streams): the packing runs in
ms_build_batch_metadata, the arithmetic in ms_kv_append_rope and
ms_mixed_step_attention.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import (attention_workspace_size, mixed_step, mixed_step_attention, mixed_step_attention_ragged,
               rope_table)

META_KEYS = ("cu_seqlens_q", "q_start_pos", "context_lens", "positions", "slot_mapping", "block_tables")
RAGGED_KEYS = ("cu_seqlens_q", "q_start_pos", "context_lens", "positions", "slot_mapping", "bt_offsets", "bt_pages")


def _keys(meta: dict):
    return RAGGED_KEYS if "bt_offsets" in meta else META_KEYS


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
    bt_offsets: object = None  # ragged block table (then block_tables holds the pages back to back)

    @property
    def ragged(self) -> bool:
        return self.bt_offsets is not None

    @property
    def h2d_bytes(self) -> int:
        return sum(int(np.asarray(self.host[k]).nbytes) for k in _keys(self.host))


def to_device(meta: dict, device, non_blocking: bool = False) -> DeviceBatch:
    import torch
    t = {}
    for k in _keys(meta):
        a = np.ascontiguousarray(meta[k], dtype=np.int32)
        if a.size == 0:
            a = np.zeros(1, dtype=np.int32)  # keep a valid device pointer for empty arrays
        src = torch.from_numpy(a)
        if non_blocking:
            src = src.pin_memory()
        t[k] = src.to(device, non_blocking=non_blocking)
    S = int(meta["num_rows"])
    ctx_total = int(np.asarray(meta["context_lens"], dtype=np.int64).sum())
    if "bt_offsets" in meta:
        return DeviceBatch(t["cu_seqlens_q"], t["q_start_pos"], t["context_lens"], t["positions"],
                           t["slot_mapping"], t["bt_pages"], S, int(meta["num_tokens"]), int(meta["num_decodes"]),
                           ctx_total, meta, bt_offsets=t["bt_offsets"])
    bt = t["block_tables"]
    stride = int(meta["bt_stride"])
    t["block_tables"] = bt.view(max(S, 1), max(stride, 1)) if S > 0 and stride > 0 else bt.view(1, 1)
    return DeviceBatch(t["cu_seqlens_q"], t["q_start_pos"], t["context_lens"], t["positions"], t["slot_mapping"],
                       t["block_tables"], S, int(meta["num_tokens"]), int(meta["num_decodes"]), ctx_total, meta)


class MetaStager:
    """Reusable pinned staging for one step's metadata: the six arrays are packed
    into one pinned host buffer and reach the device in a single copy.

    Two host/device buffer pairs alternate; a host buffer is refilled only after
    the copy that last read it has finished (an event per buffer).  Device
    buffers are reused in stream order, so the kernels of a step finish reading
    one before a later copy on the same stream overwrites it.
    """

    def __init__(self, max_rows: int, max_tokens: int, max_bt: int, device):
        self.device = device
        self.cap = 0
        self.events = [None, None]
        self.flip = 0
        self._grow(3 * max_rows + 1 + 2 * max_tokens + max_bt + 6 * 4)  # plus alignment slack

    def _grow(self, cap: int):
        import torch
        for ev in self.events:
            if ev is not None:
                ev.synchronize()
        torch.cuda.synchronize(self.device)  # earlier steps may still read the old device buffers
        self.cap = cap
        self.host = [torch.empty(cap, dtype=torch.int32).pin_memory() for _ in range(2)]
        self.dev = [torch.empty(cap, dtype=torch.int32, device=self.device) for _ in range(2)]
        self.events = [None, None]

    def stage(self, meta: dict, stream=None) -> DeviceBatch:
        import torch
        S, T, stride = int(meta["num_rows"]), int(meta["num_tokens"]), int(meta["bt_stride"])
        ragged = "bt_offsets" in meta
        n_bt = (S + 1 + int(meta["bt_offsets"][S])) if ragged else S * stride
        need = 3 * S + 1 + 2 * T + n_bt + 7 * 4
        if need > self.cap:
            self._grow(max(need, 2 * self.cap))
        i = self.flip
        self.flip ^= 1
        if self.events[i] is not None:
            self.events[i].synchronize()
        hv = self.host[i].numpy()
        views, off = {}, 0
        tabs = ((("bt_offsets", S + 1), ("bt_pages", int(meta["bt_offsets"][S]))) if ragged
                else (("block_tables", S * stride),))
        for k, n in (("cu_seqlens_q", S + 1), ("q_start_pos", S), ("context_lens", S), ("positions", T),
                     ("slot_mapping", T)) + tabs:
            n_alloc = max(n, 1)
            if off + n_alloc > self.cap:
                raise ValueError("metadata larger than the stager's capacity")
            hv[off:off + n] = np.asarray(meta[k], dtype=np.int32).reshape(-1)[:n]
            views[k] = (off, n_alloc)
            off += (n_alloc + 3) & ~3  # keep each array 16-byte aligned
        st = stream if stream is not None else torch.cuda.current_stream(self.dev[i].device)
        with torch.cuda.stream(st):
            self.dev[i][:off].copy_(self.host[i][:off], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(st)
        self.events[i] = ev
        d = {k: self.dev[i][o:o + n] for k, (o, n) in views.items()}
        ctx_total = int(np.asarray(meta["context_lens"], dtype=np.int64).sum())
        if ragged:
            return DeviceBatch(d["cu_seqlens_q"], d["q_start_pos"], d["context_lens"], d["positions"],
                               d["slot_mapping"], d["bt_pages"], S, T, int(meta["num_decodes"]), ctx_total, meta,
                               bt_offsets=d["bt_offsets"])
        bt = d["block_tables"].view(S, stride) if S > 0 and stride > 0 else d["block_tables"][:1].view(1, 1)
        return DeviceBatch(d["cu_seqlens_q"], d["q_start_pos"], d["context_lens"], d["positions"],
                           d["slot_mapping"], bt, S, T, int(meta["num_decodes"]), ctx_total, meta)


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
    """One step of one layer through ms_mixed_step (the append, then the attention, with the
    prologue inside the append's launch on small steps); returns q_rot."""
    if q_rot is None:
        q_rot = q
    T = batch.num_tokens
    mixed_step(q[:T], k[:T], v[:T], batch.positions, batch.slot_mapping, cos, sin, k_cache, v_cache, q_rot[:T],
               batch.cu_seqlens_q, batch.q_start_pos, batch.context_lens, batch.block_tables, batch.context_total,
               out[:T], workspace, bt_offsets=batch.bt_offsets if batch.ragged else None, dev_status=dev_status,
               scale=scale, stream=stream)
    return q_rot


def attend(q_rot, k_cache, v_cache, batch: DeviceBatch, out, workspace, scale=None, stream=None) -> None:
    """The attention call of a staged batch, with its padded or ragged block table."""
    if batch.ragged:
        mixed_step_attention_ragged(q_rot, k_cache, v_cache, batch.cu_seqlens_q, batch.q_start_pos,
                                    batch.context_lens, batch.bt_offsets, batch.block_tables, batch.context_total,
                                    out, workspace, scale=scale, stream=stream)
    else:
        mixed_step_attention(q_rot, k_cache, v_cache, batch.cu_seqlens_q, batch.q_start_pos, batch.context_lens,
                             batch.block_tables, batch.context_total, out, workspace, scale=scale, stream=stream)
