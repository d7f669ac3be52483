"""Python binding of the mixed-batch attention step (libmixed_step.so).

Argument marshalling only: every step of the path runs in the C++ scheduler
and the sm_103a kernels behind the C ABI declared in include/mixed_step.h.
Because the ABI takes bare addresses, each device wrapper checks its tensors'
dtype, contiguity, shape, size and device first and raises ValueError.
The functions keep the C names without the ``ms_`` prefix.  Device tensors
are torch tensors (used for memory and streams only); host metadata is numpy.

There is no fallback: if the shared library is missing or cannot be loaded,
every call raises.  Build it with ``chunked_prefill_mixed_decode_gb300.build.build()``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import numpy as np

from .build import LIB as _LIB_PATH

MS_OK, MS_ERR_ARG, MS_ERR_BUDGET, MS_ERR_NO_PAGES, MS_ERR_CUDA, MS_ERR_DEVICE = 0, -1, -2, -3, -4, -5
MS_ERR_SCRATCH = -6
STATUS_BAD_SLOT, STATUS_BAD_POSITION, STATUS_BAD_PAGE, STATUS_TIMEOUT, STATUS_BAD_META = 1, 2, 4, 8, 16
STATUS_INTERNAL = 32
PAGE_SIZE = 16

_ERR_NAMES = {MS_ERR_ARG: "MS_ERR_ARG", MS_ERR_BUDGET: "MS_ERR_BUDGET", MS_ERR_NO_PAGES: "MS_ERR_NO_PAGES",
              MS_ERR_CUDA: "MS_ERR_CUDA", MS_ERR_DEVICE: "MS_ERR_DEVICE", MS_ERR_SCRATCH: "MS_ERR_SCRATCH"}


class MixedStepError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} failed: {_ERR_NAMES.get(code, code)}")
        self.code = code


class Request(ctypes.Structure):
    _fields_ = [("cached_len", ctypes.c_int32), ("remaining_prompt", ctypes.c_int32),
                ("block_table", ctypes.POINTER(ctypes.c_int32)), ("num_pages", ctypes.c_int32)]


POLICY_DECODE_FIRST, POLICY_PREFILL_FIRST, POLICY_FAIR_SHARE = 0, 1, 2


class SchedConfig(ctypes.Structure):
    _fields_ = [("token_budget", ctypes.c_int32), ("max_chunk_per_request", ctypes.c_int32),
                ("policy", ctypes.c_int32), ("min_chunk_per_request", ctypes.c_int32),
                ("prefill_quota", ctypes.c_int32), ("decode_share_permille", ctypes.c_int32)]


class BatchInfo(ctypes.Structure):
    _fields_ = [("num_rows", ctypes.c_int32), ("num_decodes", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("bt_stride", ctypes.c_int32), ("unused_tokens", ctypes.c_int32), ("num_deferred", ctypes.c_int32)]


class EngineStats(ctypes.Structure):
    _fields_ = [("num_live", ctypes.c_int32), ("num_prefilling", ctypes.c_int32),
                ("num_free_pages", ctypes.c_int32), ("num_pages", ctypes.c_int32),
                ("max_request_pages", ctypes.c_int32), ("rounds", ctypes.c_int64)]


class GraphConfig(ctypes.Structure):
    _fields_ = [("H_q", ctypes.c_int32), ("H_kv", ctypes.c_int32), ("D", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("max_rows", ctypes.c_int32), ("max_row_pages", ctypes.c_int32),
                ("max_pos", ctypes.c_int32), ("scale", ctypes.c_float), ("num_buckets", ctypes.c_int32),
                ("buckets", ctypes.POINTER(ctypes.c_int32))]


class GraphBuffers(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in ("q", "k", "v", "cos_tab", "sin_tab", "k_cache", "v_cache", "q_rot",
                                                "out", "workspace")] + \
               [("ws_bytes", ctypes.c_size_t), ("dev_status", ctypes.c_void_p)]


_lib_handle = None
# ms_mixed_step runs the attention's prologue inside the append's launch on steps of at most
# this many rows (mixed_step.h)
FUSED_STEP_MAX_ROWS = 1024

_I32P = ctypes.POINTER(ctypes.c_int32)
_VP = ctypes.c_void_p


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it has not been built)."""
    global _lib_handle
    if _lib_handle is not None:
        return _lib_handle
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: run chunked_prefill_mixed_decode_gb300.build.build() first")
    h = ctypes.CDLL(_LIB_PATH)
    h.ms_build_batch_metadata.restype = ctypes.c_int
    h.ms_build_batch_metadata.argtypes = [
        ctypes.POINTER(Request), ctypes.c_int32, ctypes.POINTER(SchedConfig), ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int64, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P, ctypes.POINTER(BatchInfo)]
    h.ms_rope_table.restype = ctypes.c_int
    h.ms_rope_table.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_double, _VP, _VP]
    h.ms_kv_append_rope.restype = ctypes.c_int
    h.ms_kv_append_rope.argtypes = [_VP, _VP, _VP, _VP, _VP, ctypes.c_int32, _VP, _VP, ctypes.c_int32, _VP, _VP,
                                    ctypes.c_int32, _VP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                    ctypes.c_int32, _VP, _VP]
    h.ms_attention_workspace_size.restype = ctypes.c_size_t
    h.ms_attention_workspace_size.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                              ctypes.c_int32, ctypes.c_int32]
    h.ms_mixed_step_attention.restype = ctypes.c_int
    h.ms_mixed_step_attention.argtypes = [_VP, _VP, _VP, ctypes.c_int32, _VP, _VP, _VP, _VP, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _VP, _VP,
                                          ctypes.c_size_t, _VP]
    h.ms_build_batch_metadata_ragged.restype = ctypes.c_int
    h.ms_build_batch_metadata_ragged.argtypes = [
        ctypes.POINTER(Request), ctypes.c_int32, ctypes.POINTER(SchedConfig), ctypes.c_int32, ctypes.c_int32,
        ctypes.c_int64, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P, ctypes.POINTER(BatchInfo)]
    h.ms_mixed_step_attention_ragged.restype = ctypes.c_int
    h.ms_mixed_step_attention_ragged.argtypes = [_VP, _VP, _VP, ctypes.c_int32, _VP, _VP, _VP, _VP, _VP,
                                                 ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                 ctypes.c_float, _VP, _VP, ctypes.c_size_t, _VP]
    h.ms_mixed_step.restype = ctypes.c_int
    h.ms_mixed_step.argtypes = [_VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_int32, _VP, _VP, ctypes.c_int32, _VP,
                                _VP, _VP, _VP, _VP, _VP, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                ctypes.c_int32, ctypes.c_float, _VP, _VP, ctypes.c_size_t, _VP, _VP]
    h.ms_mixed_step_attention_noalloc.restype = ctypes.c_int
    h.ms_mixed_step_attention_noalloc.argtypes = [_VP, _VP, _VP, ctypes.c_int32, _VP, _VP, _VP, _VP,
                                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                                  ctypes.c_float, _VP, _VP, _VP]
    h.ms_test_attention_stall.restype = ctypes.c_int
    h.ms_test_attention_stall.argtypes = [_VP, _VP, _VP, ctypes.c_int32, _VP, _VP, _VP, _VP, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_float, _VP, _VP,
                                          ctypes.c_size_t, ctypes.c_int64, _VP]
    h.ms_test_attention_split.restype = ctypes.c_int
    h.ms_test_attention_split.argtypes = [_VP, _VP, _VP, ctypes.c_int32, _VP, _VP, _VP, _VP, _VP, ctypes.c_int64,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
                                          ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                          ctypes.c_float, _VP, _VP, ctypes.c_size_t, ctypes.c_int32, _VP]
    h.ms_cost_model_rates.restype = ctypes.c_int
    h.ms_cost_model_rates.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_float)]
    h.ms_read_status.restype = ctypes.c_int
    h.ms_read_status.argtypes = [_VP, _VP, _I32P]
    h.ms_num_sms.restype = ctypes.c_int
    h.ms_num_sms.argtypes = []
    for name, args in (
            ("ms_engine_create", [ctypes.c_int32, ctypes.POINTER(SchedConfig), ctypes.POINTER(_VP)]),
            ("ms_engine_destroy", [_VP]),
            ("ms_engine_add_request", [_VP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _I32P]),
            ("ms_engine_request_pages", [_VP, ctypes.c_int32, _I32P, ctypes.c_int32, _I32P]),
            ("ms_engine_plan", [_VP, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _I32P, _I32P, _I32P, _I32P,
                                _I32P, _I32P, _I32P, ctypes.POINTER(BatchInfo)]),
            ("ms_engine_commit", [_VP, _I32P, ctypes.c_int32, _I32P]),
            ("ms_engine_stats", [_VP, ctypes.POINTER(EngineStats)]),
            ("ms_graph_create", [ctypes.POINTER(GraphConfig), ctypes.POINTER(GraphBuffers), _VP,
                                 ctypes.POINTER(_VP)]),
            ("ms_graph_destroy", [_VP]),
            ("ms_graph_bucket", [_VP, ctypes.c_int32]),
            ("ms_graph_run", [_VP, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P, ctypes.c_int32, ctypes.c_int32,
                              ctypes.c_int32, _VP, _I32P]),
            ("ms_graph_read_status", [_VP, _VP, _I32P])):
        getattr(h, name).restype = ctypes.c_int
        getattr(h, name).argtypes = args
    h.ms_graph_workspace_size.restype = ctypes.c_size_t
    h.ms_graph_workspace_size.argtypes = [ctypes.POINTER(GraphConfig)]
    _lib_handle = h
    return h


def _check(rc: int, what: str) -> None:
    if rc != MS_OK:
        raise MixedStepError(rc, what)


def _i32(a: np.ndarray):
    return a.ctypes.data_as(_I32P)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _stream(stream) -> int:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    return int(getattr(stream, "cuda_stream", stream))


# ---------------------------------------------------------------------------- host

def build_batch_metadata(states: Sequence[tuple], block_tables: Sequence[np.ndarray], token_budget: int,
                         max_chunk_per_request: int = 0, policy: int = POLICY_DECODE_FIRST,
                         min_chunk_per_request: int = 0, prefill_quota: int = 0,
                         decode_share_permille: int = 500, ragged: bool = False) -> dict:
    """Token-budget packing + varlen metadata (ms_build_batch_metadata).

    ``states[i] = (cached_len, remaining_prompt)``; ``block_tables[i]`` is an
    int32 array of that request's physical pages.  Returns numpy int32 arrays
    and the batch summary.  With ``ragged`` (ms_build_batch_metadata_ragged)
    the block table comes as ``bt_offsets`` [rows + 1] and ``bt_pages`` (each
    row's pages in use, back to back) instead of padded ``block_tables``.
    """
    n = len(states)
    reqs, keep = _request_array(states, block_tables)
    lens = reqs["num_pages"][:n]
    cfg = SchedConfig(int(token_budget), int(max_chunk_per_request), int(policy), int(min_chunk_per_request),
                      int(prefill_quota), int(decode_share_permille))
    cap_rows = max(n, 1)
    cap_tokens = max(int(token_budget), 1)
    max_pages = max(int(lens.max()) if n else 0, 1)
    # ragged: a row reads at most its request's pages
    cap_bt = max(int(lens.sum()) if n else 0, 1) if ragged else cap_rows * max_pages
    # one output buffer; the returned arrays are views of it
    bt_sizes = (("bt_offsets", cap_rows + 1), ("bt_pages", cap_bt)) if ragged else (("block_tables", cap_bt),)
    sizes = (("cu_seqlens_q", cap_rows + 1), ("q_start_pos", cap_rows), ("context_lens", cap_rows),
             ("positions", cap_tokens), ("slot_mapping", cap_tokens)) + bt_sizes + \
        (("row_req", cap_rows), ("num_scheduled", max(n, 1)))
    # every element a returned view covers is written by the call
    buf = np.empty(sum(sz for _, sz in sizes), dtype=np.int32)
    out, off = {}, 0
    for k, sz in sizes:
        out[k] = buf[off:off + sz]
        off += sz
    info = BatchInfo()
    reqp = reqs.ctypes.data_as(ctypes.POINTER(Request))
    if ragged:
        rc = lib().ms_build_batch_metadata_ragged(reqp, n, ctypes.byref(cfg), cap_rows, cap_tokens, cap_bt,
                                                  _i32(out["cu_seqlens_q"]), _i32(out["q_start_pos"]),
                                                  _i32(out["context_lens"]), _i32(out["positions"]),
                                                  _i32(out["slot_mapping"]), _i32(out["bt_offsets"]),
                                                  _i32(out["bt_pages"]), _i32(out["row_req"]),
                                                  _i32(out["num_scheduled"]), ctypes.byref(info))
    else:
        rc = lib().ms_build_batch_metadata(reqp, n, ctypes.byref(cfg), cap_rows, cap_tokens, cap_bt,
                                           _i32(out["cu_seqlens_q"]), _i32(out["q_start_pos"]),
                                           _i32(out["context_lens"]), _i32(out["positions"]),
                                           _i32(out["slot_mapping"]), _i32(out["block_tables"]),
                                           _i32(out["row_req"]), _i32(out["num_scheduled"]), ctypes.byref(info))
    del keep
    _check(rc, "ms_build_batch_metadata_ragged" if ragged else "ms_build_batch_metadata")
    S, T, stride = info.num_rows, info.num_tokens, info.bt_stride
    if ragged:
        pages = int(out["bt_offsets"][S])
        tables = {"bt_offsets": out["bt_offsets"][: S + 1], "bt_pages": out["bt_pages"][:pages]}
    else:
        tables = {"block_tables": out["block_tables"][: S * stride].reshape(S, stride)}
    return {
        "cu_seqlens_q": out["cu_seqlens_q"][: S + 1],
        "q_start_pos": out["q_start_pos"][:S],
        "context_lens": out["context_lens"][:S],
        "positions": out["positions"][:T],
        "slot_mapping": out["slot_mapping"][:T],
        **tables,
        "bt_stride": stride,
        "row_req": out["row_req"][:S],
        "num_scheduled": out["num_scheduled"][:n],
        "num_rows": S,
        "num_decodes": info.num_decodes,
        "num_tokens": T,
        "unused_tokens": info.unused_tokens,
        "num_deferred": info.num_deferred,
    }


# ms_request as a numpy record: filled column by column instead of request by request
_REQ_DTYPE = np.dtype({"names": ["cached_len", "remaining_prompt", "block_table", "num_pages"],
                       "formats": ["<i4", "<i4", "<u8", "<i4"], "offsets": [0, 4, 8, 16],
                       "itemsize": ctypes.sizeof(Request)})


def _request_array(states, block_tables):
    """ms_request records for the requests; also returns the concatenated block
    tables, which must stay alive while the records are in use."""
    n = len(states)
    if n != len(block_tables):
        raise ValueError("one block table per request")
    reqs = np.zeros(max(n, 1), dtype=_REQ_DTYPE)
    if n == 0:
        return reqs, None
    st = np.asarray(states, dtype=np.int64).reshape(n, 2)
    lens = np.fromiter((len(bt) for bt in block_tables), dtype=np.int64, count=n)
    if (st < np.iinfo(np.int32).min).any() or (st > np.iinfo(np.int32).max).any():
        raise ValueError("request lengths out of int32 range")
    flat = np.ascontiguousarray(np.concatenate([np.asarray(bt).reshape(-1) for bt in block_tables]), dtype=np.int32) \
        if lens.sum() else np.zeros(1, dtype=np.int32)
    starts = np.concatenate(([0], np.cumsum(lens)[:-1]))
    reqs["cached_len"][:n] = st[:, 0]
    reqs["remaining_prompt"][:n] = st[:, 1]
    reqs["num_pages"][:n] = lens
    reqs["block_table"][:n] = np.where(lens > 0, flat.ctypes.data + 4 * starts, 0).astype(np.uint64)
    return reqs, flat


class Engine:
    """Multi-round engine over a page pool (ms_engine_*): full-input admission, then
    plan / device step / commit every round."""

    def __init__(self, num_pages: int, token_budget: int, max_chunk_per_request: int = 0,
                 policy: int = POLICY_DECODE_FIRST, min_chunk_per_request: int = 0, prefill_quota: int = 0,
                 decode_share_permille: int = 500):
        self._h = None
        self.token_budget = int(token_budget)
        cfg = SchedConfig(int(token_budget), int(max_chunk_per_request), int(policy), int(min_chunk_per_request),
                          int(prefill_quota), int(decode_share_permille))
        h = _VP()
        _check(lib().ms_engine_create(int(num_pages), ctypes.byref(cfg), ctypes.byref(h)), "ms_engine_create")
        self._h = h

    def __del__(self):
        if getattr(self, "_h", None) is not None and _lib_handle is not None:
            _lib_handle.ms_engine_destroy(self._h)
            self._h = None

    def add_request(self, prompt_len: int, max_new_tokens: int, cached_len: int = 0) -> int:
        """Admit a request; raises MixedStepError(MS_ERR_NO_PAGES) when the pool cannot hold it."""
        rid = ctypes.c_int32()
        _check(lib().ms_engine_add_request(self._h, int(prompt_len), int(max_new_tokens), int(cached_len),
                                           ctypes.byref(rid)), "ms_engine_add_request")
        return rid.value

    def stats(self) -> dict:
        st = EngineStats()
        _check(lib().ms_engine_stats(self._h, ctypes.byref(st)), "ms_engine_stats")
        return {k: getattr(st, k) for k, _ in EngineStats._fields_}

    def request_pages(self, request_id: int) -> np.ndarray:
        n = ctypes.c_int32()
        cap = self.stats()["max_request_pages"]
        out = np.zeros(max(cap, 1), dtype=np.int32)
        _check(lib().ms_engine_request_pages(self._h, int(request_id), _i32(out), cap, ctypes.byref(n)),
               "ms_engine_request_pages")
        return out[: n.value].copy()

    def plan(self) -> dict:
        """Pack the next round; the metadata of build_batch_metadata plus row_request_id."""
        st = self.stats()
        cap_rows = max(st["num_live"], 1)
        cap_tokens = max(self.token_budget, 1)
        cap_bt = cap_rows * max(st["max_request_pages"], 1)
        sizes = (("cu_seqlens_q", cap_rows + 1), ("q_start_pos", cap_rows), ("context_lens", cap_rows),
                 ("positions", cap_tokens), ("slot_mapping", cap_tokens), ("block_tables", cap_bt),
                 ("row_request_id", cap_rows))
        # the returned arrays are views of it; every element they cover is written by the call
        buf = np.empty(sum(sz for _, sz in sizes), dtype=np.int32)
        out, off = {}, 0
        for k, sz in sizes:
            out[k] = buf[off:off + sz]
            off += sz
        info = BatchInfo()
        rc = lib().ms_engine_plan(self._h, cap_rows, cap_tokens, cap_bt, _i32(out["cu_seqlens_q"]),
                                  _i32(out["q_start_pos"]), _i32(out["context_lens"]), _i32(out["positions"]),
                                  _i32(out["slot_mapping"]), _i32(out["block_tables"]),
                                  _i32(out["row_request_id"]), ctypes.byref(info))
        _check(rc, "ms_engine_plan")
        S, T, stride = info.num_rows, info.num_tokens, info.bt_stride
        return {
            "cu_seqlens_q": out["cu_seqlens_q"][: S + 1],
            "q_start_pos": out["q_start_pos"][:S],
            "context_lens": out["context_lens"][:S],
            "positions": out["positions"][:T],
            "slot_mapping": out["slot_mapping"][:T],
            "block_tables": out["block_tables"][: S * stride].reshape(S, stride),
            "bt_stride": stride,
            "row_request_id": out["row_request_id"][:S],
            "num_rows": S,
            "num_decodes": info.num_decodes,
            "num_tokens": T,
            "unused_tokens": info.unused_tokens,
            "num_deferred": info.num_deferred,
        }

    def commit(self) -> list:
        """Advance the planned rows; returns the ids of the requests that finished."""
        cap = max(self.stats()["num_live"], 1)
        ids = np.zeros(cap, dtype=np.int32)
        n = ctypes.c_int32()
        _check(lib().ms_engine_commit(self._h, _i32(ids), cap, ctypes.byref(n)), "ms_engine_commit")
        return ids[: n.value].tolist()


class StepGraph:
    """One captured CUDA graph per token bucket of the whole step (ms_graph_*).

    Owns fixed device buffers: ``q``, ``k``, ``v`` (write a step's new tokens
    into their first rows), ``q_rot`` and ``out``, [largest bucket, heads, D].
    ``stream`` must be a side stream (the legacy default stream cannot be
    captured)."""

    def __init__(self, k_cache, v_cache, cos, sin, H_q: int, max_rows: int, max_row_pages: int, buckets,
                 stream, scale: float = None):
        import torch
        self._h = None
        if k_cache.dim() != 4 or cos.dim() != 2:
            raise ValueError("k_cache must be [pages, H_kv, 16, D] and cos, sin [max_pos, D/2]")
        dev = k_cache.device
        num_pages, H_kv, _, D = k_cache.shape
        _pools(k_cache, v_cache, H_kv, D)
        _dev(cos, "cos", torch.float32, (cos.shape[0], D // 2))
        _dev(sin, "sin", torch.float32, cos.shape)
        _on_one_gpu("k_cache v_cache cos sin", k_cache, v_cache, cos, sin)
        self.buckets = [int(b) for b in buckets]
        B = self.buckets[-1]
        self.stream = stream
        self.q = torch.zeros((B, H_q, D), dtype=torch.bfloat16, device=dev)
        self.k = torch.zeros((B, H_kv, D), dtype=torch.bfloat16, device=dev)
        self.v = torch.zeros((B, H_kv, D), dtype=torch.bfloat16, device=dev)
        self.q_rot = torch.zeros_like(self.q)
        self.out = torch.zeros_like(self.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self._bk = np.asarray(self.buckets, dtype=np.int32)
        self._cfg = GraphConfig(H_q, H_kv, D, num_pages, int(max_rows), int(max_row_pages), int(cos.shape[0]),
                                float(scale if scale is not None else float(D) ** -0.5), len(self.buckets),
                                _i32(self._bk))
        n = lib().ms_graph_workspace_size(ctypes.byref(self._cfg))
        if n == 0:
            raise MixedStepError(MS_ERR_ARG, "ms_graph_workspace_size")
        self.workspace = torch.empty(n, dtype=torch.uint8, device=dev)
        self._keep = (k_cache, v_cache, cos, sin)
        bufs = GraphBuffers(_ptr(self.q), _ptr(self.k), _ptr(self.v), _ptr(cos), _ptr(sin), _ptr(k_cache),
                            _ptr(v_cache), _ptr(self.q_rot), _ptr(self.out), _ptr(self.workspace), n,
                            _ptr(self.status))
        h = _VP()
        _check(lib().ms_graph_create(ctypes.byref(self._cfg), ctypes.byref(bufs), _stream(stream), ctypes.byref(h)),
               "ms_graph_create")
        self._h = h

    def __del__(self):
        if getattr(self, "_h", None) is not None and _lib_handle is not None:
            _lib_handle.ms_graph_destroy(self._h)
            self._h = None

    def bucket(self, num_tokens: int) -> int:
        b = lib().ms_graph_bucket(self._h, int(num_tokens))
        _check(min(b, 0), "ms_graph_bucket")
        return b

    def run(self, meta: dict) -> int:
        """Replay the step for host metadata ``meta`` (build_batch_metadata or Engine.plan);
        returns the bucket it ran in."""
        arrs = [np.ascontiguousarray(meta[k], dtype=np.int32).reshape(-1)
                for k in ("cu_seqlens_q", "q_start_pos", "context_lens", "positions", "slot_mapping",
                          "block_tables")]
        arrs = [a if a.size else np.zeros(1, dtype=np.int32) for a in arrs]
        used = ctypes.c_int32()
        rc = lib().ms_graph_run(self._h, *[_i32(a) for a in arrs], int(meta["bt_stride"]), int(meta["num_rows"]),
                                int(meta["num_tokens"]), _stream(self.stream), ctypes.byref(used))
        _check(rc, "ms_graph_run")
        return used.value

    def read_status(self) -> int:
        v = ctypes.c_int32()
        rc = lib().ms_graph_read_status(self._h, _stream(self.stream), ctypes.byref(v))
        if rc not in (MS_OK, MS_ERR_DEVICE):
            _check(rc, "ms_graph_read_status")
        return int(v.value)


def rope_table(max_pos: int, D: int, base: float = 10000.0):
    """fp32 cos/sin tables [max_pos, D/2] on the host (ms_rope_table)."""
    cos = np.empty((max_pos, D // 2), dtype=np.float32)
    sin = np.empty((max_pos, D // 2), dtype=np.float32)
    _check(lib().ms_rope_table(int(max_pos), int(D), float(base), cos.ctypes.data, sin.ctypes.data),
           "ms_rope_table")
    return cos, sin


def attention_workspace_size(max_rows: int, max_tokens: int, max_context_total: int, H_q: int, H_kv: int,
                             D: int) -> int:
    return int(lib().ms_attention_workspace_size(int(max_rows), int(max_tokens), int(max_context_total), int(H_q),
                                                 int(H_kv), int(D)))


def num_sms() -> int:
    n = lib().ms_num_sms()
    _check(n if n < 0 else 0, "ms_num_sms")
    return n


# ---------------------------------------------------------------------------- device

def _dev(t, name: str, dtype, shape=None, min_numel: int = 0) -> None:
    """Check a tensor before its pointer crosses the C ABI, which sees only an
    address: dtype, dense row-major layout, then shape or size."""
    if t is None:
        raise ValueError(f"{name} is required")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None:
        if t.shape != shape:
            raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    elif min_numel and t.numel() < min_numel:
        raise ValueError(f"{name} must hold at least {min_numel} elements, got {t.numel()}")


def _on_one_gpu(names: str, *tensors) -> None:
    """Every tensor (None entries skipped) on the CUDA device of the first;
    ``names`` lists them, space-separated, for the error message."""
    dev = -2
    for i, t in enumerate(tensors):
        if t is None:
            continue
        d = t.get_device()
        if d < 0 or (dev != -2 and d != dev):
            name = names.split()[i]
            if d < 0:
                raise ValueError(f"{name} must be a CUDA tensor, got {t.device}")
            raise ValueError(f"{name} is on {t.device}, the other tensors on cuda:{dev}")
        dev = d


def _pools(k_cache, v_cache, H_kv: int, D: int) -> None:
    import torch
    if k_cache.dim() != 4:
        raise ValueError(f"k_cache must be [pages, H_kv, {PAGE_SIZE}, D], got {tuple(k_cache.shape)}")
    _dev(k_cache, "k_cache", torch.bfloat16, (k_cache.shape[0], H_kv, PAGE_SIZE, D))
    _dev(v_cache, "v_cache", torch.bfloat16, k_cache.shape)


def kv_append_rope(q, k, v, positions, slot_mapping, cos_tab, sin_tab, k_cache, v_cache, q_rot=None,
                   dev_status=None, stream=None) -> None:
    """Rotate q, k at absolute positions; append k, v into the paged pools (ms_kv_append_rope)."""
    import torch
    if q.dim() != 3:
        raise ValueError(f"q must be [T, H_q, D], got {tuple(q.shape)}")
    if k_cache.dim() != 4:
        raise ValueError(f"k_cache must be [pages, H_kv, {PAGE_SIZE}, D], got {tuple(k_cache.shape)}")
    T, H_q, D = q.shape
    H_kv = k_cache.shape[1]
    if q_rot is None:
        q_rot = q
    _dev(q, "q", torch.bfloat16)
    _dev(k, "k", torch.bfloat16, (T, H_kv, D))
    _dev(v, "v", torch.bfloat16, (T, H_kv, D))
    _dev(q_rot, "q_rot", torch.bfloat16, (T, H_q, D))
    _dev(positions, "positions", torch.int32, min_numel=T)
    _dev(slot_mapping, "slot_mapping", torch.int32, min_numel=T)
    if cos_tab.dim() != 2:
        raise ValueError("cos_tab must be [max_pos, D/2]")
    _dev(cos_tab, "cos_tab", torch.float32, (cos_tab.shape[0], D // 2))
    _dev(sin_tab, "sin_tab", torch.float32, cos_tab.shape)
    _pools(k_cache, v_cache, H_kv, D)
    if dev_status is not None:
        _dev(dev_status, "dev_status", torch.int32, min_numel=1)
    _on_one_gpu("q k v q_rot positions slot_mapping cos_tab sin_tab k_cache v_cache dev_status", q, k, v, q_rot,
                positions, slot_mapping, cos_tab, sin_tab, k_cache, v_cache, dev_status)
    rc = lib().ms_kv_append_rope(_ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(slot_mapping), T, _ptr(cos_tab),
                                 _ptr(sin_tab), cos_tab.shape[0], _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                 _ptr(q_rot), H_q, H_kv, D, PAGE_SIZE, _ptr(dev_status), _stream(stream))
    _check(rc, "ms_kv_append_rope")


def _attention_args(q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens, block_tables, out):
    """Shapes of an attention call, after checking its tensors."""
    import torch
    if q_rot.dim() != 3:
        raise ValueError("q_rot must be [T, H_q, D]")
    T, H_q, D = q_rot.shape
    _dev(q_rot, "q_rot", torch.bfloat16)
    if k_cache.dim() != 4:
        raise ValueError(f"k_cache must be [pages, H_kv, {PAGE_SIZE}, D], got {tuple(k_cache.shape)}")
    H_kv = k_cache.shape[1]
    _pools(k_cache, v_cache, H_kv, D)
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.shape[0] < 1:
        raise ValueError("cu_seqlens_q must be 1-D with rows + 1 entries")
    S = cu_seqlens_q.shape[0] - 1
    _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _dev(q_start_pos, "q_start_pos", torch.int32, min_numel=S)
    _dev(context_lens, "context_lens", torch.int32, min_numel=S)
    stride = block_tables.shape[1] if block_tables.dim() == 2 else block_tables.shape[0] // max(S, 1)
    _dev(block_tables, "block_tables", torch.int32, min_numel=S * stride)
    _dev(out, "out", torch.bfloat16, (T, H_q, D))
    _on_one_gpu("q_rot k_cache v_cache cu_seqlens_q q_start_pos context_lens block_tables out", q_rot, k_cache,
                v_cache, cu_seqlens_q, q_start_pos, context_lens, block_tables, out)
    return T, H_q, D, H_kv, S, stride


def mixed_step_attention(q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens, block_tables,
                         context_total: int, out, workspace, scale: float = None, stream=None) -> None:
    """Causal attention of every packed row over its paged context (ms_mixed_step_attention).

    Metadata arguments are device int32 tensors; ``block_tables`` is [rows, stride].
    ``context_total`` is the host-side sum of context_lens (bounds the workspace).
    """
    T, H_q, D, H_kv, S, stride = _attention_args(q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens,
                                                 block_tables, out)
    _dev(workspace, "workspace", None)
    _on_one_gpu("q_rot workspace", q_rot, workspace)
    if scale is None:
        scale = float(D) ** -0.5
    rc = lib().ms_mixed_step_attention(_ptr(q_rot), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                       _ptr(cu_seqlens_q), _ptr(q_start_pos), _ptr(context_lens),
                                       _ptr(block_tables), stride, S, T, int(context_total), H_q, H_kv, D,
                                       PAGE_SIZE, float(scale), _ptr(out), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "ms_mixed_step_attention")


def mixed_step_attention_ragged(q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens, bt_offsets,
                                bt_pages, context_total: int, out, workspace, scale: float = None,
                                stream=None) -> None:
    """Attention with the ragged block table (ms_mixed_step_attention_ragged): row s reads its pages
    from ``bt_pages[bt_offsets[s]:bt_offsets[s + 1]]`` (device int32 tensors)."""
    import torch
    if q_rot.dim() != 3:
        raise ValueError("q_rot must be [T, H_q, D]")
    T, H_q, D = q_rot.shape
    _dev(q_rot, "q_rot", torch.bfloat16)
    if k_cache.dim() != 4:
        raise ValueError(f"k_cache must be [pages, H_kv, {PAGE_SIZE}, D], got {tuple(k_cache.shape)}")
    H_kv = k_cache.shape[1]
    _pools(k_cache, v_cache, H_kv, D)
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.shape[0] < 1:
        raise ValueError("cu_seqlens_q must be 1-D with rows + 1 entries")
    S = cu_seqlens_q.shape[0] - 1
    _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _dev(q_start_pos, "q_start_pos", torch.int32, min_numel=S)
    _dev(context_lens, "context_lens", torch.int32, min_numel=S)
    _dev(bt_offsets, "bt_offsets", torch.int32, min_numel=S + 1)
    _dev(bt_pages, "bt_pages", torch.int32, min_numel=1)
    _dev(out, "out", torch.bfloat16, (T, H_q, D))
    _dev(workspace, "workspace", None)
    _on_one_gpu("q_rot k_cache v_cache cu_seqlens_q q_start_pos context_lens bt_offsets bt_pages out workspace",
                q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens, bt_offsets, bt_pages, out,
                workspace)
    if scale is None:
        scale = float(D) ** -0.5
    rc = lib().ms_mixed_step_attention_ragged(_ptr(q_rot), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                              _ptr(cu_seqlens_q), _ptr(q_start_pos), _ptr(context_lens),
                                              _ptr(bt_offsets), _ptr(bt_pages), bt_pages.numel(), S, T,
                                              int(context_total), H_q, H_kv, D, PAGE_SIZE, float(scale), _ptr(out),
                                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                                              _stream(stream))
    _check(rc, "ms_mixed_step_attention_ragged")


def mixed_step(q, k, v, positions, slot_mapping, cos_tab, sin_tab, k_cache, v_cache, q_rot, cu_seqlens_q,
               q_start_pos, context_lens, block_tables, context_total: int, out, workspace, bt_offsets=None,
               dev_status=None, scale: float = None, stream=None) -> None:
    """Append + attention of one step in one call (ms_mixed_step).  ``block_tables`` is the padded
    [rows, stride] table, or, with ``bt_offsets`` given, the ragged page list; the other arguments are
    those of kv_append_rope and mixed_step_attention(_ragged)."""
    import torch
    if q.dim() != 3:
        raise ValueError(f"q must be [T, H_q, D], got {tuple(q.shape)}")
    T, H_q, D = q.shape
    if k_cache.dim() != 4:
        raise ValueError(f"k_cache must be [pages, H_kv, {PAGE_SIZE}, D], got {tuple(k_cache.shape)}")
    H_kv = k_cache.shape[1]
    _dev(q, "q", torch.bfloat16)
    _dev(k, "k", torch.bfloat16, (T, H_kv, D))
    _dev(v, "v", torch.bfloat16, (T, H_kv, D))
    _dev(q_rot, "q_rot", torch.bfloat16, (T, H_q, D))
    _dev(positions, "positions", torch.int32, min_numel=T)
    _dev(slot_mapping, "slot_mapping", torch.int32, min_numel=T)
    if cos_tab.dim() != 2:
        raise ValueError("cos_tab must be [max_pos, D/2]")
    _dev(cos_tab, "cos_tab", torch.float32, (cos_tab.shape[0], D // 2))
    _dev(sin_tab, "sin_tab", torch.float32, cos_tab.shape)
    _pools(k_cache, v_cache, H_kv, D)
    if cu_seqlens_q.dim() != 1 or cu_seqlens_q.shape[0] < 1:
        raise ValueError("cu_seqlens_q must be 1-D with rows + 1 entries")
    S = cu_seqlens_q.shape[0] - 1
    _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _dev(q_start_pos, "q_start_pos", torch.int32, min_numel=S)
    _dev(context_lens, "context_lens", torch.int32, min_numel=S)
    if bt_offsets is None:
        stride = block_tables.shape[1] if block_tables.dim() == 2 else block_tables.shape[0] // max(S, 1)
        _dev(block_tables, "block_tables", torch.int32, min_numel=S * stride)
        bt_len = 0
    else:
        _dev(bt_offsets, "bt_offsets", torch.int32, min_numel=S + 1)
        _dev(block_tables, "block_tables", torch.int32, min_numel=1)
        stride, bt_len = 0, block_tables.numel()
    _dev(out, "out", torch.bfloat16, (T, H_q, D))
    _dev(workspace, "workspace", None)
    if dev_status is not None:
        _dev(dev_status, "dev_status", torch.int32, min_numel=1)
    _on_one_gpu("q k v q_rot positions slot_mapping cos_tab sin_tab k_cache v_cache cu_seqlens_q q_start_pos "
                "context_lens block_tables bt_offsets out workspace dev_status", q, k, v, q_rot, positions,
                slot_mapping, cos_tab, sin_tab, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens,
                block_tables, bt_offsets, out, workspace, dev_status)
    if scale is None:
        scale = float(D) ** -0.5
    rc = lib().ms_mixed_step(_ptr(q), _ptr(k), _ptr(v), _ptr(positions), _ptr(slot_mapping), _ptr(cos_tab),
                             _ptr(sin_tab), cos_tab.shape[0], _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                             _ptr(q_rot), _ptr(cu_seqlens_q), _ptr(q_start_pos), _ptr(context_lens),
                             _ptr(block_tables), _ptr(bt_offsets), bt_len, stride, S, T, int(context_total), H_q,
                             H_kv, D, PAGE_SIZE, float(scale), _ptr(out), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream))
    _check(rc, "ms_mixed_step")


def mixed_step_attention_noalloc(q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens, block_tables,
                                 context_total: int, out, dev_status=None, scale: float = None,
                                 stream=None) -> None:
    """The attention step without a caller workspace (ms_mixed_step_attention_noalloc).

    For callers that cannot allocate device memory on their step path; the
    step runs out of the library's 64 MiB static scratch per device.  Calls
    share that scratch, so they must not overlap on the GPU.  ``dev_status``
    (device int32, optional) receives this call's status bits.
    """
    T, H_q, D, H_kv, S, stride = _attention_args(q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens,
                                                 block_tables, out)
    if dev_status is not None:
        import torch
        _dev(dev_status, "dev_status", torch.int32, min_numel=1)
        _on_one_gpu("q_rot dev_status", q_rot, dev_status)
    if scale is None:
        scale = float(D) ** -0.5
    rc = lib().ms_mixed_step_attention_noalloc(_ptr(q_rot), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                               _ptr(cu_seqlens_q), _ptr(q_start_pos), _ptr(context_lens),
                                               _ptr(block_tables), stride, S, T, int(context_total), H_q, H_kv, D,
                                               PAGE_SIZE, float(scale), _ptr(out), _ptr(dev_status),
                                               _stream(stream))
    _check(rc, "ms_mixed_step_attention_noalloc")


def test_attention_stall(q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens, block_tables,
                         context_total: int, out, workspace, wait_limit_ns: int, scale: float = None,
                         stream=None) -> None:
    """Test hook of the bounded device waits (ms_test_attention_stall): the attention call with every
    chunk-phase producer stopped, so the chunk phase's waits run out after ``wait_limit_ns`` and set
    STATUS_TIMEOUT in the workspace's status word.  Not for production use."""
    T, H_q, D, H_kv, S, stride = _attention_args(q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens,
                                                 block_tables, out)
    _dev(workspace, "workspace", None)
    _on_one_gpu("q_rot workspace", q_rot, workspace)
    if scale is None:
        scale = float(D) ** -0.5
    rc = lib().ms_test_attention_stall(_ptr(q_rot), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                       _ptr(cu_seqlens_q), _ptr(q_start_pos), _ptr(context_lens),
                                       _ptr(block_tables), stride, S, T, int(context_total), H_q, H_kv, D,
                                       PAGE_SIZE, float(scale), _ptr(out), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(), int(wait_limit_ns),
                                       _stream(stream))
    _check(rc, "ms_test_attention_stall")


def test_attention_split(q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens, block_tables,
                         context_total: int, out, workspace, chunk_ctas: int, bt_offsets=None, scale: float = None,
                         stream=None) -> None:
    """Test hook of the SM-split cost model (ms_test_attention_split): the attention call with
    ``chunk_ctas`` CTAs starting on chunk work.  ``block_tables`` is the padded table, or with
    ``bt_offsets`` the ragged page list.  Outputs equal the ordinary call's."""
    import torch
    if q_rot.dim() != 3:
        raise ValueError("q_rot must be [T, H_q, D]")
    T, H_q, D = q_rot.shape
    H_kv = k_cache.shape[1]
    _pools(k_cache, v_cache, H_kv, D)
    S = cu_seqlens_q.shape[0] - 1
    if bt_offsets is None:
        stride = block_tables.shape[1] if block_tables.dim() == 2 else block_tables.shape[0] // max(S, 1)
        bt_len = 0
    else:
        _dev(bt_offsets, "bt_offsets", torch.int32, min_numel=S + 1)
        stride, bt_len = 0, block_tables.numel()
    _dev(block_tables, "block_tables", torch.int32, min_numel=1)
    _dev(out, "out", torch.bfloat16, (T, H_q, D))
    _dev(workspace, "workspace", None)
    _on_one_gpu("q_rot k_cache v_cache cu_seqlens_q q_start_pos context_lens block_tables bt_offsets out workspace",
                q_rot, k_cache, v_cache, cu_seqlens_q, q_start_pos, context_lens, block_tables, bt_offsets, out,
                workspace)
    if scale is None:
        scale = float(D) ** -0.5
    rc = lib().ms_test_attention_split(_ptr(q_rot), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0],
                                       _ptr(cu_seqlens_q), _ptr(q_start_pos), _ptr(context_lens),
                                       _ptr(block_tables), _ptr(bt_offsets), bt_len, stride, S, T,
                                       int(context_total), H_q, H_kv, D, PAGE_SIZE, float(scale), _ptr(out),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       int(chunk_ctas), _stream(stream))
    _check(rc, "ms_test_attention_split")


def cost_model_rates() -> tuple:
    """(rated SM clock in MHz, HBM GB/s) behind the SM split before a call has measured the clock
    (ms_cost_model_rates)."""
    mhz, gbs = ctypes.c_float(0), ctypes.c_float(0)
    _check(lib().ms_cost_model_rates(ctypes.byref(mhz), ctypes.byref(gbs)), "ms_cost_model_rates")
    return float(mhz.value), float(gbs.value)


def read_status(dev_status, stream=None) -> int:
    """Read and clear a device status word (ms_read_status); returns the status bits."""
    import torch  # noqa: F401
    v = ctypes.c_int32(0)
    rc = lib().ms_read_status(_ptr(dev_status), _stream(stream), ctypes.byref(v))
    if rc not in (MS_OK, MS_ERR_DEVICE):
        _check(rc, "ms_read_status")
    return int(v.value)
