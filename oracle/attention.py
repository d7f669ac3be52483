"""Oracle: causal attention of a packed mixed batch over the paged KV cache, fp64.

Sources: "Chunked Prefill 的 Token 预算" (zwjcode.cn), section 02 -- the chunk at
[c, c+d) reads the cached [0, c) K/V and attends causally within itself, which
equals full prefill because position i only depends on 0..i; section 07 -- the
query at chunk index i sees keys {0, 1, ..., c+i}; "Chunked Prefill: Ending the
Great Stall", section 05 -- each chunk is an ordinary causal attention call of
its queries against all keys up to the chunk's end; "Prefill head-of-line
blocking" (sference.com), "How a request actually gets served" -- a decode
reads the whole cache to produce one vector.

This is the plain definition: for the query at absolute position p and query
head h (KV head h // (H_q / H_kv)),

    s_j = scale * sum_d q[h, d] * K[j, d]       for j = 0..p
    o   = sum_j exp(s_j - max_j s_j) * V[j] / sum_j exp(s_j - max_j s_j)

with K/V row j read from page block_table[j // 16], slot j % 16.  All
arithmetic is fp64 on the bf16 input values.  Reading: scale = 1/sqrt(D).
"""
from __future__ import annotations

import numpy as np

from .rope import bf16_to_f64


def _gather(pool_bits: np.ndarray, table: np.ndarray, n_keys: int, kv_head: int, page_size: int):
    """Keys 0..n_keys-1 of one KV head, in logical order, as fp64 [n_keys, D]."""
    j = np.arange(n_keys)
    pages = np.asarray(table, dtype=np.int64)[j // page_size]
    return bf16_to_f64(pool_bits[pages, kv_head, j % page_size, :])


def attention_rows(q_rot_bits, k_pool_bits, v_pool_bits, meta, H_kv: int, scale=None,
                   select=None, page_size: int = 16):
    """fp64 outputs for selected (token, q_head) pairs of the packed batch.

    ``meta`` holds cu_seqlens_q, q_start_pos and block_tables (numpy).
    ``select`` is an iterable of (t, h); None means every pair.
    Returns {(t, h): fp64 vector [D]}.
    """
    T, H_q, D = q_rot_bits.shape
    G = H_q // H_kv
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    cu = np.asarray(meta["cu_seqlens_q"])
    c0 = np.asarray(meta["q_start_pos"])
    tables = np.asarray(meta["block_tables"])
    row_of = np.searchsorted(cu, np.arange(T), side="right") - 1
    if select is None:
        select = [(t, h) for t in range(T) for h in range(H_q)]
    groups = {}
    for t, h in select:
        groups.setdefault((int(row_of[t]), h // G), []).append((t, h))
    out = {}
    for (s, kvh), pairs in groups.items():
        n_all = int(c0[s]) + int(cu[s + 1] - cu[s])
        K = _gather(k_pool_bits, tables[s], n_all, kvh, page_size)
        V = _gather(v_pool_bits, tables[s], n_all, kvh, page_size)
        for t, h in pairs:
            pos = int(c0[s]) + (t - int(cu[s]))
            q = bf16_to_f64(q_rot_bits[t, h])
            scores = scale * (K[: pos + 1] @ q)
            w = np.exp(scores - scores.max())
            out[(t, h)] = (w @ V[: pos + 1]) / w.sum()
    return out


def attention_all(q_rot_bits, k_pool_bits, v_pool_bits, meta, H_kv: int, scale=None,
                  page_size: int = 16) -> np.ndarray:
    """fp64 output [T, H_q, D] for every token and head of the packed batch."""
    T, H_q, D = q_rot_bits.shape
    res = attention_rows(q_rot_bits, k_pool_bits, v_pool_bits, meta, H_kv, scale, None, page_size)
    out = np.zeros((T, H_q, D), dtype=np.float64)
    for (t, h), o in res.items():
        out[t, h] = o
    return out
