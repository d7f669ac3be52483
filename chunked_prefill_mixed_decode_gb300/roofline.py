"""Algorithmic work of one mixed step: what the method must compute and move.

Counts follow the pages' cost model:
* "Splitting Prefill From Decode Inside a Step", "The arithmetic of chunk
  boundaries": causal attention over a T-token prompt is about T^2/2 position
  pairs whether it runs in one pass or in chunks -- here exactly
  sum over rows of d*c + d(d+1)/2 pairs, at 4*D FLOPs per pair and query head
  (QK^T and PV, one multiply-add each per element);
* "Chunked Prefill: Ending the Great Stall", section 05: the extra cost of
  chunking is HBM traffic -- each chunk reads the KV of its whole prefix, so a
  row reads (c + d) KV tokens; for L = 4096 in chunks of 512 that is 18,432
  token reads against 4,096.

Bytes count each row's K and V once per KV head (shared by its G query heads),
Q in and O out, the append's reads and writes, and the metadata: row offsets,
positions and lengths, and each row's ceil((c + d) / 16) page ids (zwjcode
section 06), the block table in its ragged form; nothing padded or re-read.
"""
from __future__ import annotations

from typing import Iterable, Tuple

BF16 = 2


def step_counts(rows: Iterable[Tuple[int, int]], H_q: int, H_kv: int, D: int) -> dict:
    """rows: (c, d) per packed row.  Returns FLOPs and bytes of append and attention."""
    rows = [(int(c), int(d)) for c, d in rows]
    T = sum(d for _, d in rows)
    S = len(rows)
    pairs = sum(d * c + d * (d + 1) // 2 for c, d in rows)
    kv_tokens = sum(c + d for c, d in rows)
    flops = 4 * D * H_q * pairs
    pages = sum((c + d + 15) // 16 for c, d in rows)
    meta_bytes = 4 * ((S + 1) + 2 * S + (S + 1) + pages)
    attn_bytes = kv_tokens * H_kv * D * BF16 * 2 + 2 * T * H_q * D * BF16 + meta_bytes
    append_bytes = T * (2 * H_q * D * BF16 + 4 * H_kv * D * BF16 + 2 * (D // 2) * 4) + 8 * T
    dec = [(c, d) for c, d in rows if d == 1]
    chk = [(c, d) for c, d in rows if d > 1]
    return {
        "tokens": T,
        "rows": S,
        "causal_pairs": pairs,
        "kv_token_reads": kv_tokens,
        "flops": flops,
        "attn_bytes": attn_bytes,
        "append_bytes": append_bytes,
        "step_bytes": attn_bytes + append_bytes,
        "decode_kv_bytes": sum(c + d for c, d in dec) * H_kv * D * BF16 * 2,
        "chunk_flops": 4 * D * H_q * sum(d * c + d * (d + 1) // 2 for c, d in chk),
    }


def roofline_time_s(counts: dict, hbm_gbs: float, tflops: float, bytes_key: str = "step_bytes") -> dict:
    t_mem = counts[bytes_key] / (hbm_gbs * 1e9)
    t_flop = counts["flops"] / (tflops * 1e12)
    return {"t_mem_s": t_mem, "t_flop_s": t_flop, "t_roof_s": max(t_mem, t_flop),
            "bound": "hbm" if t_mem >= t_flop else "tensor"}
