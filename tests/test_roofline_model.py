"""Pins for the algorithmic work model against the pages' own numbers."""
from chunked_prefill_mixed_decode_gb300 import roofline


def test_chunked_prefill_kv_reread_matches_page():
    """"Chunked Prefill: Ending the Great Stall", section 05: L = 4,096 in chunks of 512
    reads 18,432 KV-token entries against 4,096 for a monolithic prefill (about 4.5x)."""
    chunks = [(512 * k, 512) for k in range(8)]
    assert roofline.step_counts(chunks, 1, 1, 64)["kv_token_reads"] == 18432
    assert roofline.step_counts([(0, 4096)], 1, 1, 64)["kv_token_reads"] == 4096


def test_causal_pairs_unchanged_by_chunking():
    """"Splitting Prefill From Decode Inside a Step": a T-token prompt performs about T^2/2
    position pairs whether it runs in one pass or in chunks."""
    T = 4096
    full = roofline.step_counts([(0, T)], 1, 1, 64)["causal_pairs"]
    chunked = sum(roofline.step_counts([(c, 448)], 1, 1, 64)["causal_pairs"] for c in range(0, 4032, 448))
    chunked += roofline.step_counts([(4032, 64)], 1, 1, 64)["causal_pairs"]
    assert full == chunked == T * (T + 1) // 2


def test_decode_is_two_flops_per_kv_byte_pair():
    """A decode reads each cached K and V element once and spends 2 FLOPs on each (one
    multiply-add): with G query heads sharing a KV head the FLOPs scale by G, the bytes do not."""
    c = roofline.step_counts([(999, 1)], 8, 2, 128)
    assert c["flops"] == 4 * 128 * 8 * 1000
    assert c["decode_kv_bytes"] == 1000 * 2 * 128 * 2 * 2
