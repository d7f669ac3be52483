"""Pins for the oracle's multi-round engine (page pool, full-input admission, plan/commit).

  [zwj] "Chunked Prefill 的 Token 预算" (zwjcode.cn), sections 03, 08 and 11
  [mer] "Splitting Prefill From Decode Inside a Step" (mercemay.com), "The arithmetic of chunk boundaries"
  [sar] "Chunked Prefill: Ending the Great Stall" (manishklach.github.io), sections 04 and 05
"""
import numpy as np
import pytest

import oracle
from conftest import read_golden


def test_worked_example_through_the_engine():
    """[zwj] section 03 table, driven by plan/commit: P takes 5, 5, 2 and decodes in round 4."""
    golden = read_golden("worked_example_rounds.txt")
    e = oracle.Engine(num_pages=64, token_budget=8)
    for n in (37, 64, 100):
        e.add_request(prompt_len=n, max_new_tokens=10, cached_len=n)  # running decodes
    p = e.add_request(prompt_len=12, max_new_tokens=3)
    for g in golden:
        rnd, n_dec, p_chunk, p_done, p_len, used, budget = map(int, g)
        prompt_before = {r.rid: r.rem for r in e.live}[p]
        meta = e.plan()
        rid = meta["row_request_id"]
        d = np.diff(meta["cu_seqlens_q"])
        k = int(np.flatnonzero(rid == p)[0])
        assert meta["num_decodes"] == n_dec, rnd
        chunk = int(d[k]) if prompt_before > 0 else 0  # round 4: P's row is a decode
        assert chunk == p_chunk and (k >= meta["num_decodes"]) == (prompt_before > 0), rnd
        assert budget - meta["unused_tokens"] == used, rnd
        e.commit()
        assert p_len - {r.rid: r.rem for r in e.live}[p] == p_done, rnd


def test_full_input_admission_refuses_up_front():
    """[mer] / [zwj] section 11: reserve the whole sequence at admission, so a request that
    cannot finish is refused before its first chunk instead of failing part way through."""
    e = oracle.Engine(num_pages=10, token_budget=64)
    a = e.add_request(prompt_len=80, max_new_tokens=16)     # 6 pages
    with pytest.raises(oracle.AdmissionError):
        e.add_request(prompt_len=80, max_new_tokens=16)     # 6 more: only 4 free
    assert len(e.free) == 4
    while e.live:
        e.plan()
        e.commit()
    assert sorted(e.free) == list(range(10))                # everything came back
    b = e.add_request(prompt_len=80, max_new_tokens=16)
    assert b == a + 1 and len(e.free) == 4


def test_prefix_caching_prefills_only_the_uncached_suffix():
    """[sar] section 05: with a cached prefix, only the uncached suffix is prefilled, at its
    absolute positions."""
    e = oracle.Engine(num_pages=32, token_budget=64)
    e.add_request(prompt_len=120, max_new_tokens=4, cached_len=100)
    meta = e.plan()
    assert meta["positions"].tolist() == list(range(100, 120))
    assert meta["context_lens"].tolist() == [120]


def test_random_arrivals_keep_pages_and_decodes_consistent():
    """Pages are owned by one live request or free, never both; under decode-first every
    running decode advances every round ([sar] section 04: a waiting prefill never
    displaces a decode); each request's prompt is covered exactly once and it produces
    max_new_tokens tokens."""
    rng = np.random.default_rng(9)
    e = oracle.Engine(num_pages=200, token_budget=48)
    produced = {}
    spec = {}
    for rnd in range(300):
        if rng.random() < 0.3:
            pl = int(rng.integers(1, 150))
            mn = int(rng.integers(1, 20))
            cached = int(rng.integers(0, pl + 1)) if rng.random() < 0.3 else 0
            try:
                rid = e.add_request(pl, mn, cached)
                spec[rid] = (pl, mn, cached)
                produced[rid] = {"prefill": [], "decode": 0}
            except oracle.AdmissionError:
                pass
        owned = [int(p) for r in e.live for p in r.pages]
        assert len(owned) == len(set(owned)) and not set(owned) & set(e.free)
        assert len(owned) + len(e.free) == 200
        running = [r.rid for r in e.live if r.rem == 0]
        if not e.live:
            continue
        meta = e.plan()
        d = np.diff(meta["cu_seqlens_q"])
        rids = meta["row_request_id"].tolist()
        assert set(running) <= set(rids[: meta["num_decodes"]])
        for k, rid in enumerate(rids):
            if k < meta["num_decodes"]:
                produced[rid]["decode"] += 1
            else:
                produced[rid]["prefill"].append((int(meta["q_start_pos"][k]), int(d[k])))
        for rid in e.commit():
            pl, mn, cached = spec[rid]
            segs = produced[rid]["prefill"]
            covered = sum(x for _, x in segs)
            assert covered == pl - cached
            if segs:
                assert segs[0][0] == cached
            assert produced[rid]["decode"] == mn - 1
