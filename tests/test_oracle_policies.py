"""Pins for the oracle's scheduling policies beyond decode-first.

  [sfe] "Prefill head-of-line blocking" (sference.com), "The fix" and "What comes next"
  [mer] "Splitting Prefill From Decode Inside a Step" (mercemay.com), "Choosing the priority order"
  [zwj] "Chunked Prefill 的 Token 预算" (zwjcode.cn), sections 08 and 16
"""
import numpy as np
import pytest

import oracle


def takes(rows, states):
    return {i: d for i, c, d in rows if states[i][1] > 0}


def test_floor_splits_between_long_prefills_and_expands_when_alone():
    """[sfe] "What comes next": as a floor, two long prefills take half the budget each,
    one on its own takes all of it; as a ceiling, a lone long prefill stays at the cap."""
    long2 = [(0, 600000), (0, 600000)]
    rows, unused = oracle.schedule(long2, 8192, min_chunk=4096)
    assert takes(rows, long2) == {0: 4096, 1: 4096} and unused == 0
    alone = [(0, 600000)]
    rows, unused = oracle.schedule(alone, 8192, min_chunk=4096)
    assert takes(rows, alone) == {0: 8192} and unused == 0
    rows, unused = oracle.schedule(alone, 8192, max_chunk=4096)  # the ceiling of "The fix"
    assert takes(rows, alone) == {0: 4096} and unused == 4096


def test_floor_lets_short_prompts_slip_past_a_long_one():
    """[sfe] "What comes next": a guaranteed slice per long request is all short prompts need."""
    st = [(0, 600000), (0, 500), (0, 3000)]
    rows, unused = oracle.schedule(st, 8192, min_chunk=4096)
    t = takes(rows, st)
    assert t[1] == 500 and t[2] == 3000 and t[0] == 8192 - 3500 and unused == 0
    rows, _ = oracle.schedule(st, 8192)  # plain arrival order: the long prompt takes everything
    assert takes(rows, st) == {0: 8192}


def test_concurrency_is_budget_over_threshold():
    """[sfe] "The fix": chunked_prefill_size // threshold partial prefills run at once
    (8192 // 4096 = 2, 16384 // 4096 = 4)."""
    st = [(0, 10**6)] * 6
    for budget, n in ((8192, 2), (16384, 4)):
        rows, _ = oracle.schedule(st, budget, max_chunk=4096)
        assert len(rows) == n and all(d == 4096 for _, _, d in rows)


def test_prefill_quota_prevents_starvation():
    """[zwj] section 16, exercise 3 with the section 08 remedy: reserve 25 % of the budget
    for prefill under decode traffic that never drains; the long prompt still finishes.
    Without the quota it never gets a token."""
    B, P = 16, 100
    states = [(50 + i, 0) for i in range(16)] + [(0, P)]
    for quota, expect_rounds in ((4, 25), (0, None)):
        st = list(states)
        done_in = None
        for rnd in range(1, 60):
            rows, unused = oracle.schedule(st, B, prefill_quota=quota)
            assert sum(d for _, _, d in rows) + unused == B
            n_dec = sum(1 for i, _, _ in rows if st[i][1] == 0)
            assert n_dec <= (B - quota if st[16][1] > 0 else B)
            st = oracle.commit_round(st, rows)
            st = [(c, r) for c, r in st[:16]] + [st[16]]
            if st[16][1] == 0 and done_in is None:
                done_in = rnd
        assert done_in == expect_rounds


def test_quota_defers_decodes_instead_of_failing():
    """With a quota, decodes beyond budget - quota wait (the first ones in input order run);
    the quota only holds back what the prompts can use."""
    st = [(10, 0)] * 10 + [(0, 40)]
    with pytest.raises(oracle.BudgetError):
        oracle.schedule(st, 8)
    rows, unused = oracle.schedule(st, 8, prefill_quota=2)
    assert sum(1 for i, _, _ in rows if st[i][1] == 0) == 6 and takes(rows, st) == {10: 2}
    assert [r[0] for r in rows[:6]] == list(range(6))  # the first decodes in input order
    st = [(10, 0)] * 10 + [(0, 1)]
    rows, unused = oracle.schedule(st, 8, prefill_quota=4)
    assert sum(1 for i, _, _ in rows if st[i][1] == 0) == 7 and takes(rows, st) == {10: 1} and unused == 0


def test_prefill_first_serves_prompts_before_decodes():
    """[mer]: prefill-first spends the budget on prompt chunks and runs decodes with whatever
    capacity remains."""
    st = [(37, 0), (64, 0), (100, 0), (0, 12)]
    rows, unused = oracle.schedule(st, 8, policy=oracle.PREFILL_FIRST)
    assert takes(rows, st) == {3: 8} and len(rows) == 1 and unused == 0
    st2 = [(37, 0), (64, 0), (100, 0), (0, 5)]
    rows, unused = oracle.schedule(st2, 8, policy=oracle.PREFILL_FIRST)
    assert takes(rows, st2) == {3: 5} and len(rows) == 4 and unused == 0


def test_fair_share_splits_and_gives_unused_share_away():
    """[mer]: fair share allocates the budget between the two classes so both progress; the
    share one class leaves unused goes to the other (reading: a 50 % decode share)."""
    st = [(5 + i, 0) for i in range(6)] + [(0, 12)]
    rows, unused = oracle.schedule(st, 8, policy=oracle.FAIR_SHARE)
    assert sum(1 for i, _, _ in rows if st[i][1] == 0) == 4 and takes(rows, st) == {6: 4}
    st = [(5, 0), (6, 0)] + [(0, 12)]
    rows, unused = oracle.schedule(st, 8, policy=oracle.FAIR_SHARE)
    assert takes(rows, st) == {2: 6} and unused == 0  # unused decode share went to the prompt
    st = [(5 + i, 0) for i in range(6)] + [(0, 1)]
    rows, unused = oracle.schedule(st, 8, policy=oracle.FAIR_SHARE)
    assert sum(1 for i, _, _ in rows if st[i][1] == 0) == 6 and unused == 1  # prompt left 3 over


@pytest.mark.parametrize("policy", [oracle.DECODE_FIRST, oracle.PREFILL_FIRST, oracle.FAIR_SHARE])
def test_policy_invariants_fuzz(policy):
    """[zwj] section 05 invariants for every policy: within budget, positive chunks, each
    prompt's ranges contiguous and non-overlapping, at most one row per request."""
    rng = np.random.default_rng(100 + policy)
    for trial in range(200):
        n_dec = int(rng.integers(0, 14))
        n_pr = int(rng.integers(0, 5))
        budget = int(rng.integers(1, 48))
        cap = int(rng.integers(0, 2)) * int(rng.integers(1, 20))
        floor = int(rng.integers(0, 2)) * int(rng.integers(1, 12))
        quota = int(rng.integers(0, 2)) * int(rng.integers(1, budget + 1))
        share = int(rng.integers(0, 1001))
        st = [(int(rng.integers(0, 300)), 0) for _ in range(n_dec)]
        st += [(int(rng.integers(0, 50)), int(rng.integers(1, 90))) for _ in range(n_pr)]
        order = rng.permutation(len(st))
        cur = [st[k] for k in order]
        start = list(cur)
        ranges = {i: [] for i, s in enumerate(cur) if s[1] > 0}
        for _ in range(40):
            try:
                rows, unused = oracle.schedule(cur, budget, cap, policy, floor, quota, share)
            except oracle.BudgetError:
                assert policy == oracle.DECODE_FIRST and quota == 0
                break
            used = sum(d for _, _, d in rows)
            assert used + unused == budget and all(d > 0 for _, _, d in rows)
            ids = [i for i, _, _ in rows]
            assert len(ids) == len(set(ids))
            for i, c, d in rows:
                assert c == cur[i][0]
                if cur[i][1] == 0:
                    assert d == 1
                else:
                    assert d <= cur[i][1] and (cap == 0 or d <= cap)
                    ranges[i].append((c, c + d))
            if unused > 0:
                # work-conserving: budget is left only when every request got all it may take
                for i, s in enumerate(cur):
                    got = sum(d for j, _, d in rows if j == i)
                    assert got == (1 if s[1] == 0 else (min(s[1], cap) if cap else s[1]))
            cur = oracle.commit_round(cur, rows)
        for i, rs in ranges.items():
            for (a, b), (a2, _) in zip(rs, rs[1:]):
                assert b == a2 and a < b
            if rs:
                assert rs[0][0] == start[i][0] and rs[-1][1] <= start[i][0] + start[i][1]
