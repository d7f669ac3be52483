"""Pins for the fp64 oracle: values the pages print, closed forms, invariants and
library routines -- never the oracle's own formulas retyped.

Citations name the page and section:
  [zwj]  "Chunked Prefill 的 Token 预算" (zwjcode.cn)
  [sar]  "Chunked Prefill: Ending the Great Stall" (manishklach.github.io)
  [mer]  "Splitting Prefill From Decode Inside a Step" (mercemay.com)
  [sfe]  "Prefill head-of-line blocking" (sference.com)
"""
import math

import numpy as np
import pytest

import oracle
import workloads
from conftest import read_golden


# ----------------------------------------------------------------- helpers

def run_rounds(states, budget, n_rounds, max_chunk=0):
    """Schedule and commit n rounds; returns the per-round rows and unused budgets."""
    hist = []
    for _ in range(n_rounds):
        rows, unused = oracle.schedule(states, budget, max_chunk)
        hist.append((list(states), rows, unused))
        states = oracle.commit_round(states, rows)
    return hist, states


def bits(a):
    return oracle.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))


def rand_bf16(rng, shape):
    return bits(rng.standard_normal(shape).astype(np.float32))


# ----------------------------------------------------------------- scheduler

def test_worked_example_rounds_match_page_table():
    """[zwj] section 03: budget 8, D1-D3 + a 12-token P -> P takes 5, 5, 2, decodes in round 4."""
    golden = read_golden("worked_example_rounds.txt")
    states = [(37, 0), (64, 0), (100, 0), (0, 12)]
    hist, _ = run_rounds(states, 8, len(golden))
    for (st, rows, unused), g in zip(hist, golden):
        rnd, n_dec, p_chunk, p_done, p_len, used, budget = map(int, g)
        dec_rows = [r for r in rows if st[r[0]][1] == 0]
        p_rows = [r for r in rows if r[0] == 3 and st[3][1] > 0]
        assert len(dec_rows) == n_dec, rnd
        assert (p_rows[0][2] if p_rows else 0) == p_chunk, rnd
        assert budget - unused == used, rnd
        got_done = (p_rows[0][1] + p_rows[0][2]) if p_rows else p_len
        assert got_done == p_done, rnd


def test_snippet_takes_five_five_two():
    """[zwj] section 05: the teaching scheduler's comment -- P takes 5, 5, 2 tokens."""
    states = [(37, 0), (64, 0), (100, 0), (0, 12)]
    hist, _ = run_rounds(states, 8, 3)
    assert [r[2] for _, rows, _ in hist for r in rows if r[0] == 3] == [5, 5, 2]


@pytest.mark.parametrize("budget,n_chunks", [(2048, 2), (512, 8)])
def test_4096_prompt_chunk_count(budget, n_chunks):
    """[sar] section 03: a 4,096-token prompt is two chunks at budget 2,048, eight at 512."""
    hist, final = run_rounds([(0, 4096)], budget, n_chunks + 1)
    chunks = [d for _, rows, _ in hist[:n_chunks] for (_, _, d) in rows]
    assert chunks == [budget] * n_chunks
    assert final[0] == (4096 + 1, 0)  # finished, then decoded once


def test_leftover_after_decodes():
    """[sar] section 03: 12 decodes leave 2,036 of 2,048; [zwj] section 01: 64 decodes leave 448 of 512."""
    rows, unused = oracle.schedule([(100, 0)] * 12 + [(0, 10**6)], 2048)
    assert rows[-1][2] == 2036 and unused == 0
    rows, unused = oracle.schedule([(100, 0)] * 64 + [(0, 4096)], 512)
    assert rows[-1][2] == 448 and unused == 0


def test_decode_overflow_is_an_error():
    """[zwj] section 05: more decodes than the budget raises."""
    with pytest.raises(oracle.BudgetError):
        oracle.schedule([(5, 0)] * 9, 8)
    rows, unused = oracle.schedule([(5, 0)] * 8, 8)
    assert len(rows) == 8 and unused == 0


def test_exercise_budget16_fcfs():
    """[zwj] section 16, exercise 1 (answer derived here): budget 16, 6 decodes, prompts of 18 and 5.

    Round 1: P1 takes 10.  Round 2: P1 takes its last 8, P2 takes 2.  Round 3:
    P1 now decodes (7 decodes) and P2 takes its last 3, using 10 of 16.
    """
    states = [(50 + i, 0) for i in range(6)] + [(0, 18), (0, 5)]
    hist, _ = run_rounds(states, 16, 3)
    take = [[(r[0], r[2]) for r in rows if st[r[0]][1] > 0] for st, rows, _ in hist]
    assert take == [[(6, 10)], [(6, 8), (7, 2)], [(7, 3)]]
    assert [16 - u for _, _, u in hist] == [16, 16, 10]
    assert sum(1 for r in hist[2][1] if hist[2][0][r[0]][1] == 0) == 7


def test_per_request_cap():
    """[sfe] "The fix" / [mer] build_batch: a per-request cap splits the budget across prompts.

    8192 // 4096 = two partial prefills at once (the page's Kimi example).
    """
    states = [(0, 100000), (0, 100000), (0, 100000)]
    rows, unused = oracle.schedule(states, 8192, max_chunk=4096)
    assert [(r[0], r[2]) for r in rows] == [(0, 4096), (1, 4096)] and unused == 0
    rows, unused = oracle.schedule([(0, 100000)], 8192, max_chunk=4096)
    assert rows == [(0, 0, 4096)] and unused == 4096  # a lone long prefill is capped anyway


def test_schedule_invariants_fuzz():
    """[zwj] section 05: every round within budget, chunk lengths positive, and each
    prompt's computed ranges contiguous and non-overlapping; [zwj] section 04:
    |D_t| + sum |c| <= B_tok; [sar] section 04: decodes are never displaced."""
    rng = np.random.default_rng(7)
    for trial in range(300):
        n_dec = int(rng.integers(0, 12))
        n_pr = int(rng.integers(0, 5))
        budget = int(rng.integers(max(n_dec, 1), 64))
        cap = int(rng.integers(0, 3)) * int(rng.integers(1, 20))
        states = [(int(rng.integers(0, 300)), 0) for _ in range(n_dec)]
        prompts = [(int(rng.integers(0, 50)), int(rng.integers(1, 120))) for _ in range(n_pr)]
        order = rng.permutation(len(states) + len(prompts))
        allst = states + prompts
        allst = [allst[k] for k in order]
        start = {i: s for i, s in enumerate(allst)}
        computed = {i: [] for i, s in enumerate(allst) if s[1] > 0}
        cur = allst
        for _ in range(60):
            n_d = sum(1 for s in cur if s[1] == 0)
            if n_d > budget:
                with pytest.raises(oracle.BudgetError):
                    oracle.schedule(cur, budget, cap)
                break
            rows, unused = oracle.schedule(cur, budget, cap)
            used = sum(r[2] for r in rows)
            assert used + unused == budget and used <= budget
            assert all(r[2] > 0 for r in rows)
            dec_req = [i for i, s in enumerate(cur) if s[1] == 0]
            assert [r[0] for r in rows[:len(dec_req)]] == dec_req          # decodes first, all of them
            assert all(r[2] == 1 for r in rows[:len(dec_req)])
            for i, c, d in rows[len(dec_req):]:
                assert cur[i][1] > 0 and c == cur[i][0] and d <= cur[i][1]
                if cap:
                    assert d <= cap
                computed[i].append((c, c + d))
            if unused > 0:  # leftover remains only when no prompt could take more
                for i, s in enumerate(cur):
                    if s[1] > 0:
                        took = sum(r[2] for r in rows if r[0] == i)
                        assert took == s[1] or (cap and took == cap)
            cur = oracle.commit_round(cur, rows)
        for i, ranges in computed.items():
            c0, rem0 = start[i]
            for (a, b), (a2, b2) in zip(ranges, ranges[1:]):
                assert b == a2 and a < b           # contiguous, non-overlapping
            if ranges:
                assert ranges[0][0] == c0 and ranges[-1][1] <= c0 + rem0


# ----------------------------------------------------------------- metadata

def test_chunk_5_10_metadata_matches_page():
    """[zwj] section 06: chunk [5, 10) of a 12-token prompt."""
    g = {r[0]: r[1:] for r in read_golden("chunk_metadata_5_10.txt")}
    plen, c, d = int(g["prompt_len"][0]), int(g["chunk_start"][0]), int(g["chunk_len"][0])
    table = np.array([9], dtype=np.int32)
    rows, _ = oracle.schedule([(c, plen - c)], d)
    meta = oracle.batch_metadata(rows, [table], 1)
    assert meta["positions"].tolist() == [int(x) for x in g["positions"]]
    assert meta["context_lens"].tolist() == [int(g["context_len"][0])]
    assert meta["bt_stride"] == int(g["block_table_entries_page16"][0])
    assert meta["slot_mapping"].tolist() == [9 * 16 + p for p in range(5, 10)]


def test_diagram_chunks_0_4_8_10():
    """[zwj] section 02 diagram: a 10-token prompt as chunks 0:4, 4:8, 8:10 (budget 4)."""
    hist, _ = run_rounds([(0, 10)], 4, 3)
    assert [(r[1], r[1] + r[2]) for _, rows, _ in hist for r in rows] == [(0, 4), (4, 8), (8, 10)]


def test_exercise_4_3_3_positions_and_visibility():
    """[zwj] section 16, exercise 2 with the section 07 rule: chunks [4, 3, 3] of a 10-token
    prompt have positions 0..3 | 4..6 | 7..9, context lengths 4, 7, 10, and the last
    chunk's query i sees exactly keys 0..7+i.  Visibility is read off the attention:
    with q = 0 every visible key weighs the same, and V[j] = e_j makes the output
    the indicator of the visible set divided by its size."""
    D, page = 16, 16
    table = np.array([3], dtype=np.int32)
    kp = np.zeros((4, 1, page, D), dtype=np.uint16)
    vp = np.zeros((4, 1, page, D), dtype=np.uint16)
    states = [(0, 10)]
    expect_pos = [[0, 1, 2, 3], [4, 5, 6], [7, 8, 9]]
    for k, d in enumerate([4, 3, 3]):
        rows, _ = oracle.schedule(states, d)
        meta = oracle.batch_metadata(rows, [table], 1)
        assert meta["positions"].tolist() == expect_pos[k]
        assert meta["context_lens"].tolist() == [[4, 7, 10][k]]
        T = len(meta["positions"])
        q = np.zeros((T, 1, D), dtype=np.uint16)
        kk = np.zeros((T, 1, D), dtype=np.uint16)
        vv = np.zeros((T, 1, D), dtype=np.float32)
        for t, p in enumerate(meta["positions"]):
            vv[t, 0, p] = 1.0
        _, kp, vp = oracle.kv_append(q, kk, bits(vv), meta["positions"], meta["slot_mapping"], kp, vp)
        out = oracle.attention_all(q, kp, vp, meta, H_kv=1)
        if k == 2:
            for i in range(3):
                vis = np.zeros(D)
                vis[: 7 + i + 1] = 1.0 / (7 + i + 1)
                np.testing.assert_array_equal(out[i, 0], vis)
        states = oracle.commit_round(states, rows)


def test_identity_allocation_round1_and_round4_metadata():
    """The walk-through with pages allocated in order (D1 0-2, D2 3-7, D3 8-14, P 15):
    slot = page * 16 + pos % 16 by the [zwj] section 06 definitions (values derived here)."""
    wl = workloads.identity_worked_example()
    states = [(r.cached_len, r.remaining) for r in wl.requests]
    tables = [r.block_table for r in wl.requests]
    rows, _ = oracle.schedule(states, 8)
    m = oracle.batch_metadata(rows, tables, 4, num_decodes=3)
    assert m["cu_seqlens_q"].tolist() == [0, 1, 2, 3, 8]
    assert m["positions"].tolist() == [37, 64, 100, 0, 1, 2, 3, 4]
    assert m["slot_mapping"].tolist() == [37, 112, 228, 240, 241, 242, 243, 244]
    assert m["context_lens"].tolist() == [38, 65, 101, 5]
    assert m["q_start_pos"].tolist() == [37, 64, 100, 0]
    assert m["bt_stride"] == 7
    assert m["block_tables"][3].tolist() == [15, -1, -1, -1, -1, -1, -1]
    for _ in range(3):
        states = oracle.commit_round(states, rows)
        rows, unused = oracle.schedule(states, 8)
    m = oracle.batch_metadata(rows, tables, 4, num_decodes=4)
    assert m["positions"].tolist() == [40, 67, 103, 12]
    assert m["slot_mapping"].tolist() == [40, 115, 231, 252]
    assert unused == 4


def test_missing_pages_is_an_error():
    """[mer] "The arithmetic of chunk boundaries": pages must be reserved before the chunk runs."""
    rows, _ = oracle.schedule([(30, 5)], 8)
    with pytest.raises(oracle.NoPagesError):
        oracle.batch_metadata(rows, [np.array([1, 2], dtype=np.int32)], 1)  # needs ceil(35/16) = 3


# ----------------------------------------------------------------- rotary embedding

def test_rope_table_against_library_cos_sin():
    """The fp32 table agrees with numpy's own cos/sin to within one fp32 ulp; position 0 is exact."""
    pos = np.array([0, 1, 2, 17, 4095, 28672, 131071])
    for D in (64, 128):
        cos, sin = oracle.rope_tables(pos, D)
        ang = pos[:, None].astype(np.float64) * (10000.0 ** (-np.arange(0, D, 2) / D))[None, :]
        for got, ref in ((cos, np.cos(ang)), (sin, np.sin(ang))):
            ulp = np.spacing(np.abs(ref).astype(np.float32))
            assert np.all(np.abs(got.astype(np.float64) - ref) <= ulp)
        assert np.all(cos[0] == 1.0) and np.all(sin[0] == 0.0)
        # the first pair rotates by exactly p radians (theta_0 = 1)
        assert cos[3, 0] == np.float32(math.cos(17.0))


def test_rope_matches_complex_rotation():
    """Rotate-half RoPE equals multiplying z_i = x_i + j*x_{i+D/2} by exp(j*p*theta_i)
    (a different algebra, fp64) to within one bf16 rounding."""
    rng = np.random.default_rng(3)
    for D in (64, 128):
        T, H = 40, 3
        pos = rng.integers(0, 200000, size=T)
        x = rand_bf16(rng, (T, H, D))
        cos, sin = oracle.rope_tables(pos, D)
        y = oracle.bf16_to_f64(oracle.rope_rotate(x, cos, sin))
        xf = oracle.bf16_to_f64(x)
        z = xf[..., : D // 2] + 1j * xf[..., D // 2:]
        theta = 10000.0 ** (-np.arange(0, D, 2) / D)
        rot = np.exp(1j * pos[:, None, None] * theta[None, None, :])
        ref = z * rot
        ref = np.concatenate([ref.real, ref.imag], axis=-1)
        mag = np.abs(xf[..., : D // 2]) + np.abs(xf[..., D // 2:])
        mag = np.concatenate([mag, mag], axis=-1)
        # bf16 half-ulp of the result, fp32 product rounding, and the fp32 table's
        # phase error, which grows with the angle p * theta (|p| up to 2e5 here)
        tol = 2.0 ** -8 * np.abs(ref) + 2.0 ** -20 * mag * (1 + pos[:, None, None] / 64.0)
        assert np.all(np.abs(y - ref) <= tol)


def test_rope_position_zero_is_identity_and_norm_preserved():
    rng = np.random.default_rng(4)
    x = rand_bf16(rng, (5, 2, 64))
    cos, sin = oracle.rope_tables([0] * 5, 64)
    np.testing.assert_array_equal(oracle.rope_rotate(x, cos, sin), x)
    cos, sin = oracle.rope_tables([7, 100, 1000, 5000, 9], 64)
    y = oracle.bf16_to_f64(oracle.rope_rotate(x, cos, sin))
    xf = oracle.bf16_to_f64(x)
    pair_in = xf[..., :32] ** 2 + xf[..., 32:] ** 2
    pair_out = y[..., :32] ** 2 + y[..., 32:] ** 2
    assert np.all(np.abs(np.sqrt(pair_out) - np.sqrt(pair_in)) <= 2.0 ** -7 * np.sqrt(pair_in) + 1e-30)


def test_rope_relative_position_property():
    """[zwj] section 07: attention scores depend on relative position only, so shifting
    every position by the same amount keeps q.k (to bf16 rounding) -- and resetting a
    chunk's positions to 0 (the bug the page warns about) does not."""
    rng = np.random.default_rng(5)
    D = 128
    q = rand_bf16(rng, (1, 1, D))
    k = rand_bf16(rng, (1, 1, D))

    def score(pq, pk):
        cq, sq = oracle.rope_tables([pq], D)
        ck, sk = oracle.rope_tables([pk], D)
        a = oracle.bf16_to_f64(oracle.rope_rotate(q, cq, sq))[0, 0]
        b = oracle.bf16_to_f64(oracle.rope_rotate(k, ck, sk))[0, 0]
        return float(a @ b)

    base = score(517, 500)
    assert abs(score(1517, 1500) - base) < 0.15
    assert abs(score(17, 0) - base) < 0.15
    assert abs(score(17, 500) - base) > 0.15  # query position reset to 0-based


def test_kv_append_writes_slots_only():
    rng = np.random.default_rng(6)
    D, H_kv, P = 64, 2, 6
    kp = rand_bf16(rng, (P, H_kv, 16, D))
    vp = rand_bf16(rng, (P, H_kv, 16, D))
    T = 4
    q = rand_bf16(rng, (T, 4, D))
    k = rand_bf16(rng, (T, H_kv, D))
    v = rand_bf16(rng, (T, H_kv, D))
    pos = np.array([0, 33, 34, 90])
    slots = np.array([5 * 16 + 0, 2 * 16 + 1, -1, 0 * 16 + 10])
    q_rot, kp2, vp2 = oracle.kv_append(q, k, v, pos, slots, kp, vp)
    np.testing.assert_array_equal(kp2[5, :, 0], k[0])          # position 0: unrotated
    np.testing.assert_array_equal(vp2[5, :, 0], v[0])
    np.testing.assert_array_equal(vp2[2, :, 1], v[1])          # V is a plain copy
    np.testing.assert_array_equal(vp2[0, :, 10], v[3])
    np.testing.assert_array_equal(q_rot[0], q[0])
    touched = np.zeros((P, 16), bool)
    touched[5, 0] = touched[2, 1] = touched[0, 10] = True
    tr = (0, 2, 1, 3)  # [page, slot, head, d]
    np.testing.assert_array_equal(kp2.transpose(tr)[~touched], kp.transpose(tr)[~touched])
    np.testing.assert_array_equal(vp2.transpose(tr)[~touched], vp.transpose(tr)[~touched])


# ----------------------------------------------------------------- attention

def _one_step(wl, states, rng, scale=None, kp=None, vp=None):
    tables = [r.block_table for r in wl.requests]
    rows, _ = oracle.schedule(states, wl.token_budget, wl.max_chunk)
    meta = oracle.batch_metadata(rows, tables, len(states))
    T = meta["num_tokens"]
    q = rand_bf16(rng, (T, wl.H_q, wl.D))
    k = rand_bf16(rng, (T, wl.H_kv, wl.D))
    v = rand_bf16(rng, (T, wl.H_kv, wl.D))
    q_rot, kp, vp = oracle.kv_append(q, k, v, meta["positions"], meta["slot_mapping"], kp, vp)
    out = oracle.attention_all(q_rot, kp, vp, meta, wl.H_kv, scale)
    return rows, meta, q_rot, kp, vp, out


def test_decode_with_one_key_returns_its_value():
    """A decode at c = 0 sees one key: the output is that key's V exactly."""
    rng = np.random.default_rng(8)
    wl = workloads.small_mixed(dec_ctx=(0,), prompts=(), H_q=4, H_kv=2, D=64)
    kp = rand_bf16(rng, (wl.num_pages, 2, 16, 64))
    vp = rand_bf16(rng, (wl.num_pages, 2, 16, 64))
    rows, meta, q_rot, kp, vp, out = _one_step(wl, [(0, 0)], rng, kp=kp, vp=vp)
    page = wl.requests[0].block_table[0]
    for h in range(4):
        np.testing.assert_array_equal(out[0, h], oracle.bf16_to_f64(vp[page, h // 2, 0]))


def test_zero_query_and_equal_keys_give_mean_of_visible_values():
    rng = np.random.default_rng(9)
    D, H = 64, 2
    table = np.array([4, 1, 7], dtype=np.int32)
    kp = rand_bf16(rng, (8, H, 16, D))
    vp = rand_bf16(rng, (8, H, 16, D))
    rows, _ = oracle.schedule([(20, 0)], 4)
    meta = oracle.batch_metadata(rows, [table], 1)
    vis = np.array([oracle.bf16_to_f64(vp[table[j // 16], :, j % 16]) for j in range(21)])
    q = np.zeros((1, H, D), dtype=np.uint16)
    out = oracle.attention_all(q, kp, vp, meta, H)
    np.testing.assert_allclose(out[0], vis.mean(axis=0), rtol=0, atol=1e-15)
    kp_eq = np.broadcast_to(kp[4, :, 3][None, :, None, :], kp.shape).copy()
    q = rand_bf16(rng, (1, H, D))
    out = oracle.attention_all(q, kp_eq, vp, meta, H)
    np.testing.assert_allclose(out[0], vis.mean(axis=0), rtol=0, atol=1e-15)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(10)
    D = 64
    table = np.array([2, 0], dtype=np.int32)
    kp = bits(rng.standard_normal((3, 1, 16, D)).astype(np.float32) * 0.01)
    vp = rand_bf16(rng, (3, 1, 16, D))
    q = bits(np.full((1, 1, D), 4.0, np.float32))
    kp[0, 0, 5] = bits(np.full(D, 4.0, np.float32))  # logical key 21
    rows, _ = oracle.schedule([(25, 0)], 1)
    meta = oracle.batch_metadata(rows, [table], 1)
    out = oracle.attention_all(q, kp, vp, meta, 1)
    np.testing.assert_allclose(out[0, 0], oracle.bf16_to_f64(vp[0, 0, 5]), atol=1e-12)


def test_gqa_equals_mha_with_replicated_kv_heads():
    rng = np.random.default_rng(12)
    D, Hq, Hkv, G = 64, 8, 2, 4
    table = np.array([3, 0, 5, 1], dtype=np.int32)
    kp = rand_bf16(rng, (6, Hkv, 16, D))
    vp = rand_bf16(rng, (6, Hkv, 16, D))
    rows, _ = oracle.schedule([(10, 0), (0, 50)], 60)
    meta = oracle.batch_metadata(rows, [table, table], 2)
    q = rand_bf16(rng, (meta["num_tokens"], Hq, D))
    gqa = oracle.attention_all(q, kp, vp, meta, Hkv)
    mha = oracle.attention_all(q, np.repeat(kp, G, axis=1), np.repeat(vp, G, axis=1), meta, Hq)
    np.testing.assert_array_equal(gqa, mha)


def _prompt_in_chunks(chunks, H_q=4, H_kv=2, D=64, seed=13, perm=None):
    """Prefill one prompt in the given chunks; returns its output rows [L, H_q, D] and state."""
    rng = np.random.default_rng(seed)
    L = sum(chunks)
    n_pages = -(-L // 16)
    table = np.arange(n_pages, dtype=np.int32) if perm is None else np.asarray(perm, np.int32)
    q_all = rand_bf16(rng, (L, H_q, D))
    k_all = rand_bf16(rng, (L, H_kv, D))
    v_all = rand_bf16(rng, (L, H_kv, D))
    kp = np.zeros((max(table) + 1, H_kv, 16, D), np.uint16)
    vp = np.zeros_like(kp)
    states = [(0, L)]
    outs = []
    for d in chunks:
        rows, _ = oracle.schedule(states, d)
        meta = oracle.batch_metadata(rows, [table], 1)
        p = meta["positions"]
        q_rot, kp, vp = oracle.kv_append(q_all[p], k_all[p], v_all[p], p, meta["slot_mapping"], kp, vp)
        outs.append(oracle.attention_all(q_rot, kp, vp, meta, H_kv))
        states = oracle.commit_round(states, rows)
    return np.concatenate(outs), (q_all, k_all, v_all)


@pytest.mark.parametrize("chunks", [[2, 3, 1], [4, 3, 3], [5, 5, 2], [16, 1, 17, 30]])
def test_chunked_prefill_equals_full_prefill(chunks):
    """[zwj] sections 02 and 07: chunked prefill with absolute positions equals full
    prefill; the page's debug case is chunks [2, 3, 1] of a 6-token prompt.  In fp64
    through the paged cache the match is exact."""
    L = sum(chunks)
    chunked, _ = _prompt_in_chunks(chunks)
    full, _ = _prompt_in_chunks([L])
    np.testing.assert_array_equal(chunked, full)


def test_page_permutation_invariance():
    out_a, _ = _prompt_in_chunks([20, 30, 14])
    out_b, _ = _prompt_in_chunks([20, 30, 14], perm=[3, 0, 2, 1])
    np.testing.assert_array_equal(out_a, out_b)


def test_against_torch_sdpa_causal_fp64():
    """A library routine on plain contiguous tensors: torch's scaled_dot_product_attention
    (is_causal, fp64) on the rotated prompt equals the oracle's paged chunked output."""
    torch = pytest.importorskip("torch")
    chunks = [7, 9, 16, 1, 11]
    H_q, H_kv, D = 4, 2, 64
    out, (q_all, k_all, v_all) = _prompt_in_chunks(chunks, H_q, H_kv, D, perm=[2, 0, 3, 1])
    L = sum(chunks)
    pos = np.arange(L)
    cos, sin = oracle.rope_tables(pos, D)
    q = torch.from_numpy(oracle.bf16_to_f64(oracle.rope_rotate(q_all, cos, sin)))
    k = torch.from_numpy(oracle.bf16_to_f64(oracle.rope_rotate(k_all, cos, sin)))
    v = torch.from_numpy(oracle.bf16_to_f64(v_all))
    G = H_q // H_kv
    qh = q.permute(1, 0, 2)
    kh = k.permute(1, 0, 2).repeat_interleave(G, dim=0)
    vh = v.permute(1, 0, 2).repeat_interleave(G, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, is_causal=True)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-13)


def test_mixed_batch_rows_are_independent():
    """A decode's output does not depend on what else shares the step."""
    rng = np.random.default_rng(14)
    wl = workloads.small_mixed(H_q=4, H_kv=2, D=64, dec_ctx=(40, 70), prompts=((0, 30),))
    kp = rand_bf16(rng, (wl.num_pages, 2, 16, 64))
    vp = rand_bf16(rng, (wl.num_pages, 2, 16, 64))
    tables = [r.block_table for r in wl.requests]
    states = [(r.cached_len, r.remaining) for r in wl.requests]
    rows, _ = oracle.schedule(states, wl.token_budget)
    meta = oracle.batch_metadata(rows, tables, 3)
    q = rand_bf16(rng, (meta["num_tokens"], 4, 64))
    full = oracle.attention_all(q, kp, vp, meta, 2)
    alone_rows, _ = oracle.schedule(states[:1], 1)
    alone = oracle.attention_all(q[:1], kp, vp, oracle.batch_metadata(alone_rows, tables[:1], 1), 2)
    np.testing.assert_array_equal(full[0], alone[0])
