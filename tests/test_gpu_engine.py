"""GPU parity of the multi-round driver: engine plan -> append + attention -> commit.

Random arrivals over many rounds on one small page pool, with pages freed and
handed out again: every round's metadata equals the oracle engine's, the K/V
pools stay bit-exact with the oracle's appends, and the attention output is
within |gpu - oracle| <= 1e-2 + 1e-2 * |oracle| of the fp64 oracle.
"""
import types

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from chunked_prefill_mixed_decode_gb300 import build
    build.build()
    import chunked_prefill_mixed_decode_gb300 as ms
    from chunked_prefill_mixed_decode_gb300 import step
    return torch, ms, step


# (policy, H_q, H_kv, D, budget, ceiling, floor, prefill quota, arrival seed)
CASES = [
    (0, 4, 2, 64, 40, 24, 0, 0, 50),
    (1, 8, 8, 128, 40, 24, 0, 0, 51),
    (2, 8, 1, 128, 40, 24, 0, 0, 52),
    # sference.com, "What comes next": a floor per prompt instead of a ceiling -- every waiting prompt
    # gets up to 8 tokens first, the leftover then goes out in arrival order
    (0, 8, 2, 128, 40, 0, 8, 0, 106),
    # zwjcode section 08 and section 16 exercise 3: a prefill quota against starvation -- while prompts
    # wait, decodes leave 10 of the 12 tokens to them and the rest of the decodes wait a round
    (0, 4, 1, 64, 12, 0, 0, 10, 181),
]


@pytest.mark.parametrize("policy,H_q,H_kv,D,budget,cap,floor,quota,seed", CASES)
def test_engine_rounds_match_oracle(env, policy, H_q, H_kv, D, budget, cap, floor, quota, seed):
    torch, ms, step = env
    from chunked_prefill_mixed_decode_gb300.driver import RoundDriver
    num_pages = 48
    shape = types.SimpleNamespace(num_pages=num_pages, H_q=H_q, H_kv=H_kv, page_size=16, D=D)
    k_cache, v_cache = workloads.kv_pool(shape, 31 + policy, "cuda")
    kp, vp = workloads.bf16_bits(k_cache), workloads.bf16_bits(v_cache)
    cos, sin = step.rope_tables_device(num_pages * 16 + 1, D, "cuda")
    eng = ms.Engine(num_pages, budget, max_chunk_per_request=cap, policy=policy, min_chunk_per_request=floor,
                    prefill_quota=quota)
    ref = oracle.Engine(num_pages, budget, max_chunk=cap, policy=policy, min_chunk=floor, prefill_quota=quota)
    drv = RoundDriver(eng, k_cache, v_cache, cos, sin, H_q, H_kv, D)
    rng = np.random.default_rng(seed)
    finished = admitted = 0
    shared_rounds = deferred_rounds = 0  # rounds where the floor split the budget / the quota held decodes back
    for rnd in range(40):
        for _ in range(int(rng.integers(0, 3))):
            pl, mn = int(rng.integers(1, 120)), int(rng.integers(2, 12))
            cached = int(rng.integers(0, pl + 1)) if rng.random() < 0.3 else 0
            try:
                rid = ref.add_request(pl, mn, cached)
            except oracle.AdmissionError:
                with pytest.raises(ms.MixedStepError):
                    eng.add_request(pl, mn, cached)
                continue
            assert eng.add_request(pl, mn, cached) == rid
            admitted += 1
        if not ref.live:
            continue
        rem_before = {r.rid: r.rem for r in ref.live}
        rmeta = ref.plan()
        T = rmeta["num_tokens"]
        q, k, v = workloads.step_tensors(shape, T, 900 + rnd, "cuda")
        rec = drv.step(q, k, v)
        got = rec["meta"]
        for key in ("cu_seqlens_q", "q_start_pos", "context_lens", "positions", "slot_mapping", "row_request_id"):
            np.testing.assert_array_equal(got[key], rmeta[key], err_msg=key)
        q_rot, kp, vp = oracle.kv_append(workloads.bf16_bits(q[:T]), workloads.bf16_bits(k[:T]),
                                         workloads.bf16_bits(v[:T]), rmeta["positions"], rmeta["slot_mapping"],
                                         kp, vp)
        want = oracle.attention_all(q_rot, kp, vp, rmeta, H_kv)
        out = oracle.bf16_to_f64(workloads.bf16_bits(drv.out[:T]))
        err = np.abs(out - want)
        assert (err <= ATOL + RTOL * np.abs(want)).all(), f"round {rnd}: max err {err.max():.3g}"
        np.testing.assert_array_equal(workloads.bf16_bits(drv.q_rot[:T]), q_rot)
        assert rec["finished"] == ref.commit()
        chunks = [(rid, d) for rid, d in zip(rec["row_request_id"].tolist(),
                                             np.diff(rec["cu_seqlens_q"]).tolist()) if rem_before[rid] > 0]
        if len(chunks) >= 2 and chunks[0][1] < rem_before[chunks[0][0]]:
            shared_rounds += 1  # the first prompt still had tokens left, yet a later one got some
        deferred_rounds += rec["deferred_decodes"] > 0
        finished += len(rec["finished"])
    np.testing.assert_array_equal(workloads.bf16_bits(k_cache), kp)
    np.testing.assert_array_equal(workloads.bf16_bits(v_cache), vp)
    assert admitted >= 8 and finished >= 4  # pages were released and handed out again
    if floor:
        assert shared_rounds > 0, "the floor never split the budget between two prompts"
    if quota:
        assert deferred_rounds > 0, "the quota never held a decode back"
