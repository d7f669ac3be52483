"""CUDA-graph replay with padded token buckets against eager launches and the oracle.

Two engines with the same arrivals drive two copies of one page pool: one
launches the step's kernels eagerly, the other replays the captured graph of
the step's token bucket with pad tokens (slot -1) and pad rows (d = 0).  Every
round the outputs of the real tokens are bit-identical, and within
|gpu - oracle| <= 1e-2 + 1e-2 * |oracle| of the fp64 oracle; the pools stay
bit-identical (pad tokens write nothing).
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


@pytest.mark.parametrize("H_q,H_kv,D", [(4, 2, 64), (8, 2, 128)])
def test_graph_replay_matches_eager_and_oracle(env, H_q, H_kv, D):
    torch, ms, step = env
    from chunked_prefill_mixed_decode_gb300.driver import RoundDriver
    num_pages, budget, cap = 48, 40, 24
    buckets = [8, 16, 32, 40]
    shape = types.SimpleNamespace(num_pages=num_pages, H_q=H_q, H_kv=H_kv, page_size=16, D=D)
    ka, va = workloads.kv_pool(shape, 61, "cuda")
    kb, vb = ka.clone(), va.clone()
    kp, vp = workloads.bf16_bits(ka), workloads.bf16_bits(va)
    cos, sin = step.rope_tables_device(num_pages * 16 + 1, D, "cuda")
    ea = ms.Engine(num_pages, budget, max_chunk_per_request=cap)
    eb = ms.Engine(num_pages, budget, max_chunk_per_request=cap)
    eager = RoundDriver(ea, ka, va, cos, sin, H_q, H_kv, D)
    graph = RoundDriver(eb, kb, vb, cos, sin, H_q, H_kv, D, graph_buckets=buckets, max_row_pages=num_pages)
    rng = np.random.default_rng(8)
    used_buckets, pads = set(), 0
    for rnd in range(36):
        for _ in range(int(rng.integers(0, 2))):
            pl, mn = int(rng.integers(1, 40)), int(rng.integers(2, 10))
            try:
                rid = ea.add_request(pl, mn)
            except ms.MixedStepError:
                continue
            assert eb.add_request(pl, mn) == rid
        if ea.stats()["num_live"] == 0:
            continue
        q, k, v = workloads.step_tensors(shape, budget, 700 + rnd, "cuda")
        ra = eager.step(q, k, v)
        rb = graph.step(q, k, v)
        T = ra["meta"]["num_tokens"]
        for key in ("cu_seqlens_q", "positions", "slot_mapping"):
            np.testing.assert_array_equal(ra["meta"][key], rb["meta"][key])
        assert rb["bucket"] == min(b for b in buckets if b >= T) and rb["pad_tokens"] == rb["bucket"] - T
        used_buckets.add(rb["bucket"])
        pads += rb["pad_tokens"]
        np.testing.assert_array_equal(workloads.bf16_bits(eager.out[:T]), workloads.bf16_bits(graph.out[:T]))
        meta = ra["meta"]
        q_rot, kp, vp = oracle.kv_append(workloads.bf16_bits(q[:T]), workloads.bf16_bits(k[:T]),
                                         workloads.bf16_bits(v[:T]), meta["positions"], meta["slot_mapping"], kp, vp)
        want = oracle.attention_all(q_rot, kp, vp, meta, H_kv)
        got = oracle.bf16_to_f64(workloads.bf16_bits(graph.out[:T]))
        assert (np.abs(got - want) <= ATOL + RTOL * np.abs(want)).all(), f"round {rnd}"
        assert ra["finished"] == rb["finished"]
    np.testing.assert_array_equal(workloads.bf16_bits(ka), workloads.bf16_bits(kb))
    np.testing.assert_array_equal(workloads.bf16_bits(va), workloads.bf16_bits(vb))
    np.testing.assert_array_equal(workloads.bf16_bits(kb), kp)
    np.testing.assert_array_equal(workloads.bf16_bits(vb), vp)
    assert len(used_buckets) >= 3 and pads > 0


def test_graph_rejects_oversize_steps(env):
    torch, ms, step = env
    shape = types.SimpleNamespace(num_pages=8, H_q=4, H_kv=2, page_size=16, D=64)
    kc, vc = workloads.kv_pool(shape, 3, "cuda")
    cos, sin = step.rope_tables_device(129, 64, "cuda")
    g = ms.StepGraph(kc, vc, cos, sin, 4, max_rows=4, max_row_pages=8, buckets=[8, 16],
                     stream=torch.cuda.Stream())
    meta = ms.build_batch_metadata([(0, 20)], [np.arange(8, dtype=np.int32)], 20)
    with pytest.raises(ms.MixedStepError) as e:
        g.run(meta)  # 20 tokens > largest bucket
    assert e.value.code == ms.MS_ERR_ARG
    meta = ms.build_batch_metadata([(3, 0)] * 5, [np.arange(8, dtype=np.int32)] * 5, 8)
    with pytest.raises(ms.MixedStepError):
        g.run(meta)  # 5 rows > max_rows
    meta = ms.build_batch_metadata([(3, 0)] * 3, [np.arange(8, dtype=np.int32)] * 3, 8)
    assert g.run(meta) == 8
    torch.cuda.synchronize()
    assert g.read_status() == 0
