"""Randomized GPU parity: seeded random mixed steps through every entry shape.

Each case draws a layer shape (H_q, H_kv, D with G in {1, 2, 4, 8}), a set of
decodes and prompts with random cached prefixes, a token budget and a chunk
ceiling, then runs one step through the step call (`ms_mixed_step`) or through
the append followed by the attention call, with the block table padded or
ragged.  The row count crosses the one-warp prologue's 32-row limit.  The bar
is the parity tests': metadata, q_rot and both pools bit-exact against the
fp64 oracle, attention within |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|.
"""
import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2
SHAPES = [(4, 2, 64), (8, 8, 64), (8, 1, 64), (16, 2, 64), (8, 2, 128), (8, 8, 128), (32, 8, 128), (8, 1, 128)]


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


@pytest.mark.parametrize("seed", range(48))
def test_random_mixed_step_matches_oracle(env, seed):
    """Seeds 0-23: contexts below 700 keys; seeds 24-47: up to 6000 keys (decodes split into
    several items whose partials merge; chunks over long prefixes, many 128-key tiles)."""
    torch, ms, step = env
    rng = np.random.default_rng(1000 + seed)
    H_q, H_kv, D = SHAPES[seed % len(SHAPES)]
    long_ctx = seed >= 24
    n_dec = int(rng.choice([0, 1, 3, 17, 31, 40]))
    n_prompt = int(rng.integers(0 if n_dec else 1, 4))
    dec_ctx = [int(x) for x in rng.integers(0, 6000 if long_ctx else 700, size=n_dec)]
    prompts = [(int(rng.integers(0, 3000 if long_ctx else 400)), int(rng.integers(1, 600 if long_ctx else 300)))
               for _ in range(n_prompt)]
    budget = n_dec + int(rng.integers(0, 600))
    cap = int(rng.choice([0, 0, 64, 129]))
    wl = workloads.small_mixed(seed=2000 + seed, H_q=H_q, H_kv=H_kv, D=D, dec_ctx=dec_ctx, prompts=prompts,
                               budget=budget, max_chunk=cap)
    states = [(r.cached_len, r.remaining) for r in wl.requests]
    tables = [r.block_table for r in wl.requests]
    ragged = bool(seed & 1)
    fused = bool(seed & 2)
    meta = ms.build_batch_metadata(states, tables, wl.token_budget, wl.max_chunk, ragged=ragged)
    T = meta["num_tokens"]
    if T == 0:
        pytest.skip("nothing scheduled")
    rows, _ = oracle.schedule(states, wl.token_budget, wl.max_chunk)
    ref_meta = oracle.batch_metadata(rows, tables, len(states), num_decodes=meta["num_decodes"])
    for key in ("cu_seqlens_q", "q_start_pos", "context_lens", "positions", "slot_mapping"):
        np.testing.assert_array_equal(meta[key], ref_meta[key], err_msg=key)

    b = step.to_device(meta, "cuda")
    q, k, v = workloads.step_tensors(wl, T, 3000 + seed, "cuda")
    kc, vc = workloads.kv_pool(wl, 3000 + seed, "cuda")
    k_in, v_in = workloads.bf16_bits(kc), workloads.bf16_bits(vc)
    cos, sin = step.rope_tables_device(wl.max_pos + 1, D, "cuda")
    q_rot, out = torch.empty_like(q), torch.zeros_like(q)
    ws = step.workspace_for(b, H_q, H_kv, D, "cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    if fused:
        step.run_step(q, k, v, b, cos, sin, kc, vc, out, ws, q_rot=q_rot, dev_status=status)
    else:
        ms.kv_append_rope(q, k, v, b.positions, b.slot_mapping, cos, sin, kc, vc, q_rot=q_rot, dev_status=status)
        step.attend(q_rot, kc, vc, b, out, ws)
    torch.cuda.synchronize()
    assert ms.read_status(status) == 0 and ms.read_status(ws) == 0

    q_ref, kp, vp = oracle.kv_append(workloads.bf16_bits(q), workloads.bf16_bits(k), workloads.bf16_bits(v),
                                     ref_meta["positions"], ref_meta["slot_mapping"], k_in, v_in)
    np.testing.assert_array_equal(workloads.bf16_bits(q_rot), q_ref)
    np.testing.assert_array_equal(workloads.bf16_bits(kc), kp)
    np.testing.assert_array_equal(workloads.bf16_bits(vc), vp)
    want = oracle.attention_all(q_ref, kp, vp, ref_meta, H_kv)
    got = oracle.bf16_to_f64(workloads.bf16_bits(out))
    err = np.abs(got - want)
    bad = err > ATOL + RTOL * np.abs(want)
    assert not bad.any(), (f"seed {seed} ({H_q}/{H_kv}/{D}, {meta['num_rows']} rows, {T} tokens, ragged {ragged}, "
                           f"fused {fused}): {bad.sum()} elements out of bound, max err {err.max():.3g}")
