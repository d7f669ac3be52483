"""The attention step without a caller workspace (ms_mixed_step_attention_noalloc).

Some callers of this library cannot allocate device memory for a workspace:
a serving process that hands nearly all of the GPU's memory to its KV-cache
pool at start-up has nothing left to give, and host code on the per-step path
should not call cudaMalloc because an allocation can synchronise the device
and stall other streams.  Those callers use this entry point, which runs the
same kernels out of a scratch array the library owns (64 MiB per device).

Checked here through the C ABI: its output matches the workspace entry
point's within the parity tolerance on two calls in a row (the second call
starts from whatever the first left in the shared scratch), the calls leave
free device memory unchanged, and a step too large for the scratch is refused
with MS_ERR_SCRATCH.  This file is collected last so that a failure here does
not hide the results of the other GPU tests.
"""
import numpy as np
import pytest

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


def _prepared_step(env, wl, seed):
    """Metadata, appended caches and q_rot of one step, ready for attention."""
    torch, ms, step = env
    states = [(r.cached_len, r.remaining) for r in wl.requests]
    tables = [r.block_table for r in wl.requests]
    meta = ms.build_batch_metadata(states, tables, wl.token_budget, wl.max_chunk)
    batch = step.to_device(meta, "cuda")
    T = meta["num_tokens"]
    q, k, v = workloads.step_tensors(wl, T, seed, "cuda")
    kc, vc = workloads.kv_pool(wl, seed, "cuda")
    cos, sin = step.rope_tables_device(wl.max_pos + 1, wl.D, "cuda")
    q_rot = torch.empty_like(q)
    ms.kv_append_rope(q, k, v, batch.positions, batch.slot_mapping, cos, sin, kc, vc, q_rot=q_rot)
    return batch, q_rot, kc, vc


@pytest.mark.parametrize("which", ["small_mixed", "mha7b_last_offset"])
def test_noalloc_matches_workspace_entry_point_twice(env, which):
    torch, ms, step = env
    if which == "small_mixed":
        wl = workloads.small_mixed(seed=77, H_q=8, H_kv=2, D=128)
    else:
        wl = workloads.mha7b_steps()[-1]
    batch, q_rot, kc, vc = _prepared_step(env, wl, seed=5)
    args = (q_rot, kc, vc, batch.cu_seqlens_q, batch.q_start_pos, batch.context_lens, batch.block_tables,
            batch.context_total)
    ref = torch.empty_like(q_rot)
    ws = step.workspace_for(batch, wl.H_q, wl.H_kv, wl.D, "cuda")
    ms.mixed_step_attention(*args, ref, ws)
    torch.cuda.synchronize()
    assert ms.read_status(ws) == 0
    ref_f = ref.float().cpu().numpy()
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        out = torch.full_like(q_rot, float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        ms.mixed_step_attention_noalloc(*args, out, dev_status=status)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free_before, f"call {call + 1} changed free device memory"
        assert int(status.item()) == 0, f"call {call + 1} status {int(status.item())}"
        got = out.float().cpu().numpy()
        assert np.all(np.abs(got - ref_f) <= ATOL + RTOL * np.abs(ref_f)), f"call {call + 1} differs"


def test_noalloc_refuses_a_step_larger_than_its_scratch(env):
    torch, ms, step = env
    wl = workloads.small_mixed(seed=78, H_q=8, H_kv=2, D=128)
    batch, q_rot, kc, vc = _prepared_step(env, wl, seed=6)
    out = torch.zeros_like(q_rot)
    with pytest.raises(ms.MixedStepError) as e:
        ms.mixed_step_attention_noalloc(q_rot, kc, vc, batch.cu_seqlens_q, batch.q_start_pos,
                                        batch.context_lens, batch.block_tables, 1 << 40, out)
    assert e.value.code == ms.MS_ERR_SCRATCH
    torch.cuda.synchronize()
    assert float(out.abs().sum()) == 0.0  # nothing was enqueued
