"""The SM-split cost model against a sweep of the split on the two large GQA steps.

At the start of a step the attention kernel puts some CTAs on chunk tiles and
the rest on decode items; a CTA whose queue runs dry takes the other one, so
the split moves time but not results.  The prologue picks the split from a cost
model (SM cycles per 128x128 chunk tile, decode bytes per SM cycle, both scaled
by the SM clock the previous call measured, and the HBM rate from the device's
memory clock and bus width).  ms_test_attention_split forces the split: the
test times the step over a sweep of splits and checks that the model's own
choice is within a few percent of the best one, and that a forced split leaves
the output bit for bit unchanged.
"""
import numpy as np
import pytest

import workloads

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

TOL = 0.05  # the model's split may be this much slower than the swept best
REPS = 5


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


def _median_ms(torch, fn, reps=REPS):
    fn()  # warm-up
    ts = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return float(np.median(ts))


@pytest.mark.parametrize("name", ["gqa8b_b8192", "long_bimodal_b4608"])
def test_cost_model_split_is_near_the_swept_best(env, name):
    torch, ms, step = env
    wl = workloads.CONFIGS[name]()
    states = [(r.cached_len, r.remaining) for r in wl.requests]
    tables = [r.block_table for r in wl.requests]
    meta = ms.build_batch_metadata(states, tables, wl.token_budget, wl.max_chunk, ragged=True)
    b = step.to_device(meta, "cuda")
    T = meta["num_tokens"]
    q, _, _ = workloads.step_tensors(wl, T, 5, "cuda")
    kc, vc = workloads.kv_pool(wl, 5, "cuda")
    out = torch.empty_like(q)
    ws = step.workspace_for(b, wl.H_q, wl.H_kv, wl.D, "cuda")
    n_sms = ms.num_sms()
    rated_mhz, hbm_gbs = ms.cost_model_rates()  # the model's fallback clock and its HBM cap
    assert 500 <= rated_mhz <= 5000 and 1000 <= hbm_gbs <= 20000, (rated_mhz, hbm_gbs)

    def model():
        step.attend(q, kc, vc, b, out, ws)

    def forced(n, dst=out):
        ms.test_attention_split(q, kc, vc, b.cu_seqlens_q, b.q_start_pos, b.context_lens, b.block_tables,
                                b.context_total, dst, ws, n, bt_offsets=b.bt_offsets)

    for _ in range(3):  # the first calls measure the SM clock into the workspace header
        model()
    torch.cuda.synchronize()
    hdr = ws[:256].view(torch.int32).cpu().numpy()
    n_model, mhz = int(hdr[9]), int(hdr[10])
    assert 0 <= n_model <= n_sms and 500 <= mhz <= 4000, (n_model, mhz)
    ref = out.clone()
    t_model = _median_ms(torch, model)

    times = {}
    for n in sorted(set(range(0, n_sms + 1, 16)) | {n_sms}):
        times[n] = _median_ms(torch, lambda: forced(n))
    coarse = min(times, key=times.get)
    for n in range(max(0, coarse - 12), min(n_sms, coarse + 12) + 1, 3):
        if n not in times:
            times[n] = _median_ms(torch, lambda: forced(n))
    best = min(times, key=times.get)
    sweep = ", ".join(f"{n}: {times[n]:.3f}" for n in sorted(times))
    assert t_model <= (1 + TOL) * times[best], (
        f"{name}: model split {n_model} at {mhz} MHz takes {t_model:.3f} ms, best swept split {best} "
        f"{times[best]:.3f} ms; sweep (CTAs: ms) {sweep}")
    assert ms.read_status(ws) == 0

    # the split moves time, not results
    for n in (0, n_sms):
        alt = torch.zeros_like(out)
        forced(n, alt)
        torch.cuda.synchronize()
        assert torch.equal(alt.view(torch.int16), ref.view(torch.int16)), n
    print(f"{name}: model {n_model} CTAs at {mhz} MHz {t_model:.3f} ms; best {best} {times[best]:.3f} ms; {sweep}")
