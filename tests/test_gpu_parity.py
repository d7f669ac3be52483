"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Bar: metadata, K/V pool and q_rot bit-exact; attention output within
|gpu - oracle| <= 1e-2 + 1e-2 * |oracle| elementwise (bf16 in, fp32 accumulate,
bf16 out); the GPU's chunked prefill matches its own full prefill within the
same bound.
"""
import time

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


def _states(wl):
    return [(r.cached_len, r.remaining) for r in wl.requests]


def _tables(wl):
    return [r.block_table for r in wl.requests]


class Case:
    """One step of a workload on the GPU and its oracle inputs."""

    def __init__(self, env, wl, states, seed, pool=None, dev="cuda", host_pool=True):
        torch, ms, step = env
        self.wl, self.states = wl, states
        self.meta = ms.build_batch_metadata(states, _tables(wl), wl.token_budget, wl.max_chunk)
        self.batch = step.to_device(self.meta, dev)
        T = self.meta["num_tokens"]
        self.q, self.k, self.v = workloads.step_tensors(wl, max(T, 1), seed, dev)
        if pool is None:
            pool = workloads.kv_pool(wl, seed, dev)
        self.k_cache, self.v_cache = pool
        if host_pool:  # host copies before the step
            self.k_in = workloads.bf16_bits(self.k_cache)
            self.v_in = workloads.bf16_bits(self.v_cache)
        # positions of later rounds stay within the pages each request reserved
        max_pos = max([wl.max_pos + 1] + [16 * len(r.block_table) for r in wl.requests])
        self.cos, self.sin = step.rope_tables_device(max_pos, wl.D, dev)
        self.out = torch.zeros_like(self.q)
        self.q_rot = torch.empty_like(self.q)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = step.workspace_for(self.batch, wl.H_q, wl.H_kv, wl.D, dev)

    def run(self, env):
        torch, ms, step = env
        step.run_step(self.q, self.k, self.v, self.batch, self.cos, self.sin, self.k_cache, self.v_cache, self.out,
                      self.ws, q_rot=self.q_rot, dev_status=self.status)
        torch.cuda.synchronize()
        assert ms.read_status(self.status) == 0
        assert ms.read_status(self.ws) == 0
        return self

    def oracle_append(self):
        T = self.meta["num_tokens"]
        ref_meta = oracle.batch_metadata(*oracle.schedule(self.states, self.wl.token_budget, self.wl.max_chunk)[:1],
                                         _tables(self.wl), len(self.states),
                                         num_decodes=sum(1 for s in self.states if s[1] == 0))
        for key in ("cu_seqlens_q", "positions", "slot_mapping", "context_lens", "q_start_pos"):
            np.testing.assert_array_equal(self.meta[key], ref_meta[key])
        q = workloads.bf16_bits(self.q[:T])
        k = workloads.bf16_bits(self.k[:T])
        v = workloads.bf16_bits(self.v[:T])
        return ref_meta, oracle.kv_append(q, k, v, ref_meta["positions"], ref_meta["slot_mapping"], self.k_in,
                                          self.v_in)


def _check_attention(got_bits, ref, what=""):
    got = oracle.bf16_to_f64(got_bits)
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements out of bound, max err {err.max():.3g}"
    return err.max()


def _full_parity(env, wl, states, seed):
    case = Case(env, wl, states, seed).run(env)
    T = case.meta["num_tokens"]
    ref_meta, (q_rot, kp, vp) = case.oracle_append()
    np.testing.assert_array_equal(workloads.bf16_bits(case.q_rot[:T]), q_rot)
    np.testing.assert_array_equal(workloads.bf16_bits(case.k_cache), kp)
    np.testing.assert_array_equal(workloads.bf16_bits(case.v_cache), vp)
    ref = oracle.attention_all(q_rot, kp, vp, ref_meta, wl.H_kv)
    got = workloads.bf16_bits(case.out[:T])
    n_dec = case.meta["num_decodes"]
    if n_dec:
        _check_attention(got[:n_dec], ref[:n_dec], f"{wl.name} decode rows")
    if T > n_dec:
        _check_attention(got[n_dec:], ref[n_dec:], f"{wl.name} chunk rows")
    return case


def test_worked_example_four_rounds(env):
    """The 8-token-budget walk-through (3 decodes + 12-token prompt), stepped four rounds on one pool."""
    wl = workloads.worked_example()
    states = _states(wl)
    torch = env[0]
    pool = workloads.kv_pool(wl, 1, "cuda")
    for rnd in range(4):
        case = Case(env, wl, states, 100 + rnd, pool=pool).run(env)
        T = case.meta["num_tokens"]
        ref_meta, (q_rot, kp, vp) = case.oracle_append()
        np.testing.assert_array_equal(workloads.bf16_bits(case.k_cache), kp)
        np.testing.assert_array_equal(workloads.bf16_bits(case.v_cache), vp)
        ref = oracle.attention_all(q_rot, kp, vp, ref_meta, wl.H_kv)
        _check_attention(workloads.bf16_bits(case.out[:T]), ref, f"round {rnd + 1}")
        rows, _ = oracle.schedule(states, wl.token_budget)
        states = oracle.commit_round(states, rows)
    assert states[3] == (13, 0)


@pytest.mark.parametrize("H_q,H_kv,D", [(8, 2, 128), (8, 8, 64), (4, 4, 128), (16, 2, 128), (8, 2, 64),
                                        (4, 1, 64), (8, 4, 128), (16, 2, 64)])
def test_small_mixed_all_rows(env, H_q, H_kv, D):
    """Decodes at c = 0, page boundaries and beyond a tile; chunks of 130 (several tiles), 200 at offset 300
    and a 5-token tail at offset 16."""
    wl = workloads.small_mixed(seed=H_q * 100 + H_kv * 10 + D, H_q=H_q, H_kv=H_kv, D=D)
    _full_parity(env, wl, _states(wl), seed=7)


@pytest.mark.parametrize("H_q,H_kv,D", [(4, 4, 128), (8, 2, 128), (8, 8, 64)])
def test_odd_query_tile_counts(env, H_q, H_kv, D):
    """Chunks whose 128-row query tiles come in odd numbers, so that the last work item holds a
    single tile (G = 1: 300 tokens = 3 tiles; G = 4: 70 tokens = 3 tiles, 390 = 13), next to
    decodes."""
    wl = workloads.small_mixed(seed=50 + H_q + D, H_q=H_q, H_kv=H_kv, D=D, dec_ctx=(3, 129, 640),
                               prompts=((0, 300), (50, 70), (1000, 390)))
    _full_parity(env, wl, _states(wl), seed=9)


def test_decode_only_and_chunk_only(env):
    wl = workloads.small_mixed(seed=31, H_q=8, H_kv=2, D=128, dec_ctx=(5, 64, 255, 256, 257, 1000, 2049),
                               prompts=())
    _full_parity(env, wl, _states(wl), seed=8)
    wl = workloads.small_mixed(seed=32, H_q=8, H_kv=2, D=128, dec_ctx=(), prompts=((0, 2), (700, 129), (5, 64)))
    _full_parity(env, wl, _states(wl), seed=9)


@pytest.mark.parametrize("n_dec", [3000, 8191])
def test_many_rows(env, n_dec):
    """Steps past the prologue's sort limit (2048 rows per list are ordered longest-first; more
    keep input order) up to the 8192-row maximum: decodes with short contexts and one chunk."""
    rng = np.random.default_rng(n_dec)
    ctx = tuple(int(c) for c in rng.integers(0, 80, size=n_dec))
    wl = workloads.small_mixed(seed=60, H_q=4, H_kv=2, D=64, dec_ctx=ctx, prompts=((40, 37),))
    _full_parity(env, wl, _states(wl), seed=10)


@pytest.mark.parametrize("n_dec", [30, 31, 32, 33])
def test_prologue_row_count_edges(env, n_dec):
    """Up to 32 rows the prologue is one warp (a row per lane); from 33 rows a block of warps.
    n_dec decodes plus one chunk straddle that edge."""
    rng = np.random.default_rng(70 + n_dec)
    ctx = tuple(int(c) for c in rng.integers(0, 700, size=n_dec))
    wl = workloads.small_mixed(seed=70 + n_dec, H_q=8, H_kv=2, D=128, dec_ctx=ctx, prompts=((40, 37),))
    _full_parity(env, wl, _states(wl), seed=11)


@pytest.mark.parametrize("n_dec,ragged", [(3, False), (3, True), (60, False), (60, True), (1100, True)])
def test_step_call_equals_separate_calls(env, n_dec, ragged):
    """ms_mixed_step against ms_kv_append_rope followed by the attention call, same inputs: q_rot, both
    pools and the output bit-identical, and the output within tolerance of the oracle.  Up to 32 rows the
    prologue inside the append's launch is one warp, up to 1024 rows a block of warps; past 1024 rows the
    step call launches the three kernels of the separate calls."""
    torch, ms, step = env
    rng = np.random.default_rng(90 + n_dec)
    ctx = tuple(int(c) for c in rng.integers(0, 300, size=n_dec))
    wl = workloads.small_mixed(seed=90 + n_dec, H_q=8, H_kv=2, D=64, dec_ctx=ctx, prompts=((40, 37), (0, 130)))
    states = _states(wl)
    meta = ms.build_batch_metadata(states, _tables(wl), wl.token_budget, wl.max_chunk, ragged=ragged)
    b = step.to_device(meta, "cuda")
    T = meta["num_tokens"]
    q, k, v = workloads.step_tensors(wl, T, 7, "cuda")
    cos, sin = step.rope_tables_device(wl.max_pos + 1, wl.D, "cuda")
    runs = []
    for fused in (False, True):
        kc, vc = workloads.kv_pool(wl, 7, "cuda")
        q_rot, out = torch.empty_like(q), torch.zeros_like(q)
        ws = step.workspace_for(b, wl.H_q, wl.H_kv, wl.D, "cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        if fused:
            step.run_step(q, k, v, b, cos, sin, kc, vc, out, ws, q_rot=q_rot, dev_status=status)
        else:
            ms.kv_append_rope(q, k, v, b.positions, b.slot_mapping, cos, sin, kc, vc, q_rot=q_rot,
                              dev_status=status)
            step.attend(q_rot, kc, vc, b, out, ws)
        torch.cuda.synchronize()
        assert ms.read_status(status) == 0 and ms.read_status(ws) == 0
        runs.append([workloads.bf16_bits(t) for t in (q_rot, kc, vc, out)])
    for name, sep, fus in zip(("q_rot", "k_cache", "v_cache", "out"), *runs):
        np.testing.assert_array_equal(fus, sep, err_msg=name)
    pmeta = ms.build_batch_metadata(states, _tables(wl), wl.token_budget, wl.max_chunk)
    k_in, v_in = (workloads.bf16_bits(t) for t in workloads.kv_pool(wl, 7, "cuda"))
    q_ref, kp, vp = oracle.kv_append(workloads.bf16_bits(q), workloads.bf16_bits(k), workloads.bf16_bits(v),
                                     pmeta["positions"], pmeta["slot_mapping"], k_in, v_in)
    np.testing.assert_array_equal(runs[1][0], q_ref)
    _check_attention(runs[1][3], oracle.attention_all(q_ref, kp, vp, pmeta, wl.H_kv), "step call")


def test_more_rows_than_a_step_holds_is_refused(env):
    """8193 rows: the call returns MS_ERR_ARG before any launch."""
    torch, ms, step = env
    S = 8193
    meta = {"cu_seqlens_q": np.arange(S + 1, dtype=np.int32), "q_start_pos": np.zeros(S, np.int32),
            "context_lens": np.ones(S, np.int32), "positions": np.zeros(S, np.int32),
            "slot_mapping": np.arange(S, dtype=np.int32), "block_tables": np.zeros((S, 1), np.int32),
            "num_rows": S, "num_tokens": S, "num_decodes": S, "bt_stride": 1}
    b = step.to_device(meta, "cuda")
    q = torch.zeros((S, 4, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((S, 2, 16, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(ms.MixedStepError) as e:
        ms.mixed_step_attention(q, kc, kc, b.cu_seqlens_q, b.q_start_pos, b.context_lens, b.block_tables, S,
                                torch.empty_like(q), ws)
    assert e.value.code == ms.MS_ERR_ARG


def test_more_tokens_than_a_step_holds_is_refused(env):
    """2^21 + 1 tokens in one chunk row: the call returns MS_ERR_ARG before any launch."""
    torch, ms, step = env
    T = (1 << 21) + 1
    meta = {"cu_seqlens_q": np.array([0, T], np.int32), "q_start_pos": np.zeros(1, np.int32),
            "context_lens": np.array([T], np.int32), "positions": np.zeros(1, np.int32),
            "slot_mapping": np.zeros(1, np.int32), "block_tables": np.zeros((1, 1), np.int32),
            "num_rows": 1, "num_tokens": T, "num_decodes": 0, "bt_stride": 1}
    b = step.to_device(meta, "cuda")
    q = torch.zeros((T, 1, 64), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 1, 16, 64), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(ms.MixedStepError) as e:
        ms.mixed_step_attention(q, kc, kc, b.cu_seqlens_q, b.q_start_pos, b.context_lens, b.block_tables, T,
                                torch.empty_like(q), ws)
    assert e.value.code == ms.MS_ERR_ARG


def test_chunked_prefill_matches_full_prefill_on_gpu(env):
    """zwjcode section 07: chunks [2, 3, 1] of a 6-token prompt -- and a 300-token prompt as
    [100, 37, 163] -- give the same outputs as one full prefill (same pool, same inputs)."""
    torch, ms, step = env
    for chunks, H_q, H_kv, D in (([2, 3, 1], 4, 2, 64), ([100, 37, 163], 8, 2, 128), ([129, 128, 1], 8, 8, 128)):
        L = sum(chunks)
        rng = np.random.default_rng(L)
        table = rng.permutation(-(-L // 16) + 2).astype(np.int32)
        wl = workloads.Workload("chunked_vs_full", H_q, H_kv, D, L, [workloads.Request(0, L, table)],
                                len(table))
        qa, ka, va = workloads.step_tensors(wl, L, 5, "cuda")
        cos, sin = step.rope_tables_device(L + 1, D, "cuda")

        def run(chunk_list):
            kc = torch.zeros((wl.num_pages, H_kv, 16, D), dtype=torch.bfloat16, device="cuda")
            vc = torch.zeros_like(kc)
            outs = []
            state = [(0, L)]
            for d in chunk_list:
                meta = ms.build_batch_metadata(state, [table], d)
                b = step.to_device(meta, "cuda")
                c0 = state[0][0]
                q = qa[c0:c0 + d].clone()
                out = torch.zeros_like(q)
                ws = step.workspace_for(b, H_q, H_kv, D, "cuda")
                step.run_step(q, ka[c0:c0 + d], va[c0:c0 + d], b, cos, sin, kc, vc, out, ws)
                outs.append(out)
                state = [(c0 + d, L - c0 - d)]
            torch.cuda.synchronize()
            return torch.cat(outs).float().cpu().numpy()

        full = run([L])
        chunked = run(chunks)
        assert np.all(np.abs(chunked - full) <= ATOL + RTOL * np.abs(full))


def test_status_reports_bad_slot_and_page(env):
    torch, ms, step = env
    wl = workloads.small_mixed(seed=41, H_q=4, H_kv=2, D=64, dec_ctx=(20,), prompts=())
    case = Case(env, wl, _states(wl), seed=3)
    bad_slots = torch.full_like(case.batch.slot_mapping, wl.num_pages * 16 + 5)
    ms.kv_append_rope(case.q, case.k, case.v, case.batch.positions, bad_slots, case.cos, case.sin, case.k_cache,
                      case.v_cache, q_rot=case.q_rot, dev_status=case.status)
    torch.cuda.synchronize()
    assert ms.read_status(case.status) & ms.STATUS_BAD_SLOT
    np.testing.assert_array_equal(workloads.bf16_bits(case.k_cache), case.k_in)  # nothing written
    case.batch.block_tables.fill_(wl.num_pages + 7)
    ms.mixed_step_attention(case.q_rot, case.k_cache, case.v_cache, case.batch.cu_seqlens_q,
                            case.batch.q_start_pos, case.batch.context_lens, case.batch.block_tables,
                            case.batch.context_total, case.out, case.ws)
    torch.cuda.synchronize()
    assert ms.read_status(case.ws) & ms.STATUS_BAD_PAGE
    assert ms.read_status(case.ws) == 0  # cleared by the read


@pytest.mark.parametrize("dec_ctx", [(20, 30), tuple(range(20, 60))])
def test_inconsistent_metadata_is_flagged(env, dec_ctx):
    """Both prologue shapes (one warp up to 32 rows, a block beyond) reject a row with ctx != c + d."""
    torch, ms, step = env
    wl = workloads.small_mixed(seed=42, H_q=4, H_kv=2, D=64, dec_ctx=dec_ctx, prompts=((0, 9),))
    case = Case(env, wl, _states(wl), seed=3)
    case.batch.context_lens[len(dec_ctx) // 2] += 1  # no longer c + d
    ms.mixed_step_attention(case.q, case.k_cache, case.v_cache, case.batch.cu_seqlens_q, case.batch.q_start_pos,
                            case.batch.context_lens, case.batch.block_tables, case.batch.context_total,
                            case.out, case.ws)
    torch.cuda.synchronize()
    assert ms.read_status(case.ws) & ms.STATUS_BAD_META
    # the same through the step call, whose prologue runs inside the append's launch
    step.run_step(case.q, case.k, case.v, case.batch, case.cos, case.sin, case.k_cache, case.v_cache, case.out,
                  case.ws, q_rot=case.q_rot, dev_status=case.status)
    torch.cuda.synchronize()
    assert ms.read_status(case.ws) & ms.STATUS_BAD_META
    assert ms.read_status(case.status) == 0  # the append itself was fine
    # a decode whose c + d wraps in 32 bits (c = 2^31 - 1, ctx given as the wrapped sum) is refused too
    case.batch.context_lens[len(dec_ctx) // 2] -= 1
    case.batch.q_start_pos[0] = 2**31 - 1
    case.batch.context_lens[0] = -2**31
    ms.mixed_step_attention(case.q, case.k_cache, case.v_cache, case.batch.cu_seqlens_q, case.batch.q_start_pos,
                            case.batch.context_lens, case.batch.block_tables, case.batch.context_total,
                            case.out, case.ws)
    torch.cuda.synchronize()
    assert ms.read_status(case.ws) & ms.STATUS_BAD_META


def test_append_bad_position_and_negative_slot(env):
    """A token whose position lies outside the cos/sin table writes nothing (no K, no V) and sets
    BAD_POSITION; slot -1 is the one silent "no write" value, any other negative slot sets BAD_SLOT."""
    torch, ms, step = env
    wl = workloads.small_mixed(seed=43, H_q=4, H_kv=2, D=64, dec_ctx=(20, 33), prompts=((0, 6),))
    case = Case(env, wl, _states(wl), seed=4)
    b = case.batch
    bad_pos = torch.full_like(b.positions, case.cos.shape[0] + 3)
    ms.kv_append_rope(case.q, case.k, case.v, bad_pos, b.slot_mapping, case.cos, case.sin, case.k_cache,
                      case.v_cache, q_rot=case.q_rot, dev_status=case.status)
    torch.cuda.synchronize()
    st = ms.read_status(case.status)
    assert st & ms.STATUS_BAD_POSITION and not st & ms.STATUS_BAD_SLOT, st
    np.testing.assert_array_equal(workloads.bf16_bits(case.k_cache), case.k_in)
    np.testing.assert_array_equal(workloads.bf16_bits(case.v_cache), case.v_in)
    slots = b.slot_mapping.clone()
    slots[0] = -2
    slots[1:] = -1
    ms.kv_append_rope(case.q, case.k, case.v, b.positions, slots, case.cos, case.sin, case.k_cache,
                      case.v_cache, q_rot=case.q_rot, dev_status=case.status)
    torch.cuda.synchronize()
    assert ms.read_status(case.status) == ms.STATUS_BAD_SLOT
    np.testing.assert_array_equal(workloads.bf16_bits(case.k_cache), case.k_in)
    np.testing.assert_array_equal(workloads.bf16_bits(case.v_cache), case.v_in)


# bf16 bit patterns a recycled page may hold: quiet NaN, +Inf, -Inf, NaN with every bit set
_GARBAGE = np.array([0x7FC0, 0x7F80, 0xFF80, 0xFFFF], dtype=np.uint16)


def _poison_unread_slots(case):
    """Fill every pool slot that no row of the step reads (past each row's context in its last page)
    with non-finite bf16 patterns, on the device and in the host copies the oracle starts from."""
    torch = pytest.importorskip("torch")
    meta, wl = case.meta, case.wl
    kp, vp = case.k_in.copy(), case.v_in.copy()
    n_poison = 0
    for s in range(meta["num_rows"]):
        table = wl.requests[int(meta["row_req"][s])].block_table
        L = int(meta["context_lens"][s])
        for j in range(L, 16 * len(table)):
            page, off = int(table[j // 16]), j % 16
            pat = np.resize(np.roll(_GARBAGE, j), kp.shape[-1])
            kp[page, :, off, :] = pat
            vp[page, :, off, :] = pat[::-1]
            n_poison += 1
    dev = case.k_cache.device
    case.k_cache.copy_(torch.from_numpy(kp.view(np.int16)).view(torch.bfloat16).to(dev))
    case.v_cache.copy_(torch.from_numpy(vp.view(np.int16)).view(torch.bfloat16).to(dev))
    case.k_in, case.v_in = kp, vp
    return n_poison


@pytest.mark.parametrize("H_q,H_kv,D", [(8, 2, 128), (4, 4, 64), (8, 1, 128), (8, 8, 128)])
def test_nonfinite_garbage_past_the_context_is_never_used(env, H_q, H_kv, D):
    """zwjcode section 07: the query at chunk index i sees keys 0..c+i and nothing else.  A recycled
    page holds anything, so the slots past every row's context (the tail of its last page) hold NaN
    and +-Inf bit patterns here; decode rows and chunk rows (ragged tiles at D = 64 and 128) must stay
    within tolerance of the oracle, which never reads those slots."""
    wl = workloads.small_mixed(seed=H_q * 7 + H_kv + D, H_q=H_q, H_kv=H_kv, D=D,
                               dec_ctx=(0, 5, 14, 17, 40, 100, 333),
                               prompts=((0, 70), (33, 130), (16, 5), (250, 3)))
    case = Case(env, wl, _states(wl), seed=12)
    assert _poison_unread_slots(case) > 0
    case.run(env)
    T = case.meta["num_tokens"]
    ref_meta, (q_rot, kp, vp) = case.oracle_append()
    np.testing.assert_array_equal(workloads.bf16_bits(case.k_cache), kp)
    np.testing.assert_array_equal(workloads.bf16_bits(case.v_cache), vp)
    ref = oracle.attention_all(q_rot, kp, vp, ref_meta, wl.H_kv)
    got = workloads.bf16_bits(case.out[:T])
    assert np.isfinite(oracle.bf16_to_f64(got)).all()
    n_dec = case.meta["num_decodes"]
    _check_attention(got[:n_dec], ref[:n_dec], "decode rows next to garbage")
    _check_attention(got[n_dec:], ref[n_dec:], "chunk rows next to garbage")


def test_stalled_chunk_phase_times_out_and_the_workspace_recovers(env):
    """Failure detection of the persistent kernel: with every chunk-phase producer stopped (the
    ms_test_attention_stall hook) the chunk-phase waits give up after 1 ms, the call ends, the
    status word carries STATUS_TIMEOUT, and the next ordinary call on the same workspace (whose
    kernel must allocate the tensor memory the stalled one held) matches the oracle again."""
    torch, ms, step = env
    wl = workloads.small_mixed(seed=45, H_q=8, H_kv=2, D=128)
    case = Case(env, wl, _states(wl), seed=6).run(env)
    T = case.meta["num_tokens"]
    ref_meta, (q_rot, kp, vp) = case.oracle_append()
    ref = oracle.attention_all(q_rot, kp, vp, ref_meta, wl.H_kv)
    b = case.batch
    args = (case.q_rot, case.k_cache, case.v_cache, b.cu_seqlens_q, b.q_start_pos, b.context_lens,
            b.block_tables, b.context_total)
    for attempt in range(2):
        stalled = torch.zeros_like(case.out)
        t0 = time.perf_counter()
        ms.test_attention_stall(*args, stalled, case.ws, wait_limit_ns=1_000_000)
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 10.0
        assert ms.read_status(case.ws) & ms.STATUS_TIMEOUT, f"attempt {attempt}: no timeout recorded"
        again = torch.zeros_like(case.out)
        ms.mixed_step_attention(*args, again, case.ws)
        torch.cuda.synchronize()
        assert ms.read_status(case.ws) == 0
        _check_attention(workloads.bf16_bits(again[:T]), ref, f"call after stall {attempt}")


def _ragged_batch(env, wl, states, dev="cuda"):
    torch, ms, step = env
    meta = ms.build_batch_metadata(states, _tables(wl), wl.token_budget, wl.max_chunk, ragged=True)
    return meta, step.to_device(meta, dev)


@pytest.mark.parametrize("H_q,H_kv,D", [(8, 2, 128), (8, 4, 64), (4, 4, 128)])
def test_ragged_block_table_matches_padded_and_oracle(env, H_q, H_kv, D):
    """zwjcode section 06 gives each row ceil((c+d)/B) block-table entries: the ragged form passes exactly
    those.  Its attention output equals the padded call's bit for bit (the same pages are read) and the
    oracle's within tolerance."""
    torch, ms, step = env
    wl = workloads.small_mixed(seed=H_q * 3 + H_kv + D, H_q=H_q, H_kv=H_kv, D=D)
    case = Case(env, wl, _states(wl), seed=21).run(env)
    T = case.meta["num_tokens"]
    rmeta, rb = _ragged_batch(env, wl, _states(wl))
    assert rb.ragged and rb.block_tables.numel() < case.batch.block_tables.numel()
    out = torch.zeros_like(case.out)
    ws = step.workspace_for(rb, wl.H_q, wl.H_kv, wl.D, "cuda")
    step.attend(case.q_rot[:T], case.k_cache, case.v_cache, rb, out[:T], ws)
    torch.cuda.synchronize()
    assert ms.read_status(ws) == 0
    np.testing.assert_array_equal(workloads.bf16_bits(out[:T]), workloads.bf16_bits(case.out[:T]))
    ref_meta, (q_rot, kp, vp) = case.oracle_append()
    ref = oracle.attention_all(q_rot, kp, vp, ref_meta, wl.H_kv)
    _check_attention(workloads.bf16_bits(out[:T]), ref, "ragged")


def test_ragged_row_short_of_pages_is_flagged(env):
    """A row whose offsets give it fewer pages than ceil(context/16) makes the step compute nothing and
    set BAD_META; so does an offset past the end of the page list."""
    torch, ms, step = env
    wl = workloads.small_mixed(seed=44, H_q=8, H_kv=2, D=128, dec_ctx=(20, 40), prompts=((0, 33),))
    case = Case(env, wl, _states(wl), seed=4).run(env)
    rmeta, rb = _ragged_batch(env, wl, _states(wl))
    ws = step.workspace_for(rb, wl.H_q, wl.H_kv, wl.D, "cuda")
    for bad in ("short", "past_end"):
        off = rb.bt_offsets.clone()
        if bad == "short":
            off[1] -= 1  # row 0 loses a page (row 1 gains one)
        else:
            off[-1] += 5
        b2 = step.DeviceBatch(rb.cu_seqlens_q, rb.q_start_pos, rb.context_lens, rb.positions, rb.slot_mapping,
                              rb.block_tables, rb.num_rows, rb.num_tokens, rb.num_decodes, rb.context_total,
                              rb.host, bt_offsets=off)
        out = torch.zeros_like(case.out)
        step.attend(case.q_rot, case.k_cache, case.v_cache, b2, out, ws)
        torch.cuda.synchronize()
        assert ms.read_status(ws) & ms.STATUS_BAD_META, bad


@pytest.mark.slow
@pytest.mark.parametrize("name", ["gqa8b_b8192", "long_bimodal_b4608"])
def test_full_size_ragged_equals_padded(env, name):
    """The full-size step with the ragged block table gives the padded call's output bit for bit."""
    torch, ms, step = env
    wl = workloads.CONFIGS[name]()
    case = Case(env, wl, _states(wl), seed=23, host_pool=False).run(env)
    T = case.meta["num_tokens"]
    rmeta, rb = _ragged_batch(env, wl, _states(wl))
    out = torch.zeros_like(case.out)
    ws = step.workspace_for(rb, wl.H_q, wl.H_kv, wl.D, "cuda")
    step.attend(case.q_rot[:T], case.k_cache, case.v_cache, rb, out[:T], ws)
    torch.cuda.synchronize()
    assert ms.read_status(ws) == 0
    assert torch.equal(out[:T].view(torch.int16), case.out[:T].view(torch.int16))


# ------------------------------------------------------------------ full-size configurations (sampled)

def _sampled_parity(env, wl, seed, n_dec_rows=48, n_chunk_tokens=48, heads=None):
    """Full-size step on the GPU; oracle on sampled (token, head) pairs.

    The sampled rows' pages are gathered from the device pool before and after
    the step: the oracle appends the rows' new tokens into the "before" copy,
    which must equal the "after" copy bit for bit, then attends from it."""
    torch, ms, step = env
    states = _states(wl)
    case = Case(env, wl, states, seed, host_pool=False)
    meta = case.meta
    T, n_dec = meta["num_tokens"], meta["num_decodes"]
    rng = np.random.default_rng(seed)
    H_q = wl.H_q
    heads = heads or sorted(set(rng.integers(0, H_q, size=4).tolist()) | {0, H_q - 1})
    dec_rows = sorted(set(rng.choice(n_dec, size=min(n_dec, n_dec_rows), replace=False).tolist())) if n_dec else []
    chunk_tok = sorted(set(rng.choice(np.arange(n_dec, T), size=min(T - n_dec, n_chunk_tokens),
                                      replace=False).tolist()) | ({n_dec, T - 1} if T > n_dec else set()))
    forced = _hardest_tokens(meta, wl.H_q // wl.H_kv)
    every = sorted(set(dec_rows) | set(chunk_tok) | forced)
    # decodes past LONG_KEYS keys go through _long_decode_parity (one row's pages at a time)
    long_dec = [t for t in every if t < n_dec and meta["context_lens"][t] > LONG_KEYS]
    tokens = [t for t in every if t not in set(long_dec)]
    ref_meta = oracle.batch_metadata(oracle.schedule(states, wl.token_budget, wl.max_chunk)[0], _tables(wl),
                                     len(states), num_decodes=n_dec)
    for key in ("cu_seqlens_q", "positions", "slot_mapping", "context_lens", "q_start_pos"):
        np.testing.assert_array_equal(meta[key], ref_meta[key])
    cu = ref_meta["cu_seqlens_q"]
    row_of = np.searchsorted(cu, np.arange(T), side="right") - 1
    rows = sorted(set(row_of[tokens].tolist()))
    bts = ref_meta["block_tables"]
    pages = np.unique(np.concatenate([bts[s][bts[s] >= 0] for s in rows]))
    remap = np.full(wl.num_pages, -1, dtype=np.int64)
    remap[pages] = np.arange(len(pages))
    pidx = torch.from_numpy(pages.astype(np.int64)).to(case.k_cache.device)
    k_pre = workloads.bf16_bits(case.k_cache.index_select(0, pidx))
    v_pre = workloads.bf16_bits(case.v_cache.index_select(0, pidx))
    case.run(env)
    k_post = workloads.bf16_bits(case.k_cache.index_select(0, pidx))
    v_post = workloads.bf16_bits(case.v_cache.index_select(0, pidx))
    sub_meta = {"cu_seqlens_q": cu, "q_start_pos": ref_meta["q_start_pos"],
                "block_tables": np.where(bts >= 0, remap[np.maximum(bts, 0)], -1)}
    tok_rows = [t for t in range(T) if row_of[t] in set(rows)]
    q = workloads.bf16_bits(case.q[tok_rows])
    k = workloads.bf16_bits(case.k[tok_rows])
    v = workloads.bf16_bits(case.v[tok_rows])
    pos = ref_meta["positions"][tok_rows]
    slots = ref_meta["slot_mapping"][tok_rows]
    sub_slots = remap[slots // 16] * 16 + slots % 16
    q_rot_sub, kp_ref, vp_ref = oracle.kv_append(q, k, v, pos, sub_slots, k_pre, v_pre)
    np.testing.assert_array_equal(k_post, kp_ref)
    np.testing.assert_array_equal(v_post, vp_ref)
    np.testing.assert_array_equal(workloads.bf16_bits(case.q_rot[tok_rows]), q_rot_sub)
    q_rot_full = np.zeros((T, H_q, wl.D), np.uint16)
    q_rot_full[tok_rows] = q_rot_sub
    select = [(t, h) for t in tokens for h in heads]
    ref = oracle.attention_rows(q_rot_full, kp_ref, vp_ref, sub_meta, wl.H_kv, select=select)
    got = workloads.bf16_bits(case.out)
    g = np.stack([got[t, h] for t, h in select])
    r = np.stack([ref[(t, h)] for t, h in select])
    _check_attention(g, r, wl.name)
    if long_dec:
        _long_decode_parity(env, case, ref_meta, long_dec, sorted({0, H_q - 1}))
    return len(tokens) + len(long_dec)


LONG_KEYS = 32768


def _long_decode_parity(env, case, ref_meta, rows, heads):
    """Decode rows too long to copy the pool around (64K-128K keys): the row's appended slot is checked
    bit-exact against the oracle's rotation of its token, then the oracle attends over the row's own
    pages of one KV head at a time, gathered from the device pool after the step."""
    torch, ms, step = env
    wl = case.wl
    G = wl.H_q // wl.H_kv
    dev = case.k_cache.device
    got = workloads.bf16_bits(case.out)
    for t in rows:  # a decode row's token index is its row index
        ctx = int(ref_meta["context_lens"][t])
        n_pages = -(-ctx // 16)
        table = ref_meta["block_tables"][t][:n_pages].astype(np.int64)
        slot = int(ref_meta["slot_mapping"][t])
        zero = np.zeros((1,) + tuple(case.k_cache.shape[1:]), np.uint16)
        q_rot1, k1, v1 = oracle.kv_append(workloads.bf16_bits(case.q[t:t + 1]), workloads.bf16_bits(case.k[t:t + 1]),
                                          workloads.bf16_bits(case.v[t:t + 1]), ref_meta["positions"][t:t + 1],
                                          np.array([slot % 16]), zero, zero)
        np.testing.assert_array_equal(workloads.bf16_bits(case.q_rot[t:t + 1]), q_rot1)
        page = torch.tensor([slot // 16], device=dev)
        np.testing.assert_array_equal(workloads.bf16_bits(case.k_cache.index_select(0, page))[0, :, slot % 16],
                                      k1[0, :, slot % 16])
        np.testing.assert_array_equal(workloads.bf16_bits(case.v_cache.index_select(0, page))[0, :, slot % 16],
                                      v1[0, :, slot % 16])
        pidx = torch.from_numpy(table).to(dev)
        for kvh in sorted({h // G for h in heads}):
            kp = workloads.bf16_bits(case.k_cache.index_select(0, pidx)[:, kvh:kvh + 1])
            vp = workloads.bf16_bits(case.v_cache.index_select(0, pidx)[:, kvh:kvh + 1])
            sub = {"cu_seqlens_q": np.array([0, 1]), "q_start_pos": np.array([ctx - 1]),
                   "block_tables": np.arange(n_pages)[None, :]}
            hs = [h for h in heads if h // G == kvh]
            ref = oracle.attention_rows(q_rot1[:, kvh * G:(kvh + 1) * G], kp, vp, sub, 1,
                                        select=[(0, h - kvh * G) for h in hs])
            g = np.stack([got[t, h] for h in hs])
            r = np.stack([ref[(0, h - kvh * G)] for h in hs])
            _check_attention(g, r, f"{wl.name} decode row {t} ({ctx} keys)")


def _hardest_tokens(meta, G):
    """Tokens every full-size check includes besides its random sample: the longest decode row
    (which also has the most splits to merge), every decode of 64K keys or more, and the first and
    last two tokens of the first and last 128-row query tile of every chunk row (the tile that
    starts the causal diagonal and the one that ends the chunk, with its ragged tail)."""
    cu, c0 = meta["cu_seqlens_q"], meta["q_start_pos"]
    n_dec = meta["num_decodes"]
    out = set()
    if n_dec:
        ctx = meta["context_lens"][:n_dec]
        out.add(int(np.argmax(ctx)))
        out |= {int(s) for s in np.nonzero(ctx >= 65536)[0]}
    tpt = 128 // G
    for s in range(n_dec, meta["num_rows"]):
        a, b = int(cu[s]), int(cu[s + 1])
        if b - a < 2:
            continue
        last_tile = a + ((b - a - 1) // tpt) * tpt
        for t in (a, a + 1, min(a + tpt, b) - 2, min(a + tpt, b) - 1, last_tile, last_tile + 1, b - 2, b - 1):
            if a <= t < b:
                out.add(t)
    return out


@pytest.mark.slow
@pytest.mark.parametrize("name", ["mha7b_b512", "mha13b_b2048", "gqa8b_b8192", "long_bimodal_b4608"])
def test_full_size_config_sampled(env, name):
    wls = workloads.CONFIGS[name]()
    if isinstance(wls, list):
        wls = [wls[0], wls[-1]] + workloads.mha7b_steps(include_tail=True)[-1:]
    else:
        wls = [wls]
    for i, wl in enumerate(wls):
        _sampled_parity(env, wl, seed=17 + i)
