"""Host-side checks of the C ABI (no GPU): the library builds, loads and exports
every declared entry point; the C++ scheduler and rope table are bit-exact with
the oracle; error codes follow the header."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import workloads
from conftest import ROOT


@pytest.fixture(scope="module")
def ms():
    from chunked_prefill_mixed_decode_gb300 import build
    build.build()
    import chunked_prefill_mixed_decode_gb300 as ms
    return ms


def header_symbols():
    syms = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            syms += re.findall(r"MS_API\s+[\w\s\*]+?\b(ms_\w+)\s*\(", text)
    return syms


def test_library_exports_every_declared_symbol(ms):
    syms = header_symbols()
    assert len(syms) >= 7
    lib = ctypes.CDLL(ms.build.LIB)
    for s in syms:
        assert hasattr(lib, s), s


def _oracle_meta(states, tables, budget, cap=0):
    rows, unused = oracle.schedule(states, budget, cap)
    n_dec = sum(1 for s in states if s[1] == 0)
    m = oracle.batch_metadata(rows, tables, len(states), num_decodes=n_dec)
    m["unused_tokens"] = unused
    return m


def _assert_meta_equal(got, ref):
    for k in ("cu_seqlens_q", "q_start_pos", "context_lens", "positions", "slot_mapping", "row_req",
              "num_scheduled"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    np.testing.assert_array_equal(got["block_tables"], ref["block_tables"])
    for k in ("bt_stride", "num_rows", "num_tokens", "num_decodes", "unused_tokens"):
        assert got[k] == ref[k], k


def test_worked_example_rounds_bit_exact(ms):
    wl = workloads.worked_example()
    tables = [r.block_table for r in wl.requests]
    states = [(r.cached_len, r.remaining) for r in wl.requests]
    for _ in range(4):
        got = ms.build_batch_metadata(states, tables, wl.token_budget)
        ref = _oracle_meta(states, tables, wl.token_budget)
        _assert_meta_equal(got, ref)
        rows, _ = oracle.schedule(states, wl.token_budget)
        states = oracle.commit_round(states, rows)


@pytest.mark.parametrize("name", ["mha7b_b512", "mha13b_b2048", "gqa8b_b8192", "long_bimodal_b4608"])
def test_config_metadata_bit_exact(ms, name):
    wls = workloads.CONFIGS[name]()
    wls = wls if isinstance(wls, list) else [wls]
    for wl in wls[:3]:
        tables = [r.block_table for r in wl.requests]
        states = [(r.cached_len, r.remaining) for r in wl.requests]
        got = ms.build_batch_metadata(states, tables, wl.token_budget, wl.max_chunk)
        _assert_meta_equal(got, _oracle_meta(states, tables, wl.token_budget, wl.max_chunk))


def test_scheduler_fuzz_bit_exact(ms):
    rng = np.random.default_rng(21)
    for trial in range(400):
        n = int(rng.integers(0, 12))
        budget = int(rng.integers(0, 40))
        cap = int(rng.integers(0, 3)) * int(rng.integers(1, 9))
        states, tables = [], []
        for _ in range(n):
            c = int(rng.integers(0, 100))
            rem = 0 if rng.random() < 0.5 else int(rng.integers(1, 60))
            need = -(-(c + max(rem, 1)) // 16)
            short = rng.random() < 0.08
            n_pages = max(0, need - int(rng.integers(1, 3))) if short else need + int(rng.integers(0, 3))
            tables.append(rng.integers(0, 1000, size=n_pages).astype(np.int32))
            states.append((c, rem))
        try:
            ref = _oracle_meta(states, tables, budget, cap)
            err = None
        except oracle.BudgetError:
            err = ms.MS_ERR_BUDGET
        except oracle.NoPagesError:
            err = ms.MS_ERR_NO_PAGES
        if err is None:
            _assert_meta_equal(ms.build_batch_metadata(states, tables, budget, cap), ref)
        else:
            with pytest.raises(ms.MixedStepError) as e:
                ms.build_batch_metadata(states, tables, budget, cap)
            assert e.value.code == err


@pytest.mark.parametrize("policy", [0, 1, 2])
def test_policies_fuzz_bit_exact(ms, policy):
    """Every scheduling policy and limit: the C++ scheduler's rows and metadata equal the oracle's."""
    rng = np.random.default_rng(400 + policy)
    for trial in range(300):
        n = int(rng.integers(0, 12))
        budget = int(rng.integers(0, 40))
        cap = int(rng.integers(0, 2)) * int(rng.integers(1, 16))
        floor = int(rng.integers(0, 2)) * int(rng.integers(1, 12))
        quota = int(rng.integers(0, 2)) * int(rng.integers(0, budget + 1))
        share = int(rng.integers(0, 1001))
        states, tables = [], []
        for _ in range(n):
            c = int(rng.integers(0, 100))
            rem = 0 if rng.random() < 0.5 else int(rng.integers(1, 60))
            need = -(-(c + max(rem, 1)) // 16)
            tables.append(rng.integers(0, 1000, size=need).astype(np.int32))
            states.append((c, rem))
        kw = dict(policy=policy, min_chunk=floor, prefill_quota=quota, decode_share=share)
        try:
            rows, unused = oracle.schedule(states, budget, cap, **kw)
            n_dec = sum(1 for i, _, d in rows if states[i][1] == 0)
            ref = oracle.batch_metadata(rows, tables, n, num_decodes=n_dec)
            ref["unused_tokens"] = unused
            err = None
        except oracle.BudgetError:
            err = ms.MS_ERR_BUDGET
        if err is None:
            got = ms.build_batch_metadata(states, tables, budget, cap, policy, floor, quota, share)
            _assert_meta_equal(got, ref)
            n_decodes = sum(1 for s_ in states if s_[1] == 0)
            assert got["num_deferred"] == n_decodes - ref["num_decodes"]
        else:
            with pytest.raises(ms.MixedStepError) as e:
                ms.build_batch_metadata(states, tables, budget, cap, policy, floor, quota, share)
            assert e.value.code == err


def test_rope_table_bit_exact_with_oracle(ms):
    for D in (64, 128):
        max_pos = 131073
        cos, sin = ms.rope_table(max_pos, D)
        pos = np.array([0, 1, 2, 5, 15, 16, 17, 448, 4095, 6000, 28672, 32767, 65536, 100003, 131072])
        oc, os_ = oracle.rope_tables(pos, D)
        np.testing.assert_array_equal(cos[pos], oc)
        np.testing.assert_array_equal(sin[pos], os_)


def test_argument_errors(ms):
    lib = ms.lib()
    assert lib.ms_rope_table(0, 64, 10000.0, None, None) == ms.MS_ERR_ARG
    assert lib.ms_kv_append_rope(*([None] * 5), 1, None, None, 1, None, None, 1, None, 4, 3, 64, 16, None,
                                 None) == ms.MS_ERR_ARG  # H_q % H_kv != 0
    assert lib.ms_kv_append_rope(*([None] * 5), 0, None, None, 1, None, None, 1, None, 4, 2, 64, 16, None,
                                 None) == ms.MS_OK  # T == 0 is a no-op
    assert lib.ms_mixed_step_attention(None, None, None, 1, None, None, None, None, 1, 0, 0, 0, 4, 2, 96, 16,
                                       0.1, None, None, 0, None) == ms.MS_ERR_ARG  # D = 96
    assert lib.ms_mixed_step_attention(None, None, None, 1, None, None, None, None, 1, 0, 0, 0, 4, 2, 64, 16,
                                       0.1, None, None, 0, None) == ms.MS_OK  # empty step
    assert lib.ms_mixed_step_attention(None, None, None, 1, None, None, None, None, 1, 0, 0, 0, 12, 4, 64, 16,
                                       0.1, None, None, 0, None) == ms.MS_ERR_ARG  # G = 3 unsupported
    # capacity too small -> MS_ERR_ARG, budget overflow -> MS_ERR_BUDGET
    bt = np.arange(4, dtype=np.int32)
    with pytest.raises(ms.MixedStepError) as e:
        ms.build_batch_metadata([(3, 0)] * 3, [bt] * 3, 2)
    assert e.value.code == ms.MS_ERR_BUDGET
    with pytest.raises(ms.MixedStepError) as e:
        ms.build_batch_metadata([(60, 10)], [bt], 8)  # needs ceil(68/16) = 5 pages
    assert e.value.code == ms.MS_ERR_NO_PAGES


def test_workspace_size_grows_with_context(ms):
    a = ms.attention_workspace_size(65, 512, 64 * 4096, 32, 32, 128)
    b = ms.attention_workspace_size(65, 512, 2 * 64 * 4096, 32, 32, 128)
    assert 0 < a < b
    assert ms.attention_workspace_size(1, 1, 0, 4, 2, 96) == 0


def _engine_pair(ms, num_pages, budget, **kw):
    okw = dict(max_chunk=kw.get("max_chunk_per_request", 0), policy=kw.get("policy", 0),
               min_chunk=kw.get("min_chunk_per_request", 0), prefill_quota=kw.get("prefill_quota", 0),
               decode_share=kw.get("decode_share_permille", 500))
    return ms.Engine(num_pages, budget, **kw), oracle.Engine(num_pages, budget, **okw)


@pytest.mark.parametrize("policy", [0, 1, 2])
def test_engine_simulation_bit_exact(ms, policy):
    """Random arrivals over many rounds: the C++ engine's admissions, metadata, finished ids and
    pool counts equal the oracle engine's at every round."""
    rng = np.random.default_rng(700 + policy)
    for trial in range(6):
        budget = int(rng.integers(8, 96))
        kw = dict(max_chunk_per_request=int(rng.integers(0, 2)) * int(rng.integers(1, 40)), policy=policy,
                  min_chunk_per_request=int(rng.integers(0, 2)) * int(rng.integers(1, 16)),
                  prefill_quota=int(rng.integers(0, 2)) * int(rng.integers(1, budget)) if policy == 0 else 0,
                  decode_share_permille=int(rng.integers(0, 1001)))
        num_pages = int(rng.integers(20, 300))
        got, ref = _engine_pair(ms, num_pages, budget, **kw)
        rounds = 0
        for rnd in range(150):
            for _ in range(int(rng.integers(0, 3))):
                pl = int(rng.integers(1, 200))
                mn = int(rng.integers(2, 30))
                cached = int(rng.integers(0, pl + 1)) if rng.random() < 0.25 else 0
                try:
                    want = ref.add_request(pl, mn, cached)
                except oracle.AdmissionError:
                    with pytest.raises(ms.MixedStepError) as e:
                        got.add_request(pl, mn, cached)
                    assert e.value.code == ms.MS_ERR_NO_PAGES
                    continue
                assert got.add_request(pl, mn, cached) == want
                np.testing.assert_array_equal(got.request_pages(want), ref.live[-1].pages)
            if not ref.live:
                continue
            try:
                r = ref.plan()
            except oracle.BudgetError:
                with pytest.raises(ms.MixedStepError) as e:
                    got.plan()
                assert e.value.code == ms.MS_ERR_BUDGET
                break
            g = got.plan()
            for k in ("cu_seqlens_q", "q_start_pos", "context_lens", "positions", "slot_mapping",
                      "row_request_id"):
                np.testing.assert_array_equal(g[k], r[k], err_msg=k)
            np.testing.assert_array_equal(g["block_tables"], r["block_tables"])
            assert g["num_decodes"] == r["num_decodes"] and g["unused_tokens"] == r["unused_tokens"]
            assert got.commit() == ref.commit()
            rounds += 1
            st = got.stats()
            assert st["num_live"] == len(ref.live) and st["num_free_pages"] == len(ref.free)
            assert st["rounds"] == rounds


def test_engine_argument_errors(ms):
    e = ms.Engine(8, 16)
    for args in ((0, 4, 0), (10, 0, 0), (10, 4, 11), (10, 1, 10), (10, 4, -1)):
        with pytest.raises(ms.MixedStepError) as err:
            e.add_request(*args)
        assert err.value.code == ms.MS_ERR_ARG
        with pytest.raises(ValueError):
            oracle.Engine(8, 16).add_request(*args)
    with pytest.raises(ms.MixedStepError) as err:
        e.commit()  # no plan yet
    assert err.value.code == ms.MS_ERR_ARG
    with pytest.raises(ms.MixedStepError) as err:
        e.add_request(120, 20)  # 9 pages > 8
    assert err.value.code == ms.MS_ERR_NO_PAGES
    assert e.stats()["num_free_pages"] == 8


def test_graph_config_errors(ms):
    """Invalid graph configs are refused before any CUDA call."""
    import ctypes
    bk = np.array([16, 32], dtype=np.int32)
    ok = ms.GraphConfig(4, 2, 64, 8, 4, 8, 128, 0.125, 2, bk.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)))
    assert ms.lib().ms_graph_workspace_size(ctypes.byref(ok)) > 0
    for field, bad in (("D", 96), ("max_rows", 0), ("max_rows", 8193), ("num_buckets", 0), ("H_kv", 3)):
        cfg = ms.GraphConfig.from_buffer_copy(ok)
        setattr(cfg, field, bad)
        assert ms.lib().ms_graph_workspace_size(ctypes.byref(cfg)) == 0, field
    desc = np.array([32, 16], dtype=np.int32)
    cfg = ms.GraphConfig.from_buffer_copy(ok)
    cfg.buckets = desc.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    assert ms.lib().ms_graph_workspace_size(ctypes.byref(cfg)) == 0  # buckets must ascend
    h = ctypes.c_void_p()
    bufs = ms.GraphBuffers()
    assert ms.lib().ms_graph_create(ctypes.byref(ok), ctypes.byref(bufs), None, ctypes.byref(h)) == ms.MS_ERR_ARG
    assert ms.lib().ms_graph_destroy(None) == ms.MS_OK


def test_request_marshalling_edge_cases(ms):
    """The binding packs requests column by column: tables of any integer dtype
    and layout, empty tables, empty rounds, and bad lengths behave as the
    oracle and the header say."""
    rng = np.random.default_rng(17)
    states = [(0, 5), (16, 0), (3, 0), (0, 0)]
    tables = [rng.permutation(8).astype(np.int64)[:1],       # int64 input, cast to int32
              np.arange(40, 42, dtype=np.int32)[::-1].copy(),
              np.asarray([7]),                              # platform int
              np.zeros(0, dtype=np.int32)]                  # empty table, no tokens scheduled
    ref_rows, _ = oracle.schedule(states[:3], 16)
    ref = oracle.batch_metadata(ref_rows, [np.asarray(t, dtype=np.int32) for t in tables[:3]], 3)
    got = ms.build_batch_metadata(states[:3], tables[:3], 16)
    for k in ("cu_seqlens_q", "q_start_pos", "context_lens", "positions", "slot_mapping"):
        np.testing.assert_array_equal(got[k], ref[k])
    np.testing.assert_array_equal(got["block_tables"], ref["block_tables"])
    # the returned arrays are views of one fresh buffer per call: two calls share nothing
    again = ms.build_batch_metadata(states[:3], tables[:3], 16)
    again["positions"][:] = -1
    np.testing.assert_array_equal(got["positions"], ref["positions"])
    # an empty round
    empty = ms.build_batch_metadata([], [], 8)
    assert empty["num_rows"] == 0 and empty["num_tokens"] == 0
    # one table per request
    with pytest.raises(ValueError):
        ms.build_batch_metadata(states[:2], tables[:1], 16)
    # lengths beyond int32
    with pytest.raises(ValueError):
        ms.build_batch_metadata([(2 ** 31, 0)], [tables[1]], 16)


def test_device_wrappers_check_tensors_before_the_call(ms):
    """The ABI sees only addresses, so the binding checks dtype, layout, shape,
    size and device of every tensor first; a bad one raises ValueError and no
    pointer reaches the library (CPU tensors end at the device check)."""
    torch = pytest.importorskip("torch")
    T, H_q, H_kv, D, P = 5, 4, 2, 64, 3
    bf = torch.bfloat16
    good = dict(q=torch.zeros((T, H_q, D), dtype=bf), k=torch.zeros((T, H_kv, D), dtype=bf),
                v=torch.zeros((T, H_kv, D), dtype=bf), positions=torch.zeros(T, dtype=torch.int32),
                slot_mapping=torch.zeros(T, dtype=torch.int32), cos_tab=torch.zeros((32, D // 2)),
                sin_tab=torch.zeros((32, D // 2)), k_cache=torch.zeros((P, H_kv, 16, D), dtype=bf),
                v_cache=torch.zeros((P, H_kv, 16, D), dtype=bf))
    bad_append = [
        ("q", torch.zeros((T, H_q, D)), "q must be torch.bfloat16"),
        ("k", torch.zeros((T, H_kv + 1, D), dtype=bf), "k must have shape"),
        ("positions", torch.zeros(T, dtype=torch.int64), "positions must be torch.int32"),
        ("slot_mapping", torch.zeros(T - 1, dtype=torch.int32), "at least 5"),
        ("cos_tab", torch.zeros((32, D)), "cos_tab must have shape"),
        ("v_cache", torch.zeros((P, H_kv, D, 16), dtype=bf).transpose(2, 3), "v_cache must be contiguous"),
        ("k_cache", torch.zeros((P, H_kv, 8, D), dtype=bf), "k_cache must have shape"),
    ]
    for name, t, msg in bad_append:
        with pytest.raises(ValueError, match=msg):
            ms.kv_append_rope(**{**good, name: t})
    with pytest.raises(ValueError, match="CUDA"):
        ms.kv_append_rope(**good)

    S = 2
    att = dict(q_rot=good["q"], k_cache=good["k_cache"], v_cache=good["v_cache"],
               cu_seqlens_q=torch.tensor([0, 1, T], dtype=torch.int32),
               q_start_pos=torch.zeros(S, dtype=torch.int32), context_lens=torch.ones(S, dtype=torch.int32),
               block_tables=torch.zeros((S, 2), dtype=torch.int32), context_total=2,
               out=torch.zeros((T, H_q, D), dtype=bf), workspace=torch.zeros(256, dtype=torch.uint8))
    bad_attention = [
        ("out", torch.zeros((T, H_q, D)), "out must be torch.bfloat16"),
        ("out", torch.zeros((T - 1, H_q, D), dtype=bf), "out must have shape"),
        ("context_lens", torch.ones(S - 1, dtype=torch.int32), "context_lens must hold at least 2"),
        ("block_tables", torch.zeros((S, 2), dtype=torch.int64), "block_tables must be torch.int32"),
        ("cu_seqlens_q", torch.zeros((1, 3), dtype=torch.int32), "cu_seqlens_q must be 1-D"),
        ("v_cache", torch.zeros((P, H_kv, 16, D)), "v_cache must be torch.bfloat16"),
    ]
    for name, t, msg in bad_attention:
        with pytest.raises(ValueError, match=msg):
            ms.mixed_step_attention(**{**att, name: t})
        kw = {k: v for k, v in att.items() if k != "workspace"}
        with pytest.raises(ValueError, match=msg):
            ms.mixed_step_attention_noalloc(**{**kw, name: t})
    with pytest.raises(ValueError, match="CUDA"):
        ms.mixed_step_attention(**att)


def test_page_ids_a_row_reads_must_be_valid(ms):
    """A page id below 0 (which could turn a slot into the "no write" value -1)
    or one whose slots overflow int32 is refused with MS_ERR_ARG; ids the step
    does not read are not looked at."""
    ok = ms.build_batch_metadata([(16, 0)], [np.asarray([3, 5, -1], dtype=np.int32)], 8)
    np.testing.assert_array_equal(ok["slot_mapping"], [5 * 16])
    for bad in ([3, -1], [-2, 5], [3, 2 ** 31 // 16]):
        with pytest.raises(ms.MixedStepError) as e:
            ms.build_batch_metadata([(16, 0)], [np.asarray(bad, dtype=np.int32)], 8)
        assert e.value.code == ms.MS_ERR_ARG
    with pytest.raises(ms.MixedStepError) as e:  # a chunk row reads every page up to its last token
        ms.build_batch_metadata([(0, 40)], [np.asarray([0, -1, 2], dtype=np.int32)], 64)
    assert e.value.code == ms.MS_ERR_ARG


# ------------------------------------------------------------------ ragged block tables

def _expand_ragged(got):
    """The ragged block table (bt_offsets, bt_pages) as the padded [rows, stride] table."""
    S, stride = got["num_rows"], got["bt_stride"]
    out = np.full((S, stride), -1, dtype=np.int32)
    off = got["bt_offsets"]
    assert off[0] == 0 and np.all(np.diff(off) >= 0) and off[S] == got["bt_pages"].size
    for s in range(S):
        out[s, : off[s + 1] - off[s]] = got["bt_pages"][off[s]: off[s + 1]]
    return out


def _assert_ragged_meta_equal(got, ref):
    """zwjcode section 06: row s holds ceil((c+d)/16) pages -- exactly that many in the ragged form."""
    need = -(-np.asarray(got["context_lens"], dtype=np.int64) // 16)
    np.testing.assert_array_equal(np.diff(got["bt_offsets"]), need)
    padded = dict(got)
    padded["block_tables"] = _expand_ragged(got)
    _assert_meta_equal(padded, ref)


@pytest.mark.parametrize("name", ["worked_example_b8", "mha7b_b512", "mha13b_b2048", "gqa8b_b8192",
                                  "long_bimodal_b4608"])
def test_ragged_metadata_matches_oracle_expanded(ms, name):
    wls = workloads.CONFIGS[name]()
    wls = wls if isinstance(wls, list) else [wls]
    for wl in wls[:3]:
        tables = [r.block_table for r in wl.requests]
        states = [(r.cached_len, r.remaining) for r in wl.requests]
        got = ms.build_batch_metadata(states, tables, wl.token_budget, wl.max_chunk, ragged=True)
        _assert_ragged_meta_equal(got, _oracle_meta(states, tables, wl.token_budget, wl.max_chunk))


def test_ragged_scheduler_fuzz_and_errors(ms):
    rng = np.random.default_rng(22)
    for trial in range(300):
        n = int(rng.integers(0, 12))
        budget = int(rng.integers(0, 40))
        cap = int(rng.integers(0, 3)) * int(rng.integers(1, 9))
        states, tables = [], []
        for _ in range(n):
            c = int(rng.integers(0, 100))
            rem = 0 if rng.random() < 0.5 else int(rng.integers(1, 60))
            need = -(-(c + max(rem, 1)) // 16)
            short = rng.random() < 0.08
            n_pages = max(0, need - int(rng.integers(1, 3))) if short else need + int(rng.integers(0, 3))
            tables.append(rng.integers(0, 1000, size=n_pages).astype(np.int32))
            states.append((c, rem))
        try:
            ref = _oracle_meta(states, tables, budget, cap)
            err = None
        except oracle.BudgetError:
            err = ms.MS_ERR_BUDGET
        except oracle.NoPagesError:
            err = ms.MS_ERR_NO_PAGES
        if err is None:
            _assert_ragged_meta_equal(ms.build_batch_metadata(states, tables, budget, cap, ragged=True), ref)
        else:
            with pytest.raises(ms.MixedStepError) as e:
                ms.build_batch_metadata(states, tables, budget, cap, ragged=True)
            assert e.value.code == err


def test_ragged_scheduler_refuses_too_small_page_capacity(ms):
    """Three decodes of 2, 1 and 3 pages need 6 entries: capacity 5 is MS_ERR_ARG, 6 is enough."""
    lib = ms.lib()
    states = [(20, 0), (3, 0), (40, 0)]
    tables = [np.arange(4, dtype=np.int32), np.arange(4, 8, dtype=np.int32), np.arange(8, 12, dtype=np.int32)]
    reqs = (ms.Request * 3)()
    for i, ((c, r), t) in enumerate(zip(states, tables)):
        reqs[i] = ms.Request(c, r, t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), len(t))
    cfg = ms.SchedConfig(8, 0, 0, 0, 0, 500)
    arr = {k: np.zeros(16, dtype=np.int32) for k in ("cu", "qs", "ctx", "pos", "slot", "off", "pages", "rr", "ns")}
    info = ms.BatchInfo()
    p = {k: v.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) for k, v in arr.items()}
    for cap, want in ((5, ms.MS_ERR_ARG), (6, ms.MS_OK)):
        rc = lib.ms_build_batch_metadata_ragged(reqs, 3, ctypes.byref(cfg), 3, 8, cap, p["cu"], p["qs"], p["ctx"],
                                                p["pos"], p["slot"], p["off"], p["pages"], p["rr"], p["ns"],
                                                ctypes.byref(info))
        assert rc == want, (cap, rc)
    assert arr["off"][:4].tolist() == [0, 2, 3, 6]
    assert arr["pages"][:6].tolist() == [0, 1, 4, 8, 9, 10]
