"""Seeded synthetic inputs for the mixed-batch attention step.

This module is the only code shared by the CUDA path's callers (tests, bench)
and the fp64 oracle.  It draws inputs and nothing else: request states (cached
prefix length ``c`` and remaining prompt tokens), physical page assignments,
and bf16 tensors.  It holds none of the method's arithmetic -- no scheduling,
no rotary embedding, no attention.

Workload shapes follow the pages on chunked prefill:

* the 8-token-budget walk-through (3 decodes + one 12-token prompt) of
  "Chunked Prefill 的 Token 预算" (zwjcode.cn), section 03;
* a 7B-like layer at budget 512 = 64 decodes + a 448-token chunk, the split of
  a 4096-token prompt given in section 01 of the same page;
* 13B-like, 8B-GQA-like and long-context bimodal layers, whose decode context
  mixes follow the bimodal traffic described in "Prefill head-of-line blocking"
  (sference.com), "Why the median looks fine".

Conventions (the plainest reading where the pages are silent):

* a decode's "ctx" is ``c``, the tokens already cached; its query sits at
  absolute position ``c`` and it appends one token there;
* a prompt row is ``(c, remaining)``: ``c`` tokens are cached, ``remaining``
  still need prefill;
* every request owns ``ceil((c + max(remaining, 1)) / 16)`` physical pages,
  reserved up front, drawn from a seeded random permutation of the pool;
* tensor values are N(0, 1) rounded to bf16; cached pages hold N(0, 1) values
  that stand in for already-rotated keys.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional, Sequence

import numpy as np

PAGE = 16


@dataclasses.dataclass
class Request:
    cached_len: int          # c: tokens already in the KV cache
    remaining: int           # 0 => running decode, > 0 => waiting prompt tokens
    block_table: np.ndarray  # int32 physical page ids, logical order


@dataclasses.dataclass
class Workload:
    name: str
    H_q: int
    H_kv: int
    D: int
    token_budget: int
    requests: List[Request]
    num_pages: int
    max_chunk: int = 0
    page_size: int = PAGE
    seed: int = 0

    @property
    def max_pos(self) -> int:
        """One past the largest absolute position any token of this state can take."""
        return max(r.cached_len + max(r.remaining, 1) for r in self.requests)


def _pages_for(n_tokens: int) -> int:
    return (n_tokens + PAGE - 1) // PAGE


def assign_pages(states: Sequence[tuple], rng: np.random.Generator,
                 reserve: Optional[Sequence[int]] = None) -> tuple:
    """Give each (c, remaining) state its own pages from a random permutation.

    ``reserve[i]`` (optional) is the token capacity to reserve for request i;
    by default it is ``c + max(remaining, 1)``.
    """
    need = []
    for i, (c, rem) in enumerate(states):
        cap = reserve[i] if reserve is not None else c + max(rem, 1)
        need.append(_pages_for(cap))
    total = int(sum(need))
    perm = rng.permutation(total).astype(np.int32)
    reqs, off = [], 0
    for (c, rem), n in zip(states, need):
        reqs.append(Request(int(c), int(rem), perm[off:off + n].copy()))
        off += n
    return reqs, total


def worked_example(seed: int = 1, reserve_tokens: int = 24) -> Workload:
    """Budget 8, decodes D1-D3 at c = 37, 64, 100 and one 12-token prompt P.

    Pages are reserved for several future rounds (``reserve_tokens`` beyond c)
    so the same pool can be stepped through the four rounds of the walk-through.
    """
    rng = np.random.default_rng(seed)
    states = [(37, 0), (64, 0), (100, 0), (0, 12)]
    reserve = [c + max(r, 1) + reserve_tokens for c, r in states]
    reqs, total = assign_pages(states, rng, reserve)
    return Workload("worked_example_b8", 4, 2, 64, 8, reqs, total, seed=seed)


def identity_worked_example() -> Workload:
    """The walk-through with pages allocated in order (D1: 0-2, D2: 3-7, D3: 8-14, P: 15)."""
    states = [(37, 0), (64, 0), (100, 0), (0, 12)]
    reqs, off = [], 0
    for c, rem in states:
        n = _pages_for(c + max(rem, 1) + 3)
        reqs.append(Request(c, rem, np.arange(off, off + n, dtype=np.int32)))
        off += n
    return Workload("worked_example_identity", 4, 2, 64, 8, reqs, off)


def mha7b_steps(seed: int = 2, include_tail: bool = False) -> List[Workload]:
    """7B-like MHA layer (H 32, D 128), budget 512: 64 decodes + a 448-token chunk.

    The 4096-token prompt sits at prefix offsets 0, 448, ..., 3584 (nine steps);
    ``include_tail`` adds the final 64-token step at offset 4032.
    """
    rng = np.random.default_rng(seed)
    dec_c = rng.integers(512, 4096, size=64, endpoint=True)
    offsets = [448 * k for k in range(9)] + ([4032] if include_tail else [])
    # one pool shared by all steps: the prompt owns 4096 tokens of pages
    states = [(int(c), 0) for c in dec_c] + [(0, 4096)]
    base, total = assign_pages(states, rng, [int(c) + 1 for c in dec_c] + [4096])
    out = []
    for off in offsets:
        reqs = [Request(r.cached_len, r.remaining, r.block_table) for r in base[:-1]]
        reqs.append(Request(off, 4096 - off, base[-1].block_table))
        out.append(Workload(f"mha7b_b512_off{off}", 32, 32, 128, 512, reqs, total, seed=seed))
    return out


def mha13b(seed: int = 3) -> Workload:
    """13B-like MHA layer (H 40, D 128), budget 2048: 128 decodes at c = 2048 + a 1920 chunk at 2048."""
    rng = np.random.default_rng(seed)
    states = [(2048, 0)] * 128 + [(2048, 1920)]
    reqs, total = assign_pages(states, rng)
    return Workload("mha13b_b2048", 40, 40, 128, 2048, reqs, total, seed=seed)


def gqa8b(seed: int = 4) -> Workload:
    """8B-like GQA layer (H_q 32, H_kv 8, D 128), budget 8192.

    256 decodes with c ~ lognormal(median 1500, sigma 1) clamped to [1, 16384],
    a whole 3968-token prompt at c = 0 and a 3968-token chunk at c = 6000.
    """
    rng = np.random.default_rng(seed)
    ctx = np.clip(np.round(rng.lognormal(math.log(1500.0), 1.0, size=256)), 1, 16384).astype(int)
    states = [(int(c), 0) for c in ctx] + [(0, 3968), (6000, 3968)]
    reqs, total = assign_pages(states, rng)
    return Workload("gqa8b_b8192", 32, 8, 128, 8192, reqs, total, seed=seed)


def long_bimodal(seed: int = 5) -> Workload:
    """Long-context bimodal GQA layer (H_q 32, H_kv 8, D 128), budget 4608.

    The last 4096-token chunk of a 32768-token prompt (c = 28672) plus 512
    decodes: 461 with c ~ U[200, 800] and 51 with c ~ U[65536, 131072].
    """
    rng = np.random.default_rng(seed)
    short = rng.integers(200, 800, size=461, endpoint=True)
    long_ = rng.integers(65536, 131072, size=51, endpoint=True)
    ctx = np.concatenate([short, long_])
    rng.shuffle(ctx)
    states = [(int(c), 0) for c in ctx] + [(28672, 4096)]
    reqs, total = assign_pages(states, rng)
    return Workload("long_bimodal_b4608", 32, 8, 128, 4608, reqs, total, seed=seed)


def small_mixed(seed: int = 11, H_q: int = 8, H_kv: int = 2, D: int = 128,
                dec_ctx: Sequence[int] = (0, 1, 15, 16, 17, 130, 300, 777),
                prompts: Sequence[tuple] = ((0, 130), (300, 200), (16, 5)),
                budget: Optional[int] = None, max_chunk: int = 0) -> Workload:
    """A small mixed batch spanning several 128-key tiles with ragged tails.

    Default: 8 decodes (including c = 0 and page-boundary contexts) and three
    prompts: a 130-token whole prompt, a 200-token chunk at offset 300 and a
    5-token tail chunk at offset 16.
    """
    rng = np.random.default_rng(seed)
    states = [(int(c), 0) for c in dec_ctx] + [(int(c), int(r)) for c, r in prompts]
    reqs, total = assign_pages(states, rng)
    if budget is None:
        budget = len(dec_ctx) + sum(r for _, r in prompts)
    return Workload(f"small_mixed_s{seed}", H_q, H_kv, D, budget, reqs, total, max_chunk, seed=seed)


CONFIGS = {
    "worked_example_b8": worked_example,
    "mha7b_b512": mha7b_steps,
    "mha13b_b2048": mha13b,
    "gqa8b_b8192": gqa8b,
    "long_bimodal_b4608": long_bimodal,
}


# --------------------------------------------------------------------------- tensors

@dataclasses.dataclass
class Arrival:
    """A multi-round scenario: running decodes, then one long prompt arrives.

    decode_ctx     cached prompt lengths of the running decodes (admitted fully cached)
    decode_new     tokens each decode generates (long enough to outlast the run)
    prompt_len     the long prompt that arrives at round ``arrival_round``
    """
    name: str
    H_q: int
    H_kv: int
    D: int
    decode_ctx: List[int]
    decode_new: int
    prompt_len: int
    prompt_new: int
    arrival_round: int
    tail_rounds: int


def long_prompt_arrival(seed: int = 2, prompt_len: int = 16384) -> Arrival:
    """7B-like MHA layer (H 32, D 128): 64 decodes with c ~ U[512, 4096] are streaming
    when a 16384-token prompt arrives at round 16 (the moment a long prompt lands)."""
    rng = np.random.default_rng(seed)
    ctx = [int(c) for c in rng.integers(512, 4096, size=64, endpoint=True)]
    return Arrival("mha7b_arrival16k", 32, 32, 128, ctx, 240, prompt_len, 8, 16, 16)


def _torch():
    import torch  # local import: the oracle-only tests do not need torch at import time
    return torch


def step_tensors(wl: Workload, n_tokens: int, seed: int, device="cpu"):
    """q [n, H_q, D], k and v [n, H_kv, D] for the step's new tokens: bf16 N(0, 1)."""
    torch = _torch()
    g = torch.Generator(device=device).manual_seed(int(seed))
    n = max(int(n_tokens), 0)
    shape_q = (n, wl.H_q, wl.D)
    shape_kv = (n, wl.H_kv, wl.D)
    q = torch.randn(shape_q, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    k = torch.randn(shape_kv, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn(shape_kv, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    return q, k, v


def kv_pool(wl: Workload, seed: int, device="cpu"):
    """K and V page pools [num_pages, H_kv, 16, D], bf16 N(0, 1) (cached prefixes)."""
    torch = _torch()
    g = torch.Generator(device=device).manual_seed(int(seed) + 1000003)
    shape = (wl.num_pages, wl.H_kv, wl.page_size, wl.D)
    kc = torch.empty(shape, device=device, dtype=torch.bfloat16)
    vc = torch.empty(shape, device=device, dtype=torch.bfloat16)
    # fill in slabs to bound the fp32 temporary on large pools
    slab = max(1, (1 << 26) // (wl.H_kv * wl.page_size * wl.D))
    for dst in (kc, vc):
        for p0 in range(0, wl.num_pages, slab):
            p1 = min(wl.num_pages, p0 + slab)
            dst[p0:p1] = torch.randn((p1 - p0,) + shape[1:], generator=g, device=device,
                                     dtype=torch.float32).to(torch.bfloat16)
    return kc, vc


def bf16_bits(t) -> np.ndarray:
    """bf16 torch tensor -> numpy uint16 bit patterns (on the host)."""
    torch = _torch()
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
