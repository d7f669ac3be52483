"""Oracle: a multi-round driver over a page pool with full-input admission.

Sources: "Splitting Prefill From Decode Inside a Step", "The arithmetic of
chunk boundaries" -- a sequence's cache grows chunk by chunk, and its
allocation must be reserved before the first chunk, or it fails part way
through its prompt, which is worse than failing at admission; "Chunked
Prefill 的 Token 预算" (zwjcode.cn), section 11 -- admission checks the
complete input length against the KV capacity (scheduler_reserve_full_isl),
and section 08 -- each round schedules, runs the step, then commits KV and
request progress together; "Chunked Prefill: Ending the Great Stall",
section 05 -- the per-request state is its cached length and chunk offset.

Readings where the pages are silent:
* a request of prompt_len tokens, cached_len of them already in the cache,
  asking for max_new_tokens, reserves ceil((prompt_len + max_new_tokens) / 16)
  pages at admission, or is refused;
* pages come from a last-in-first-out free list that starts as
  [num_pages - 1, ..., 1, 0] and pops from the end, so the first request gets
  pages 0, 1, 2, ...; a finished request pushes its pages back in block-table
  order;
* the last prefill chunk yields the first generated token; each decode round
  yields one more; a request finishes when it has max_new_tokens tokens.
  A request admitted with its whole prompt cached has generated one token
  (it is a running decode), so it must ask for at least two.
"""
from __future__ import annotations

import dataclasses
from typing import List

import numpy as np

from .schedule import DECODE_FIRST, batch_metadata, schedule


class AdmissionError(ValueError):
    """The pool cannot hold the request's full input plus its new tokens."""


@dataclasses.dataclass
class Live:
    rid: int
    c: int
    rem: int
    gen: int
    max_new: int
    pages: np.ndarray


class Engine:
    def __init__(self, num_pages: int, token_budget: int, max_chunk: int = 0, policy: int = DECODE_FIRST,
                 min_chunk: int = 0, prefill_quota: int = 0, decode_share: int = 500, page_size: int = 16):
        self.page = page_size
        self.num_pages = num_pages
        self.free: List[int] = list(range(num_pages - 1, -1, -1))
        self.cfg = dict(max_chunk=max_chunk, policy=policy, min_chunk=min_chunk, prefill_quota=prefill_quota,
                        decode_share=decode_share)
        self.budget = token_budget
        self.live: List[Live] = []
        self.next_id = 0
        self.planned = None

    def add_request(self, prompt_len: int, max_new_tokens: int, cached_len: int = 0) -> int:
        if prompt_len < 1 or max_new_tokens < 1 or not 0 <= cached_len <= prompt_len or \
                (cached_len == prompt_len and max_new_tokens < 2):
            raise ValueError("bad request lengths")
        need = -(-(prompt_len + max_new_tokens) // self.page)
        if need > len(self.free):
            raise AdmissionError(f"needs {need} pages, {len(self.free)} free")
        pages = np.array([self.free.pop() for _ in range(need)], dtype=np.int32)
        rem = prompt_len - cached_len
        rid = self.next_id
        self.next_id += 1
        self.live.append(Live(rid, cached_len, rem, 1 if rem == 0 else 0, max_new_tokens, pages))
        return rid

    def plan(self):
        """Pack the next round over the live requests (arrival order)."""
        states = [(r.c, r.rem) for r in self.live]
        rows, unused = schedule(states, self.budget, self.cfg["max_chunk"], self.cfg["policy"],
                                self.cfg["min_chunk"], self.cfg["prefill_quota"], self.cfg["decode_share"])
        n_dec = sum(1 for i, _, _ in rows if states[i][1] == 0)
        meta = batch_metadata(rows, [r.pages for r in self.live], len(self.live), num_decodes=n_dec,
                              page_size=self.page)
        meta["unused_tokens"] = unused
        meta["row_request_id"] = np.array([self.live[i].rid for i, _, _ in rows], dtype=np.int32)
        self.planned = rows
        return meta

    def commit(self) -> List[int]:
        """Advance every planned row; finished requests free their pages.  Returns their ids."""
        if self.planned is None:
            raise ValueError("commit without plan")
        for i, c, d in self.planned:
            r = self.live[i]
            if r.rem == 0:
                r.c += 1
                r.gen += 1
            else:
                r.c += d
                r.rem -= d
                if r.rem == 0:
                    r.gen = 1
        self.planned = None
        finished = [r for r in self.live if r.gen >= r.max_new]
        for r in finished:
            self.free.extend(int(p) for p in r.pages)
        self.live = [r for r in self.live if r.gen < r.max_new]
        return [r.rid for r in finished]
