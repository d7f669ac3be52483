"""Oracle: decode-first token-budget packing and the per-step metadata.

Sources (the pages on chunked prefill):

* "Chunked Prefill 的 Token 预算" (zwjcode.cn), section 04: one round obeys
  |D_t| + sum over chunks |c| <= B_tok; section 05: more decodes than the
  budget is an error, prompts are served first-come-first-served, each takes
  the smaller of what it still needs and what is left, and packing stops once
  nothing is left; section 08: running decodes are placed first (one token
  each), then the leftover budget is filled with prefill chunks, then the step
  runs and KV plus request progress are committed together.
* "Chunked Prefill: Ending the Great Stall", sections 03-04: decode-maximal
  rule -- every running decode first, then the largest chunk that fits the
  leftover for each waiting prefill in queue order.
* "Splitting Prefill From Decode Inside a Step", "Chunked prefill as a rate
  control": an optional per-prefill chunk size also caps the take.
* "Prefill head-of-line blocking" (sference.com), "The fix": the per-request
  cap (--long-prefill-token-threshold) on tokens one prefill may take per round.
* zwjcode section 06: the metadata of a chunk covering positions [c, c+d) --
  positions c..c+d-1 (never reset to 0), one physical slot per new token,
  ceil((c+d)/B) block-table entries, and context_len = c + d after the round.

Readings where the pages are silent: rows are all decodes in input order, then
chunks in input (FCFS) order; block_tables rows are padded with -1 to the
largest row's page count; a slot is page_id * page_size + pos % page_size.
"""
from __future__ import annotations

from typing import Sequence

import numpy as np


class BudgetError(ValueError):
    """More running decodes than the round's token budget."""


class NoPagesError(ValueError):
    """A request's block table cannot address the tokens scheduled for it."""


DECODE_FIRST, PREFILL_FIRST, FAIR_SHARE = 0, 1, 2


def schedule(states: Sequence[tuple], token_budget: int, max_chunk: int = 0, policy: int = DECODE_FIRST,
             min_chunk: int = 0, prefill_quota: int = 0, decode_share: int = 500):
    """Pack one round.

    ``states[i] = (cached_len, remaining)``; remaining == 0 marks a running
    decode.  Returns ``(rows, unused)`` where rows is a list of
    ``(request_index, c, d)`` -- decode rows first, in input order, then
    chunk rows in input order -- and unused the budget left over.

    Policies ("Splitting Prefill From Decode Inside a Step", "Choosing the
    priority order"):
      DECODE_FIRST   every running decode, then prompts in arrival order take
                     what is left (zwjcode sections 05 and 08);
      PREFILL_FIRST  prompts take the budget first, decodes whatever remains;
      FAIR_SHARE     decodes may use decode_share / 1000 of the budget and
                     prompts the rest; what one class leaves unused goes to
                     the other.
    Per-prompt limits ("Prefill head-of-line blocking", "The fix" and "What
    comes next"): max_chunk caps one prompt's take per round (a ceiling);
    min_chunk is a floor -- every waiting prompt first gets up to min_chunk
    tokens in arrival order, then the leftover is handed out in arrival order.
    prefill_quota (zwjcode section 08, "reserve a prefill quota"; section 16,
    exercise 3): while prompts wait, decodes use at most budget - min(quota,
    what the prompts can take) tokens and the others wait for a later round.  Without a quota, DECODE_FIRST
    treats more decodes than the budget as an error (zwjcode section 05);
    the other policies defer them.
    """
    decodes = [i for i, (_, rem) in enumerate(states) if rem == 0]
    prompts = [i for i, (_, rem) in enumerate(states) if rem > 0]
    B = token_budget

    def prompt_takes(allowance):
        """Tokens per prompt (arrival order) out of `allowance`, with floor and ceiling."""
        take = {i: 0 for i in prompts}
        left = allowance
        limit = {i: states[i][1] if max_chunk <= 0 else min(states[i][1], max_chunk) for i in prompts}
        if min_chunk > 0:  # pass 1: the floor
            for i in prompts:
                if left == 0:
                    break
                t = min(limit[i], min_chunk, left)
                take[i] += t
                left -= t
        for i in prompts:  # the leftover, in arrival order
            if left == 0:
                break
            t = min(limit[i] - take[i], left)
            take[i] += t
            left -= t
        return take, allowance - left

    if policy == DECODE_FIRST:
        # the quota reserves only what the waiting prompts can use this round
        demand = sum(states[i][1] if max_chunk <= 0 else min(states[i][1], max_chunk) for i in prompts)
        dec_cap = B - min(prefill_quota, demand) if prefill_quota > 0 else B
        if prefill_quota <= 0 and len(decodes) > B:
            raise BudgetError(f"{len(decodes)} decodes exceed the token budget {B}")
        n_dec = min(len(decodes), max(dec_cap, 0))
        take, used_p = prompt_takes(B - n_dec)
    elif policy == PREFILL_FIRST:
        take, used_p = prompt_takes(B)
        n_dec = min(len(decodes), B - used_p)
    elif policy == FAIR_SHARE:
        dec_allow = (B * decode_share) // 1000
        n_dec = min(len(decodes), dec_allow)
        take, used_p = prompt_takes(B - n_dec)
        n_dec = min(len(decodes), B - used_p)  # prompts left some over: decodes may take it
    else:
        raise ValueError(f"unknown policy {policy}")
    rows = [(i, int(states[i][0]), 1) for i in decodes[:n_dec]]
    rows += [(i, int(states[i][0]), take[i]) for i in prompts if take[i] > 0]
    used = n_dec + sum(take.values())
    return rows, B - used


def batch_metadata(rows, block_tables: Sequence[np.ndarray], n_requests: int,
                   num_decodes: int = 0, page_size: int = 16):
    """Varlen metadata of one packed round, as plain int32 arrays.

    ``num_decodes`` is the number of leading rows that are running decodes.
    """
    S = len(rows)
    cu = np.zeros(S + 1, dtype=np.int32)
    q_start = np.zeros(S, dtype=np.int32)
    ctx = np.zeros(S, dtype=np.int32)
    row_req = np.zeros(S, dtype=np.int32)
    num_sched = np.zeros(n_requests, dtype=np.int32)
    positions, slots = [], []
    n_pages_row = []
    for s, (i, c, d) in enumerate(rows):
        bt = block_tables[i]
        need = -(-(c + d) // page_size)
        if len(bt) < need:
            raise NoPagesError(f"request {i} needs {need} pages for context {c + d}, has {len(bt)}")
        cu[s + 1] = cu[s] + d
        q_start[s] = c
        ctx[s] = c + d
        row_req[s] = i
        num_sched[i] = d
        n_pages_row.append(need)
        for j in range(d):
            pos = c + j
            positions.append(pos)
            slots.append(int(bt[pos // page_size]) * page_size + pos % page_size)
    stride = max(n_pages_row) if n_pages_row else 0
    tables = np.full((S, stride), -1, dtype=np.int32)
    for s, (i, _, _) in enumerate(rows):
        tables[s, :n_pages_row[s]] = block_tables[i][:n_pages_row[s]]
    return {
        "cu_seqlens_q": cu,
        "q_start_pos": q_start,
        "context_lens": ctx,
        "positions": np.asarray(positions, dtype=np.int32),
        "slot_mapping": np.asarray(slots, dtype=np.int32),
        "block_tables": tables,
        "bt_stride": stride,
        "row_req": row_req,
        "num_scheduled": num_sched,
        "num_rows": S,
        "num_decodes": int(num_decodes),
        "num_tokens": int(cu[-1]),
    }


def commit_round(states: Sequence[tuple], rows):
    """The caller's commit after the step: progress advances by what ran.

    A decode advances one position; a chunk advances c by d and removes d
    tokens from the prompt, which starts decoding in the next round once
    nothing remains (zwjcode section 03, round 4).
    """
    new = [list(s) for s in states]
    for i, c, d in rows:
        if new[i][1] == 0:
            new[i][0] = c + 1
        else:
            new[i][0] = c + d
            new[i][1] -= d
    return [tuple(s) for s in new]
