"""fp64 CPU oracle for the mixed-batch attention step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, calls or links anything here, and this
package imports nothing from the product path: the two share only the seeded
input generator ``workloads.py``.

Each function follows the pages on chunked prefill as plainly as possible,
in the pages' order and notation:

* ``schedule``  -- decode-first token-budget packing ("Chunked Prefill 的 Token
  预算", zwjcode.cn, sections 03-05 and 08; "Chunked Prefill: Ending the Great
  Stall", sections 03-04; "Splitting Prefill From Decode Inside a Step",
  "Chunked prefill as a rate control") and the per-step metadata of section 06
  of the zwjcode page;
* ``rope``      -- rotary embedding at absolute positions (zwjcode section 07)
  and the paged K/V append through ``slot_mapping`` (zwjcode section 06);
* ``attention`` -- causal attention of every query at absolute position p over
  keys 0..p read through the block table (zwjcode sections 02 and 07);
* ``engine``    -- a multi-round driver over a page pool that reserves a
  request's full input plus its new tokens at admission (zwjcode section 11;
  "Splitting Prefill From Decode Inside a Step").

Pins (tests/test_oracle.py) tie every function to values the pages print,
closed forms, invariants and library routines.  No function here is
"parity unpinned".
"""
from .schedule import (BudgetError, NoPagesError, schedule, batch_metadata, commit_round, DECODE_FIRST,
                       PREFILL_FIRST, FAIR_SHARE)
from .rope import bf16_to_f64, f32_to_bf16_bits, rope_tables, rope_rotate, kv_append
from .attention import attention_rows, attention_all
from .engine import AdmissionError, Engine

__all__ = [
    "BudgetError", "NoPagesError", "schedule", "batch_metadata", "commit_round", "DECODE_FIRST",
    "PREFILL_FIRST", "FAIR_SHARE",
    "bf16_to_f64", "f32_to_bf16_bits", "rope_tables", "rope_rotate", "kv_append",
    "attention_rows", "attention_all", "AdmissionError", "Engine",
]
