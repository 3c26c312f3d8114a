"""Oracle for the attention-scored KV decode path: a plain, slow float64 CPU statement.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import or execute anything in
this package.  The product path (the C-ABI library and its Python binding) never
imports it, and this package imports nothing from the product path: the two share
no code, no tables and no helpers.

What it computes, each piece citing the page passage it follows:

* ``e4m3``       - the E4M3 value table and the per-position quantiser
                   (Flash-MoE "Context Optimization", FP8 KV Cache > How It Works).
* ``attention``  - masked decode attention with an explicit softmax, and the two
                   per-step masses (token: sum over heads; block: max over heads of
                   the in-block mass) ("Context views at marginal cost", Tier 1 and
                   Fact 3; "Per-Head Attention as a Scoring Signal", Fix: score per
                   head, place per block; "Context Optimization", H2O > How It Works).
* ``cache``      - the cache bookkeeping: append log with absolute positions, window /
                   H2O residency, next_position, cumulative + EMA score tables and
                   block selection ("Context Optimization", Sliding Window Attention
                   and H2O KV Cache Eviction; "LLM mechanics III", sections 1, 3, 5).
* ``slot_cache`` - the incremental W-slot cache of "LLM mechanics III" (slots, absolute
                   positions and processed count kept apart), used to pin the window
                   bookkeeping against a full sliding-mask recompute.
* ``selection``  - sort-based top-k with ties to the lower block id, and the H2O
                   protected regions.
* ``snapkv``     - SnapKV prefill scoring: observation-window votes, max-pooled with
                   kernel 7 ("Context views at marginal cost", per-system reductions).
* ``memory``     - the KV memory arithmetic ("Context Optimization", Memory Budget
                   Calculator).

Parity status per function is listed in each module header.
"""

from . import e4m3, attention, selection, memory, slot_cache, snapkv, cache  # noqa: F401
from .cache import OracleKV  # noqa: F401
