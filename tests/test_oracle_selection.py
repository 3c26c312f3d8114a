"""Pins of the oracle's block selection.

Pinned to: brute force over every k-subset of up to 12 blocks (the kept set maximises
the score sum, ties broken towards lower ids lexicographically); H2O protected
regions worked by hand ("Context Optimization", H2O > The Algorithm: sinks = first 4
tokens, recent = last quarter of the budget)."""
import itertools

import numpy as np
import pytest

from oracle import selection
from oracle.cache import OracleKV


def _brute(cands, scores, k):
    """Best k-subset: highest multiset of scores, then lowest ids (sorted id tuple)."""
    best = None
    for sub in itertools.combinations(sorted(cands), min(k, len(cands))):
        key = (sorted((scores[c] for c in sub), reverse=True), [-c for c in sub])
        # compare: larger score profile first, then lexicographically smaller ids
        if best is None or key[0] > best[0][0] or (key[0] == best[0][0] and list(sub) < best[1]):
            best = (key, list(sub))
    return best[1]


@pytest.mark.parametrize("seed", range(40))
def test_top_k_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 13))
    cands = sorted(rng.choice(100, size=n, replace=False).tolist())
    # few distinct values so that ties are frequent
    scores = {c: float(rng.integers(0, 4)) / 4 for c in cands}
    for k in range(0, n + 2):
        assert selection.top_k_blocks(cands, scores, k) == _brute(cands, scores, k)


def test_ties_prefer_lower_block_id():
    assert selection.top_k_blocks([5, 2, 9], {5: 1.0, 2: 1.0, 9: 1.0}, 2) == [2, 5]


def test_h2o_protection_by_hand():
    # 40 blocks resident, next position 640 (blocks 0..39), budget 10 blocks (160 tokens),
    # recent = ceil(0.25*160) = 40 tokens = positions 600..639 = blocks 37, 38, 39,
    # sinks = first 4 tokens = block 0; room for 6 heavy hitters
    cands = list(range(40))
    scores = {c: float(c % 7) for c in cands}
    keep = selection.h2o_keep(cands, scores, 10, 640, 4, selection.recent_token_count(160, 0.25), 16)
    assert len(keep) == 10
    assert {0, 37, 38, 39} <= set(keep)
    heavy = [c for c in keep if c not in (0, 37, 38, 39)]
    assert sorted(heavy) == [5, 6, 13, 20, 27, 34]


def test_h2o_under_budget_keeps_all():
    assert selection.h2o_keep([1, 2, 3], {1: 0, 2: 0, 3: 0}, 5, 60, 4, 8) == [1, 2, 3]


def test_recent_region_partial_tail_block():
    # next = 650 (block 40 partially filled), recent 40 tokens = 610..649 -> blocks 38, 39, 40
    assert selection.protected_blocks(range(41), 650, 4, 40) == [0, 38, 39, 40]


def test_oracle_h2o_eviction_keeps_budget():
    rng = np.random.default_rng(9)
    o = OracleKV(num_layers=1, num_q_heads=2, num_kv_heads=1, head_dim=8, num_seqs=1,
                 max_positions=400, kv_format="f32", h2o_budget_tokens=64)
    o.append(0, 0, rng.normal(size=(300, 1, 8)), rng.normal(size=(300, 1, 8)))
    for t in range(40):
        o.append(0, 0, rng.normal(size=(1, 1, 8)), rng.normal(size=(1, 1, 8)))
        o.attend(0, 0, rng.normal(size=(2, 8)))
        o.accumulate()
        keep = o.select(0, o.h2o_budget_blocks, protect=True, apply=True)
        assert len(keep) <= 4 and 0 in keep
        nxt = int(o.next_position[0, 0])
        assert (nxt - 1) // 16 in keep                  # the current block is recent
        assert o.resident_block_ids(0) == keep
