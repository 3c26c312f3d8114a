"""Pins of the oracle's summed block scores and the selections that use them.

token_sum (H2O's accumulated score, "Context Optimization", H2O > How It Works, at
block granularity) and tova (the latest query's weight, "Context views at marginal
cost", per-system reductions), both summed over a block's entries:
- s_blk equals the sum of the token cumulative table over the block's positions;
- t_blk sums, over all blocks, to layers x query heads on every step (each softmax row
  sums to one), and is zero for blocks nothing attended in the latest step (left the
  window);
- keeping the top n-1 blocks by tova evicts exactly the argmin block, the highest id
  among equal minima (brute force);
- top-k by either score equals the brute-force best k-subset on tiny inputs.
"""
import itertools

import numpy as np
import pytest

from oracle.cache import OracleKV


def _run(window, steps=30, prefill=37, seed=5):
    rng = np.random.default_rng(seed)
    L, hq, hkv, D = 2, 4, 2, 16
    o = OracleKV(num_layers=L, num_q_heads=hq, num_kv_heads=hkv, head_dim=D, num_seqs=1,
                 max_positions=prefill + steps, kv_format="f32", window=window)
    for l in range(L):
        o.append(l, 0, rng.normal(size=(prefill, hkv, D)), rng.normal(size=(prefill, hkv, D)))
    for t in range(steps):
        for l in range(L):
            o.append(l, 0, rng.normal(size=(1, hkv, D)), rng.normal(size=(1, hkv, D)))
            o.attend(l, 0, rng.normal(size=(hq, D)) * 2)
        o.accumulate()
        yield o, L * hq


@pytest.mark.parametrize("window", [0, 20, 48])
def test_token_sum_is_block_sum_of_cumulative(window):
    for o, _ in _run(window):
        sc = o.scores[0]
        n = int(o.next_position[0, 0])
        for k in range(-(-n // 16)):
            assert abs(sc.s_blk[k] - sc.c_tok[16 * k:min(n, 16 * k + 16)].sum()) <= 1e-12


@pytest.mark.parametrize("window", [0, 20, 48])
def test_tova_sums_to_layers_times_heads_and_forgets_the_past(window):
    for o, lh in _run(window):
        sc = o.scores[0]
        n = int(o.next_position[0, 0])
        nb = -(-n // 16)
        assert abs(sc.t_blk[:nb].sum() - lh) <= 1e-9
        if window:
            lo = n - window
            for k in range(nb):
                if 16 * k + 16 <= lo:                # wholly out of the window
                    assert sc.t_blk[k] == 0.0


def test_tova_keeps_all_but_the_argmin():
    for o, _ in _run(0):
        cand = o.resident_block_ids(0)
        t = o.scores[0].t_blk
        keep = o.select(0, len(cand) - 1, score_kind="tova")
        lowest = min(t[c] for c in cand)
        evict = max(c for c in cand if t[c] == lowest)
        assert sorted(set(cand) - set(keep)) == [evict]


@pytest.mark.parametrize("kind", ["token_sum", "tova"])
def test_top_k_is_the_best_subset(kind):
    for o, _ in _run(0, steps=6, prefill=120):
        cand = o.resident_block_ids(0)
        table = o.scores[0].s_blk if kind == "token_sum" else o.scores[0].t_blk
        for k in (1, 3, len(cand) - 2):
            keep = o.select(0, k, score_kind=kind)
            best = max(itertools.combinations(cand, k), key=lambda sub: (sum(table[c] for c in sub),
                                                                        [-c for c in sub]))
            assert sorted(keep) == sorted(best)
