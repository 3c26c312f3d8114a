"""Pins of the oracle's side-car views ("Context views at marginal cost", Tier 1: a
bounded per-span record, viewed by filtering the kept table).

- Threshold view: with theta just under the k-th best score (scores distinct), the
  filter keeps exactly the top k.  With theta = -1 it keeps every resident block.
- Trajectory ring: its newest column is t_blk.  The ring summed over its last n
  columns equals the growth of s_blk over those n steps, a different route through
  the tables.
- Layer profile: each row equals that layer's block mass summed over the logged
  steps.  It never exceeds the cumulative block score, which takes the max over
  layers every step.
"""
import numpy as np
import pytest

from oracle.cache import OracleKV


def _run(window=0, steps=24, prefill=45, seed=9, traj=8, layers=(0, 2)):
    rng = np.random.default_rng(seed)
    L, hq, hkv, D = 3, 4, 2, 16
    o = OracleKV(num_layers=L, num_q_heads=hq, num_kv_heads=hkv, head_dim=D, num_seqs=1,
                 max_positions=prefill + steps, kv_format="f32", window=window, traj_len=traj,
                 profile_layers=layers)
    for l in range(L):
        o.append(l, 0, rng.normal(size=(prefill, hkv, D)), rng.normal(size=(prefill, hkv, D)))
    hist, masses = [], []
    for t in range(steps):
        for l in range(L):
            o.append(l, 0, rng.normal(size=(1, hkv, D)), rng.normal(size=(1, hkv, D)))
            o.attend(l, 0, rng.normal(size=(hq, D)) * 2)
        masses.append({l: dict(o.block_mass(l, 0)) for l in range(L)})
        o.accumulate()
        hist.append(o.scores[0].s_blk.copy())
        yield o, hist, masses


def test_threshold_is_top_k_just_below_the_kth():
    for o, _, _ in _run():
        cand = o.resident_block_ids(0)
        c = o.scores[0].c_blk
        vals = sorted((c[b] for b in cand), reverse=True)
        for k in (1, 2, len(cand) // 2):
            theta = vals[k - 1] - 1e-12 if vals[k - 1] - 1e-12 > vals[k] else None
            if theta is None:
                continue
            assert o.filter_blocks(0, "cumulative", theta) == sorted(o.select(0, k))
        assert o.filter_blocks(0, "tova", -1.0) == cand


@pytest.mark.parametrize("window", [0, 30])
def test_trajectory_ring(window):
    for o, hist, _ in _run(window=window):
        sc = o.scores[0]
        tr = sc.trajectory()
        nb = len(sc.t_blk)
        assert np.array_equal(tr[:nb, -1], sc.t_blk[:nb])
        n = min(sc.traj_len, len(hist) - 1)
        if n:
            grown = hist[-1] - hist[-1 - n]
            assert np.allclose(tr[:, -n:].sum(axis=1)[:len(grown)], grown, rtol=0, atol=1e-12)


def test_layer_profiles():
    for o, _, masses in _run():
        sc = o.scores[0]
        for i, l in enumerate(sc.profile_layers):
            ref = np.zeros(sc.prof.shape[1])
            for step in masses:
                for k, m in step[l].items():
                    ref[k] += m
            assert np.allclose(sc.prof[i], ref, rtol=0, atol=1e-12)
            assert np.all(sc.prof[i] <= sc.c_blk + 1e-12)


def _head_run(L=2, hq=4, hkv=2, window=0, steps=20, prefill=37, heads=((0, 1), (1, 3)), seed=5):
    rng = np.random.default_rng(seed)
    D = 16
    o = OracleKV(num_layers=L, num_q_heads=hq, num_kv_heads=hkv, head_dim=D, num_seqs=1,
                 max_positions=prefill + steps, kv_format="f32", window=window, profile_heads=heads)
    for l in range(L):
        o.append(l, 0, rng.normal(size=(prefill, hkv, D)), rng.normal(size=(prefill, hkv, D)))
    for t in range(steps):
        for l in range(L):
            o.append(l, 0, rng.normal(size=(1, hkv, D)), rng.normal(size=(1, hkv, D)))
            o.attend(l, 0, rng.normal(size=(hq, D)) * 2)
        o.accumulate()
    return o


@pytest.mark.parametrize("window", [0, 21])
def test_head_profiles_hold_one_unit_of_weight_per_step(window):
    """A head's weights sum to one over the resident entries every step, so its
    profile summed over the blocks equals the number of steps; and a single head's
    in-block sum never exceeds the block mass (the max over heads and layers), so the
    profile stays under the cumulative block score."""
    o = _head_run(window=window)
    sc = o.scores[0]
    for i in range(len(sc.profile_heads)):
        assert abs(sc.hprof[i].sum() - sc.steps) <= 1e-12 * sc.steps
        assert np.all(sc.hprof[i] <= sc.c_blk + 1e-12)


def test_head_profile_of_the_only_head_is_the_cumulative_block_score():
    """With one layer and one query head the block mass is that head's in-block sum,
    so the head's profile is the cumulative block score itself."""
    o = _head_run(L=1, hq=1, hkv=1, heads=((0, 0),))
    sc = o.scores[0]
    assert np.array_equal(sc.hprof[0], sc.c_blk)
