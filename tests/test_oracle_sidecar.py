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
