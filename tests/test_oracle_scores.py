"""Pins of the oracle's score tables (cumulative and EMA, token and block level).

Pinned to: the cumulative equals the sum of the logged per-step masses; the EMA equals
its closed form (1-d) * sum_t d^(T-t) x_t (a different formula from the recursive
update the oracle runs); per step the token scores add up to layers x query heads
(each softmax row sums to one); block scores lie in [0, 1] per layer and their sum per
step is at least 1; tokens that leave the window keep their cumulative and decay.
"""
import numpy as np
import pytest

from oracle.cache import OracleKV


def _run(window, steps=40, prefill=21, seed=0, d=0.9):
    rng = np.random.default_rng(seed)
    L, hq, hkv, D = 2, 4, 2, 16
    o = OracleKV(num_layers=L, num_q_heads=hq, num_kv_heads=hkv, head_dim=D, num_seqs=2,
                 max_positions=prefill + steps, kv_format="f32", window=window, ema_decay=d)
    for b in range(2):
        for l in range(L):
            o.append(l, b, rng.normal(size=(prefill, hkv, D)), rng.normal(size=(prefill, hkv, D)))
    logs = []
    for t in range(steps):
        for b in range(2):
            for l in range(L):
                o.append(l, b, rng.normal(size=(1, hkv, D)), rng.normal(size=(1, hkv, D)))
                o.attend(l, b, rng.normal(size=(hq, D)) * 2)
        logs.append(o.accumulate())
    return o, logs


@pytest.mark.parametrize("window", [0, 5, 16, 24])
def test_cumulative_is_sum_of_step_masses(window):
    o, logs = _run(window)
    for b in range(2):
        n = int(o.next_position[0, b])
        c = np.zeros(n)
        cb = np.zeros(-(-n // 16))
        for step in logs:
            x, y = step[b]
            c[:len(x)] += x
            cb[:len(y)] += y
        assert np.max(np.abs(o.scores[b].c_tok[:n] - c)) < 1e-12
        assert np.max(np.abs(o.scores[b].c_blk[:len(cb)] - cb)) < 1e-12


@pytest.mark.parametrize("window", [0, 7])
def test_ema_closed_form(window):
    d = 0.9
    o, logs = _run(window, d=d)
    T = len(logs)
    for b in range(2):
        n = int(o.next_position[0, b])
        e = np.zeros(n)
        for t, step in enumerate(logs, start=1):
            x, _ = step[b]
            full = np.zeros(n)
            full[:len(x)] = x
            e += (1 - d) * d ** (T - t) * full
        assert np.max(np.abs(o.scores[b].e_tok[:n] - e)) < 1e-12


def test_token_scores_sum_to_layers_times_heads():
    o, logs = _run(6)
    for step in logs:
        for b in range(2):
            x, y = step[b]
            assert abs(x.sum() - 2 * 4) < 1e-12
            assert np.all(y >= 0) and np.all(y <= 1 + 1e-15)
            assert y.sum() >= 1 - 1e-12


def test_left_window_entries_decay_and_keep_cumulative():
    o, logs = _run(4, steps=30)
    for b in range(2):
        # position 0 left the window long ago: its cumulative is frozen at what
        # prefill-era steps gave it (0: it was never resident during decode)
        assert o.scores[b].c_tok[0] == 0.0
        # the position that left the window most recently still has mass, decaying
        nxt = int(o.next_position[0, b])
        p_old = nxt - 5
        assert o.scores[b].c_tok[p_old] > 0
        x_last = logs[-1][b][0][p_old]
        assert x_last == 0.0


def test_accumulate_requires_every_layer():
    o = OracleKV(num_layers=2, num_q_heads=2, num_kv_heads=1, head_dim=4, num_seqs=1,
                 max_positions=4, kv_format="f32")
    for l in range(2):
        o.append(l, 0, np.ones((1, 1, 4)), np.ones((1, 1, 4)))
    o.attend(0, 0, np.ones((2, 4)))
    with pytest.raises(ValueError):
        o.accumulate()
