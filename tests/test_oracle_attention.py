"""Pins of the oracle's decode attention and per-step masses.

Pinned to: torch.nn.functional.scaled_dot_product_attention in float64 (a library
routine the oracle does not use) for no window / a window covering everything; the
window-1 closed form (the output is the current token's value, every head puts all
of its mass on it); softmax rows summing to one; block-mass bounds.
"""
import numpy as np
import pytest
import torch

from oracle import attention
from oracle.cache import OracleKV


def _sdpa(q, k, v):
    """Reference: one query per head, GQA by repeating KV heads, float64."""
    hq, d = q.shape
    n, hkv, _ = k.shape
    g = hq // hkv
    qt = torch.from_numpy(q)[:, None, :]                       # [Hq, 1, D]
    kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(g, 0)   # [Hq, n, D]
    vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(g, 0)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)
    return out[:, 0, :].numpy()


@pytest.mark.parametrize("hq,hkv,d,n", [(4, 2, 16, 1), (4, 2, 16, 37), (32, 4, 128, 300), (8, 8, 64, 5)])
def test_matches_sdpa(hq, hkv, d, n):
    rng = np.random.default_rng(hq * 1000 + n)
    q = rng.normal(size=(hq, d))
    k = rng.normal(size=(n, hkv, d))
    v = rng.normal(size=(n, hkv, d))
    out, w = attention.decode_attention(q, k, v)
    assert np.max(np.abs(out - _sdpa(q, k, v))) < 1e-12
    assert np.max(np.abs(w.sum(axis=1) - 1.0)) < 1e-12


def test_gqa_mapping_head_to_kv_head():
    # only KV head 1 carries signal: query heads 2,3 (group 1 of G=2) must see it
    rng = np.random.default_rng(1)
    q = rng.normal(size=(4, 8))
    k = rng.normal(size=(6, 2, 8))
    v = np.zeros((6, 2, 8))
    v[:, 1, :] = 1.0
    out, _ = attention.decode_attention(q, k, v)
    assert np.allclose(out[:2], 0.0) and np.allclose(out[2:], 1.0)


def test_empty_cache_rejected():
    with pytest.raises(ValueError):
        attention.decode_attention(np.zeros((4, 8)), np.zeros((0, 2, 8)), np.zeros((0, 2, 8)))


def test_window_one_closed_form():
    """W = 1: each step attends only the token just written."""
    o = OracleKV(num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=16, num_seqs=1,
                 max_positions=20, kv_format="f32", window=1)
    rng = np.random.default_rng(2)
    for t in range(20):
        for l in range(2):
            k = rng.normal(size=(1, 2, 16)).astype(np.float32).astype(np.float64)
            v = rng.normal(size=(1, 2, 16)).astype(np.float32).astype(np.float64)
            o.append(l, 0, k, v)
            out, w, pos = o.attend(l, 0, rng.normal(size=(4, 16)))
            assert list(pos) == [t]
            assert np.array_equal(out, np.repeat(v[0], 2, axis=0))
            _, tau = o.token_mass(l, 0)
            assert tau[0] == 4.0                     # every head's whole mass
            assert o.block_mass(l, 0) == {t // 16: 1.0}
        o.accumulate()


def test_block_mass_bounds_and_sum():
    rng = np.random.default_rng(4)
    w = rng.dirichlet(np.ones(50), size=6)           # 6 heads, rows sum to 1
    pos = np.arange(100, 150)
    bm = attention.block_step_mass(w, pos, 16)
    assert set(bm) == {6, 7, 8, 9}
    vals = np.array(list(bm.values()))
    assert np.all(vals >= 0) and np.all(vals <= 1 + 1e-15)
    assert vals.sum() >= 1 - 1e-12                    # max over heads >= any one head's share
    # hand check of one block: max over heads of in-block sums
    sel = (pos // 16) == 7
    assert bm[7] == np.max(w[:, sel].sum(axis=1))


def test_token_mass_sums_to_heads():
    rng = np.random.default_rng(6)
    q = rng.normal(size=(8, 32))
    k = rng.normal(size=(40, 2, 32))
    _, w = attention.decode_attention(q, k, k)
    assert abs(attention.token_step_mass(w).sum() - 8.0) < 1e-12


def test_block_mass_brute_force_any_order():
    """Block masses equal a per-block loop written out by hand, for positions in any
    order and blocks with gaps (an H2O residency)."""
    rng = np.random.default_rng(8)
    pos = np.concatenate([np.arange(0, 20), np.arange(64, 90), np.arange(200, 205)])
    perm = rng.permutation(len(pos))
    w = rng.dirichlet(np.ones(len(pos)), size=5)
    bm = attention.block_step_mass(w[:, perm], pos[perm], 16)
    assert set(bm) == {0, 1, 4, 5, 12}
    for k in bm:
        best = 0.0
        for h in range(5):
            s = 0.0
            for j in range(len(pos)):
                if pos[j] // 16 == k:
                    s += w[h, j]
            best = max(best, s)
        assert abs(bm[k] - best) <= 1e-15
