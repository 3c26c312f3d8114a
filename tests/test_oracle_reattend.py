"""Pins of the oracle's Tier-2 re-attend ("Context views at marginal cost", Tier 2 and
Fact 3: a new query attends over the cached K and V of a selected subset only).

- Listing every resident block gives the full attention, exactly.
- A subset gives the full attention with every other entry masked out of the softmax
  (logits set to -inf): a different formulation from the oracle's gather.
- A single listed entry gives that entry's V for every head of its group.
"""
import numpy as np
import pytest

from oracle.cache import OracleKV


def _cache(window=0, n=70, seed=3):
    rng = np.random.default_rng(seed)
    o = OracleKV(num_layers=1, num_q_heads=4, num_kv_heads=2, head_dim=8, num_seqs=1, max_positions=n + 4,
                 kv_format="f32", window=window)
    k = rng.standard_normal((n, 2, 8))
    v = rng.standard_normal((n, 2, 8))
    o.append(0, 0, k, v)
    return o, rng


def _masked_reference(o, q, blocks):
    """Full attention over the resident entries, logits of unlisted entries -inf."""
    pos = o.resident_positions(0, 0)
    k, v = o.stored_kv(0, 0, pos)
    g = q.shape[0] // k.shape[1]
    out = np.zeros_like(q)
    inside = np.isin(pos // 16, np.asarray(blocks))
    for h in range(q.shape[0]):
        s = k[:, h // g, :] @ q[h] / np.sqrt(q.shape[1])
        s = np.where(inside, s, -np.inf)
        a = np.exp(s - s[inside].max())
        a /= a.sum()
        out[h] = a @ v[:, h // g, :]
    return out


@pytest.mark.parametrize("window", [0, 40])
def test_all_blocks_is_full_attention(window):
    o, rng = _cache(window=window)
    q = rng.standard_normal((4, 8))
    full, _, pos_full = o.attend(0, 0, q)
    got, _, pos = o.attend_blocks(0, 0, q, o.resident_block_ids(0))
    assert np.array_equal(pos, pos_full)
    assert np.allclose(got, full, rtol=0, atol=1e-15)


@pytest.mark.parametrize("blocks", [[0], [1, 3], [0, 2, 4], [4]])
def test_subset_is_masked_full_attention(blocks):
    o, rng = _cache()
    q = rng.standard_normal((4, 8))
    got, w, pos = o.attend_blocks(0, 0, q, blocks)
    assert set(int(p) // 16 for p in pos) == set(blocks)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12)
    assert np.allclose(got, _masked_reference(o, q, blocks), rtol=0, atol=1e-12)


def test_single_entry_returns_its_value():
    # 65 entries: block 4 holds only position 64
    o, rng = _cache(n=65)
    q = rng.standard_normal((4, 8))
    got, w, pos = o.attend_blocks(0, 0, q, [4])
    assert list(pos) == [64]
    _, v = o.stored_kv(0, 0, np.array([64]))
    for h in range(4):
        assert np.allclose(got[h], v[0, h // 2], rtol=0, atol=1e-15)
