"""Pin of the window bookkeeping: incremental slot cache vs full sliding-mask recompute.

"LLM mechanics III", section 2 and section 5: a two-layer float64 network with 16-wide
layers and additive absolute sinusoidal positions; the incremental cache must match
the full recompute under the sliding mask to 1e-12 for windows 1, 4 and none, lengths
1, 2, 8, 17, seeds 7, 19, 41 (36 cases), with chunked input as a further axis; invalid
windows, token IDs and all-masked rows are rejected.  The full recompute here uses
torch.nn.functional.scaled_dot_product_attention with a boolean mask, a routine the
oracle does not use.  The oracle's decode cache (``OracleKV``) is also checked
against the slot cache on decode streams: same outputs, same slot -> position map.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle.cache import OracleKV
from oracle.slot_cache import SlotCache

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_figures.json")))
TOL = GOLD["sliding_cache_error"]["tolerance"]
VOCAB, WIDTH, HEADS = 24, 16, 2


class ToyNet:
    """Two float64 attention layers (residual), 16 wide, 2 heads of width 8."""

    def __init__(self, seed):
        rng = np.random.default_rng(seed)
        self.emb = rng.normal(size=(VOCAB, WIDTH))
        self.w = [[rng.normal(size=(WIDTH, WIDTH)) / 4 for _ in range(3)] for _ in range(2)]

    def embed(self, ids, positions):
        ids = np.asarray(ids)
        if ids.size and (ids.min() < 0 or ids.max() >= VOCAB):
            raise ValueError("invalid token id")
        i = np.arange(WIDTH // 2)
        ang = np.asarray(positions)[:, None] / (10000.0 ** (2 * i / WIDTH))
        pe = np.concatenate([np.sin(ang), np.cos(ang)], axis=1)
        return self.emb[ids] + pe

    def qkv(self, layer, x):
        wq, wk, wv = self.w[layer]
        sh = lambda t: t.reshape(t.shape[0], HEADS, WIDTH // HEADS)
        return sh(x @ wq), sh(x @ wk), sh(x @ wv)

    def full(self, ids, window):
        """Every position at once, sliding mask by absolute position in every layer."""
        n = len(ids)
        x = self.embed(ids, np.arange(n))
        i = torch.arange(n)[:, None]
        j = torch.arange(n)[None, :]
        mask = j <= i
        if window is not None:
            mask &= j >= i - (window - 1)
        for layer in range(2):
            q, k, v = self.qkv(layer, x)
            qt, kt, vt = (torch.from_numpy(t).permute(1, 0, 2) for t in (q, k, v))
            o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
            x = x + o.permute(1, 0, 2).reshape(n, WIDTH).numpy()
        return x

    def incremental(self, ids, window, chunk):
        caches = [SlotCache(window, HEADS, WIDTH // HEADS) for _ in range(2)]
        outs = []
        for s in range(0, len(ids), chunk):
            part = ids[s:s + chunk]
            x = self.embed(part, np.arange(caches[0].next_position, caches[0].next_position + len(part)))
            for layer in range(2):
                q, k, v = self.qkv(layer, x)
                o = caches[layer].attend_append(q, k, v)
                x = x + o.reshape(len(part), WIDTH)
            outs.append(x)
        return np.concatenate(outs), caches


@pytest.mark.parametrize("seed", [7, 19, 41])
@pytest.mark.parametrize("length", [1, 2, 8, 17])
@pytest.mark.parametrize("window", [1, 4, None])
def test_incremental_matches_full_mask(seed, length, window):
    net = ToyNet(seed)
    ids = np.random.default_rng(seed + length).integers(0, VOCAB, size=length)
    ref = net.full(ids, window)
    for chunk in sorted({1, 3, length}):
        got, caches = net.incremental(ids, window, chunk)
        assert np.max(np.abs(got - ref)) <= TOL
        for c in caches:
            assert c.next_position == length            # processed count, never reset
            _, _, pos = c.entries()
            keep = length if window is None else min(window, length)
            assert sorted(pos) == list(range(length - keep, length))
            if window is not None:                      # slot = position % W
                for s in range(window):
                    if c.slot_pos[s] >= 0:
                        assert c.slot_pos[s] % window == s


def test_slot_zero_can_hold_position_twenty():
    c = SlotCache(4, 1, 2)
    for _ in range(21):
        c.attend_append(np.ones((1, 1, 2)), np.ones((1, 1, 2)), np.ones((1, 1, 2)))
    assert c.slot_pos[0] == 20


@pytest.mark.parametrize("bad", [0, -1, 2.5, True])
def test_invalid_window_rejected(bad):
    with pytest.raises(ValueError):
        SlotCache(bad, 1, 2)


def test_invalid_token_rejected():
    with pytest.raises(ValueError):
        ToyNet(7).incremental(np.array([3, VOCAB]), 4, 1)


def test_all_masked_row_rejected():
    with pytest.raises(ValueError):
        OracleKV(num_layers=1, num_q_heads=2, num_kv_heads=1, head_dim=4, num_seqs=1,
                 max_positions=4).attend(0, 0, np.zeros((2, 4)))


@pytest.mark.parametrize("window", [1, 4, 5, 16, 20, 0])
def test_oracle_cache_matches_slot_cache(window):
    """The parity oracle's residency rule (mask over the full log) equals the
    incremental slot cache on a decode stream, including chunked appends."""
    rng = np.random.default_rng(window + 100)
    hq, hkv, d, n_prefill, steps = 4, 2, 8, 23, 30
    o = OracleKV(num_layers=1, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_seqs=1,
                 max_positions=n_prefill + steps, kv_format="f32", window=window)
    sc = SlotCache(window if window else None, hkv, d)
    # prefill in chunks of 7: oracle appends; slot cache appends (its outputs unused)
    for s in range(0, n_prefill, 7):
        m = min(7, n_prefill - s)
        k = rng.normal(size=(m, hkv, d)).astype(np.float32).astype(np.float64)
        v = rng.normal(size=(m, hkv, d)).astype(np.float32).astype(np.float64)
        o.append(0, 0, k, v)
        sc.attend_append(np.zeros((m, hq, d)), k, v)
    for t in range(steps):
        k = rng.normal(size=(1, hkv, d)).astype(np.float32).astype(np.float64)
        v = rng.normal(size=(1, hkv, d)).astype(np.float32).astype(np.float64)
        q = rng.normal(size=(hq, d))
        o.append(0, 0, k, v)
        out, w, pos = o.attend(0, 0, q)
        ref = sc.attend_append(q[None], k, v)[0]
        assert np.max(np.abs(out - ref)) <= TOL
        _, _, spos = sc.entries()
        assert sorted(spos) == list(pos)
        if window:
            assert all(o.slot_of(p) == p % window for p in pos)
        o.accumulate()
