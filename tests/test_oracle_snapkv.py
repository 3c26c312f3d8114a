"""Pins of the oracle's SnapKV prefill scoring ("Context views at marginal cost", the
per-system reductions: observation window of the last 32 prompt queries, votes pooled
per token and head, max-pool kernel 7).

- Votes against a second construction: a dense logit matrix per head with -inf above
  the causal diagonal, a softmax over keys, and a sum over queries, in float64 torch.
  The oracle instead loops over queries and restricts the keys.
- Each head's votes sum to the number of queries, and the newest token's vote comes
  from the newest query alone.
- With one query and kernel 1, the recorded masses are the decode attend's masses for
  that query.
- The pool against scipy.ndimage.maximum_filter1d (contiguous positions) and against
  a dense -inf-padded filter (positions with gaps).
- A planted key lifts every position within 3 of it, across a block edge, so a
  neighbouring block's mass rises to the planted vote.
- Window mode sees the last W positions only.  Out-of-range windows raise.
"""
import numpy as np
import pytest
import scipy.ndimage
import torch

from oracle import attention, snapkv
from oracle.cache import OracleKV


def _cache(n=90, window=0, fmt="f32", seed=3, hq=4, hkv=2, d=16, layers=1):
    rng = np.random.default_rng(seed)
    o = OracleKV(num_layers=layers, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, num_seqs=1,
                 max_positions=n + 8, kv_format=fmt, window=window)
    for l in range(layers):
        o.append(l, 0, rng.normal(size=(n, hkv, d)), rng.normal(size=(n, hkv, d)))
    return o, rng


def _torch_votes(q_obs, obs_pos, k, key_pos):
    q = torch.from_numpy(np.asarray(q_obs, np.float64))          # [n_obs, Hq, D]
    kk = torch.from_numpy(np.asarray(k, np.float64))            # [n, Hkv, D]
    hq, hkv, d = q.shape[1], kk.shape[1], q.shape[2]
    kk = kk.repeat_interleave(hq // hkv, dim=1)                  # [n, Hq, D]
    s = torch.einsum("ihd,jhd->hij", q, kk) / np.sqrt(d)         # [Hq, n_obs, n]
    mask = torch.from_numpy(np.asarray(key_pos)[None, :] > np.asarray(obs_pos)[:, None])
    s = s.masked_fill(mask[None], float("-inf"))
    return torch.softmax(s, dim=-1).sum(dim=1).numpy()           # [Hq, n]


@pytest.mark.parametrize("n_obs,fmt", [(32, "f32"), (5, "e4m3"), (1, "bf16")])
def test_votes_match_dense_causal_softmax(n_obs, fmt):
    o, rng = _cache(fmt=fmt)
    q = rng.normal(size=(n_obs, 4, 16)) * 1.5
    votes, pooled, pos = o.prefill_score(0, 0, q)
    k, _ = o.stored_kv(0, 0, pos)
    ref = _torch_votes(q, np.arange(90 - n_obs, 90), k, pos)
    assert np.max(np.abs(votes - ref)) < 1e-12
    assert np.allclose(votes.sum(axis=1), n_obs, rtol=0, atol=1e-12)
    # the newest token is seen by the newest query only
    _, w = attention.decode_attention(q[-1], k, k)
    assert np.allclose(votes[:, -1], w[:, -1], rtol=0, atol=1e-15)
    assert np.all(pooled >= votes)


def test_one_query_kernel_one_is_the_decode_attend():
    o, rng = _cache(n=70)
    q = rng.normal(size=(4, 16))
    o.prefill_score(0, 0, q[None], kernel=1)
    tau_p, bm_p = o.token_mass(0, 0)[1].copy(), dict(o.block_mass(0, 0))
    o.attend(0, 0, q)
    tau_a, bm_a = o.token_mass(0, 0)[1], o.block_mass(0, 0)
    assert np.allclose(tau_p, tau_a, rtol=0, atol=1e-15)
    assert bm_p.keys() == bm_a.keys()
    assert max(abs(bm_p[b] - bm_a[b]) for b in bm_a) < 1e-15


def test_pool_matches_scipy_filters():
    rng = np.random.default_rng(11)
    v = rng.random(size=(3, 57))
    pos = np.arange(100, 157)
    got = snapkv.max_pool(v, pos, 7)
    assert np.array_equal(got, scipy.ndimage.maximum_filter1d(v, size=7, axis=1, mode="nearest"))
    # resident positions with gaps (blocks 0, 2 and 3 of 16): neighbours across a gap
    # are absent, as in a dense filter with -inf in the gap
    pos = np.concatenate([np.arange(0, 16), np.arange(32, 64)])
    v = rng.random(size=(2, len(pos)))
    dense = np.full((2, 64), -np.inf)
    dense[:, pos] = v
    ref = scipy.ndimage.maximum_filter1d(dense, size=7, axis=1, mode="constant", cval=-np.inf)[:, pos]
    assert np.array_equal(snapkv.max_pool(v, pos, 7), ref)


def test_planted_key_lifts_its_neighbours_across_a_block_edge():
    """Every query of head group 0 matches the key at position 48 (first entry of block
    3), so its vote dominates.  Positions 45..51 take that vote after pooling, so block
    2 (positions 32..47) gets a block mass of at least 3 x the planted vote."""
    n, d = 80, 16
    o, rng = _cache(n=n, d=d)
    key = np.zeros((1, 2, d))
    key[0, 0, 0] = 40.0
    o.k_vals[0, 0, 48] = key[0]
    q = rng.normal(size=(8, 4, d)) * 0.1
    q[:, 0:2, 0] = 1.0                              # heads 0, 1 read KV head 0
    votes, pooled, pos = o.prefill_score(0, 0, q)
    planted = votes[0, 48]
    assert planted > 7.9 and np.argmax(votes[0]) == 48
    for j in range(n):
        if abs(j - 48) <= 3:
            assert pooled[0, j] == planted
        elif abs(j - 48) > 6:
            assert pooled[0, j] < 0.1
    bm = o.block_mass(0, 0)
    assert bm[2] >= 3 * planted and bm[3] >= 4 * planted


def test_window_sees_the_last_w_positions():
    o, rng = _cache(n=90, window=40)
    q = rng.normal(size=(6, 4, 16))
    votes, pooled, pos = o.prefill_score(0, 0, q)
    assert np.array_equal(pos, np.arange(50, 90))
    k, _ = o.stored_kv(0, 0, pos)
    assert np.max(np.abs(votes - _torch_votes(q, np.arange(84, 90), k, pos))) < 1e-12
    tau = o.token_mass(0, 0)[1]
    assert np.allclose(tau, pooled.sum(axis=0), rtol=0, atol=1e-15)
    with pytest.raises(ValueError):
        o.prefill_score(0, 0, rng.normal(size=(41, 4, 16)))


def test_feeds_the_score_tables_as_a_first_step():
    o, rng = _cache(n=50, layers=2)
    q = [rng.normal(size=(4, 4, 16)) for _ in range(2)]
    pooled = [o.prefill_score(l, 0, q[l])[1] for l in range(2)]
    with pytest.raises(ValueError):
        o.prefill_score(0, 0, rng.normal(size=(51, 4, 16)))
    o.accumulate()
    sc = o.scores[0]
    assert sc.steps == 1
    assert np.allclose(sc.c_tok[:50], pooled[0].sum(axis=0) + pooled[1].sum(axis=0), rtol=0, atol=1e-12)
    for b in range(4):
        sel = slice(16 * b, min(16 * b + 16, 50))
        y = max(np.max(pooled[l][:, sel].sum(axis=1)) for l in range(2))
        assert abs(sc.c_blk[b] - y) < 1e-12


def test_planted_workload_keeps_the_fact_and_its_left_neighbour():
    """"Per-Head Attention as a Scoring Signal", Example: on a scaled-down copy of the
    planted workload (8192-token prompt, retrieval key at 4096, the first entry of
    block 256), SnapKV scoring alone ranks the anchor, the fact and the recent blocks
    into the kept set.  The pool carries the fact's vote to positions 4093..4095, so
    block 255 is kept as well."""
    import workloads
    wl = workloads.scaled_down("bf16-b1-ctx131072-planted", context=8192, retrieval_pos=4096,
                               num_layers=2, steps=1, prefill_chunk=0)
    inp = workloads.Inputs(wl, device="cpu")
    o = OracleKV(num_layers=wl.num_layers, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                 head_dim=wl.head_dim, num_seqs=1, max_positions=wl.max_positions, kv_format="bf16")
    fact_head = 2 * wl.group                       # KV head 2 carries the retrieval key
    for l in range(wl.num_layers):
        k, v = inp.prefill_kv(l, 0)
        o.append(l, 0, workloads.as_f64(k), workloads.as_f64(v))
        votes, pooled, pos = o.prefill_score(l, 0, workloads.as_f64(inp.obs_q(l, 32)[0]))
        f = wl.retrieval_pos
        assert np.argmax(votes[fact_head]) == f
        assert np.all(pooled[fact_head, f - 3: f + 4] == votes[fact_head, f])
    o.accumulate()
    keep = set(o.select(0, wl.keep_k(len(o.resident_block_ids(0)))))
    anchor = {p // 16 for p in range(51)}
    recent = {p // 16 for p in range(wl.context - 100, wl.context)}
    assert anchor <= keep and recent <= keep
    assert {255, 256} <= keep
