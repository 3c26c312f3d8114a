"""SnapKV prefill scoring: observation-window votes, max-pooled along the tokens.

Test infrastructure only (see the package docstring).

Source: "Context views at marginal cost", the per-system reductions, SnapKV entry.
Once, when prefill ends, the prompt's last N queries (the observation window, N = 32)
each attend over the prompt.  Their weights are pooled into one score per prompt
token per head.  That score is then max-pooled along the tokens with a kernel of 7,
so a key that scores high lifts its neighbours too.

Readings taken where the page leaves a step open:
  * an observation query at absolute position p attends causally, over the resident
    entries at positions <= p.  The cache is the prompt: all of it, its last W
    positions under a window, or the entries of the resident blocks under H2O.
    Logits are q.k/sqrt(D) and the softmax is per head, as in the decode attend;
  * a token's vote for head h sums the weights that the observation queries of head h
    give it;
  * the max-pool is per head: stride 1, output as long as the input, and at each
    position the largest vote among the resident positions within 3 of it. Neighbours
    outside the resident entries are absent, not padded;
  * the pooled votes feed the reductions of one decode step's weights: the token mass
    sums over heads, and the block mass is the max over heads of the in-block sum.
    So the score tables take them as their first step.

Everything is float64.  Parity: pinned by tests/test_oracle_snapkv.py.  The pins are:
  * every head's votes sum to the number of observation queries;
  * the newest token's vote comes from the newest query alone;
  * with one query and kernel 1, the votes are the decode weights;
  * the pool equals scipy's maximum filter, and a planted key lifts exactly the
    positions within 3 of it;
  * brute force recomputes a small case.
"""

import numpy as np

from . import attention


def observation_votes(q_obs, obs_pos, k, key_pos):
    """Per-head votes of the observation queries.

    q_obs: [n_obs, Hq, D] queries at absolute positions obs_pos [n_obs]; k: [n, Hkv, D]
    the stored keys at positions key_pos [n] (ascending).  Query i attends over the
    keys with key_pos <= obs_pos[i].  Returns votes [Hq, n]: sum over i of query i's
    weights (0 for keys a query does not see)."""
    q_obs = np.asarray(q_obs, np.float64)
    k = np.asarray(k, np.float64)
    key_pos = np.asarray(key_pos, np.int64)
    n_obs, hq, _ = q_obs.shape
    votes = np.zeros((hq, k.shape[0]))
    for i in range(n_obs):
        seen = key_pos <= int(obs_pos[i])
        _, w = attention.decode_attention(q_obs[i], k[seen], k[seen])   # values unused
        votes[:, seen] += w
    return votes


def max_pool(votes, key_pos, kernel=7):
    """Per head, the largest vote among the positions within kernel // 2 of each
    position (positions not listed in key_pos are absent)."""
    votes = np.asarray(votes, np.float64)
    key_pos = np.asarray(key_pos, np.int64)
    r = kernel // 2
    out = np.empty_like(votes)
    for j in range(len(key_pos)):
        near = np.abs(key_pos - key_pos[j]) <= r
        out[:, j] = np.max(votes[:, near], axis=1)
    return out
