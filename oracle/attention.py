"""Masked decode attention with an explicit softmax, and the per-step masses.

Test infrastructure only (see the package docstring).

Sources:
  * "Context views at marginal cost", section 7, Fact 3: attending a query over
    cached keys and values is the QK^T, softmax, V read, which is the floor of the
    method.  The logit scale is not given on the pages; the textbook 1/sqrt(D) is
    used, applied to the dot product.
  * Flash-MoE "Context Optimization", H2O > How It Works, step 1: post-softmax
    scores are summed per position over all query heads, and query heads share
    KV heads (GQA).  Query head h reads KV head floor(h / G), G = Hq / Hkv.
  * "Per-Head Attention as a Scoring Signal", Fix: score per head, place per
    block: each head's weights score the 16-token blocks separately and a block
    stays if any head weights it, so the block mass of one step is the maximum over
    heads of each head's in-block sum.

Everything is float64.  Parity: pinned by tests/test_oracle_attention.py (rows sum
to one, window-1 closed form, equality with torch scaled_dot_product_attention in
float64, block-mass bounds).
"""

import numpy as np


def decode_attention(q, k, v):
    """One decode query per head over n cached entries.

    q: [Hq, D]; k, v: [n, Hkv, D] (the stored values, already dequantised).
    Returns (out [Hq, D], weights [Hq, n]).  Raises on an empty cache, which is the
    all-masked row that "LLM mechanics III" section 5 rejects.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    hq, d = q.shape
    n, hkv, dk = k.shape
    if n == 0:
        raise ValueError("all-masked attention row: the cache holds no entry")
    if dk != d or v.shape != k.shape or hq % hkv:
        raise ValueError("shape mismatch")
    g = hq // hkv
    out = np.empty((hq, d), dtype=np.float64)
    weights = np.empty((hq, n), dtype=np.float64)
    inv_sqrt_d = 1.0 / np.sqrt(d)
    for h in range(hq):
        kvh = h // g
        logits = (k[:, kvh, :] @ q[h]) * inv_sqrt_d
        m = np.max(logits)
        e = np.exp(logits - m)
        a = e / np.sum(e)
        weights[h] = a
        out[h] = a @ v[:, kvh, :]
    return out, weights


def token_step_mass(weights):
    """Per-entry mass of one step of one layer: the sum over query heads."""
    return np.sum(np.asarray(weights, dtype=np.float64), axis=0)


def block_step_mass(weights, positions, block_tokens=16):
    """Per-block mass of one step of one layer.

    For each block id k = floor(position / block_tokens) present among the entries,
    the maximum over query heads of that head's summed weight over the block's
    entries.  Returns a dict {block id: mass}.
    """
    weights = np.asarray(weights, dtype=np.float64)
    positions = np.asarray(positions, dtype=np.int64)
    blocks = positions // block_tokens
    # group the entries by block (a stable sort keeps each block's entries in order),
    # sum each head's weights over every group, then take the max over heads
    order = np.argsort(blocks, kind="stable")
    ids, starts = np.unique(blocks[order], return_index=True)
    per_head = np.add.reduceat(weights[:, order], starts, axis=1)     # [Hq, blocks]
    best = np.max(per_head, axis=0)
    return {int(k): float(m) for k, m in zip(ids, best)}
