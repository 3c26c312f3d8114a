"""Block selection: top-k by score with ties to the lower block id, plus H2O protection.

Test infrastructure only (see the package docstring).

Sources:
  * "Per-Head Attention as a Scoring Signal", Combined placement decision: the
    highest-scoring (sequence, 16-token block) units stay resident, the rest go to
    the host tier.  The tie rule (lower block id first) is the reading taken here.
  * Flash-MoE "Context Optimization", H2O > The Algorithm and How It Works, steps 2-3:
    the first few tokens (sinks, typically 4) and the most recent tokens (the last
    quarter of the budget) are always kept, the remainder of the budget goes to the
    highest cumulative scores, and eviction runs once the resident count exceeds the
    budget.  Counts here are in 16-token blocks (the reading taken here: the block is
    the placement unit, so the budget of 2048 tokens is 128 blocks).

Parity: pinned by tests/test_oracle_selection.py (brute force over every k-subset of
up to 12 blocks; protected-region cases worked by hand).
"""

import math


def top_k_blocks(candidates, scores, k):
    """The k best candidates, best = larger score, ties = lower block id.

    candidates: iterable of int block ids; scores: mapping id -> float.
    Returns the kept ids in ascending order.  If k >= len(candidates) all are kept.
    """
    cand = sorted(set(int(c) for c in candidates))
    if k < 0:
        raise ValueError("k must be >= 0")
    ranked = sorted(cand, key=lambda c: (-float(scores[c]), c))
    return sorted(ranked[:k])


def protected_blocks(candidates, next_position, sink_tokens, recent_tokens, block_tokens=16):
    """Blocks holding a sink token (position < sink_tokens) or a recent token
    (position >= next_position - recent_tokens), restricted to the candidates."""
    cand = set(int(c) for c in candidates)
    prot = set()
    for p in range(min(sink_tokens, next_position)):
        prot.add(p // block_tokens)
    for p in range(max(0, next_position - recent_tokens), next_position):
        prot.add(p // block_tokens)
    return sorted(prot & cand)


def h2o_keep(candidates, scores, budget_blocks, next_position, sink_tokens, recent_tokens,
             block_tokens=16):
    """H2O keep set in block units.

    If the candidates fit the budget nothing is evicted.  Otherwise the protected
    blocks are kept and the rest of the budget is filled by score (ties to the lower
    id) among the unprotected candidates.
    """
    cand = sorted(set(int(c) for c in candidates))
    if len(cand) <= budget_blocks:
        return cand
    prot = protected_blocks(cand, next_position, sink_tokens, recent_tokens, block_tokens)
    rest = [c for c in cand if c not in set(prot)]
    room = max(0, budget_blocks - len(prot))
    return sorted(prot + top_k_blocks(rest, scores, room))


def recent_token_count(budget_tokens, recent_frac):
    """Recent region size in tokens: the last recent_frac of the budget, rounded up."""
    return int(math.ceil(recent_frac * budget_tokens))
