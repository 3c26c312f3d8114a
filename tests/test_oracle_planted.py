"""Pin of the oracle's selection on the planted four-head-type workload.

"Per-Head Attention as a Scoring Signal", Example: 128K Context Document QA and the
Combined placement decision: the blocks that stay resident are the anchor blocks
(system prompt at the start), the block holding the retrieved fact and the recent
tail.  A scaled-down copy of the planted workload (8192-token context, retrieval key
at 4096, 2 layers, 2 steps) must keep exactly those blocks among its top 10%.
"""
import numpy as np

import workloads
from oracle.cache import OracleKV


def test_planted_selection_keeps_anchor_fact_and_recent():
    wl = workloads.scaled_down("bf16-b1-ctx131072-planted", context=8192, retrieval_pos=4096,
                               num_layers=2, steps=2, prefill_chunk=0)
    inp = workloads.Inputs(wl, device="cpu")
    o = OracleKV(num_layers=wl.num_layers, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                 head_dim=wl.head_dim, num_seqs=1, max_positions=wl.max_positions, kv_format="bf16")
    for l in range(wl.num_layers):
        k, v = inp.prefill_kv(l, 0)
        o.append(l, 0, workloads.as_f64(k), workloads.as_f64(v))
    for t in range(wl.steps):
        for l in range(wl.num_layers):
            k, v = inp.step_kv(l, t)
            o.append(l, 0, workloads.as_f64(k[0]), workloads.as_f64(v[0]))
            o.attend(l, 0, workloads.as_f64(inp.step_q(l, t)[0]))
        o.accumulate()
    cands = o.resident_block_ids(0)
    keep = set(o.select(0, wl.keep_k(len(cands))))
    anchor = {p // 16 for p in range(51)}
    fact = {wl.retrieval_pos // 16}
    recent = {p // 16 for p in range(wl.context - 100, wl.context + wl.steps)}
    assert anchor <= keep
    assert fact <= keep
    assert recent <= keep
    # and those blocks out-score every unplanted block by a wide margin
    c = o.scores[0].c_blk
    planted = sorted(anchor | fact | recent)
    others = [b for b in cands if b not in set(planted)]
    assert min(c[b] for b in planted) > 2 * np.median([c[b] for b in others])
