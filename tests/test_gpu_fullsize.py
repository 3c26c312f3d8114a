"""GPU parity at the configured full sizes, in the launch configuration bench.py times.

The decode steps go through append_attend, a layer's append and attend in one launch
where the context allows, and accumulate_select, as bench.py's step does.  The oracle
follows a sample of the sequences from their first token:
- 35B bf16 (8 x 4096) and FP8 (16 x 32768, window 4096): every output row, the
  masses, the score tables, the selection and the stored codes of the sampled
  sequences, every step; for FP8 also the Tier-2 re-attend over the kept blocks.
- Ragged FP8 with H2O (64 sequences up to 32768, budget 2048, eviction applied): the
  same for one sampled sequence over the first steps, from the full-context first
  step to the evicted steady state.
- 397B bf16 (1 x 131072, planted heads): float64 over the whole cache would need
  tens of GB on the host, so one layer is recomputed exactly. All properties that hold
  at any size are checked: every head's weights sum to one (sum of the entry masses
  = Hq), block masses lie in [0, 1], and the selection keeps the anchor, fact and
  recent blocks.
Bars as in test_gpu_parity.
"""
import dataclasses

import numpy as np
import pytest
import torch

import attention_scored_kv_gb300 as kvs
import workloads
from oracle import attention
from tests import harness

pytestmark = pytest.mark.gpu


def _bench_path_check(wl, oseqs, steps):
    run = harness.Run(wl, oracle_seqs=oseqs, kernel=kvs.KERNEL_TENSOR, fused=True)
    run.prefill()
    worst = 0.0
    for t in range(steps):
        res = run.decode_step(select=False, accumulate=False)
        worst = max(worst, res["out_err"])
        harness.check_masses(run)                  # read through the block table: before eviction
        keep = run.accumulate_select()
        harness.check_scores(run)
        harness.check_selection(run, keep)
    harness.check_storage(run)
    assert worst <= harness.OUT_TOL[wl.kv_format], worst
    assert run.cache.get_status() == 0, run.cache.last_error()
    return run


def test_fullsize_bf16_b8_ctx4096():
    wl = dataclasses.replace(workloads.get("bf16-b8-ctx4096"), steps=3)
    _bench_path_check(wl, oseqs=[0, 5], steps=3)


def test_fullsize_e4m3_b16_ctx32768_window4096():
    wl = dataclasses.replace(workloads.get("e4m3-b16-ctx32768-window4096"), steps=3)
    run = _bench_path_check(wl, oseqs=[0, 9], steps=3)
    assert run.cache.layout().attend_kernel == kvs.KERNEL_TENSOR
    # Tier-2 re-attend of a new query over the blocks a selection keeps (k = 64 of 257)
    lay = run.cache.layout()
    ids, cnt = run.cache.select_blocks(wl.keep_k(257), keep_capacity=lay.max_blocks)
    worst = 0.0
    for l in (0, wl.num_layers - 1):
        q = run.inp.step_q(l, wl.steps + 5)
        got = run.cache.attend_blocks(l, q, ids, cnt)
        qf = workloads.as_f64(q)
        for i, s in enumerate(run.oseqs):
            ref, _, _ = run.oracle.attend_blocks(l, i, qf[s], ids[s, : int(cnt[s])].cpu().numpy())
            worst = max(worst, harness.rel_err_rows(got[s].double().cpu().numpy(), ref))
    assert worst <= harness.OUT_TOL[wl.kv_format], worst
    assert run.cache.get_status() == 0


def test_fullsize_e4m3_b64_ragged_h2o2048():
    wl = dataclasses.replace(workloads.get("e4m3-b64-ragged-h2o2048"), steps=3)
    lens = workloads.Inputs(wl, device="cpu").prefill_lengths()
    mid = int(np.argsort(lens)[len(lens) // 2])       # a sequence of median length
    _bench_path_check(wl, oseqs=[mid], steps=3)


def test_fullsize_bf16_b1_ctx131072_planted():
    wl = dataclasses.replace(workloads.get("bf16-b1-ctx131072-planted"), steps=2)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR, fused=True)
    run.prefill()
    L, Hq = wl.num_layers, wl.num_q_heads
    for t in range(wl.steps):
        run.decode_step(select=False, accumulate=False)
        sv = harness.StateView(run.cache, wl)    # one read-back of this step's state
        # every head's weights sum to one: the entry masses of a layer sum to Hq
        n = int(wl.context) + t + 1
        pos = np.arange(n)
        page, slot = sv.page_slot(0, pos)
        for l in range(L):
            tau = sv.token_mass(l)[page, slot].astype(np.float64)
            assert abs(tau.sum() - Hq) <= 1e-3 * Hq, (t, l, tau.sum())
            bm = sv.block_mass(l)[0, : (n + 15) // 16]
            assert bm.min() >= 0.0 and bm.max() <= 1.0 + 1e-6
        keep, cnt = run.cache.accumulate_select(wl.keep_k((n + 15) // 16),
                                                keep_capacity=run.cache.layout().max_blocks)
    # one layer exactly, last step: the stored bf16 values are the inputs themselves
    l = L // 2
    kp, vp = run.inp.prefill_kv(l, 0)
    ks = [run.inp.step_kv(l, t) for t in range(wl.steps)]
    k = np.concatenate([workloads.as_f64(kp)] + [workloads.as_f64(a[0]) for a, _ in ks])
    v = np.concatenate([workloads.as_f64(vp)] + [workloads.as_f64(b[0]) for _, b in ks])
    q = workloads.as_f64(run.inp.step_q(l, wl.steps - 1)[0])
    ref, w = attention.decode_attention(q, k, v)
    got = run.last_out[l][0].double().cpu().numpy()
    err = harness.rel_err_rows(got, ref)
    assert err <= harness.OUT_TOL[wl.kv_format], err
    n = k.shape[0]
    page, slot = sv.page_slot(0, np.arange(n))
    tau = sv.token_mass(l)[page, slot].astype(np.float64)
    assert np.max(np.abs(tau - attention.token_step_mass(w))) <= harness.SCORE_TOL
    bref = attention.block_step_mass(w, np.arange(n))
    bm = sv.block_mass(l)[0]
    assert max(abs(float(bm[kb]) - m) for kb, m in bref.items()) <= harness.SCORE_TOL
    # the planted blocks are kept: anchor keys 0-50, the fact at the retrieval key and
    # the recent tail ("Per-Head Attention as a Scoring Signal", Example)
    kept = set(int(x) for x in keep[0, : int(cnt[0])].cpu().numpy())
    anchor = {p // 16 for p in range(51)}
    fact = {wl.retrieval_pos // 16}
    recent = {p // 16 for p in range(wl.context - 100, wl.context + wl.steps)}
    assert anchor <= kept and fact <= kept and recent <= kept
    assert run.cache.get_status() == 0
