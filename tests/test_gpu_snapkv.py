"""GPU parity of SnapKV prefill scoring against the oracle ("Context views at marginal
cost", the per-system reductions: observation window, votes per token and head,
max-pool kernel 7).

For every layer, kvs_prefill_score is called with the queries of the prompt's last
n_obs positions, and its entry and block masses are compared with the oracle's.  Then
kvs_accumulate_scores folds them into the tables as their first step, and decode
steps and selections continue from there.  The cases span a window that wraps, no
window, 8 KV heads with planted heads, a ragged H2O batch whose first selection
evicts (SnapKV's one-shot compression), n_obs of 32, 7 and 1, and the 32K-context
FP8 batch at full size.

Bar: these masses sum the weights of n_obs queries and are then max-pooled, so they
reach tens to hundreds (a vote is at most n_obs per head, a pooled in-block sum at most
16 n_obs), where the decode step's masses stay below the number of heads.  The GPU
computes them in float32, whose error is relative: a logit of magnitude |s| <= 32
(log2 units) carries at most ~|s| 2^-23 of rounding, i.e. a relative weight error of
<= 32 * 2^-23 * ln 2 = 2.6e-6, and summing up to 512 positive float32 terms adds a few
2^-24 more.  So the decode bar gains a relative term, |got - ref| <= 1e-4 + RHO |ref|
with RHO = 1e-5, for every storage format (the E4M3 path converts the bf16 queries to
f16, which is exact in f16's normal range, and its keys' E4M3 values are exact in f16
too).  Measured worst relative error: about 6e-7 for both formats.  The bar applies to
masses, tables and the selection's cut-off band; kept sets must be equal except near
the cut-off.
"""
import dataclasses

import numpy as np
import pytest
import torch

import attention_scored_kv_gb300 as kvs
import workloads
from tests import harness
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu


RHO = 1e-5


def _snap_run(wl, n_obs, oseqs, steps):
    rho = RHO
    run = harness.Run(wl, oracle_seqs=oseqs, kernel=kvs.KERNEL_TENSOR, obs_window=32)
    run.prefill()
    worst = run.prefill_score(n_obs, rel=rho)
    harness.check_scores(run, rel=rho)
    keep = run.select()                        # H2O: the one-shot compression
    harness.check_selection(run, keep, rel=rho)
    for t in range(steps):
        res = run.decode_step(select=False)
        assert res["out_err"] <= harness.OUT_TOL[wl.kv_format]
        harness.check_masses(run)              # a decode step's masses: the decode bar
        harness.check_scores(run, rel=rho)
        harness.check_selection(run, run.select(), rel=rho)
    harness.check_storage(run)
    assert run.cache.get_status() == 0, run.cache.last_error()
    return run, worst


@pytest.mark.parametrize("name,n_obs", [("e4m3-window", 32), ("e4m3-window", 7), ("bf16", 32), ("bf16", 1),
                                        ("e4m3-nowindow", 32), ("bf16-hkv8", 32), ("e4m3-h2o", 32)])
def test_prefill_score_against_oracle(name, n_obs):
    wl = SMALL[name]
    _snap_run(wl, n_obs, list(range(wl.batch)), steps=2)


def test_prefill_score_fullsize_e4m3_b16_ctx32768_window4096():
    """The 32K-context FP8 batch (window 4096), 32 observation queries per sequence:
    the masses of two sampled sequences in every layer, then one decode step."""
    wl = dataclasses.replace(workloads.get("e4m3-b16-ctx32768-window4096"), steps=1)
    _snap_run(wl, 32, [0, 9], steps=1)


def test_prefill_score_over_more_sequences_than_one_launch_takes():
    """A call of 530 sequences runs as launches of at most 512 (one launch's scoring
    scratch holds 512 sequences).  Ragged short prompts of 2 to 6 blocks (no eviction
    at this budget) put many (sequence, KV head) groups into each CTA's share;
    sequences on both sides of the split follow the oracle."""
    wl = workloads.scaled_down("e4m3-b64-ragged-h2o2048", name="snap-530", num_layers=1, batch=530,
                               context_range=(40, 90), h2o_budget_tokens=256, steps=1, prefill_chunk=0)
    _snap_run(wl, 32, [0, 1, 511, 512, 529], steps=1)


def test_prefill_score_is_deterministic_and_leaves_the_cache():
    """Two calls give the same bytes; the K/V storage and positions are untouched."""
    wl = SMALL["e4m3-window"]
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR, obs_window=32)
    run.prefill()
    c = run.cache
    kp = c.read_state(kvs.STATE_K_PAGES, 1).clone()
    q = run.inp.obs_q(1, 32)
    c.prefill_score(1, q)
    a = (c.read_state(kvs.STATE_TOKEN_MASS, 1).clone(), c.read_state(kvs.STATE_BLOCK_MASS, 1).clone())
    c.prefill_score(1, q)
    b = (c.read_state(kvs.STATE_TOKEN_MASS, 1), c.read_state(kvs.STATE_BLOCK_MASS, 1))
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
    assert torch.equal(kp, c.read_state(kvs.STATE_K_PAGES, 1))
    assert c.get_status() == 0


def test_prefill_score_rejects_bad_calls():
    wl = SMALL["e4m3-window"]                   # window 256, prompts of 700
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR, obs_window=16)
    c = run.cache
    q = run.inp.obs_q(0, 16)
    with pytest.raises(kvs.KVSError):           # nothing appended yet: fewer entries than n_obs
        c.prefill_score(0, q)
    run.prefill()
    with pytest.raises(kvs.KVSError):           # more than obs_window
        c.prefill_score(0, run.inp.obs_q(0, 17))
    with pytest.raises(kvs.KVSError):
        c.prefill_score(wl.num_layers, q)
    c.prefill_score(0, q)
    off = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    off.prefill()
    with pytest.raises(kvs.KVSError):           # scoring scratch not configured
        off.cache.prefill_score(0, q)
    assert c.get_status() == 0 and off.cache.get_status() == 0
