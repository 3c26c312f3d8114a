"""GPU parity of the side-car views against the oracle ("Context views at marginal
cost", Tier 1): the trajectory ring of the TOVA block score, the per-layer profiles,
the threshold filter, and the score snapshot (export, import, resume).

The ring is shorter than the run, so it wraps; the workloads span a window that blocks
leave, H2O eviction, and no eviction at all.  Bars as in test_gpu_parity: 1e-4
absolute on scores; filtered sets equal except blocks whose oracle score lies within
1e-4 of theta; snapshots bit-exact.
"""
import dataclasses

import numpy as np
import pytest
import torch

import attention_scored_kv_gb300 as kvs
from tests import harness
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu

TRAJ = 4
PROF = (0, 1)
_KINDS = ((kvs.SCORE_CUMULATIVE, "cumulative", "c_blk"), (kvs.SCORE_EMA, "ema", "e_blk"),
          (kvs.SCORE_TOKEN_SUM, "token_sum", "s_blk"), (kvs.SCORE_TOVA, "tova", "t_blk"))


def _views(run):
    wl, lay = run.wl, run.cache.layout()
    traj = run.cache.read_state(kvs.STATE_TRAJECTORY).cpu().numpy().view(np.float32)
    prof = run.cache.read_state(kvs.STATE_LAYER_PROFILE).cpu().numpy().view(np.float64)
    return (traj.reshape(wl.batch, lay.max_blocks, TRAJ), prof.reshape(wl.batch, lay.max_blocks, len(PROF)))


def _check_views(run):
    traj, prof = _views(run)
    worst = 0.0
    for i, s in enumerate(run.oseqs):
        sc = run.oracle.scores[i]
        ref = sc.trajectory()
        n = ref.shape[0]
        worst = max(worst, float(np.max(np.abs(traj[s, :n].astype(np.float64) - ref))))
        assert not traj[s, n:].any()
        worst = max(worst, float(np.max(np.abs(prof[s, :n] - sc.prof.T))))
    assert worst <= harness.SCORE_TOL, worst
    return worst


@pytest.mark.parametrize("name,fused", [("e4m3-window", False), ("e4m3-window", True), ("bf16", False),
                                        ("e4m3-h2o", True)])
def test_trajectory_and_profiles_against_oracle(name, fused):
    """Every step: the ring read oldest first (zero where a block was not updated, before
    the first step and after a block left), and each profiled layer's summed block
    mass.  fused runs the bench's step (append_attend, accumulate_select)."""
    wl = dataclasses.replace(SMALL[name], steps=min(SMALL[name].steps, 9))
    run = harness.Run(wl, oracle_seqs=list(range(wl.batch)), kernel=kvs.KERNEL_TENSOR, fused=fused,
                      traj_len=TRAJ, profile_layers=PROF)
    run.prefill()
    traj, prof = _views(run)
    assert not traj.any() and not prof.any()
    for t in range(wl.steps):
        if fused:
            run.decode_step(select=False, accumulate=False)
            run.accumulate_select()
        else:
            run.decode_step(select=True)
        _check_views(run)
    assert run.cache.get_status() == 0, run.cache.last_error()


@pytest.mark.parametrize("name", ["e4m3-window", "e4m3-h2o"])
def test_filter_blocks_against_oracle(name):
    """The blocks above theta, for every score kind, at thetas between the scores (the
    median and the quartiles of the resident blocks' oracle scores) and at +-inf."""
    wl = dataclasses.replace(SMALL[name], steps=min(SMALL[name].steps, 6))
    run = harness.Run(wl, oracle_seqs=list(range(wl.batch)), kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    lay = run.cache.layout()
    for t in range(wl.steps):
        run.decode_step(select=True)
        for kind, okind, table in _KINDS:
            res = [sorted(run.oracle.resident_block_ids(i)) for i in range(wl.batch)]
            tabs = [getattr(run.oracle.scores[i], table) for i in range(wl.batch)]
            vals = np.concatenate([tabs[i][res[i]] for i in range(wl.batch)])
            for theta in (float(np.median(vals)), float(np.quantile(vals, 0.25)), float(np.quantile(vals, 0.75)),
                          -np.inf, np.inf):
                ids, cnt = run.cache.filter_blocks(theta, score_kind=kind, capacity=lay.max_blocks)
                ids, cnt = ids.cpu().numpy(), cnt.cpu().numpy()
                for i, s in enumerate(run.oseqs):
                    got = list(ids[s, : cnt[s]])
                    assert got == sorted(got)
                    ref = run.oracle.filter_blocks(i, okind, theta)
                    for k in set(got) ^ set(ref):
                        assert abs(tabs[i][k] - theta) <= harness.SCORE_TOL, (okind, theta, k, tabs[i][k])
                    if theta == -np.inf:
                        assert got == res[i]
                    if theta == np.inf:
                        assert got == []
    assert run.cache.get_status() == 0, run.cache.last_error()


def test_filter_capacity_overflow_flags_error():
    """More blocks pass than the output holds: the first `capacity` ids are written,
    the count is the full number, and the device error word says capacity."""
    wl = dataclasses.replace(SMALL["bf16"], steps=1)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    run.decode_step(select=False)
    ids, cnt = run.cache.filter_blocks(-np.inf, capacity=3)
    assert wl.window == 0 and wl.context_range is None
    assert cnt.cpu().tolist() == [(wl.context + 1 + 15) // 16] * wl.batch
    assert ids.cpu().tolist() == [[0, 1, 2]] * wl.batch
    assert run.cache.get_status() == kvs._abi.ERR_CAPACITY
    run.cache.clear_error()
    assert run.cache.get_status() == 0


_SNAP_ITEMS = (kvs.STATE_C_TOKEN, kvs.STATE_E_TOKEN, kvs.STATE_C_BLOCK, kvs.STATE_E_BLOCK, kvs.STATE_S_BLOCK,
               kvs.STATE_T_BLOCK, kvs.STATE_STEPS, kvs.STATE_TRAJECTORY, kvs.STATE_LAYER_PROFILE)


def _score_state(cache):
    return {w: cache.read_state(w).cpu() for w in _SNAP_ITEMS}


@pytest.mark.parametrize("host", [False, True])
def test_snapshot_round_trip(host):
    """Export, reset (every table back to zero), import: every score table and the
    step counts come back bit-exact; a sub-range copies only its own rows."""
    wl = dataclasses.replace(SMALL["e4m3-window"], steps=5)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR, traj_len=TRAJ, profile_layers=PROF)
    run.prefill()
    for t in range(wl.steps):
        run.decode_step(select=False)
    c = run.cache
    before = _score_state(c)
    dst = torch.empty(c.snapshot_bytes(wl.batch), dtype=torch.uint8, pin_memory=True) if host else None
    snap = c.export_scores(dst=dst)
    torch.cuda.synchronize()
    c.reset()
    zero = _score_state(c)
    assert not zero[kvs.STATE_C_BLOCK].any() and not zero[kvs.STATE_STEPS].any()
    c.import_scores(snap)
    after = _score_state(c)
    for w in _SNAP_ITEMS:
        assert torch.equal(before[w], after[w]), w
    # sequence 1 alone into a reset cache: its rows only
    part = c.export_scores(seq_begin=1, n_seqs=1)
    assert part.numel() == c.snapshot_bytes(1) < snap.numel()
    c.reset()
    c.import_scores(part, seq_begin=1, n_seqs=1)
    one = _score_state(c)
    for w in (kvs.STATE_C_BLOCK, kvs.STATE_TRAJECTORY, kvs.STATE_LAYER_PROFILE):
        a, b = before[w].view(wl.batch, -1), one[w].view(wl.batch, -1)
        assert torch.equal(a[1], b[1]) and not b[0].any() and not b[2].any(), w
    with pytest.raises(kvs.KVSError):
        c.import_scores(part[:-1], seq_begin=0, n_seqs=1)
    assert c.get_status() == 0, c.last_error()


def test_snapshot_resume_matches_uninterrupted_run():
    """Checkpoint and resume: a second cache holds the same KV (the same appends and
    attends, without scoring), imports the first cache's snapshot of step 3, and then
    scores steps 3..5; every table equals the uninterrupted run's bit for bit."""
    wl = dataclasses.replace(SMALL["e4m3-window"], steps=6)
    a = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR, traj_len=TRAJ, profile_layers=PROF)
    b = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR, traj_len=TRAJ, profile_layers=PROF)
    a.prefill()
    b.prefill()
    snap = None
    for t in range(wl.steps):
        if t == 3:
            snap = a.cache.export_scores()
            b.cache.import_scores(snap)
        a.decode_step(select=False)
        b.decode_step(select=False, accumulate=t >= 3)
    sa, sb = _score_state(a.cache), _score_state(b.cache)
    for w in _SNAP_ITEMS:
        assert torch.equal(sa[w], sb[w]), w
    assert a.cache.get_status() == 0 and b.cache.get_status() == 0


HEADS = ((0, 3), (1, 0), (1, 13), (0, 31))      # (layer, query head): four KV groups


def _check_head_profiles(run, heads, rel=0.0):
    wl, lay = run.wl, run.cache.layout()
    got = run.cache.read_state(kvs.STATE_HEAD_PROFILE).cpu().numpy().view(np.float64)
    got = got.reshape(wl.batch, lay.max_blocks, len(heads))
    worst = 0.0
    for i, s in enumerate(run.oseqs):
        ref = run.oracle.scores[i].hprof            # [heads][blocks]
        n = ref.shape[1]
        worst = max(worst, float(np.max(np.abs(got[s, :n] - ref.T) / (harness.SCORE_TOL + rel * np.abs(ref.T)))))
    assert worst <= 1.0, worst


@pytest.mark.parametrize("name,fused,kernel", [("e4m3-window", True, kvs.KERNEL_TENSOR),
                                               ("bf16", False, kvs.KERNEL_TENSOR),
                                               ("e4m3-h2o", True, kvs.KERNEL_TENSOR),
                                               ("bf16", False, kvs.KERNEL_GENERAL)])
def test_head_profiles_against_oracle(name, fused, kernel):
    """Per-head profiles ("Context views at marginal cost", Tier 1 views: "within head
    H" of a retrieval-head subset) of four (layer, head) pairs, every step, through the
    separate calls, the bench's fused step, the general kernel and H2O eviction."""
    wl = dataclasses.replace(SMALL[name], steps=min(SMALL[name].steps, 9))
    run = harness.Run(wl, oracle_seqs=list(range(wl.batch)), kernel=kernel, fused=fused, profile_heads=HEADS)
    run.prefill()
    for t in range(wl.steps):
        if fused:
            run.decode_step(select=False, accumulate=False)
            run.accumulate_select()
        else:
            run.decode_step(select=True)
        _check_head_profiles(run, HEADS)
    assert run.cache.get_status() == 0, run.cache.last_error()


def test_head_profiles_after_snapkv_scoring():
    """SnapKV prefill scoring as the first step: the profiled heads' pooled in-block votes
    start the profiles, then decode steps add their weights."""
    wl = dataclasses.replace(SMALL["e4m3-window"], steps=3)
    run = harness.Run(wl, oracle_seqs=list(range(wl.batch)), kernel=kvs.KERNEL_TENSOR, obs_window=32,
                      profile_heads=HEADS)
    run.prefill()
    run.prefill_score(16, rel=1e-5)
    _check_head_profiles(run, HEADS, rel=1e-5)         # pooled votes: the SnapKV bar
    for t in range(wl.steps):
        run.decode_step(select=False)
        _check_head_profiles(run, HEADS, rel=1e-5)
    assert run.cache.get_status() == 0, run.cache.last_error()
