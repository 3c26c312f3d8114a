"""Scattered sequences through every call of the C ABI, against the oracle.

A serving batch rarely occupies a contiguous range of the cache's sequences, so every
per-sequence call also takes a list of sequence ids (kvs_seqs in list form: the ids in
host memory for the library's checks and plans, and in device memory for its kernels).
Here the list {5, 0, 11} (out of 12 sequences, not in ascending order) is driven
through append, attend (with the optional per-position token-mass output), the fused
append + attend, accumulate, select, the fused accumulate + select, the threshold
filter, the block-list re-attend, SnapKV prefill scoring, score export / import and
reset, and compared with the oracle tracking those three sequences at the decode
bars.  The sequences not listed must come through untouched.  An H2O cache with
eviction runs the list {3, 0} the same way.
"""
import dataclasses

import numpy as np
import pytest
import torch

import attention_scored_kv_gb300 as kvs
import workloads
from tests import harness

pytestmark = pytest.mark.gpu

IDS = [5, 0, 11]
WL = workloads.scaled_down("e4m3-b16-ctx32768-window4096", name="seq-ids-window", num_layers=2, batch=12,
                           context=300, window=128, steps=8, prefill_chunk=64)
H2O = workloads.scaled_down("e4m3-b64-ragged-h2o2048", name="seq-ids-h2o", num_layers=2, batch=5,
                            context_range=(100, 400), h2o_budget_tokens=128, steps=10, prefill_chunk=128)


def _rows(t, ids):
    return t[torch.tensor(ids, device=t.device)].contiguous()


def _list_step(run, ids, seq, fused):
    """One decode step of the listed sequences only: every layer through the list form,
    outputs and per-position token masses against the oracle; then accumulate."""
    wl, c, t = run.wl, run.cache, run.step
    oidx = [run.oseqs.index(s) for s in ids]
    worst = 0.0
    for l in range(wl.num_layers):
        k, v = run.inp.step_kv(l, t)
        q = run.inp.step_q(l, t)
        k, v, q = _rows(k, ids), _rows(v, ids), _rows(q, ids)
        tm = torch.full((len(ids), wl.max_positions), -7.0, dtype=torch.float32, device="cuda")
        if fused:
            out = c.append_attend(l, k, v, q, seq_ids=seq, tok_mass_out=tm)
        else:
            c.append_kv(l, k, v, seq_ids=seq)
            out = c.decode_attend(l, q, seq_ids=seq, tok_mass_out=tm)
        kf, vf, qf = workloads.as_f64(k), workloads.as_f64(v), workloads.as_f64(q)
        tmh = tm.cpu().numpy().astype(np.float64)
        for i, oi in enumerate(oidx):
            run.oracle.append(l, oi, kf[i], vf[i])
            ref, _, _ = run.oracle.attend(l, oi, qf[i])
            worst = max(worst, harness.rel_err_rows(out[i].double().cpu().numpy(), ref))
            pos, tau = run.oracle.token_mass(l, oi)
            assert np.max(np.abs(tmh[i, pos] - tau)) <= harness.SCORE_TOL, (l, ids[i])
            others = np.ones(wl.max_positions, bool)
            others[pos] = False
            assert np.all(tmh[i, others] == -7.0), "positions not resident must be left as they were"
    assert worst <= harness.OUT_TOL[wl.kv_format], worst
    c.accumulate_scores(seq_ids=seq)
    run.oracle.accumulate(seqs=oidx)
    run.step += 1


def _select_list(run, ids, seq, fused_acc=False):
    """select (or, with fused_acc, accumulate + select) on the list; kept sets against
    the oracle's."""
    wl, c = run.wl, run.cache
    oidx = [run.oseqs.index(s) for s in ids]
    lay = c.layout()
    if wl.h2o_budget_tokens > 0:
        kb = wl.h2o_budget_tokens // 16
        fn = c.accumulate_select if fused_acc else c.select_blocks
        ids_t, cnt = fn(kb, seq_ids=seq, flags=kvs.SELECT_PROTECT | kvs.SELECT_APPLY)
        ora = {s: run.oracle.select(oi, kb, protect=True, apply=True) for s, oi in zip(ids, oidx)}
    else:
        ks = [wl.keep_k(len(run.oracle.resident_block_ids(oi))) for oi in oidx]
        kt = torch.tensor(ks, dtype=torch.int32, device="cuda")
        fn = c.accumulate_select if fused_acc else c.select_blocks
        ids_t, cnt = fn(kt, seq_ids=seq, keep_capacity=lay.max_blocks)
        ora = {s: run.oracle.select(oi, k) for s, oi, k in zip(ids, oidx, ks)}
    ids_h, cnt_h = ids_t.cpu().numpy(), cnt.cpu().numpy()
    gpu = {s: list(ids_h[i, :cnt_h[i]]) for i, s in enumerate(ids)}
    harness.check_selection(run, (gpu, ora))
    return ids_t, cnt


def _untouched(before, after, ids):
    for s in range(len(before)):
        if s not in ids:
            assert before[s] == after[s], ("a sequence outside the list moved", s)


def test_scattered_sequences_window_cache():
    run = harness.Run(WL, oracle_seqs=IDS, kernel=kvs.KERNEL_TENSOR, obs_window=32)
    run.prefill()
    c = run.cache
    seq = kvs.SeqIds(IDS)
    nxt0 = harness.StateView(c, WL).next_position(0).copy()

    # SnapKV prefill scoring on the list, folded in as the first step
    for l in range(WL.num_layers):
        q = _rows(run.inp.obs_q(l, 16), IDS)
        c.prefill_score(l, q, seq_ids=seq)
        for i, s in enumerate(IDS):
            run.oracle.prefill_score(l, run.oseqs.index(s), workloads.as_f64(q[i]))
    harness.check_masses(run, rel=1e-5)
    c.accumulate_scores(seq_ids=seq)
    run.oracle.accumulate(seqs=[run.oseqs.index(s) for s in IDS])
    harness.check_scores(run, rel=1e-5)

    for t in range(6):
        _list_step(run, IDS, seq, fused=(t % 2 == 1))
        harness.check_masses(run)
        harness.check_scores(run, rel=1e-5)
        keep, cnt = _select_list(run, IDS, seq)
    harness.check_storage(run)
    nxt1 = harness.StateView(c, WL).next_position(0).copy()
    _untouched(nxt0, nxt1, IDS)
    assert all(nxt1[s] == nxt0[s] + 6 for s in IDS)

    # threshold filter on the list, at the median of each sequence's resident scores
    sv = harness.StateView(c, WL)
    cblk = sv.table(kvs.STATE_C_BLOCK)
    theta = float(np.median([cblk[s, b] for s in IDS for b in run.oracle.resident_block_ids(run.oseqs.index(s))]))
    fids, fcnt = c.filter_blocks(theta, seq_ids=seq)
    fids, fcnt = fids.cpu().numpy(), fcnt.cpu().numpy()
    for i, s in enumerate(IDS):
        ref = run.oracle.filter_blocks(run.oseqs.index(s), "cumulative", theta)
        got = list(fids[i, :fcnt[i]])
        sc = run.oracle.scores[run.oseqs.index(s)].c_blk
        for b in set(got) ^ set(ref):
            assert abs(sc[b] - theta) <= harness.SCORE_TOL, (s, b)

    # Tier-2 re-attend over the kept blocks of the list
    for l in range(WL.num_layers):
        q = _rows(run.inp.step_q(l, 50), IDS)
        out = c.attend_blocks(l, q, keep, cnt, seq_ids=seq)
        kh, ch = keep.cpu().numpy(), cnt.cpu().numpy()
        for i, s in enumerate(IDS):
            ref, _, _ = run.oracle.attend_blocks(l, run.oseqs.index(s), workloads.as_f64(q[i]), kh[i, :ch[i]])
            assert harness.rel_err_rows(out[i].double().cpu().numpy(), ref) <= harness.OUT_TOL[WL.kv_format]

    # fused accumulate + select on the list (one more list step first)
    for l in range(WL.num_layers):
        k, v = run.inp.step_kv(l, run.step)
        q = run.inp.step_q(l, run.step)
        c.append_attend(l, _rows(k, IDS), _rows(v, IDS), _rows(q, IDS), seq_ids=seq)
        for i, s in enumerate(IDS):
            oi = run.oseqs.index(s)
            run.oracle.append(l, oi, workloads.as_f64(_rows(k, IDS))[i], workloads.as_f64(_rows(v, IDS))[i])
            run.oracle.attend(l, oi, workloads.as_f64(_rows(q, IDS))[i])
    run.oracle.accumulate(seqs=[run.oseqs.index(s) for s in IDS])
    run.step += 1
    _select_list(run, IDS, seq, fused_acc=True)
    harness.check_scores(run, rel=1e-5)

    # export in list order equals the per-sequence exports; import into other sequences
    snap = c.export_scores(seq_ids=[11, 5]).cpu()
    one11 = c.export_scores(seq_begin=11, n_seqs=1).cpu()
    one5 = c.export_scores(seq_begin=5, n_seqs=1).cpu()
    c.import_scores(snap.cuda(), seq_ids=[2, 7])
    assert torch.equal(c.export_scores(seq_ids=[2, 7]).cpu(), snap)
    assert torch.equal(c.export_scores(seq_begin=2, n_seqs=1).cpu(), one11)
    assert torch.equal(c.export_scores(seq_begin=7, n_seqs=1).cpu(), one5)

    # reset on a list empties exactly those sequences
    before = harness.StateView(c, WL).next_position(1).copy()
    c.reset(seq_ids=[11, 0])
    after = harness.StateView(c, WL).next_position(1).copy()
    assert after[11] == 0 and after[0] == 0 and after[5] == before[5]
    _untouched(before, after, [11, 0])
    assert c.get_status() == 0, c.last_error()


def test_scattered_sequences_h2o_eviction():
    ids = [3, 0]
    run = harness.Run(H2O, oracle_seqs=ids, kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    seq = kvs.SeqIds(ids)
    c = run.cache
    nxt0 = harness.StateView(c, H2O).next_position(0).copy()
    for t in range(8):
        _list_step(run, ids, seq, fused=(t % 2 == 0))
        harness.check_masses(run)
        harness.check_scores(run)
        _select_list(run, ids, seq, fused_acc=False)
    harness.check_storage(run)
    _untouched(nxt0, harness.StateView(c, H2O).next_position(0).copy(), ids)
    assert c.get_status() == 0, c.last_error()


def test_sequence_lists_are_checked():
    run = harness.Run(dataclasses.replace(WL, num_layers=1), oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    c = run.cache
    q = _rows(run.inp.step_q(0, 0), [1, 1])
    with pytest.raises(kvs.KVSError) as e:                   # a repeated id
        c.decode_attend(0, q, seq_ids=[1, 1])
    assert e.value.status == 1
    with pytest.raises(kvs.KVSError) as e:                   # an id beyond max_seqs
        c.decode_attend(0, q, seq_ids=[1, 12])
    assert e.value.status == 1
    with pytest.raises(ValueError):                          # rows and ids disagree
        c.decode_attend(0, q, seq_ids=[1, 2, 3])
    assert c.get_status() == 0
