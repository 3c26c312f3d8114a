"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Sizes are small enough for the oracle to follow every sequence and every step, yet
span several 16-token blocks, several CTAs per sequence and ragged tails.  Bars:
E4M3 codes, scales, slots and absolute positions bit-exact; attention output within
2e-3 (bf16 / E4M3 inputs) or 1e-4 (f32) max relative error per (sequence, head) row;
masses and score tables within 1e-4 absolute; kept block sets equal except for
blocks whose oracle score lies within 1e-4 of the cut-off.
"""
import dataclasses

import numpy as np
import pytest
import torch

import attention_scored_kv_gb300 as kvs
import workloads
from tests import harness

pytestmark = pytest.mark.gpu


def _full_check(wl, kernel=kvs.KERNEL_AUTO, steps=None, every=1, fused=False):
    run = harness.Run(wl, oracle_seqs=list(range(wl.batch)), kernel=kernel, fused=fused)
    run.prefill()
    worst = 0.0
    n = wl.steps if steps is None else steps
    for t in range(n):
        res = run.decode_step(select=False)
        worst = max(worst, res["out_err"])
        check = t % every == 0 or t == n - 1
        if check:   # masses are read through the block table, so before any eviction
            harness.check_masses(run)
            harness.check_scores(run)
        keep = run.select()
        if check:
            harness.check_selection(run, keep)
    harness.check_storage(run)
    assert worst <= harness.OUT_TOL[wl.kv_format], worst
    assert run.cache.get_status() == 0, run.cache.last_error()
    return run, worst


# ------------------------------------------------------------------ tiny (general kernel)
@pytest.mark.parametrize("seed", [7, 19, 41])
def test_tiny_f32_window4(seed):
    wl = workloads.scaled_down("tiny-f32-window4", name="tiny-%d" % seed, seed=seed)
    run, _ = _full_check(wl)
    assert run.cache.layout().attend_kernel == kvs.KERNEL_GENERAL


# ------------------------------------------------------------------ tensor-core kernel
SMALL = {
    "bf16": workloads.scaled_down("bf16-b8-ctx4096", num_layers=2, batch=3, context=300, steps=12),
    "e4m3-window": workloads.scaled_down("e4m3-b16-ctx32768-window4096", num_layers=2, batch=3, context=700,
                                         window=256, steps=12, prefill_chunk=128),
    "e4m3-nowindow": workloads.scaled_down("e4m3-b16-ctx32768-window4096", num_layers=2, batch=2, context=513,
                                           window=0, steps=6, prefill_chunk=0),
    "bf16-hkv8": workloads.scaled_down("bf16-b1-ctx131072-planted", num_layers=2, batch=2, context=1000,
                                       retrieval_pos=500, steps=6, prefill_chunk=0),
    "e4m3-h2o": workloads.scaled_down("e4m3-b64-ragged-h2o2048", num_layers=2, batch=5, context_range=(100, 700),
                                      h2o_budget_tokens=256, steps=40, prefill_chunk=256),
    # 16 sequences of 65 resident blocks: several blocks per CTA and about 9 CTAs per
    # sequence, the shape of the 32K-context batch at a smaller window
    "e4m3-b16-window": workloads.scaled_down("e4m3-b16-ctx32768-window4096", num_layers=2, batch=16,
                                             context=2500, window=1024, steps=6, prefill_chunk=512),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_tensor_kernel_small(name):
    wl = SMALL[name]
    run, worst = _full_check(wl, kernel=kvs.KERNEL_TENSOR, every=3)
    assert run.cache.layout().attend_kernel == kvs.KERNEL_TENSOR


@pytest.mark.parametrize("name", ["bf16", "e4m3-window", "e4m3-nowindow", "e4m3-b16-window", "e4m3-h2o"])
def test_fused_append_attend_against_oracle(name):
    """append_attend (one launch per layer where the context allows; two calls for H2O)
    against the oracle, every step."""
    _full_check(SMALL[name], kernel=kvs.KERNEL_TENSOR, every=3, fused=True)


def _state(cache, L):
    names = [kvs.STATE_K_PAGES, kvs.STATE_V_PAGES, kvs.STATE_POSITIONS, kvs.STATE_TOKEN_MASS, kvs.STATE_BLOCK_MASS,
             kvs.STATE_NEXT_POSITION]
    if cache.cfg.kv_dtype == kvs.E4M3:
        names += [kvs.STATE_K_SCALES, kvs.STATE_V_SCALES]
    return {(n, l): cache.read_state(n, l).cpu() for n in names for l in range(L)}


@pytest.mark.parametrize("name,steps", [("e4m3-b16-window", 20), ("bf16", 18), ("e4m3-nowindow", 17)])
def test_fused_append_attend_is_bitwise_the_two_calls(name, steps):
    """The single-launch form stores the same bytes and computes the same outputs and
    masses, bit for bit, as append_kv followed by decode_attend (the window wraps and
    blocks fill and start during these steps)."""
    wl = dataclasses.replace(SMALL[name], steps=steps)
    a = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    b = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR, fused=True)
    a.prefill()
    b.prefill()
    for t in range(steps):
        a.decode_step(select=False)
        b.decode_step(select=False)
        for l in range(wl.num_layers):
            assert torch.equal(a.last_out[l], b.last_out[l]), (t, l)
    sa, sb = _state(a.cache, wl.num_layers), _state(b.cache, wl.num_layers)
    for key in sa:
        assert torch.equal(sa[key], sb[key]), key
    for n in (kvs.STATE_C_TOKEN, kvs.STATE_E_TOKEN, kvs.STATE_C_BLOCK, kvs.STATE_E_BLOCK):
        assert torch.equal(a.cache.read_state(n).cpu(), b.cache.read_state(n).cpu()), n
    assert a.cache.get_status() == 0 and b.cache.get_status() == 0


def test_fused_append_attend_from_an_empty_cache():
    """The first token of every sequence through append_attend (no entry before it), then
    a few more: one block per sequence, fewer blocks than CTAs."""
    wl = workloads.scaled_down("e4m3-b16-ctx32768-window4096", name="fused-empty", num_layers=2, batch=4,
                               context=0, window=64, steps=20, prefill_chunk=0)
    _full_check(wl, kernel=kvs.KERNEL_TENSOR, every=1, fused=True)


@pytest.mark.parametrize("name,kind,krule", [
    ("e4m3-b16-window", kvs.SCORE_CUMULATIVE, "per-seq"),
    ("e4m3-b16-window", kvs.SCORE_TOVA, "per-seq"),
    ("bf16", kvs.SCORE_TOKEN_SUM, 3),
    ("e4m3-h2o", kvs.SCORE_TOVA, "h2o"),
    ("bf16", kvs.SCORE_EMA, 3),
    ("e4m3-nowindow", kvs.SCORE_EMA, 0),
    ("e4m3-window", kvs.SCORE_CUMULATIVE, 10 ** 6),
    ("e4m3-h2o", kvs.SCORE_CUMULATIVE, "h2o"),
    ("e4m3-h2o", kvs.SCORE_EMA, "h2o"),
])
def test_accumulate_select_is_bitwise_the_two_calls(name, kind, krule):
    """accumulate_select (one launch) keeps the same ids and writes the same tables, bit
    for bit, as accumulate_scores then select_blocks: per-sequence and uniform k, k = 0,
    k above the block count, cumulative and EMA keys, H2O protection with eviction."""
    wl = dataclasses.replace(SMALL[name], steps=min(SMALL[name].steps, 12))
    runs = [harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR) for _ in range(2)]
    for r in runs:
        r.prefill()
    h2o = krule == "h2o"
    for t in range(wl.steps):
        outs = []
        for j, r in enumerate(runs):
            r.decode_step(select=False, accumulate=False)
            c = r.cache
            cap = c.layout().max_blocks
            if h2o:
                k, flags = wl.h2o_budget_tokens // 16, kvs.SELECT_PROTECT | kvs.SELECT_APPLY
            elif krule == "per-seq":
                k = torch.tensor([(3 * s + t) % 9 for s in range(wl.batch)], dtype=torch.int32, device="cuda")
                flags = 0
            else:
                k, flags = krule, 0
            if j == 0:
                c.accumulate_scores()
                ids, cnt = c.select_blocks(k, score_kind=kind, flags=flags, keep_capacity=cap)
            else:
                ids, cnt = c.accumulate_select(k, score_kind=kind, flags=flags, keep_capacity=cap)
            outs.append((ids.cpu(), cnt.cpu()))
        assert torch.equal(outs[0][1], outs[1][1]), t
        for s in range(wl.batch):
            n = int(outs[0][1][s])
            assert torch.equal(outs[0][0][s, :n], outs[1][0][s, :n]), (t, s)
    a, b = runs[0].cache, runs[1].cache
    for n in (kvs.STATE_C_TOKEN, kvs.STATE_E_TOKEN, kvs.STATE_C_BLOCK, kvs.STATE_E_BLOCK, kvs.STATE_STEPS,
              kvs.STATE_S_BLOCK, kvs.STATE_T_BLOCK):
        assert torch.equal(a.read_state(n).cpu(), b.read_state(n).cpu()), n
    if h2o:
        # the same blocks stay resident; which free page a block gets depends on the order
        # in which evicted pages were pushed (atomics), in either form
        bta = a.read_state(kvs.STATE_BLOCK_TABLE).cpu().view(torch.int32)
        btb = b.read_state(kvs.STATE_BLOCK_TABLE).cpu().view(torch.int32)
        assert torch.equal(bta >= 0, btb >= 0)
    assert a.get_status() == 0 and b.get_status() == 0


@pytest.mark.parametrize("name", ["e4m3-window", "bf16", "e4m3-h2o"])
def test_token_sum_and_tova_scores_against_oracle(name):
    """The summed block scores (H2O token sum, TOVA latest weight) and the selections by
    them, against the oracle, every step (window: blocks leave it; H2O: eviction by the
    cumulative score as the workload says, then TOVA and token-sum selections read
    only)."""
    wl = dataclasses.replace(SMALL[name], steps=min(SMALL[name].steps, 10))
    run = harness.Run(wl, oracle_seqs=list(range(wl.batch)), kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    lay = run.cache.layout()
    for t in range(wl.steps):
        run.decode_step(select=False)
        sv = harness.StateView(run.cache, wl)
        sb = sv.raw(kvs.STATE_S_BLOCK).view(np.float64).reshape(wl.batch, lay.max_blocks)
        tb = sv.raw(kvs.STATE_T_BLOCK).view(np.float64).reshape(wl.batch, lay.max_blocks)
        for i, s in enumerate(run.oseqs):
            sc = run.oracle.scores[i]
            n = len(sc.s_blk)
            assert np.max(np.abs(sb[s, :n] - sc.s_blk)) <= harness.SCORE_TOL
            assert np.max(np.abs(tb[s, :n] - sc.t_blk)) <= harness.SCORE_TOL
        for kind, table, okind in ((kvs.SCORE_TOVA, "t_blk", "tova"), (kvs.SCORE_TOKEN_SUM, "s_blk", "token_sum")):
            ncand = run.candidate_counts() if not wl.h2o_budget_tokens else \
                [len(run.oracle.resident_block_ids(i)) for i in range(wl.batch)]
            ks = torch.tensor([max(1, int(n) // 2) for n in ncand], dtype=torch.int32, device="cuda")
            ids, cnt = run.cache.select_blocks(ks, score_kind=kind, keep_capacity=lay.max_blocks)
            ids, cnt = ids.cpu().numpy(), cnt.cpu().numpy()
            gpu = {s: list(ids[s, :cnt[s]]) for s in range(wl.batch)}
            ora = {s: run.oracle.select(i, int(ks[s].item()), score_kind=okind) for i, s in enumerate(run.oseqs)}
            harness.check_selection(run, (gpu, ora), table=table)
        run.select()                                  # the workload's own rule (H2O: evicts)
    assert run.cache.get_status() == 0, run.cache.last_error()


def _reattend_check(run, keep_ids, keep_cnt, t_query):
    """attend_blocks over the kept blocks of every oracle sequence against the oracle's
    Tier-2 re-attend, with a query the cache has not seen; returns the worst error and
    the largest change from full attention (reported, not a bar)."""
    wl = run.wl
    worst, moved = 0.0, 0.0
    for l in range(wl.num_layers):
        q = run.inp.step_q(l, t_query)
        got = run.cache.attend_blocks(l, q, keep_ids, keep_cnt)
        full = run.cache.decode_attend(l, q)     # note: refreshes this layer's step masses
        qf = workloads.as_f64(q)
        for i, s in enumerate(run.oseqs):
            blocks = keep_ids[s, : int(keep_cnt[s])].cpu().numpy()
            ref, _, pos = run.oracle.attend_blocks(l, i, qf[s], blocks)
            worst = max(worst, harness.rel_err_rows(got[s].double().cpu().numpy(), ref))
            moved = max(moved, float((got[s] - full[s]).abs().max()))
    return worst, moved


@pytest.mark.parametrize("name", ["e4m3-b16-window", "bf16", "bf16-hkv8", "e4m3-h2o"])
def test_attend_blocks_against_oracle(name):
    """Tier-2 re-attend over the blocks a selection kept, against the oracle, on the
    tensor-core kernel (window, no window, 8 KV heads, H2O pages)."""
    wl = dataclasses.replace(SMALL[name], steps=min(SMALL[name].steps, 4))
    run = harness.Run(wl, oracle_seqs=list(range(wl.batch)), kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    for t in range(wl.steps - 1):
        run.decode_step(select=False)
        run.select()
    run.decode_step(select=False)
    lay = run.cache.layout()
    ncand = run.candidate_counts() if not wl.h2o_budget_tokens else [lay.max_blocks] * wl.batch
    ks = torch.tensor([max(1, wl.keep_k(int(n)) // 2) for n in ncand], dtype=torch.int32, device="cuda")
    ids, cnt = run.cache.select_blocks(ks, keep_capacity=lay.max_blocks)
    # the oracle keeps its own residency; re-attend reads both sides' kept blocks
    worst, moved = _reattend_check(run, ids, cnt, t_query=wl.steps)
    assert worst <= harness.OUT_TOL[wl.kv_format], worst
    assert moved > 0.0                           # a strict subset changes the output
    assert run.cache.get_status() == 0, run.cache.last_error()


def test_attend_blocks_over_every_block_is_full_attention():
    wl = dataclasses.replace(SMALL["e4m3-window"], steps=2)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    run.decode_step(select=False)
    lay = run.cache.layout()
    ids, cnt = run.cache.select_blocks(10 ** 6, keep_capacity=lay.max_blocks)   # keeps all
    for l in range(wl.num_layers):
        q = run.inp.step_q(l, 5)
        full = run.cache.decode_attend(l, q)
        got = run.cache.attend_blocks(l, q, ids, cnt)
        assert float((got - full).abs().max()) <= 1e-5


def test_attend_blocks_reports_a_bad_block_id():
    wl = dataclasses.replace(SMALL["e4m3-window"], steps=2)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    run.decode_step(select=False)
    lay = run.cache.layout()
    ids, cnt = run.cache.select_blocks(4, keep_capacity=lay.max_blocks)
    bad = ids.clone()
    bad[0, 0] = lay.max_blocks + 7                # out of range: reported, left out
    run.cache.attend_blocks(0, run.inp.step_q(0, 5), bad, cnt)
    assert run.cache.get_status() == kvs._abi.ERR_STATE
    run.cache.clear_error()
    assert run.cache.get_status() == 0


def _many(name, batch, **changes):
    """SMALL[name] with more sequences: forty, more than a CTA each."""
    wl = SMALL[name]
    return workloads.scaled_down(wl.name.replace("-small", ""), **{**_fields(wl), "batch": batch, **changes})


@pytest.mark.parametrize("name", ["bf16", "bf16-hkv8", "e4m3-window", "e4m3-h2o"])
def test_attend_blocks_many_sequences_against_oracle(name):
    """Tier-2 re-attend with 40 sequences against the oracle on three of them."""
    wl = _many(name, 40, steps=3)
    run = harness.Run(wl, oracle_seqs=[0, 17, 39], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    for t in range(wl.steps - 1):
        run.decode_step(select=False)
        run.select()
    run.decode_step(select=False)
    lay = run.cache.layout()
    ncand = run.candidate_counts() if not wl.h2o_budget_tokens else [lay.max_blocks] * wl.batch
    ks = torch.tensor([max(1, wl.keep_k(int(n)) // 2) for n in ncand], dtype=torch.int32, device="cuda")
    ids, cnt = run.cache.select_blocks(ks, keep_capacity=lay.max_blocks)
    worst, moved = _reattend_check(run, ids, cnt, t_query=wl.steps)
    assert worst <= harness.OUT_TOL[wl.kv_format], worst
    assert moved > 0.0
    assert run.cache.get_status() == 0, run.cache.last_error()


def test_attend_blocks_long_lists_many_sequences():
    """Lists of 107 blocks, 40 sequences: every block kept equals full attention, and
    the oracle agrees."""
    wl = _many("e4m3-nowindow", 40, context=1700, steps=2)
    run = harness.Run(wl, oracle_seqs=[0, 39], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    run.decode_step(select=False)
    lay = run.cache.layout()
    ids, cnt = run.cache.select_blocks(10 ** 6, keep_capacity=lay.max_blocks)   # keeps all
    assert int(cnt.min()) > 100
    worst, _ = _reattend_check(run, ids, cnt, t_query=7)
    assert worst <= harness.OUT_TOL[wl.kv_format], worst
    for l in range(wl.num_layers):
        q = run.inp.step_q(l, 9)
        full = run.cache.decode_attend(l, q)
        got = run.cache.attend_blocks(l, q, ids, cnt)
        for b in range(wl.batch):                 # both within the bar of the oracle
            err = harness.rel_err_rows(got[b].double().cpu().numpy(), full[b].double().cpu().numpy())
            assert err <= 2 * harness.OUT_TOL[wl.kv_format], (b, err)
    assert run.cache.get_status() == 0, run.cache.last_error()


def test_attend_blocks_many_sequences_reports_a_bad_block_id():
    wl = _many("e4m3-window", 40, steps=2)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    run.decode_step(select=False)
    lay = run.cache.layout()
    ids, cnt = run.cache.select_blocks(4, keep_capacity=lay.max_blocks)
    bad = ids.clone()
    bad[3, 1] = lay.max_blocks + 7                # out of range: reported, left out
    run.cache.attend_blocks(0, run.inp.step_q(0, 5), bad, cnt)
    assert run.cache.get_status() == kvs._abi.ERR_STATE
    run.cache.clear_error()
    assert run.cache.get_status() == 0


@pytest.mark.parametrize("name", ["bf16", "e4m3-window", "e4m3-h2o"])
def test_general_kernel_on_tensor_shapes(name):
    wl = SMALL[name]
    wl = workloads.scaled_down(wl.name.replace("-small", ""), **{**_fields(wl), "steps": 6})
    run, _ = _full_check(wl, kernel=kvs.KERNEL_GENERAL, every=2)
    assert run.cache.layout().attend_kernel == kvs.KERNEL_GENERAL


def _fields(wl):
    import dataclasses
    d = dataclasses.asdict(wl)
    d.pop("name")
    return d


def test_tensor_and_general_agree():
    wl = SMALL["e4m3-window"]
    outs = []
    for kern in (kvs.KERNEL_TENSOR, kvs.KERNEL_GENERAL):
        run = harness.Run(wl, oracle_seqs=[], kernel=kern)
        run.prefill()
        for _ in range(3):
            run.decode_step(select=False)
        outs.append(torch.stack([run.last_out[l] for l in range(wl.num_layers)]).double().cpu().numpy())
    assert harness.rel_err_rows(outs[0], outs[1]) <= 2e-3


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("window,context,kernel", [
    (1, 5, kvs.KERNEL_GENERAL),          # window 1: only the token just written
    (4, 1, kvs.KERNEL_GENERAL),          # a single prefilled token
    (20, 57, kvs.KERNEL_GENERAL),        # window not a multiple of 16: blocks straddle pages
    (16, 33, kvs.KERNEL_TENSOR),         # one page per sequence, wraps every 16 steps
    (32, 0, kvs.KERNEL_TENSOR),          # empty prefill: decode from the first token
])
def test_window_edges(window, context, kernel):
    base = "tiny-f32-window4" if kernel == kvs.KERNEL_GENERAL else "e4m3-b16-ctx32768-window4096"
    ch = dict(window=window, context=context, steps=20, prefill_chunk=7 if context else 0)
    if kernel == kvs.KERNEL_TENSOR:
        ch.update(num_layers=2, batch=2)
    wl = workloads.scaled_down(base, name="edge-w%d-c%d" % (window, context), **ch)
    _full_check(wl, kernel=kernel)


def test_prefill_chunk_longer_than_window():
    wl = workloads.scaled_down("e4m3-b16-ctx32768-window4096", name="chunk-gt-window", num_layers=1, batch=2,
                               context=300, window=64, steps=3, prefill_chunk=200)
    _full_check(wl, kernel=kvs.KERNEL_TENSOR)


def test_many_sequences_per_cta():
    # 200 short sequences: several sequence boundaries inside one CTA's share
    wl = workloads.scaled_down("e4m3-b16-ctx32768-window4096", name="many-seqs", num_layers=1, batch=200,
                               context=20, window=0, steps=2, prefill_chunk=0)
    run = harness.Run(wl, oracle_seqs=[0, 1, 99, 199], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    for _ in range(wl.steps):
        res = run.decode_step()
        assert res["out_err"] <= 2e-3
        harness.check_masses(run)
        harness.check_scores(run)
    assert run.cache.get_status() == 0


# ------------------------------------------------------------------ errors
def test_attend_on_empty_cache_is_rejected():
    wl = SMALL["bf16"]
    c = kvs.KVCache(harness.make_config(wl))
    q = torch.zeros((wl.batch, wl.num_q_heads, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvs.KVSError) as e:
        c.decode_attend(0, q)
    assert e.value.status == 3


def test_capacity_is_enforced():
    wl = workloads.scaled_down("bf16-b8-ctx4096", num_layers=1, batch=1, context=0, steps=4)
    c = kvs.KVCache(harness.make_config(wl))
    k = torch.zeros((1, 5, wl.num_kv_heads, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvs.KVSError) as e:
        c.append_kv(0, k, k)
    assert e.value.status == 2
    # a failed call leaves the state unchanged
    assert harness.StateView(c, wl).next_position(0)[0] == 0


def test_eviction_needs_h2o_mode():
    wl = SMALL["bf16"]
    c = kvs.KVCache(harness.make_config(wl))
    with pytest.raises(kvs.KVSError) as e:
        c.select_blocks(4, flags=kvs.SELECT_APPLY)
    assert e.value.status == 1


def test_layers_must_agree_at_accumulate():
    wl = workloads.scaled_down("bf16-b8-ctx4096", num_layers=2, batch=1, context=0, steps=4)
    c = kvs.KVCache(harness.make_config(wl))
    k = torch.zeros((1, 1, wl.num_kv_heads, wl.head_dim), dtype=torch.bfloat16, device="cuda")
    c.append_kv(0, k, k)
    with pytest.raises(kvs.KVSError) as e:
        c.accumulate_scores()
    assert e.value.status == 7


def test_bounded_wait_reports_timeout_and_recovers():
    """spin_limit -1: a CTA that is not the last of its sequence to arrive gives up at
    once and flags KVS_ERR_TIMEOUT; the context is usable again after clear_error."""
    wl = workloads.scaled_down("e4m3-b16-ctx32768-window4096", name="timeout", num_layers=1, batch=1,
                               context=4096, window=0, steps=1, prefill_chunk=0)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR, spin_limit=-1)
    run.prefill()
    run.decode_step(select=False)
    assert run.cache.get_status() == 5          # KVS_ERR_TIMEOUT
    run.cache.clear_error()
    assert run.cache.get_status() == 0
