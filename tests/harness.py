"""Drive one workload through the CUDA path (C ABI via the binding) and the oracle.

The GPU side runs every sequence of the workload; the oracle tracks a chosen subset
(``oracle_seqs``) on the same seeded inputs.  After each step the GPU state is read
back (codes, scales, positions, masses, score tables, kept blocks) and compared with
the oracle, position by position, at the tolerances stated in the check functions.
"""

import ctypes

import numpy as np
import torch

import attention_scored_kv_gb300 as kvs
import workloads
from oracle.cache import OracleKV

OUT_TOL = {"f32": 1e-4, "bf16": 2e-3, "e4m3": 2e-3}   # max relative error per (seq, head) row
SCORE_TOL = 1e-4                                       # absolute, masses and score tables
_FMT = {"f32": kvs.F32, "bf16": kvs.BF16, "e4m3": kvs.E4M3}


def make_config(wl, kernel=kvs.KERNEL_AUTO, spin_limit=0, traj_len=0, profile_layers=(), obs_window=0,
                profile_heads=()):
    heads = [l * 65536 + h for l, h in profile_heads] + [0] * (4 - len(profile_heads))
    return kvs.config_init(
        n_profile_heads=len(profile_heads), profile_heads=(ctypes.c_int32 * 4)(*heads),
        obs_window=obs_window, traj_len=traj_len, profile_layers=sum(1 << l for l in profile_layers),
        num_layers=wl.num_layers, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
        max_seqs=wl.batch, max_positions=wl.max_positions, window=wl.window, block_tokens=wl.block_tokens,
        h2o_budget_tokens=wl.h2o_budget_tokens, h2o_sink_tokens=wl.h2o_sink_tokens,
        h2o_recent_frac=wl.h2o_recent_frac, ema_decay=wl.ema_decay, kv_dtype=_FMT[wl.kv_format],
        in_dtype=_FMT[wl.in_dtype], kernel=kernel, spin_limit=spin_limit)


def make_oracle(wl, n, traj_len=0, profile_layers=(), profile_heads=()):
    return OracleKV(traj_len=traj_len, profile_layers=tuple(profile_layers), profile_heads=tuple(profile_heads),num_layers=wl.num_layers, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                    head_dim=wl.head_dim, num_seqs=n, max_positions=wl.max_positions, kv_format=wl.kv_format,
                    window=wl.window, h2o_budget_tokens=wl.h2o_budget_tokens,
                    h2o_sink_tokens=wl.h2o_sink_tokens, h2o_recent_frac=wl.h2o_recent_frac,
                    ema_decay=wl.ema_decay, block_tokens=wl.block_tokens)


def rel_err_rows(got, ref):
    """max over rows (last axis = head_dim) of max|got - ref| / max|ref|."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.max(np.abs(got - ref), axis=-1)
    den = np.maximum(np.max(np.abs(ref), axis=-1), 1e-30)
    return float(np.max(num / den))


class StateView:
    """GPU state of one step, read back once, indexed by absolute position."""

    def __init__(self, cache, wl):
        self.cache, self.wl = cache, wl
        self.lay = cache.layout()
        self._cache = {}

    def raw(self, what, layer=0):
        key = (what, layer)
        if key not in self._cache:
            self._cache[key] = self.cache.read_state(what, layer).cpu().numpy()
        return self._cache[key]

    def block_table(self):
        return self.raw(kvs.STATE_BLOCK_TABLE).view(np.int32).reshape(self.wl.batch, self.lay.max_blocks)

    def page_slot(self, s, positions):
        positions = np.asarray(positions, np.int64)
        if self.lay.mode == kvs.MODE_WINDOW:
            w = positions % self.wl.window
            return s * self.lay.pages_per_seq + w // 16, w % 16
        if self.lay.mode == kvs.MODE_H2O:
            return self.block_table()[s, positions // 16].astype(np.int64), positions % 16
        return s * self.lay.pages_per_seq + positions // 16, positions % 16

    def positions(self, layer):
        return self.raw(kvs.STATE_POSITIONS, layer).view(np.int64).reshape(-1, 16)

    def next_position(self, layer):
        return self.raw(kvs.STATE_NEXT_POSITION, layer).view(np.int64)

    def token_mass(self, layer):
        return self.raw(kvs.STATE_TOKEN_MASS, layer).view(np.float32).reshape(-1, 16)

    def block_mass(self, layer):
        return self.raw(kvs.STATE_BLOCK_MASS, layer).view(np.float32).reshape(self.wl.batch, self.lay.max_blocks)

    def table(self, what):
        a = self.raw(what).view(np.float64)
        per = self.wl.max_positions if what in (kvs.STATE_C_TOKEN, kvs.STATE_E_TOKEN) else self.lay.max_blocks
        return a.reshape(self.wl.batch, per)

    def codes(self, which, layer):
        """Raw page bytes as [num_pages, Hkv, 16, head_dim * element bytes]."""
        what = kvs.STATE_K_PAGES if which == "k" else kvs.STATE_V_PAGES
        return self.raw(what, layer).reshape(self.lay.num_pages, self.wl.num_kv_heads, 16, -1)

    def scales(self, which, layer):
        what = kvs.STATE_K_SCALES if which == "k" else kvs.STATE_V_SCALES
        return self.raw(what, layer).view(np.float32).reshape(-1, 16)


class Run:
    """One workload on the GPU, with the oracle tracking ``oracle_seqs``."""

    def __init__(self, wl, oracle_seqs=(0,), kernel=kvs.KERNEL_AUTO, device="cuda", spin_limit=0, fused=False,
                 traj_len=0, profile_layers=(), obs_window=0, profile_heads=()):
        self.wl = wl
        self.fused = fused            # decode steps through append_attend (one call per layer)
        self.inp = workloads.Inputs(wl, device=device)
        self.cache = kvs.KVCache(make_config(wl, kernel, spin_limit, traj_len, profile_layers, obs_window,
                                             profile_heads))
        self.oseqs = list(oracle_seqs)
        self.oracle = (make_oracle(wl, len(self.oseqs), traj_len, profile_layers, profile_heads) if self.oseqs
                       else None)
        self.lens = self.inp.prefill_lengths()
        self.step = 0
        self.last_out = {}

    # ------------------------------------------------------------------ prefill
    def prefill(self):
        wl, c = self.wl, self.cache
        chunk = wl.prefill_chunk or max(int(self.lens.max()), 1)
        uniform = wl.context_range is None
        for l in range(wl.num_layers):
            if uniform:
                if wl.context == 0:
                    continue
                ks, vs = zip(*[self.inp.prefill_kv(l, s) for s in range(wl.batch)])
                k = torch.stack(ks)
                v = torch.stack(vs)
                for a in range(0, wl.context, chunk):
                    c.append_kv(l, k[:, a:a + chunk].contiguous(), v[:, a:a + chunk].contiguous())
                for i, s in enumerate(self.oseqs):
                    self._oracle_append_chunks(l, i, k[s], v[s], chunk)
                del k, v
            else:
                for s in range(wl.batch):
                    k, v = self.inp.prefill_kv(l, s)
                    for a in range(0, k.shape[0], chunk):
                        c.append_kv(l, k[None, a:a + chunk].contiguous(), v[None, a:a + chunk].contiguous(),
                                    seq_begin=s)
                    if s in self.oseqs:
                        self._oracle_append_chunks(l, self.oseqs.index(s), k, v, chunk)

    def prefill_score(self, n_obs, rel=0.0):
        """SnapKV scoring of every layer on both sides, then the accumulate (the tables'
        first step); checks the block and entry masses of the oracle's sequences
        against the bar tol + rel * |ref| before the accumulate."""
        wl, c = self.wl, self.cache
        qs = [self.inp.obs_q(l, n_obs) for l in range(wl.num_layers)]
        for l in range(wl.num_layers):
            c.prefill_score(l, qs[l])
            for i, s in enumerate(self.oseqs):
                self.oracle.prefill_score(l, i, workloads.as_f64(qs[l][s]))
        worst = check_masses(self, rel=rel)
        c.accumulate_scores()
        self.oracle.accumulate()
        return worst

    def _oracle_append_chunks(self, l, i, k, v, chunk):
        kf, vf = workloads.as_f64(k), workloads.as_f64(v)
        for a in range(0, kf.shape[0], chunk):
            self.oracle.append(l, i, kf[a:a + chunk], vf[a:a + chunk])

    # ------------------------------------------------------------------ one decode step
    def decode_step(self, select=True, compare_outputs=True, accumulate=True):
        """Run one step on both sides; returns a dict of oracle-vs-GPU results."""
        wl, c, t = self.wl, self.cache, self.step
        res = {"out_err": 0.0}
        for l in range(wl.num_layers):
            k, v = self.inp.step_kv(l, t)
            q = self.inp.step_q(l, t)
            if self.fused:
                out = c.append_attend(l, k, v, q)
            else:
                c.append_kv(l, k, v)
                out = c.decode_attend(l, q)
            self.last_out[l] = out
            if self.oracle is not None:
                kf, vf, qf = workloads.as_f64(k), workloads.as_f64(v), workloads.as_f64(q)
                for i, s in enumerate(self.oseqs):
                    self.oracle.append(l, i, kf[s], vf[s])
                    ref, _, _ = self.oracle.attend(l, i, qf[s])
                    if compare_outputs:
                        got = out[s].double().cpu().numpy()
                        res["out_err"] = max(res["out_err"], rel_err_rows(got, ref))
        if accumulate:
            c.accumulate_scores()
            if self.oracle is not None:
                res["oracle_step"] = self.oracle.accumulate()
        if select:
            res["keep"] = self.select()
        self.step += 1
        return res

    def select(self):
        """Select on both sides with the workload's rule; returns (gpu, oracle) keep lists."""
        wl, c = self.wl, self.cache
        sv = StateView(c, wl)
        lay = sv.lay
        if wl.h2o_budget_tokens > 0:
            kb = wl.h2o_budget_tokens // 16
            ids, cnt = c.select_blocks(kb, flags=kvs.SELECT_PROTECT | kvs.SELECT_APPLY)
            ks = None
        else:
            ncand = self.candidate_counts()
            ks = torch.tensor([wl.keep_k(int(n)) for n in ncand], dtype=torch.int32, device="cuda")
            ids, cnt = c.select_blocks(ks, keep_capacity=lay.max_blocks)
        ids, cnt = ids.cpu().numpy(), cnt.cpu().numpy()
        gpu = {s: list(ids[s, :cnt[s]]) for s in range(wl.batch)}
        ora = {}
        if self.oracle is not None:
            for i, s in enumerate(self.oseqs):
                if wl.h2o_budget_tokens > 0:
                    ora[s] = self.oracle.select(i, wl.h2o_budget_tokens // 16, protect=True, apply=True)
                else:
                    ora[s] = self.oracle.select(i, int(ks[s].item()))
        return gpu, ora

    def accumulate_select(self):
        """The bench's end of a step: accumulate_select on the GPU (one launch); the
        oracle accumulates, then selects with the same rule as select()."""
        wl, c = self.wl, self.cache
        lay = c.layout()
        if self.oracle is not None:
            self.oracle.accumulate()
        if wl.h2o_budget_tokens > 0:
            ids, cnt = c.accumulate_select(wl.h2o_budget_tokens // 16, flags=kvs.SELECT_PROTECT | kvs.SELECT_APPLY)
            ks = None
        else:
            ks = torch.tensor([wl.keep_k(int(n)) for n in self.candidate_counts()], dtype=torch.int32, device="cuda")
            ids, cnt = c.accumulate_select(ks, keep_capacity=lay.max_blocks)
        ids, cnt = ids.cpu().numpy(), cnt.cpu().numpy()
        gpu = {s: list(ids[s, :cnt[s]]) for s in range(wl.batch)}
        ora = {}
        if self.oracle is not None:
            for i, s in enumerate(self.oseqs):
                if wl.h2o_budget_tokens > 0:
                    ora[s] = self.oracle.select(i, wl.h2o_budget_tokens // 16, protect=True, apply=True)
                else:
                    ora[s] = self.oracle.select(i, int(ks[s].item()))
        return gpu, ora

    def candidate_counts(self):
        """Resident blocks per sequence, from the host-side rule of the mode."""
        wl = self.wl
        out = []
        for s in range(wl.batch):
            nxt = int(self.lens[s]) + self.step + 1
            lo = max(0, nxt - wl.window) if wl.window else 0
            out.append((nxt - 1) // 16 - lo // 16 + 1)
        return out


# ---------------------------------------------------------------------- checks
def check_storage(run, layers=None, exact=True):
    """E4M3 codes and scales bit-exact, positions exact, for the oracle's sequences."""
    wl, sv, o = run.wl, StateView(run.cache, run.wl), run.oracle
    bad = []
    for l in (range(wl.num_layers) if layers is None else layers):
        pos_arr = sv.positions(l)
        nxt = sv.next_position(l)
        for i, s in enumerate(run.oseqs):
            assert nxt[s] == o.next_position[l, i], ("next_position", l, s, nxt[s], o.next_position[l, i])
            rp = o.resident_positions(l, i)
            page, slot = sv.page_slot(s, rp)
            assert np.array_equal(pos_arr[page, slot], rp), ("positions", l, s)
            if wl.kv_format == "e4m3":
                for which in ("k", "v"):
                    codes = sv.codes(which, l)[page, :, slot, :]
                    ref = (o.k_codes if which == "k" else o.v_codes)[l, i, rp]
                    if not np.array_equal(codes, ref):
                        n = int(np.sum(codes != ref))
                        bad.append((which, l, s, n))
                    sc = sv.scales(which, l)[page, slot].astype(np.float64)
                    rsc = (o.k_scale if which == "k" else o.v_scale)[l, i, rp]
                    assert np.array_equal(sc, rsc), ("scales", which, l, s)
            elif wl.kv_format == "bf16":
                vals = np.ascontiguousarray(sv.codes("k", l)).view(np.uint16)
                got = vals[page, :, slot, :].astype(np.uint32) << 16
                ref = o.k_vals[l, i, rp].astype(np.float32).view(np.uint32)
                assert np.array_equal(got, ref), ("bf16 K copy", l, s)
    assert not bad, ("E4M3 code mismatches (cache, layer, seq, count)", bad[:8])


def check_masses(run, tol=SCORE_TOL, rel=0.0):
    """Entry masses and block masses of every layer of the last step: |got - ref| <=
    tol + rel * |ref| (rel > 0 for prefill-scored masses, which sum many queries)."""
    wl, sv, o = run.wl, StateView(run.cache, run.wl), run.oracle
    worst = 0.0
    for l in range(wl.num_layers):
        tm, bm = sv.token_mass(l), sv.block_mass(l)
        for i, s in enumerate(run.oseqs):
            pos, tau = o.token_mass(l, i)
            page, slot = sv.page_slot(s, pos)
            worst = max(worst, float(np.max(np.abs(tm[page, slot] - tau) / (tol + rel * np.abs(tau)))))
            for k, m in o.block_mass(l, i).items():
                worst = max(worst, abs(float(bm[s, k]) - m) / (tol + rel * abs(m)))
    assert worst <= 1.0, ("mass error over the bar", worst)
    return worst


def check_scores(run, tol=SCORE_TOL, rel=0.0):
    """Cumulative and EMA tables, token and block level, for the oracle's sequences."""
    wl, sv, o = run.wl, StateView(run.cache, run.wl), run.oracle
    errs = {}
    for name, what, attr in (("C_tok", kvs.STATE_C_TOKEN, "c_tok"), ("E_tok", kvs.STATE_E_TOKEN, "e_tok"),
                             ("C_blk", kvs.STATE_C_BLOCK, "c_blk"), ("E_blk", kvs.STATE_E_BLOCK, "e_blk")):
        g = sv.table(what)
        e = 0.0
        for i, s in enumerate(run.oseqs):
            ref = getattr(o.scores[i], attr)
            n = min(len(ref), g.shape[1])
            e = max(e, float(np.max(np.abs(g[s, :n] - ref[:n]) / (tol + rel * np.abs(ref[:n])))))
        errs[name] = e
    steps = sv.raw(kvs.STATE_STEPS).view(np.int32)
    for i, s in enumerate(run.oseqs):
        assert steps[s] == o.scores[i].steps
    assert all(v <= 1.0 for v in errs.values()), ("score error over the bar", errs)
    return errs


def check_selection(run, keep, tol=SCORE_TOL, table="c_blk", rel=0.0):
    """Same kept set except blocks whose oracle score is within tol of the cut-off
    (the lowest score kept on score alone; protected H2O blocks do not set it)."""
    from oracle import selection
    gpu, ora = keep
    wl = run.wl
    for i, s in enumerate(run.oseqs):
        g, r = set(int(x) for x in gpu[s]), set(int(x) for x in ora[s])
        assert list(gpu[s]) == sorted(gpu[s]), "keep ids must ascend"
        if g == r:
            continue
        sc = getattr(run.oracle.scores[i], table)
        prot = set()
        if wl.h2o_budget_tokens > 0:
            nxt = int(run.oracle.next_position[0, i])
            prot = set(selection.protected_blocks(range(len(sc)), nxt, wl.h2o_sink_tokens,
                                                  run.oracle.h2o_recent_tokens))
        by_score = r - prot
        cut = min(sc[k] for k in by_score) if by_score else 0.0
        for k in g ^ r:
            assert abs(sc[k] - cut) <= tol + rel * abs(cut), ("selection differs beyond the cut-off band", s, k,
                                                              sc[k], cut)
        assert len(g) == len(r), ("kept counts differ", s, len(g), len(r))
