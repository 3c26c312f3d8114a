"""The oracle's KV cache: append log, residency, attend, masses, scores, selection.

Test infrastructure only (see the package docstring).

What one decode step computes (per layer l and sequence b, then per step):
  a1  append: the new token's K and V are stored (FP8: codes + one scale per position
      per cache, ``oracle.e4m3``), at absolute position p = next_position[l][b];
      next_position advances by the number of new tokens.
      ("Context Optimization", FP8 KV Cache > How It Works and Sliding Window
      Attention > Design; "LLM mechanics III", sections 1 and 5.)
  a2  attend: the query of every head attends over the resident entries.
      Window W: position p is resident while p >= next_position - W (the current
      token included, "LLM mechanics III" section 1).  H2O: every entry of a
      resident 16-token block ("Context Optimization", H2O).  No window: all.
  a3  masses: token mass = sum over query heads of the weights; block mass = max over
      query heads of the in-block weight sum ("Per-Head Attention as a Scoring
      Signal", Fix: score per head, place per block).
  a4  accumulate (once per step, after every layer): token score x_p = sum over
      layers of the token masses; block score y_k = max over layers of the block
      masses; cumulative C += x and EMA E = d*E + (1-d)*x for every tracked entry
      (every position < next_position, every block holding one), x = 0 where nothing
      attended ("Context views at marginal cost", Tier 1: EMA + Cumulative kept as
      O(1)-per-entry running reductions; "Context Optimization", H2O step 1).
  a5  select: top-k resident blocks by C (or E) with ties to the lower block id;
      with H2O the sink and recent blocks are protected and eviction may be applied.
  re-attend (Tier 2): a later query attends over the entries of the kept blocks only.

Where the pages leave a step open, the module docstrings of ``attention``,
``selection`` and ``e4m3`` state the reading taken.
Everything is float64 and written out plainly; no blocking or reordering.
"""

import numpy as np

from . import attention, e4m3, selection, snapkv


class ScoreTables:
    """Cumulative and EMA tables of one sequence, per token and per block, plus two
    block scores summed over the block's entries:

    - s_blk: sum over steps and entries of the entry scores x, i.e. the accumulated
      attention summed over heads, layers and the block's tokens (H2O's score, "Context
      Optimization", H2O > How It Works step 1, at block granularity);
    - t_blk: the same sum for the latest step only (TOVA's latest-query weight, summed
      over heads and layers rather than averaged: the same ranking; "Context views at
      marginal cost", the per-system reductions).
    """

    def __init__(self, max_positions, block_tokens=16, ema_decay=0.9, traj_len=0, profile_layers=(),
                 profile_heads=()):
        self.block_tokens = block_tokens
        self.d = float(ema_decay)
        nb = -(-max_positions // block_tokens)
        # side-car views ("Context views at marginal cost", Tier 1): a ring of the last
        # traj_len steps' t_blk ("when was the span hot"), and per profiled layer the
        # sum over steps of that layer's block mass ("within layer L")
        self.traj_len = traj_len
        self.traj = np.zeros((traj_len, nb))
        self.profile_layers = tuple(profile_layers)
        self.prof = np.zeros((len(self.profile_layers), nb))
        # per-head profiles ("within head H" of a retrieval-head subset): per profiled
        # (layer, query head), the sum over steps of that head's in-block weight
        self.profile_heads = tuple(profile_heads)
        self.hprof = np.zeros((len(self.profile_heads), nb))
        self.c_tok = np.zeros(max_positions)
        self.e_tok = np.zeros(max_positions)
        self.c_blk = np.zeros(nb)
        self.e_blk = np.zeros(nb)
        self.s_blk = np.zeros(nb)
        self.t_blk = np.zeros(nb)
        self.steps = 0

    def trajectory(self):
        """[nb][traj_len]: t_blk of the last traj_len steps, oldest first (0 before the
        first step)."""
        out = np.zeros((self.traj.shape[1], self.traj_len))
        for j in range(self.traj_len):
            step = self.steps - self.traj_len + j          # 0-based step index
            if step >= 0:
                out[:, j] = self.traj[step % self.traj_len]
        return out

    def update(self, tracked_positions, x_tok, y_blk, layer_blk=None, head_blk=None):
        """One step.  x_tok: float64 array over positions 0..tracked_positions-1 with
        the step's token scores (0 where nothing attended); y_blk: float64 array over
        the blocks holding a tracked position, likewise.  Every tracked entry is
        updated: C += x, E = d*E + (1-d)*x."""
        d = self.d
        n = tracked_positions
        nb = -(-n // self.block_tokens)
        x = np.asarray(x_tok, np.float64)
        y = np.asarray(y_blk, np.float64)
        if x.shape != (n,) or y.shape != (nb,):
            raise ValueError("score arrays must cover exactly the tracked entries")
        self.c_tok[:n] = self.c_tok[:n] + x
        self.e_tok[:n] = d * self.e_tok[:n] + (1.0 - d) * x
        self.c_blk[:nb] = self.c_blk[:nb] + y
        self.e_blk[:nb] = d * self.e_blk[:nb] + (1.0 - d) * y
        t = np.zeros(nb)
        for j in range(n):                          # sum of x over each block's entries
            t[j // self.block_tokens] += x[j]
        self.s_blk[:nb] = self.s_blk[:nb] + t
        self.t_blk[:nb] = t
        if self.traj_len:
            self.traj[self.steps % self.traj_len, :] = 0.0
            self.traj[self.steps % self.traj_len, :nb] = t
        for i, l in enumerate(self.profile_layers):
            for k, m in layer_blk[l].items():
                self.prof[i, k] += m
        for i in range(len(self.profile_heads)):
            for k, m in head_blk[i].items():
                self.hprof[i, k] += m
        self.steps += 1


class OracleKV:
    """Float64 model of the whole path for ``num_seqs`` sequences."""

    def __init__(self, *, num_layers, num_q_heads, num_kv_heads, head_dim, num_seqs,
                 max_positions, kv_format="bf16", window=0, h2o_budget_tokens=0,
                 h2o_sink_tokens=4, h2o_recent_frac=0.25, ema_decay=0.9, block_tokens=16, traj_len=0,
                 profile_layers=(), profile_heads=()):
        if num_q_heads % num_kv_heads:
            raise ValueError("num_q_heads must be a multiple of num_kv_heads")
        if window < 0:
            raise ValueError("window must be >= 0 (0 = none)")
        if kv_format not in ("f32", "bf16", "e4m3"):
            raise ValueError("kv_format")
        self.L, self.Hq, self.Hkv, self.D = num_layers, num_q_heads, num_kv_heads, head_dim
        self.B, self.P = num_seqs, max_positions
        self.fmt = kv_format
        self.block = block_tokens
        # H2O takes priority over the window when both are set
        # ("Context Optimization", H2O vs Sliding Window).
        if h2o_budget_tokens > 0:
            self.mode = "h2o"
            self.window = 0
        elif window > 0:
            self.mode = "window"
            self.window = window
        else:
            self.mode = "none"
            self.window = 0
        self.h2o_budget_tokens = h2o_budget_tokens
        self.h2o_budget_blocks = h2o_budget_tokens // block_tokens
        self.h2o_sink_tokens = h2o_sink_tokens
        self.h2o_recent_tokens = selection.recent_token_count(h2o_budget_tokens, h2o_recent_frac)
        self.next_position = np.zeros((num_layers, num_seqs), dtype=np.int64)
        shape = (num_layers, num_seqs, max_positions, num_kv_heads, head_dim)
        if kv_format == "e4m3":
            self.k_codes = np.zeros(shape, dtype=np.uint8)
            self.v_codes = np.zeros(shape, dtype=np.uint8)
            self.k_scale = np.zeros(shape[:3])
            self.v_scale = np.zeros(shape[:3])
        else:
            # bf16 and f32 inputs are binary32 numbers: float32 storage is exact
            self.k_vals = np.zeros(shape, dtype=np.float32)
            self.v_vals = np.zeros(shape, dtype=np.float32)
        self.resident_blocks = [set() for _ in range(num_seqs)]      # H2O mode only
        self.profile_heads = tuple((int(l), int(h)) for l, h in profile_heads)
        self.scores = [ScoreTables(max_positions, block_tokens, ema_decay, traj_len, profile_layers,
                                   self.profile_heads)
                       for _ in range(num_seqs)]
        self._head_blk = {}      # (l, b, h) -> {block: in-block weight of head h} of the latest attend
        self._tok_mass = {}      # (l, b) -> (positions, token mass) of the latest attend
        self._blk_mass = {}      # (l, b) -> {block: mass} of the latest attend
        self._attended = set()   # (l, b) attended since the last accumulate

    # ---------------------------------------------------------------- a1 append
    def append(self, layer, seq, k, v):
        """k, v: [n_new, Hkv, D] exact input values.  Returns the absolute positions."""
        k = np.asarray(k, np.float64)
        v = np.asarray(v, np.float64)
        n = k.shape[0]
        past = int(self.next_position[layer, seq])
        if past + n > self.P:
            raise ValueError("position capacity exceeded")
        pos = np.arange(past, past + n)
        if self.fmt == "e4m3":
            kc, ks = e4m3.quantise_positions(k)
            vc, vs = e4m3.quantise_positions(v)
            self.k_codes[layer, seq, pos] = kc
            self.v_codes[layer, seq, pos] = vc
            self.k_scale[layer, seq, pos] = ks
            self.v_scale[layer, seq, pos] = vs
        else:
            self.k_vals[layer, seq, pos] = k
            self.v_vals[layer, seq, pos] = v
        if self.mode == "h2o":
            for p in pos:
                self.resident_blocks[seq].add(int(p) // self.block)
        self.next_position[layer, seq] = past + n
        return pos

    def slot_of(self, position):
        """Storage slot of an absolute position (window: p % W; otherwise p)."""
        return position % self.window if self.mode == "window" else position

    # ---------------------------------------------------------------- residency
    def resident_positions(self, layer, seq):
        nxt = int(self.next_position[layer, seq])
        if self.mode == "window":
            return np.arange(max(0, nxt - self.window), nxt)
        if self.mode == "h2o":
            p = np.arange(nxt)
            keep = np.isin(p // self.block, np.array(sorted(self.resident_blocks[seq]), np.int64))
            return p[keep]
        return np.arange(nxt)

    def resident_block_ids(self, seq, layer=0):
        pos = self.resident_positions(layer, seq)
        return sorted(set(int(p) // self.block for p in pos))

    def stored_kv(self, layer, seq, positions):
        """Dequantised float64 K, V of the given positions: [n, Hkv, D] each."""
        if self.fmt == "e4m3":
            k = e4m3.dequantise(self.k_codes[layer, seq, positions], self.k_scale[layer, seq, positions])
            v = e4m3.dequantise(self.v_codes[layer, seq, positions], self.v_scale[layer, seq, positions])
            return k, v
        return (self.k_vals[layer, seq, positions].astype(np.float64),
                self.v_vals[layer, seq, positions].astype(np.float64))

    # ---------------------------------------------------------------- a2/a3 attend
    def attend(self, layer, seq, q):
        """q: [Hq, D].  Returns (out [Hq, D], weights [Hq, n], positions [n])."""
        pos = self.resident_positions(layer, seq)
        k, v = self.stored_kv(layer, seq, pos)
        out, w = attention.decode_attention(q, k, v)
        self._tok_mass[(layer, seq)] = (pos, attention.token_step_mass(w))
        self._blk_mass[(layer, seq)] = attention.block_step_mass(w, pos, self.block)
        self._record_heads(layer, seq, w, pos)
        self._attended.add((layer, seq))
        return out, w, pos

    def _record_heads(self, layer, seq, w, pos):
        # one head's in-block weight sum: the block mass of that head alone
        for l, h in self.profile_heads:
            if l == layer:
                self._head_blk[(l, seq, h)] = attention.block_step_mass(w[h:h + 1], pos, self.block)

    def attend_blocks(self, layer, seq, q, block_ids):
        """Tier-2 re-attend ("Context views at marginal cost", Tier 2 and Fact 3): a new
        query attends over the cached K and V of a selected subset only, here the
        resident entries of the listed blocks (the blocks a selection kept).  Softmax
        over that subset; no mass is recorded.  Returns (out [Hq, D], weights [Hq, n],
        positions [n])."""
        pos = self.resident_positions(layer, seq)
        keep = np.isin(pos // self.block, np.asarray(sorted(set(int(b) for b in block_ids)), np.int64))
        pos = pos[keep]
        k, v = self.stored_kv(layer, seq, pos)
        out, w = attention.decode_attention(q, k, v)
        return out, w, pos

    def prefill_score(self, layer, seq, q_obs, kernel=7):
        """SnapKV prefill scoring (``oracle.snapkv``): the last n_obs prompt queries
        q_obs [n_obs, Hq, D] (positions next_position - n_obs .. next_position - 1)
        attend causally over the resident entries; the votes are max-pooled (kernel 7)
        and recorded as this layer's step masses, as an attend records its weights.
        Returns (votes [Hq, n], pooled [Hq, n], positions [n])."""
        q_obs = np.asarray(q_obs, np.float64)
        nxt = int(self.next_position[layer, seq])
        n_obs = q_obs.shape[0]
        if n_obs < 1 or n_obs > nxt or (self.mode == "window" and n_obs > self.window):
            raise ValueError("the observation window must hold 1 .. min(prompt, window) queries")
        pos = self.resident_positions(layer, seq)
        k, _ = self.stored_kv(layer, seq, pos)
        votes = snapkv.observation_votes(q_obs, np.arange(nxt - n_obs, nxt), k, pos)
        pooled = snapkv.max_pool(votes, pos, kernel)
        self._tok_mass[(layer, seq)] = (pos, attention.token_step_mass(pooled))
        self._blk_mass[(layer, seq)] = attention.block_step_mass(pooled, pos, self.block)
        self._record_heads(layer, seq, pooled, pos)
        self._attended.add((layer, seq))
        return votes, pooled, pos

    def token_mass(self, layer, seq):
        """(positions, token mass) of the last attend of (layer, seq)."""
        return self._tok_mass[(layer, seq)]

    def block_mass(self, layer, seq):
        """{block: mass} of the last attend of (layer, seq)."""
        return self._blk_mass[(layer, seq)]

    # ---------------------------------------------------------------- a4 accumulate
    def accumulate(self, seqs=None):
        """Fold the masses of every layer into the score tables.  Returns per sequence
        the step's (x_tok, y_blk) arrays over the tracked positions / blocks."""
        seqs = range(self.B) if seqs is None else seqs
        result = {}
        for b in seqs:
            nxt = set(int(self.next_position[l, b]) for l in range(self.L))
            if len(nxt) != 1:
                raise ValueError("layers disagree on next_position at accumulate")
            n = nxt.pop()
            x_tok = np.zeros(n)
            y_blk = np.zeros(-(-n // self.block))
            layer_blk = {}
            for l in range(self.L):
                if (l, b) not in self._attended:
                    raise ValueError("layer %d of sequence %d was not attended this step" % (l, b))
                self._attended.discard((l, b))
                pos, tau = self._tok_mass[(l, b)]
                x_tok[pos] += tau                      # sum over layers
                for k, m in self._blk_mass[(l, b)].items():
                    y_blk[k] = max(y_blk[k], m)        # max over layers
                layer_blk[l] = self._blk_mass[(l, b)]
            head_blk = [self._head_blk[(l, b, h)] for l, h in self.profile_heads]
            self.scores[b].update(n, x_tok, y_blk, layer_blk, head_blk)
            result[b] = (x_tok, y_blk)
        return result

    # ---------------------------------------------------------------- side-car views
    def filter_blocks(self, seq, score_kind, theta):
        """Threshold view ("Context views at marginal cost", Tier 1: a view is a filter
        of the kept table, a_s > theta): the resident blocks whose score exceeds theta,
        ascending."""
        table = {"cumulative": self.scores[seq].c_blk, "ema": self.scores[seq].e_blk,
                 "token_sum": self.scores[seq].s_blk, "tova": self.scores[seq].t_blk}[score_kind]
        return [c for c in self.resident_block_ids(seq) if table[c] > theta]

    # ---------------------------------------------------------------- a5 select
    def select(self, seq, k, score_kind="cumulative", protect=False, apply=False):
        """Kept block ids (ascending) by a block score: "cumulative" (C of the block
        mass), "ema", "token_sum" (H2O: accumulated entry scores summed over the block)
        or "tova" (the latest step's entry scores summed over the block; keeping the top
        k is evicting the argmin until k remain).  protect: H2O sink/recent protection
        with k as the block budget; apply: evict the unkept blocks (H2O mode only)."""
        cand = self.resident_block_ids(seq)
        table = {"cumulative": self.scores[seq].c_blk, "ema": self.scores[seq].e_blk,
                 "token_sum": self.scores[seq].s_blk, "tova": self.scores[seq].t_blk}[score_kind]
        scores = {c: table[c] for c in cand}
        nxt = int(self.next_position[0, seq])
        if protect:
            keep = selection.h2o_keep(cand, scores, k, nxt, self.h2o_sink_tokens,
                                      self.h2o_recent_tokens, self.block)
        else:
            keep = selection.top_k_blocks(cand, scores, k)
        if apply:
            if self.mode != "h2o":
                raise ValueError("eviction applies to the H2O mode only")
            self.resident_blocks[seq] = set(keep)
        return keep
