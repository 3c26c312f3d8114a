"""Incremental sliding-window slot cache ("LLM mechanics III").

Test infrastructure only (see the package docstring).

Source: "LLM mechanics III: why is a four-slot cache not four-token recomputation?"
  * section 1, Define the window: position i reads positions i-(W-1) .. i (the
    current token included), clipped at the start of the sequence;
  * section 1 (incremental path): per-layer keys and values are stored together
    with their absolute positions, new entries are appended, keys outside the window
    are masked, the output is computed and then only the last W entries are kept;
    the temporary concatenation may exceed W entries;
  * section 3, Cache slots are not positions: a slot index says nothing about the
    position it holds (slot 0 may hold position 20);
  * section 5, Keep three indices separate: the processed-token count
    (next_position) advances by the number of new tokens and is never reset by
    eviction; invalid windows and all-masked rows are rejected.
Flash-MoE "Context Optimization", Sliding Window Attention > Design gives the slot
rule: position p is written to slot p % W, overwriting in place.

This module exists to pin the window bookkeeping used by ``oracle.cache`` against a
full sliding-mask recompute (tests/test_oracle_window.py).  Float64 throughout.
"""

import numpy as np


class SlotCache:
    """One layer's W-slot cache.  window=None means no eviction."""

    def __init__(self, window, kv_heads, head_dim):
        if window is not None:
            if isinstance(window, bool) or not isinstance(window, (int, np.integer)) or window < 1:
                raise ValueError("window must be an integer >= 1 or None")
            window = int(window)
        self.window = window
        self.kv_heads = kv_heads
        self.head_dim = head_dim
        self.next_position = 0                       # processed-token count
        cap = window if window is not None else 0
        self.slot_k = np.zeros((cap, kv_heads, head_dim))
        self.slot_v = np.zeros((cap, kv_heads, head_dim))
        self.slot_pos = np.full(cap, -1, dtype=np.int64)   # absolute position per slot
        # without a window the cache is a growing list in position order
        self._all_k, self._all_v, self._all_pos = [], [], []

    def entries(self):
        """(k, v, positions) of every retained entry, in slot order."""
        if self.window is None:
            if not self._all_pos:
                return (np.zeros((0, self.kv_heads, self.head_dim)),) * 2 + (np.zeros(0, np.int64),)
            return np.stack(self._all_k), np.stack(self._all_v), np.array(self._all_pos, np.int64)
        used = self.slot_pos >= 0
        return self.slot_k[used], self.slot_v[used], self.slot_pos[used]

    def attend_append(self, q, k, v):
        """Append m new entries and attend each new query over its window.

        q: [m, Hq, D]; k, v: [m, Hkv, D].  Returns out [m, Hq, D].
        """
        q = np.asarray(q, np.float64)
        k = np.asarray(k, np.float64)
        v = np.asarray(v, np.float64)
        m = q.shape[0]
        past = self.next_position
        new_pos = np.arange(past, past + m, dtype=np.int64)
        old_k, old_v, old_pos = self.entries()
        tk = np.concatenate([old_k, k], axis=0)     # temporary, may exceed W entries
        tv = np.concatenate([old_v, v], axis=0)
        tpos = np.concatenate([old_pos, new_pos])
        hq = q.shape[1]
        g = hq // self.kv_heads
        out = np.empty_like(q)
        for i in range(m):
            p = new_pos[i]
            allowed = tpos <= p
            if self.window is not None:
                allowed &= tpos >= p - (self.window - 1)
            if not allowed.any():
                raise ValueError("all-masked attention row")
            for h in range(hq):
                kv = h // g
                logits = (tk[allowed, kv, :] @ q[i, h]) / np.sqrt(self.head_dim)
                e = np.exp(logits - logits.max())
                a = e / e.sum()
                out[i, h] = a @ tv[allowed, kv, :]
        # retain: position p goes to slot p % W (the last W entries survive)
        for i in range(m):
            p = int(new_pos[i])
            if self.window is None:
                self._all_k.append(k[i].copy())
                self._all_v.append(v[i].copy())
                self._all_pos.append(p)
            else:
                s = p % self.window
                self.slot_k[s] = k[i]
                self.slot_v[s] = v[i]
                self.slot_pos[s] = p
        self.next_position = past + m               # never reset by eviction
        return out
