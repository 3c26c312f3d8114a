"""Workload recipes and their seeded input streams.

Every tensor is drawn from its own ``torch.Generator`` seeded by a 64-bit mix of
(workload seed, tensor kind, layer, sequence or step), so any slice of any workload
can be regenerated on its own, on the CPU or on the GPU (the two devices give
different but individually reproducible streams).  Values are drawn as float32
N(0, 1) and rounded to the input dtype (bf16 round-to-nearest-even) before anyone
sees them.

Workloads (shapes from the pages: "Context Optimization" Memory Savings table for the
10 x 4 x 128 and 15 x 8 x 128 full-attention stacks; "Per-Head Attention as a Scoring
Signal" for the four head types and the 16-token block):

  tiny-f32-window4              1 seq, 2 layers, 4/2 heads, D 16, f32, window 4,
                                64 tokens decoded one at a time, keep 2 blocks
  bf16-b8-ctx4096               10 layers, 32/4 heads, D 128, bf16, 8 seqs at 4096,
                                256 steps, no window, keep 50% of blocks
  e4m3-b16-ctx32768-window4096  same stack, E4M3 cache, 16 seqs at 32768, window
                                4096 (circular slots), 128 steps, keep 25%
  bf16-b1-ctx131072-planted     15 layers, 64/8 heads, D 128, bf16, 1 seq at 131072,
                                four planted head types per layer, 32 steps, keep 10%
  e4m3-b64-ragged-h2o2048       10 layers, 32/4 heads, E4M3, 64 seqs of length
                                U[1024, 32768], 16-token pages, H2O budget 2048
                                tokens applied every step for 512 steps, 5% of keys x4
"""

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_layers: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    batch: int
    context: int                      # prefill length of every sequence
    steps: int                        # decode steps
    context_range: tuple = None       # (lo, hi) inclusive: ragged prefill lengths
    window: int = 0                   # 0 = none
    kv_format: str = "bf16"           # cache storage: f32 | bf16 | e4m3
    in_dtype: str = "bf16"            # Q/K/V input dtype: f32 | bf16
    block_tokens: int = 16
    ema_decay: float = 0.9
    keep_frac: float = 0.5            # k = max(1, floor(keep_frac * candidates))
    keep_fixed: int = 0               # k fixed (overrides keep_frac when > 0)
    h2o_budget_tokens: int = 0
    h2o_sink_tokens: int = 4
    h2o_recent_frac: float = 0.25
    seed: int = 0
    planted: bool = False             # four planted head types per layer
    retrieval_pos: int = 65536        # planted retrieval key (cosine 0.9)
    heavy_frac: float = 0.0           # fraction of keys scaled by heavy_scale
    heavy_scale: float = 4.0
    prefill_chunk: int = 0            # longest prefill append (0 = whole prefill)

    @property
    def group(self):
        return self.num_q_heads // self.num_kv_heads

    @property
    def max_context(self):
        return self.context_range[1] if self.context_range else self.context

    @property
    def max_positions(self):
        return self.max_context + self.steps

    def keep_k(self, n_candidates):
        if self.keep_fixed > 0:
            return self.keep_fixed
        return max(1, int(math.floor(self.keep_frac * n_candidates)))


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny-f32-window4", num_layers=2, num_q_heads=4, num_kv_heads=2, head_dim=16,
                 batch=1, context=0, steps=64, window=4, kv_format="f32", in_dtype="f32",
                 keep_fixed=2, seed=7),
        Workload("bf16-b8-ctx4096", num_layers=10, num_q_heads=32, num_kv_heads=4, head_dim=128,
                 batch=8, context=4096, steps=256, kv_format="bf16", keep_frac=0.5, seed=1002),
        Workload("e4m3-b16-ctx32768-window4096", num_layers=10, num_q_heads=32, num_kv_heads=4,
                 head_dim=128, batch=16, context=32768, steps=128, window=4096, kv_format="e4m3",
                 keep_frac=0.25, seed=1003, prefill_chunk=4096),
        Workload("bf16-b1-ctx131072-planted", num_layers=15, num_q_heads=64, num_kv_heads=8,
                 head_dim=128, batch=1, context=131072, steps=32, kv_format="bf16", keep_frac=0.1,
                 seed=1004, planted=True, prefill_chunk=16384),
        Workload("e4m3-b64-ragged-h2o2048", num_layers=10, num_q_heads=32, num_kv_heads=4,
                 head_dim=128, batch=64, context=0, context_range=(1024, 32768), steps=512,
                 kv_format="e4m3", h2o_budget_tokens=2048, seed=1005, heavy_frac=0.05,
                 prefill_chunk=8192),
    ]
}


def get(name):
    return WORKLOADS[name]


def scaled_down(base_name, **changes):
    """A smaller copy of a named workload (same structure, other sizes)."""
    base = WORKLOADS[base_name]
    return dataclasses.replace(base, name=changes.pop("name", base.name + "-small"), **changes)


# --------------------------------------------------------------------------- seeds
_TAGS = {"q": 1, "k": 2, "v": 3, "pk": 4, "pv": 5, "heavy_p": 6, "heavy_s": 7,
         "lengths": 8, "planted_u": 9, "oq": 10}


def _splitmix64(x):
    x = (x + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
    z = x
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
    return z ^ (z >> 31)


def tensor_seed(seed, tag, *idx):
    h = _splitmix64(seed & 0xFFFFFFFFFFFFFFFF)
    for v in (_TAGS[tag],) + tuple(idx):
        h = _splitmix64(h ^ (int(v) & 0xFFFFFFFFFFFFFFFF))
    return h & 0x7FFFFFFFFFFFFFFF


_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


class Inputs:
    """Input stream of one workload on one device."""

    def __init__(self, wl, device="cpu", seed=None):
        self.wl = wl
        self.device = torch.device(device)
        self.seed = wl.seed if seed is None else seed
        self.dtype = _DT[wl.in_dtype]

    # ---- raw draws
    def _gen(self, tag, *idx):
        g = torch.Generator(device=self.device)
        g.manual_seed(tensor_seed(self.seed, tag, *idx))
        return g

    def _randn(self, shape, tag, *idx):
        return torch.randn(shape, generator=self._gen(tag, *idx), device=self.device,
                           dtype=torch.float32)

    def _rand(self, shape, tag, *idx):
        return torch.rand(shape, generator=self._gen(tag, *idx), device=self.device,
                          dtype=torch.float32)

    # ---- structure
    def prefill_lengths(self):
        """Prefill length of every sequence (ints)."""
        wl = self.wl
        if wl.context_range is None:
            return np.full(wl.batch, wl.context, dtype=np.int64)
        rng = np.random.default_rng(tensor_seed(self.seed, "lengths"))
        lo, hi = wl.context_range
        return rng.integers(lo, hi + 1, size=wl.batch).astype(np.int64)

    def _planted_u(self, layer, group):
        u = self._randn((self.wl.head_dim,), "planted_u", layer, group)
        return u / torch.linalg.vector_norm(u)

    @staticmethod
    def _set_cos(k, u, c):
        """Rotate the rows of k (float32 [..., D]) to cosine c with unit u, norms kept."""
        norm = torch.linalg.vector_norm(k, dim=-1, keepdim=True)
        perp = k - (k @ u)[..., None] * u
        perp = perp / torch.linalg.vector_norm(perp, dim=-1, keepdim=True)
        return norm * (math.sqrt(1.0 - c * c) * perp + c * u)

    def _plant_keys(self, k, layer, positions, decoded):
        """Planted head types on KV heads 0..3 ("Per-Head Attention as a Scoring Signal",
        The Four Types of Attention Heads): recency (last 100 prefill keys and every
        decoded key), anchor (keys 0-50), retrieval (key retrieval_pos, cosine 0.9), syntactic
        (every 7th key).  k: float32 [n, Hkv, D]; positions: int64 [n]."""
        ctx = self.wl.context
        pos = positions.to(self.device)
        rules = [
            (0, (pos >= ctx - 100) | torch.full_like(pos, bool(decoded), dtype=torch.bool), 0.5),
            (1, pos <= 50, 0.5),
            (2, pos == self.wl.retrieval_pos, 0.9),
            (3, (pos % 7) == 0, 0.5),
        ]
        for kvh, mask, c in rules:
            if kvh >= self.wl.num_kv_heads or not bool(mask.any()):
                continue
            u = self._planted_u(layer, kvh)
            rows = k[mask, kvh, :]
            k[mask, kvh, :] = self._set_cos(rows, u, c)
        return k

    def _heavy(self, k, tag, *idx):
        """Scale a heavy_frac fraction of the positions' keys (all KV heads) by heavy_scale."""
        wl = self.wl
        if wl.heavy_frac <= 0:
            return k
        sel = self._rand((k.shape[0],), tag, *idx) < wl.heavy_frac
        return torch.where(sel[:, None, None], k * wl.heavy_scale, k)

    # ---- streams
    def prefill_kv(self, layer, seq):
        """K, V of sequence seq's prefill in one layer: [len, Hkv, D] each (input dtype)."""
        wl = self.wl
        n = int(self.prefill_lengths()[seq])
        shape = (n, wl.num_kv_heads, wl.head_dim)
        k = self._randn(shape, "pk", layer, seq)
        v = self._randn(shape, "pv", layer, seq)
        if wl.planted:
            k = self._plant_keys(k, layer, torch.arange(n, dtype=torch.int64), decoded=False)
        k = self._heavy(k, "heavy_p", layer, seq)
        return k.to(self.dtype), v.to(self.dtype)

    def step_q(self, layer, step):
        """Queries of decode step ``step`` (0-based) in one layer: [B, Hq, D]."""
        wl = self.wl
        q = self._randn((wl.batch, wl.num_q_heads, wl.head_dim), "q", layer, step)
        if wl.planted:
            for kvh in range(min(4, wl.num_kv_heads)):
                u = self._planted_u(layer, kvh)
                q[:, kvh * wl.group, :] = math.sqrt(wl.head_dim) * u
        return q.to(self.dtype)

    def obs_q(self, layer, n_obs):
        """Queries of the last n_obs prefill positions in one layer (SnapKV's observation
        window): [B, n_obs, Hq, D], oldest first; planted heads as in step_q."""
        wl = self.wl
        q = self._randn((wl.batch, n_obs, wl.num_q_heads, wl.head_dim), "oq", layer)
        if wl.planted:
            for kvh in range(min(4, wl.num_kv_heads)):
                u = self._planted_u(layer, kvh)
                q[:, :, kvh * wl.group, :] = math.sqrt(wl.head_dim) * u
        return q.to(self.dtype)

    def step_kv(self, layer, step):
        """New K, V of decode step ``step`` in one layer: [B, 1, Hkv, D] each."""
        wl = self.wl
        shape = (wl.batch, 1, wl.num_kv_heads, wl.head_dim)
        k = self._randn(shape, "k", layer, step)
        v = self._randn(shape, "v", layer, step)
        if wl.planted:
            lens = self.prefill_lengths()
            for b in range(wl.batch):
                pos = torch.tensor([int(lens[b]) + step], dtype=torch.int64)
                k[b] = self._plant_keys(k[b], layer, pos, decoded=True)
        if wl.heavy_frac > 0:
            k = torch.stack([self._heavy(k[b], "heavy_s", layer, step, b) for b in range(wl.batch)])
        return k.to(self.dtype), v.to(self.dtype)


def as_f64(t):
    """Exact float64 numpy copy of a (bf16 or f32) tensor."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)
