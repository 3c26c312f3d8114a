"""Python binding of libkvs, the attention-scored KV cache decode path for GB300.

Thin marshalling over the C ABI in include/kvs.h: each method takes torch tensors that
already live on the GPU, checks their dtype / shape / contiguity and passes raw device
pointers and the current CUDA stream to the library.  Every step of the path (append,
attend with the fused mass epilogue, accumulate, select) runs in the library's CUDA
kernels; PyTorch provides device memory and streams only.  If libkvs.so is missing the
calls raise: there is no CPU or PyTorch fallback.
"""

import ctypes

import torch

from . import _abi
from ._abi import (  # noqa: F401
    F32, BF16, E4M3, SCORE_CUMULATIVE, SCORE_EMA, SCORE_TOKEN_SUM, SCORE_TOVA, KERNEL_AUTO, KERNEL_GENERAL,
    KERNEL_TENSOR,
    MODE_NONE, MODE_WINDOW, MODE_H2O, SELECT_PROTECT, SELECT_APPLY, Config, Layout,
)
from ._abi import (  # noqa: F401
    STATE_K_PAGES, STATE_V_PAGES, STATE_K_SCALES, STATE_V_SCALES, STATE_POSITIONS, STATE_NEXT_POSITION,
    STATE_TOKEN_MASS, STATE_BLOCK_MASS, STATE_C_TOKEN, STATE_E_TOKEN, STATE_C_BLOCK, STATE_E_BLOCK, STATE_STEPS,
    STATE_BLOCK_TABLE, STATE_S_BLOCK, STATE_T_BLOCK, STATE_TRAJECTORY, STATE_LAYER_PROFILE, STATE_HEAD_PROFILE,
)

_TORCH_DT = {F32: torch.float32, BF16: torch.bfloat16}


class KVSError(RuntimeError):
    def __init__(self, status, message):
        self.status = status
        super().__init__("%s: %s" % (_abi.STATUS_NAMES.get(status, status), message))


def lib():
    return _abi.load()


def config_init(**fields):
    """A kvs_config with the library defaults, then the given fields."""
    cfg = Config()
    lib().kvs_config_init(ctypes.byref(cfg))
    for k, v in fields.items():
        setattr(cfg, k, v)
    return cfg


def validate_config(cfg):
    """(status, message) of the host-side config check."""
    buf = ctypes.create_string_buffer(512)
    st = lib().kvs_validate_config(ctypes.byref(cfg), buf, len(buf))
    return st, buf.value.decode()


def workspace_bytes(cfg):
    return int(lib().kvs_workspace_bytes(ctypes.byref(cfg)))


def status_string(status):
    return lib().kvs_status_string(status).decode()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _need(t, name, dtype, shape):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


class SeqIds:
    """A list of distinct sequence ids for calls that work on scattered sequences (a
    serving batch whose active sequences are not contiguous).  Holds the ids twice, as
    kvs_seqs wants them: in host memory, which the library reads during each call (its
    checks and launch plans), and in device memory, which its kernels read.  Build it
    once and reuse it: building copies the ids to the device."""

    def __init__(self, ids, device="cuda"):
        ids = [int(x) for x in ids]
        if not ids:
            raise ValueError("SeqIds needs at least one id")
        self.ids = ids
        self.host = (ctypes.c_int32 * len(ids))(*ids)
        self.dev = torch.tensor(ids, dtype=torch.int32, device=device)

    def __len__(self):
        return len(self.ids)


def _seqs(seq_begin, count, seq_ids):
    """kvs_seqs of a call: the list (a SeqIds or a sequence of ints) when given, else the
    range [seq_begin, seq_begin + count)."""
    if seq_ids is None:
        return _abi.Seqs(int(seq_begin), int(count), None, None), None
    ids = seq_ids if isinstance(seq_ids, SeqIds) else SeqIds(seq_ids)
    if count is not None and int(count) != len(ids):
        raise ValueError("%d rows of inputs for %d sequence ids" % (count, len(ids)))
    return _abi.Seqs(0, len(ids), ctypes.addressof(ids.host), ids.dev.data_ptr()), ids


class KVCache:
    """A kvs context bound to a workspace this object owns (a torch uint8 tensor).

    Every per-sequence method takes the sequences either as a range (seq_begin and the
    row count of its tensors, or n_seqs) or as seq_ids, a SeqIds or a list of distinct
    sequence ids in any order; rows of inputs and outputs follow that order."""

    def __init__(self, cfg, device=None, stream=None):
        st, msg = validate_config(cfg)
        if st != _abi.OK:
            raise KVSError(st, msg)
        self.cfg = cfg
        self.device = torch.device("cuda") if device is None else torch.device(device)
        nbytes = workspace_bytes(cfg)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self._ctx = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            st = lib().kvs_create(ctypes.byref(cfg), _ptr(self.workspace), nbytes, _stream(stream),
                                  ctypes.byref(self._ctx))
        if st != _abi.OK:
            raise KVSError(st, "kvs_create failed")
        self.in_dtype = _TORCH_DT[cfg.in_dtype]
        L, Hq, Hkv, D = cfg.num_layers, cfg.num_q_heads, cfg.num_kv_heads, cfg.head_dim
        self.shape = (L, Hq, Hkv, D)

    def __del__(self):
        if getattr(self, "_ctx", None) and self._ctx.value:
            try:
                lib().kvs_destroy(self._ctx)
            except Exception:
                pass
            self._ctx = None

    def _check(self, st):
        if st != _abi.OK:
            raise KVSError(st, lib().kvs_last_error(self._ctx).decode())

    def _count(self, seq_begin, n_seqs, seq_ids):
        if seq_ids is not None:
            return len(seq_ids)
        return self.cfg.max_seqs - seq_begin if n_seqs is None else n_seqs

    # ---- the path
    def reset(self, seq_begin=0, n_seqs=None, stream=None, seq_ids=None):
        n = self._count(seq_begin, n_seqs, seq_ids)
        sq, keep = _seqs(seq_begin, n, seq_ids)
        self._check(lib().kvs_reset(self._ctx, sq, _stream(stream)))

    def append_kv(self, layer, k, v, seq_begin=0, stream=None, seq_ids=None):
        """k, v: [n_seqs, n_new, Hkv, D] in the input dtype."""
        _, _, Hkv, D = self.shape
        n_seqs, n_new = int(k.shape[0]), int(k.shape[1])
        _need(k, "k", self.in_dtype, (n_seqs, n_new, Hkv, D))
        _need(v, "v", self.in_dtype, (n_seqs, n_new, Hkv, D))
        sq, keep = _seqs(seq_begin, n_seqs, seq_ids)
        self._check(lib().kvs_append_kv(self._ctx, layer, sq, n_new, _ptr(k), _ptr(v), _stream(stream)))

    def _tok_out(self, n_seqs, tok_mass_out):
        if tok_mass_out is not None:
            _need(tok_mass_out, "tok_mass_out", torch.float32, (n_seqs, self.cfg.max_positions))
            return _ptr(tok_mass_out)
        return None

    def decode_attend(self, layer, q, out=None, seq_begin=0, stream=None, seq_ids=None, tok_mass_out=None):
        """q: [n_seqs, Hq, D] in the input dtype; returns out [n_seqs, Hq, D] float32.
        tok_mass_out: optional float32 CUDA tensor [n_seqs, max_positions] that also
        receives every resident entry's mass at its absolute position."""
        _, Hq, _, D = self.shape
        n_seqs = int(q.shape[0])
        _need(q, "q", self.in_dtype, (n_seqs, Hq, D))
        if out is None:
            out = torch.empty((n_seqs, Hq, D), dtype=torch.float32, device=q.device)
        _need(out, "out", torch.float32, (n_seqs, Hq, D))
        sq, keep = _seqs(seq_begin, n_seqs, seq_ids)
        self._check(lib().kvs_decode_attend(self._ctx, layer, sq, _ptr(q), _ptr(out),
                                            self._tok_out(n_seqs, tok_mass_out), _stream(stream)))
        return out

    def append_attend(self, layer, k, v, q, out=None, seq_begin=0, stream=None, seq_ids=None, tok_mass_out=None):
        """append_kv of one token per sequence then decode_attend, in one launch where
        the context allows.  k, v: [n_seqs, 1, Hkv, D]; q: [n_seqs, Hq, D]."""
        _, Hq, Hkv, D = self.shape
        n_seqs = int(q.shape[0])
        _need(k, "k", self.in_dtype, (n_seqs, 1, Hkv, D))
        _need(v, "v", self.in_dtype, (n_seqs, 1, Hkv, D))
        _need(q, "q", self.in_dtype, (n_seqs, Hq, D))
        if out is None:
            out = torch.empty((n_seqs, Hq, D), dtype=torch.float32, device=q.device)
        _need(out, "out", torch.float32, (n_seqs, Hq, D))
        sq, keep = _seqs(seq_begin, n_seqs, seq_ids)
        self._check(lib().kvs_append_attend(self._ctx, layer, sq, _ptr(k), _ptr(v), _ptr(q), _ptr(out),
                                            self._tok_out(n_seqs, tok_mass_out), _stream(stream)))
        return out

    def attend_blocks(self, layer, q, block_ids, block_count, out=None, seq_begin=0, stream=None, seq_ids=None):
        """Re-attend q over the resident entries of the listed blocks only (for example
        the keep_ids and keep_count of select_blocks).  block_ids: int32 CUDA tensor
        [n_seqs, stride]; block_count: int32 CUDA tensor [n_seqs]."""
        _, Hq, _, D = self.shape
        n_seqs = int(q.shape[0])
        _need(q, "q", self.in_dtype, (n_seqs, Hq, D))
        stride = int(block_ids.shape[1])
        _need(block_ids, "block_ids", torch.int32, (n_seqs, stride))
        _need(block_count, "block_count", torch.int32, (n_seqs,))
        if out is None:
            out = torch.empty((n_seqs, Hq, D), dtype=torch.float32, device=q.device)
        _need(out, "out", torch.float32, (n_seqs, Hq, D))
        sq, keep = _seqs(seq_begin, n_seqs, seq_ids)
        self._check(lib().kvs_attend_blocks(self._ctx, layer, sq, _ptr(block_ids), stride, _ptr(block_count),
                                            _ptr(q), _ptr(out), _stream(stream)))
        return out

    def decode_attend_static_scratch(self, layer, q, out=None, seq_begin=0, stream=None, seq_ids=None,
                                     tok_mass_out=None):
        """decode_attend with the exchange area in the library's own fixed array instead
        of this cache's workspace (for callers that cannot supply device memory)."""
        _, Hq, _, D = self.shape
        n_seqs = int(q.shape[0])
        _need(q, "q", self.in_dtype, (n_seqs, Hq, D))
        if out is None:
            out = torch.empty((n_seqs, Hq, D), dtype=torch.float32, device=q.device)
        _need(out, "out", torch.float32, (n_seqs, Hq, D))
        sq, keep = _seqs(seq_begin, n_seqs, seq_ids)
        self._check(lib().kvs_decode_attend_static_scratch(self._ctx, layer, sq, _ptr(q), _ptr(out),
                                                           self._tok_out(n_seqs, tok_mass_out), _stream(stream)))
        return out

    def prefill_score(self, layer, q_obs, seq_begin=0, stream=None, seq_ids=None):
        """SnapKV prefill scoring of one layer: q_obs [n_seqs, n_obs, Hq, D] bf16 CUDA
        tensor, the queries of each prompt's last n_obs positions."""
        if not isinstance(q_obs, torch.Tensor) or not q_obs.is_cuda or q_obs.dim() != 4:
            raise TypeError("q_obs must be a 4-d CUDA tensor")
        L, Hq, Hkv, D = self.shape
        n, n_obs = q_obs.shape[0], q_obs.shape[1]
        _need(q_obs, "q_obs", torch.bfloat16, (n, n_obs, Hq, D))
        sq, keep = _seqs(seq_begin, n, seq_ids)
        self._check(lib().kvs_prefill_score(self._ctx, layer, sq, _ptr(q_obs), n_obs, _stream(stream)))

    def accumulate_scores(self, seq_begin=0, n_seqs=None, stream=None, seq_ids=None):
        n = self._count(seq_begin, n_seqs, seq_ids)
        sq, keep = _seqs(seq_begin, n, seq_ids)
        self._check(lib().kvs_accumulate_scores(self._ctx, sq, _stream(stream)))

    def _keep_buffers(self, n, keep_capacity, keep_ids, keep_count, k):
        cap = self.layout().max_blocks if keep_capacity is None else keep_capacity
        if keep_ids is None:
            keep_ids = torch.full((n, cap), -1, dtype=torch.int32, device=self.device)
        if keep_count is None:
            keep_count = torch.zeros(n, dtype=torch.int32, device=self.device)
        _need(keep_ids, "keep_ids", torch.int32, (n, cap))
        _need(keep_count, "keep_count", torch.int32, (n,))
        if isinstance(k, torch.Tensor):
            _need(k, "k", torch.int32, (n,))
            kp, ku = _ptr(k), 0
        else:
            kp, ku = None, int(k)
        return cap, keep_ids, keep_count, kp, ku

    def select_blocks(self, k, seq_begin=0, n_seqs=None, score_kind=SCORE_CUMULATIVE, flags=0, keep_capacity=None,
                      keep_ids=None, keep_count=None, stream=None, seq_ids=None):
        """k: an int (same for every sequence) or an int32 CUDA tensor [n_seqs].
        Returns (keep_ids [n_seqs, keep_capacity] int32, keep_count [n_seqs] int32)."""
        n = self._count(seq_begin, n_seqs, seq_ids)
        cap, keep_ids, keep_count, kp, ku = self._keep_buffers(n, keep_capacity, keep_ids, keep_count, k)
        sq, keep = _seqs(seq_begin, n, seq_ids)
        self._check(lib().kvs_select_blocks(self._ctx, sq, kp, ku, score_kind, flags, _ptr(keep_ids), cap,
                                            _ptr(keep_count), _stream(stream)))
        return keep_ids, keep_count

    def accumulate_select(self, k, seq_begin=0, n_seqs=None, score_kind=SCORE_CUMULATIVE, flags=0,
                          keep_capacity=None, keep_ids=None, keep_count=None, stream=None, seq_ids=None):
        """accumulate_scores then select_blocks (same arguments and results as the
        latter), in one launch for sequences of at most 512 resident blocks."""
        n = self._count(seq_begin, n_seqs, seq_ids)
        cap, keep_ids, keep_count, kp, ku = self._keep_buffers(n, keep_capacity, keep_ids, keep_count, k)
        sq, keep = _seqs(seq_begin, n, seq_ids)
        self._check(lib().kvs_accumulate_select(self._ctx, sq, kp, ku, score_kind, flags, _ptr(keep_ids), cap,
                                                _ptr(keep_count), _stream(stream)))
        return keep_ids, keep_count

    def filter_blocks(self, theta, seq_begin=0, n_seqs=None, score_kind=SCORE_CUMULATIVE, capacity=None,
                      ids=None, count=None, stream=None, seq_ids=None):
        """Resident blocks whose score exceeds theta.  Returns (ids [n_seqs, capacity]
        int32, count [n_seqs] int32), ids ascending."""
        n = self._count(seq_begin, n_seqs, seq_ids)
        cap = self.layout().max_blocks if capacity is None else capacity
        if ids is None:
            ids = torch.full((n, cap), -1, dtype=torch.int32, device=self.device)
        if count is None:
            count = torch.zeros(n, dtype=torch.int32, device=self.device)
        _need(ids, "ids", torch.int32, (n, cap))
        _need(count, "count", torch.int32, (n,))
        sq, keep = _seqs(seq_begin, n, seq_ids)
        self._check(lib().kvs_filter_blocks(self._ctx, sq, score_kind, float(theta), _ptr(ids), cap, _ptr(count),
                                            _stream(stream)))
        return ids, count

    # ---- score snapshot
    def snapshot_bytes(self, n_seqs):
        return int(lib().kvs_scores_snapshot_bytes(self._ctx, n_seqs))

    def export_scores(self, seq_begin=0, n_seqs=None, dst=None, stream=None, seq_ids=None):
        """The score tables of the sequences as one uint8 tensor (CUDA unless dst, a
        contiguous uint8 tensor on the device or in pinned host memory, is given)."""
        n = self._count(seq_begin, n_seqs, seq_ids)
        nb = self.snapshot_bytes(n)
        if dst is None:
            dst = torch.empty(nb, dtype=torch.uint8, device=self.device)
        if dst.dtype != torch.uint8 or not dst.is_contiguous() or dst.numel() < nb:
            raise ValueError("dst must be a contiguous uint8 tensor of at least %d bytes" % nb)
        sq, keep = _seqs(seq_begin, n, seq_ids)
        self._check(lib().kvs_export_scores(self._ctx, sq, _ptr(dst), dst.numel(), _stream(stream)))
        return dst

    def import_scores(self, src, seq_begin=0, n_seqs=None, stream=None, seq_ids=None):
        n = self._count(seq_begin, n_seqs, seq_ids)
        if src.dtype != torch.uint8 or not src.is_contiguous():
            raise ValueError("src must be a contiguous uint8 tensor")
        sq, keep = _seqs(seq_begin, n, seq_ids)
        self._check(lib().kvs_import_scores(self._ctx, sq, _ptr(src), src.numel(), _stream(stream)))

    # ---- inspection
    def read_state(self, what, layer=0, stream=None):
        """A raw copy (uint8 CUDA tensor) of one state array; see kvs_state_item."""
        n = int(lib().kvs_state_bytes(self._ctx, what))
        if n == 0:
            raise KVSError(_abi.ERR_INVALID_ARGUMENT, "state item %d not available" % what)
        dst = torch.empty(n, dtype=torch.uint8, device=self.device)
        self._check(lib().kvs_read_state(self._ctx, what, layer, _ptr(dst), n, _stream(stream)))
        return dst

    def layout(self):
        lay = Layout()
        self._check(lib().kvs_get_layout(self._ctx, ctypes.byref(lay)))
        return lay

    def get_status(self, stream=None):
        """Synchronise and return the device status code (0 = OK)."""
        return lib().kvs_get_status(self._ctx, _stream(stream))

    def clear_error(self, stream=None):
        self._check(lib().kvs_clear_error(self._ctx, _stream(stream)))

    def last_error(self):
        return lib().kvs_last_error(self._ctx).decode()
