"""ctypes declarations of libkvs (include/kvs.h).  Argument marshalling only."""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libkvs.so")
LIB_DEBUG_PATH = os.path.join(HERE, "_lib", "libkvs_debug.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "kvs.h")

# kvs_status
OK, ERR_INVALID_ARGUMENT, ERR_CAPACITY, ERR_EMPTY_CACHE, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED, ERR_STATE = range(8)
STATUS_NAMES = {0: "OK", 1: "INVALID_ARGUMENT", 2: "CAPACITY", 3: "EMPTY_CACHE", 4: "CUDA", 5: "TIMEOUT",
                6: "UNSUPPORTED", 7: "STATE"}
# kvs_dtype
F32, BF16, E4M3 = 0, 1, 2
# kvs_score_kind
SCORE_CUMULATIVE, SCORE_EMA, SCORE_TOKEN_SUM, SCORE_TOVA = 0, 1, 2, 3
# kvs_kernel
KERNEL_AUTO, KERNEL_GENERAL, KERNEL_TENSOR = 0, 1, 2
# kvs_mode
MODE_NONE, MODE_WINDOW, MODE_H2O = 0, 1, 2
# select flags
SELECT_PROTECT, SELECT_APPLY = 1, 2
# kvs_state_item
(STATE_K_PAGES, STATE_V_PAGES, STATE_K_SCALES, STATE_V_SCALES, STATE_POSITIONS, STATE_NEXT_POSITION,
 STATE_TOKEN_MASS, STATE_BLOCK_MASS, STATE_C_TOKEN, STATE_E_TOKEN, STATE_C_BLOCK, STATE_E_BLOCK, STATE_STEPS,
 STATE_BLOCK_TABLE, STATE_S_BLOCK, STATE_T_BLOCK, STATE_TRAJECTORY, STATE_LAYER_PROFILE, STATE_HEAD_PROFILE) = range(19)


class Config(ctypes.Structure):
    _fields_ = [
        ("num_layers", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("max_seqs", ctypes.c_int32), ("max_positions", ctypes.c_int32),
        ("window", ctypes.c_int32), ("block_tokens", ctypes.c_int32), ("h2o_budget_tokens", ctypes.c_int32),
        ("h2o_sink_tokens", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("kernel", ctypes.c_int32),
        ("spin_limit", ctypes.c_int32), ("kv_dtype", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
        ("traj_len", ctypes.c_int32), ("profile_layers", ctypes.c_uint32), ("obs_window", ctypes.c_int32),
        ("n_profile_heads", ctypes.c_int32), ("profile_heads", ctypes.c_int32 * 4), ("reserved_i", ctypes.c_int32),
        ("h2o_recent_frac", ctypes.c_double), ("ema_decay", ctypes.c_double),
        ("reserved_d", ctypes.c_double * 2),
    ]


class Layout(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("num_pages", ctypes.c_int32), ("pages_per_seq", ctypes.c_int32),
                ("max_blocks", ctypes.c_int32), ("attend_kernel", ctypes.c_int32), ("attend_grid", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 2)]


class Seqs(ctypes.Structure):
    """kvs_seqs: a range (h_ids = d_ids = NULL) or a host + device list of ids."""
    _fields_ = [("begin", ctypes.c_int32), ("count", ctypes.c_int32), ("h_ids", ctypes.c_void_p),
                ("d_ids", ctypes.c_void_p)]


_P = ctypes.c_void_p
_I = ctypes.c_int32
_S = Seqs
_SIGS = {
    "kvs_config_init": (None, [ctypes.POINTER(Config)]),
    "kvs_validate_config": (_I, [ctypes.POINTER(Config), ctypes.c_char_p, ctypes.c_size_t]),
    "kvs_workspace_bytes": (ctypes.c_size_t, [ctypes.POINTER(Config)]),
    "kvs_create": (_I, [ctypes.POINTER(Config), _P, ctypes.c_size_t, _P, ctypes.POINTER(_P)]),
    "kvs_destroy": (_I, [_P]),
    "kvs_reset": (_I, [_P, _S, _P]),
    "kvs_append_kv": (_I, [_P, _I, _S, _I, _P, _P, _P]),
    "kvs_decode_attend": (_I, [_P, _I, _S, _P, _P, _P, _P]),
    "kvs_append_attend": (_I, [_P, _I, _S, _P, _P, _P, _P, _P, _P]),
    "kvs_attend_blocks": (_I, [_P, _I, _S, _P, _I, _P, _P, _P, _P]),
    "kvs_decode_attend_static_scratch": (_I, [_P, _I, _S, _P, _P, _P, _P]),
    "kvs_accumulate_scores": (_I, [_P, _S, _P]),
    "kvs_prefill_score": (_I, [_P, _I, _S, _P, _I, _P]),
    "kvs_select_blocks": (_I, [_P, _S, _P, _I, _I, ctypes.c_uint32, _P, _I, _P, _P]),
    "kvs_accumulate_select": (_I, [_P, _S, _P, _I, _I, ctypes.c_uint32, _P, _I, _P, _P]),
    "kvs_filter_blocks": (_I, [_P, _S, _I, ctypes.c_double, _P, _I, _P, _P]),
    "kvs_scores_snapshot_bytes": (ctypes.c_size_t, [_P, _I]),
    "kvs_export_scores": (_I, [_P, _S, _P, ctypes.c_size_t, _P]),
    "kvs_import_scores": (_I, [_P, _S, _P, ctypes.c_size_t, _P]),
    "kvs_state_bytes": (ctypes.c_size_t, [_P, _I]),
    "kvs_read_state": (_I, [_P, _I, _I, _P, ctypes.c_size_t, _P]),
    "kvs_get_layout": (_I, [_P, ctypes.POINTER(Layout)]),
    "kvs_get_status": (_I, [_P, _P]),
    "kvs_clear_error": (_I, [_P, _P]),
    "kvs_last_error": (ctypes.c_char_p, [_P]),
    "kvs_status_string": (ctypes.c_char_p, [_I]),
    "kvs_abi_version": (_I, []),
    "kvs_build_info": (ctypes.c_uint32, []),
}

_lib = None


def load(path=None):
    """Load libkvs.so once (libkvs_debug.so when KVS_LIB_VARIANT=debug).  Raises if it
    has not been built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if path is None:
        path = LIB_DEBUG_PATH if os.environ.get("KVS_LIB_VARIANT", "") == "debug" else LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError("libkvs.so is not built (%s); run python -m attention_scored_kv_gb300.build" % path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib
