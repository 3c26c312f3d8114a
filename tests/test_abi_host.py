"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
entry point include/kvs.h declares, and validates configs and sizes workspaces on
the host.  No call here touches a CUDA device."""
import ctypes
import os
import re

import pytest

import attention_scored_kv_gb300 as kvs
from attention_scored_kv_gb300 import _abi
from oracle import memory

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built_library():
    if not os.path.exists(_abi.LIB_PATH):
        from attention_scored_kv_gb300 import build
        build.build()
    kvs.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "kvs.h")).read()
    return sorted(set(re.findall(r"KVS_API\s+[\w\s\*]+?\b(kvs_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert len(names) >= 18
    lib = ctypes.CDLL(_abi.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    # and the binding's declarations cover exactly the header's entry points
    assert sorted(_abi._SIGS) == names


def test_abi_version_and_status_strings():
    assert kvs.lib().kvs_abi_version() == 2
    for s in range(8):
        assert kvs.status_string(s)
    assert kvs.status_string(3).startswith("empty cache")


def cfg35b(**kw):
    base = dict(num_layers=10, num_q_heads=32, num_kv_heads=4, head_dim=128, max_seqs=16, max_positions=32896)
    base.update(kw)
    return kvs.config_init(**base)


@pytest.mark.parametrize("field,value,status", [
    ("window", -1, _abi.ERR_INVALID_ARGUMENT),          # invalid window ("LLM mechanics III", section 5)
    ("head_dim", 96, _abi.ERR_UNSUPPORTED),
    ("num_kv_heads", 5, _abi.ERR_INVALID_ARGUMENT),
    ("block_tokens", 32, _abi.ERR_UNSUPPORTED),
    ("h2o_budget_tokens", 100, _abi.ERR_INVALID_ARGUMENT),
    ("ema_decay", 1.0, _abi.ERR_INVALID_ARGUMENT),
    ("h2o_recent_frac", 1.5, _abi.ERR_INVALID_ARGUMENT),
    ("max_seqs", 0, _abi.ERR_INVALID_ARGUMENT),
    ("kv_dtype", 7, _abi.ERR_INVALID_ARGUMENT),
    ("in_dtype", _abi.E4M3, _abi.ERR_INVALID_ARGUMENT),
    ("traj_len", -1, _abi.ERR_INVALID_ARGUMENT),
    ("traj_len", 257, _abi.ERR_INVALID_ARGUMENT),
    ("profile_layers", 1 << 10, _abi.ERR_INVALID_ARGUMENT),     # layer 10 of 10
    ("profile_layers", 0b11111, _abi.ERR_INVALID_ARGUMENT),     # five layers
])
def test_invalid_configs_rejected(field, value, status):
    cfg = cfg35b(**{field: value})
    st, msg = kvs.validate_config(cfg)
    assert st == status and msg
    assert kvs.workspace_bytes(cfg) == 0


def test_sidecar_workspace():
    """The trajectory ring (float32 per block and step) and the layer profiles (float64
    per block and profiled layer) add their bytes to the workspace."""
    base = kvs.workspace_bytes(cfg35b())
    mb = -(-32896 // 16)
    grown = kvs.workspace_bytes(cfg35b(traj_len=64, profile_layers=0b1001))
    assert kvs.validate_config(cfg35b(traj_len=64, profile_layers=0b1001))[0] == _abi.OK
    assert grown - base >= 16 * mb * (64 * 4 + 2 * 8)
    assert grown - base <= 16 * mb * (64 * 4 + 2 * 8) + 2 * 256


def test_reserved_fields_must_be_zero():
    cfg = cfg35b()
    cfg.reserved_i = 1
    assert kvs.validate_config(cfg)[0] == _abi.ERR_INVALID_ARGUMENT


def test_bf16_cache_needs_bf16_inputs():
    assert kvs.validate_config(cfg35b(kv_dtype=_abi.BF16, in_dtype=_abi.F32))[0] == _abi.ERR_UNSUPPORTED


def test_tensor_kernel_shape_gate():
    assert kvs.validate_config(cfg35b(kernel=_abi.KERNEL_TENSOR))[0] == _abi.OK
    assert kvs.validate_config(cfg35b(kernel=_abi.KERNEL_TENSOR, head_dim=64))[0] == _abi.ERR_UNSUPPORTED
    assert kvs.validate_config(cfg35b(kernel=_abi.KERNEL_TENSOR, window=100))[0] == _abi.ERR_UNSUPPORTED
    assert kvs.validate_config(cfg35b(kernel=_abi.KERNEL_TENSOR, in_dtype=_abi.F32, kv_dtype=_abi.E4M3))[0] == _abi.ERR_UNSUPPORTED
    assert kvs.validate_config(cfg35b(kernel=_abi.KERNEL_GENERAL, head_dim=64))[0] == _abi.OK


def test_h2o_with_window_is_accepted_and_h2o_wins():
    # "Context Optimization", H2O vs Sliding Window: H2O takes priority when both are set
    cfg = cfg35b(window=4096, h2o_budget_tokens=2048, kv_dtype=_abi.E4M3)
    assert kvs.validate_config(cfg)[0] == _abi.OK
    # H2O sizes its page pool for every position, not for the window
    h2o = kvs.workspace_bytes(cfg)
    win = kvs.workspace_bytes(cfg35b(window=4096, kv_dtype=_abi.E4M3))
    assert h2o > win


def test_workspace_holds_the_pages_formula():
    """The K/V page storage equals the Memory Budget Calculator's figure for the
    resident positions (scales included for E4M3)."""
    for fmt, dt in (("e4m3", _abi.E4M3), ("bf16", _abi.BF16)):
        cfg = cfg35b(window=4096, kv_dtype=dt, max_seqs=1)
        ws = kvs.workspace_bytes(cfg)
        kv = memory.kv_cache_bytes(10, 4, 128, fmt, context=32896, window=4096, with_scales=True)
        assert ws >= kv
        # the rest (positions, masses, score tables, scratch) is bounded
        assert ws - kv < 64 * 2 ** 20


def test_workspace_grows_with_format():
    sizes = [kvs.workspace_bytes(cfg35b(kv_dtype=dt, in_dtype=_abi.BF16 if dt != _abi.F32 else _abi.F32))
             for dt in (_abi.E4M3, _abi.BF16, _abi.F32)]
    assert sizes[0] < sizes[1] < sizes[2]


def test_debug_library_exports_the_same_symbols_and_says_so():
    """The KVS_DEBUG build (device bounds checks, poisoned scratch) is a second library
    with the same entry points; kvs_build_info tells the two apart."""
    names = declared_symbols()
    dbg = ctypes.CDLL(_abi.LIB_DEBUG_PATH)
    for n in names:
        assert hasattr(dbg, n), n
    dbg.kvs_build_info.restype = ctypes.c_uint32
    rel = ctypes.CDLL(_abi.LIB_PATH)
    rel.kvs_build_info.restype = ctypes.c_uint32
    assert dbg.kvs_build_info() & 1 and not rel.kvs_build_info() & 1


def test_nvtx_ranges_are_switched_on_by_the_environment():
    """With KVS_NVTX=1 every call opens an NVTX range (no tool attached: no effect) and
    kvs_build_info reports it; host-only calls behave as before."""
    import subprocess
    import sys
    code = ("import attention_scored_kv_gb300 as kvs\n"
            "lib = kvs.lib()\n"
            "assert lib.kvs_build_info() & 2\n"
            "cfg = kvs.config_init(num_layers=2, num_q_heads=8, num_kv_heads=1, head_dim=128)\n"
            "assert kvs.validate_config(cfg)[0] == 0 and kvs.workspace_bytes(cfg) > 0\n"
            "print('NVTX_OK')\n")
    env = dict(os.environ, KVS_NVTX="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "NVTX_OK" in r.stdout, r.stderr
    assert not kvs.lib().kvs_build_info() & 2
