"""The KVS_DEBUG build on the GPU (libkvs_debug.so, loaded with KVS_LIB_VARIANT=debug).

It compiles device-side bounds checks into the kernels for the indices the host cannot
check (sequence ids read from a device list, pages, block ids), and fills the
workspace regions that must be written before they are read with NaN.  A child
process (the library is loaded once per process) runs a small case through the fused
and the separate calls and through SnapKV prefill scoring against the oracle with that
build, then hands the kernels a
device list whose ids disagree with the host list: the bounds checks must record
KVS_ERR_STATE instead of touching memory out of range, and the context must stay
usable after kvs_clear_error.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import ctypes, dataclasses
import torch
import attention_scored_kv_gb300 as kvs
from attention_scored_kv_gb300 import _abi
from tests import harness
from tests.test_gpu_parity import SMALL

lib = kvs.lib()
assert lib._name.endswith("libkvs_debug.so"), lib._name
assert lib.kvs_build_info() & 1
for name, fused in (("e4m3-window", True), ("bf16", False), ("e4m3-h2o", True)):
    wl = dataclasses.replace(SMALL[name], steps=4)
    run = harness.Run(wl, oracle_seqs=list(range(wl.batch)), kernel=kvs.KERNEL_TENSOR, fused=fused)
    run.prefill()
    for t in range(wl.steps):
        if fused:
            res = run.decode_step(select=False, accumulate=False)
            keep = run.accumulate_select()
        else:
            res = run.decode_step(select=True)
            keep = res["keep"]
        assert res["out_err"] <= harness.OUT_TOL[wl.kv_format], res["out_err"]
        harness.check_masses(run)
        harness.check_scores(run)
        harness.check_selection(run, keep)
    assert run.cache.get_status() == 0, run.cache.last_error()

# SnapKV prefill scoring: its scratch (row partials, per-group sums) starts NaN-filled,
# so a read of a slot the launch did not write shows up in the masses
from tests.test_gpu_snapkv import RHO
for name in ("e4m3-window", "bf16-hkv8"):
    wl = dataclasses.replace(SMALL[name], steps=1)
    run = harness.Run(wl, oracle_seqs=list(range(wl.batch)), kernel=kvs.KERNEL_TENSOR, obs_window=32)
    run.prefill()
    run.prefill_score(32, rel=RHO)
    harness.check_scores(run, rel=RHO)
    assert run.cache.get_status() == 0, run.cache.last_error()

# a device list that disagrees with the host list: id 9 of 3 sequences
wl = dataclasses.replace(SMALL["e4m3-window"], steps=1)
run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
run.prefill()
c = run.cache
host = (ctypes.c_int32 * 2)(0, 1)
dev = torch.tensor([0, 9], dtype=torch.int32, device="cuda")
seqs = _abi.Seqs(0, 2, ctypes.addressof(host), dev.data_ptr())
stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
assert lib.kvs_accumulate_scores(c._ctx, seqs, stream) == 0
st = c.get_status()
assert st == 7 and "bounds" in c.last_error(), (st, c.last_error())
c.clear_error()
assert c.get_status() == 0
run.decode_step(select=False)
assert c.get_status() == 0, c.last_error()
print("DEBUG_BUILD_OK")
'''


def test_debug_build_parity_and_bounds_checks():
    env = dict(os.environ, KVS_LIB_VARIANT="debug")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "DEBUG_BUILD_OK" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
