"""The allocation-free attend entry point against the regular one.

kvs_decode_attend_static_scratch exists for callers that cannot get device memory
when they run a decode step (a runtime whose memory was handed out once at start-up,
code that must not enter the CUDA allocator): it keeps the attend's exchange area in
an array compiled into the library instead of the context's workspace.  This test
calls it through the C ABI, twice in a row on every layer, and checks that its output
and the step masses it leaves match what kvs_decode_attend produces on the same cache
and queries, within the tolerances the parity tests use.  The file sorts last so that a
failure here cannot hide another test's result; it also passes run on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import attention_scored_kv_gb300 as kvs
import workloads
from tests import harness

pytestmark = pytest.mark.gpu


def _masses(cache, layer):
    tm = cache.read_state(kvs.STATE_TOKEN_MASS, layer).cpu().numpy().view(np.float32).copy()
    bm = cache.read_state(kvs.STATE_BLOCK_MASS, layer).cpu().numpy().view(np.float32).copy()
    return tm, bm


def test_static_scratch_attend_matches_workspace_attend():
    wl = workloads.scaled_down("e4m3-b16-ctx32768-window4096", name="static-scratch", num_layers=2, batch=3,
                               context=700, window=256, steps=4, prefill_chunk=128)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    run.decode_step(select=False)
    cache = run.cache
    lib = kvs.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):                                  # two calls in a row
        for layer in range(wl.num_layers):
            q = run.inp.step_q(layer, 50 + call)
            ref = cache.decode_attend(layer, q)
            ref_tm, ref_bm = _masses(cache, layer)
            out = torch.full_like(ref, float("nan"))
            st = lib.kvs_decode_attend_static_scratch(cache._ctx, layer, 0, wl.batch, ctypes.c_void_p(q.data_ptr()),
                                                      ctypes.c_void_p(out.data_ptr()), stream)
            assert st == 0, cache.last_error()
            got_tm, got_bm = _masses(cache, layer)
            assert harness.rel_err_rows(out.double().cpu().numpy(), ref.double().cpu().numpy()) <= 2e-3
            assert np.max(np.abs(got_tm - ref_tm)) <= harness.SCORE_TOL
            assert np.max(np.abs(got_bm - ref_bm)) <= harness.SCORE_TOL
    assert cache.get_status() == 0, cache.last_error()


def test_static_scratch_rejects_general_kernel_contexts():
    wl = workloads.get("tiny-f32-window4")
    cache = kvs.KVCache(harness.make_config(wl))
    k = torch.zeros((1, 1, wl.num_kv_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    for layer in range(wl.num_layers):
        cache.append_kv(layer, k, k)
    q = torch.zeros((1, wl.num_q_heads, wl.head_dim), dtype=torch.float32, device="cuda")
    with pytest.raises(kvs.KVSError) as e:
        cache.decode_attend_static_scratch(0, q)
    assert e.value.status == 6
