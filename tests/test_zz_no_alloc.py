"""The allocation-free attend entry point against the regular one.

kvs_decode_attend_static_scratch exists for callers that cannot get device memory
when they run a decode step (a runtime whose memory was handed out once at start-up,
code that must not enter the CUDA allocator): it keeps the attend's exchange area in
an array compiled into the library instead of the context's workspace.  These tests
call it through the C ABI and compare it with kvs_decode_attend on the same cache and
queries.  Both run the same kernel with the same launch plan, so the output and the
step masses must agree bit for bit.  Between the reference call and the static call a
third attend with another query overwrites the stored masses, so the comparison sees
what the static call itself wrote.  The file sorts last so that a failure here cannot
hide another test's result; it also passes run on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import attention_scored_kv_gb300 as kvs
from attention_scored_kv_gb300 import _abi
import workloads
from tests import harness

pytestmark = pytest.mark.gpu


def _masses(cache, layer):
    tm = cache.read_state(kvs.STATE_TOKEN_MASS, layer).cpu().numpy().view(np.float32).copy()
    bm = cache.read_state(kvs.STATE_BLOCK_MASS, layer).cpu().numpy().view(np.float32).copy()
    return tm, bm


def _static_call(cache, layer, q, out, n_seqs):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    seqs = _abi.Seqs(0, n_seqs, None, None)                     # the range [0, n_seqs)
    return kvs.lib().kvs_decode_attend_static_scratch(cache._ctx, layer, seqs, ctypes.c_void_p(q.data_ptr()),
                                                      ctypes.c_void_p(out.data_ptr()), None, stream)


def _compare_on(run, calls=2):
    """Per layer and call: reference attend, an attend with another query, then the
    static call with the first query; output and masses must equal the reference."""
    cache, wl = run.cache, run.wl
    for call in range(calls):                              # two calls in a row
        for layer in range(wl.num_layers):
            q = run.inp.step_q(layer, 50 + call)
            ref = cache.decode_attend(layer, q).clone()
            ref_tm, ref_bm = _masses(cache, layer)
            cache.decode_attend(layer, run.inp.step_q(layer, 99))      # other masses in the state
            other_tm, _ = _masses(cache, layer)
            assert not np.array_equal(other_tm, ref_tm)
            out = torch.full_like(ref, float("nan"))
            st = _static_call(cache, layer, q, out, wl.batch)
            assert st == 0, cache.last_error()
            got_tm, got_bm = _masses(cache, layer)
            assert torch.equal(out, ref), (call, layer)
            assert np.array_equal(got_tm, ref_tm), (call, layer)
            assert np.array_equal(got_bm, ref_bm), (call, layer)
    assert cache.get_status() == 0, cache.last_error()


def test_static_scratch_attend_matches_workspace_attend():
    """Whole CTAs per sequence (3 sequences on the 32K-context FP8 shape, window 256)."""
    wl = workloads.scaled_down("e4m3-b16-ctx32768-window4096", name="static-scratch", num_layers=2, batch=3,
                               context=700, window=256, steps=4, prefill_chunk=128)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    run.decode_step(select=False)
    _compare_on(run)


def test_static_scratch_attend_split_plan():
    """More sequences than CTAs: the blocks of all sequences are split on the device
    (several sequences per CTA), the other launch plan of the same kernel."""
    wl = workloads.scaled_down("e4m3-b16-ctx32768-window4096", name="static-scratch-split", num_layers=1,
                               batch=200, context=40, window=64, steps=2, prefill_chunk=0)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    assert wl.batch > run.cache.layout().attend_grid
    run.prefill()
    run.decode_step(select=False)
    _compare_on(run)


def test_static_scratch_refuses_a_launch_beyond_the_array():
    """64 query heads and 120 sequences need more exchange area than the 8 MiB array
    ((grid + 120) x 64 x 128 x 4 bytes of output rows alone): KVS_ERR_CAPACITY, and the
    output buffer is left as it was."""
    wl = workloads.scaled_down("bf16-b1-ctx131072-planted", name="static-scratch-big", num_layers=1, batch=120,
                               context=20, steps=1, prefill_chunk=0, retrieval_pos=10)
    run = harness.Run(wl, oracle_seqs=[], kernel=kvs.KERNEL_TENSOR)
    run.prefill()
    q = run.inp.step_q(0, 0)
    out = torch.full((wl.batch, wl.num_q_heads, wl.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    st = _static_call(run.cache, 0, q, out, wl.batch)
    assert st == 2, (st, run.cache.last_error())                  # KVS_ERR_CAPACITY
    assert torch.isnan(out).all()
    assert run.cache.get_status() == 0


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
