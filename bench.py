#!/usr/bin/env python
"""Benchmark of the fused attend + score + select decode step on GB300.

One step = for every layer: append the new token's K/V (E4M3 quantise + circular
write) and decode-attend with the fused mass epilogue; then accumulate the score
tables and select the blocks to keep.  Default workload: E4M3 cache, 16 sequences
at 32768 context, window 4096, 10 layers x 32/4 heads x 128 (the 35B-shaped stack).

Reported (one JSON line from rank 0):
  value      decode steps/s of the whole batch, inputs resident in HBM, each step one
             replay of a CUDA graph holding that step's launches (device-timed), with
             at most eight steps in flight, as a serving loop keeps a few (unbounded_queue:
             the same steps with the host running arbitrarily far ahead)
  e2e        the same through the binding with host buffers: every step copies its
             Q/K/V from pinned host memory and reads back the outputs and kept ids
  roofline   the attend kernel alone: algorithmic KV bytes per launch / mean launch
             time (CUDA events around a graph of back-to-back launches), against the
             measured HBM copy bandwidth
  cpu_baseline  the float64 oracle on the host cores, on a bounded sample

--impl reference runs only the oracle (the slow CPU program this path replaces) and
prints the same metric for it.  Multi-GPU (torchrun): every rank runs an independent
replica on its own sequences (weak scaling, no collective in the data path).
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "fused attend+score decode: KV-scan GB/s (% of HBM peak) and decode steps/s"
DEFAULT_WORKLOAD = "e4m3-b16-ctx32768-window4096"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=50)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    p.add_argument("--e2e-steps", type=int, default=500)
    p.add_argument("--attend-reps", type=int, default=20)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-steps", type=int, default=8)
    return p.parse_args()


# --------------------------------------------------------------------------- distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if args.impl == "ours":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    elif args.impl == "ours":
        torch.cuda.set_device(0)
    return world, rank, local


IN_FLIGHT = 8


def replay_in_flight(graph_of, n, in_flight=IN_FLIGHT):
    """Replay graph_of(i) for i < n, enqueuing replay i only once replay i - in_flight
    has finished.  A serving loop needs a step's outputs to form a later step's inputs,
    so it keeps only a few steps in flight.  With the host enqueuing freely, a thousand
    step graphs pile up in the launch queue, and the same steps measured about 7 %
    slower on GB300 (235 against 218 us per decode step; 2 to 32 in flight all measured
    218).  Eight in flight leave the host about 1.7 ms to absorb a pause of its own."""
    ev = [torch.cuda.Event() for _ in range(in_flight)]
    for i in range(n):
        if i >= in_flight:
            ev[i % in_flight].synchronize()
        graph_of(i).replay()
        ev[i % in_flight].record()


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", ident], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_median": statistics.median(power) if power else None}


# --------------------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def profiled_traffic(kernel_files, profile):
    """DRAM bytes per launch from a committed ncu summary, or None once any of the
    kernel's sources has changed since the capture (the summary records the first 16
    hex digits of each file's sha256 and a traffic_bytes_per_launch line)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    text = open(path).read()
    for f in kernel_files:
        digest = hashlib.sha256(open(os.path.join(ROOT, f), "rb").read()).hexdigest()[:16]
        if "%s %s" % (os.path.basename(f), digest) not in text:
            return None
    for line in text.splitlines():
        if line.startswith("traffic_bytes_per_launch:"):
            return int(line.split(":")[1])
    return None


def kv_bytes_per_entry(wl):
    """Algorithmic bytes the attend reads per resident entry per layer: K and V of all
    KV heads, plus one float32 scale each for E4M3 ("Context Optimization", Memory
    Budget Calculator: elements x bytes, plus about 4 bytes of scale per position per
    cache)."""
    elem = {"f32": 4, "bf16": 2, "e4m3": 1}[wl.kv_format]
    b = 2 * wl.num_kv_heads * wl.head_dim * elem
    if wl.kv_format == "e4m3":
        b += 2 * 4
    return b


def resident_entries(wl, next_pos):
    """Entries an attend launch scans per sequence at next_pos (window: the last W)."""
    if wl.window:
        return min(next_pos, wl.window)
    if wl.h2o_budget_tokens:
        return None
    return next_pos


def make_config(kvs, wl):
    fmt = {"f32": kvs.F32, "bf16": kvs.BF16, "e4m3": kvs.E4M3}
    return kvs.config_init(
        num_layers=wl.num_layers, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads, head_dim=wl.head_dim,
        max_seqs=wl.batch, max_positions=wl.max_positions, window=wl.window, block_tokens=wl.block_tokens,
        h2o_budget_tokens=wl.h2o_budget_tokens, h2o_sink_tokens=wl.h2o_sink_tokens,
        h2o_recent_frac=wl.h2o_recent_frac, ema_decay=wl.ema_decay, kv_dtype=fmt[wl.kv_format],
        in_dtype=fmt[wl.in_dtype], obs_window=OBS_WINDOW if snapkv_capable(wl) else 0)


OBS_WINDOW = 32      # SnapKV's observation window


def snapkv_capable(wl):
    """Prefill scoring runs on the tensor-core configurations."""
    return wl.head_dim == 128 and wl.in_dtype == "bf16" and wl.num_q_heads == 8 * wl.num_kv_heads \
        and wl.kv_format in ("bf16", "e4m3")


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def prefill(cache, inp, wl):
    """Fill every sequence with its prefill tokens by appends (chunked as the workload says)."""
    lens = inp.prefill_lengths()
    chunk = wl.prefill_chunk or max(int(lens.max()), 1)
    for l in range(wl.num_layers):
        if wl.context_range is None:
            if wl.context == 0:
                continue
            ks, vs = zip(*[inp.prefill_kv(l, s) for s in range(wl.batch)])
            k, v = torch.stack(ks), torch.stack(vs)
            for a in range(0, wl.context, chunk):
                cache.append_kv(l, k[:, a:a + chunk].contiguous(), v[:, a:a + chunk].contiguous())
            del k, v
        else:
            for s in range(wl.batch):
                k, v = inp.prefill_kv(l, s)
                for a in range(0, k.shape[0], chunk):
                    cache.append_kv(l, k[None, a:a + chunk].contiguous(), v[None, a:a + chunk].contiguous(),
                                    seq_begin=s)


# --------------------------------------------------------------------------- GPU arm
def run_ours(args, world, rank, local):
    import attention_scored_kv_gb300 as kvs
    if not os.path.exists(kvs._abi.LIB_PATH):
        from attention_scored_kv_gb300 import build
        build.build()
    dev = torch.device("cuda", torch.cuda.current_device())
    wl0 = workloads.get(args.workload)
    eager = 2
    # positions the device advances (eager + warm-up + timed twice + e2e steps) plus those the
    # host-side checks advance while the step graphs are captured (128 + 64 graphs)
    total_steps = eager + 2 * args.warmup + 2 * args.steps + args.e2e_steps + 128 + 64 + 64
    wl = workloads.scaled_down(args.workload, name=wl0.name, steps=total_steps, seed=wl0.seed + 1000 * rank)
    cache = kvs.KVCache(make_config(kvs, wl), device=dev)
    inp = workloads.Inputs(wl, device=dev)
    lay = cache.layout()

    # ---- prefill (untimed)
    t0 = time.time()
    prefill(cache, inp, wl)
    torch.cuda.synchronize()
    prefill_s = time.time() - t0

    # ---- step inputs resident in HBM: NI distinct draws, cycled
    L, B, Hq, Hkv, D = wl.num_layers, wl.batch, wl.num_q_heads, wl.num_kv_heads, wl.head_dim
    NI = min(wl0.steps, 128)
    dt = torch.bfloat16 if wl.in_dtype == "bf16" else torch.float32
    Q = torch.empty((NI, L, B, Hq, D), dtype=dt, device=dev)
    K = torch.empty((NI, L, B, 1, Hkv, D), dtype=dt, device=dev)
    V = torch.empty_like(K)
    for t in range(NI):
        for l in range(L):
            Q[t, l] = inp.step_q(l, t)
            k, v = inp.step_kv(l, t)
            K[t, l], V[t, l] = k, v
    OUT = torch.empty((L, B, Hq, D), dtype=torch.float32, device=dev)
    keep_ids = torch.full((B, lay.max_blocks), -1, dtype=torch.int32, device=dev)
    keep_cnt = torch.zeros(B, dtype=torch.int32, device=dev)
    if wl.h2o_budget_tokens:
        k_sel, flags = wl.h2o_budget_tokens // 16, kvs.SELECT_PROTECT | kvs.SELECT_APPLY
    else:
        res_blocks = (wl.window // 16 + 1) if wl.window else lay.max_blocks
        k_sel, flags = wl0.keep_k(res_blocks), 0
    launches = {"n": 0}
    # append + attend is one launch per layer with the tensor-core attend when every
    # sequence can have CTAs of its own; otherwise append and attend are two.  H2O adds
    # one page allocation per step (the first layer to reach a new position).  accumulate
    # + select is one launch up to 512 resident blocks per sequence.
    fused = lay.attend_kernel == kvs.KERNEL_TENSOR and B <= lay.attend_grid
    res_bound = (wl.window // 16 + 1) if wl.window else (
        wl.h2o_budget_tokens // 16 + 2 if wl.h2o_budget_tokens else lay.max_blocks)
    per_step_launches = ((L if fused else 2 * L) + (1 if res_bound <= 512 else 2)
                         + (1 if wl.h2o_budget_tokens else 0))

    def step(t, q=None, k=None, v=None, out=None, ids=None, cnt=None):
        q = Q[t] if q is None else q
        k = K[t] if k is None else k
        v = V[t] if v is None else v
        out = OUT if out is None else out
        ids = keep_ids if ids is None else ids
        cnt = keep_cnt if cnt is None else cnt
        for l in range(L):
            cache.append_attend(l, k[l], v[l], q[l], out=out[l])   # append + attend of one layer
        cache.accumulate_select(k_sel, flags=flags, keep_ids=ids, keep_count=cnt)
        launches["n"] += per_step_launches

    for t in range(eager):
        step(t % NI)
    torch.cuda.synchronize()
    assert cache.get_status() == 0, cache.last_error()

    graphs = []
    for t in range(NI):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(t)
        graphs.append(g)

    replay_in_flight(lambda i: graphs[(eager + i) % NI], args.warmup)
    torch.cuda.synchronize()

    # ---- timed region (device time, CUDA events; max over ranks)
    sampler = ClockSampler(dev)
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    replay_in_flight(lambda i: graphs[(eager + args.warmup + i) % NI], args.steps)
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    status = cache.get_status()
    assert status == 0, "device status %d: %s" % (status, cache.last_error())
    steps_per_s = world * args.steps / (ms / 1e3)

    # ---- the same number of steps with the host enqueuing without bound (reported beside
    # the value, not used for it)
    barrier(world)
    torch.cuda.synchronize()
    u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    u0.record()
    for i in range(args.steps):
        graphs[(eager + args.warmup + args.steps + i) % NI].replay()
    u1.record()
    torch.cuda.synchronize()
    ums = max_over_ranks(u0.elapsed_time(u1), world, dev)
    assert cache.get_status() == 0, cache.last_error()

    # ---- attend kernel alone: graph of L back-to-back launches (layers rotate so every
    # launch reads a layer not touched for L-1 launches; L x per-layer KV > L2)
    ga = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ga):
        for l in range(L):
            cache.decode_attend(l, Q[0, l], out=OUT[l])
    for _ in range(2):
        ga.replay()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    replay_in_flight(lambda i: ga, args.attend_reps)
    a1.record()
    torch.cuda.synchronize()
    attend_us = a0.elapsed_time(a1) * 1e3 / (args.attend_reps * L)

    # ---- Tier-2 re-attend over the blocks the last step kept: graph of L launches
    reattend = None
    if lay.attend_kernel == kvs.KERNEL_TENSOR:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for l in range(L):
                cache.attend_blocks(l, Q[1, l], keep_ids, keep_cnt, out=OUT[l])
        for _ in range(2):
            gr.replay()
        torch.cuda.synchronize()
        r0, r1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        r0.record()
        replay_in_flight(lambda i: gr, args.attend_reps)
        r1.record()
        torch.cuda.synchronize()
        reattend_us = r0.elapsed_time(r1) * 1e3 / (args.attend_reps * L)
        kept = int(keep_cnt.sum().item())
        assert cache.get_status() == 0, cache.last_error()
    nxt = cache.read_state(kvs.STATE_NEXT_POSITION, 0).cpu().numpy().view(np.int64)
    if wl.h2o_budget_tokens:
        bt = cache.read_state(kvs.STATE_BLOCK_TABLE).cpu().numpy().view(np.int32).reshape(B, lay.max_blocks)
        entries = 0
        for s in range(B):
            nb = int(np.sum(bt[s] >= 0))
            entries += nb * 16 - (16 - int(nxt[s]) % 16) % 16
    else:
        entries = sum(resident_entries(wl, int(n)) for n in nxt)
    bytes_per_launch = entries * kv_bytes_per_entry(wl)
    hbm, peak_kind = peaks()
    achieved = bytes_per_launch / (attend_us * 1e-6) / 1e9
    if lay.attend_kernel == kvs.KERNEL_TENSOR:
        # resident entries of the kept blocks (a sequence's first and last block may be partial)
        ids_h, cnt_h = keep_ids.cpu().numpy(), keep_cnt.cpu().numpy()
        rent = 0
        for s in range(B):
            nx = int(nxt[s])
            lo = max(0, nx - wl.window) if wl.window else 0
            for kb in ids_h[s, : int(cnt_h[s])]:
                rent += max(0, min(nx, 16 * int(kb) + 16) - max(lo, 16 * int(kb)))
        rbytes = rent * kv_bytes_per_entry(wl)
        reattend = {"blocks_kept": kept, "kv_bytes_per_launch": int(rbytes), "launch_us": round(reattend_us, 3),
                    "kv_gbs": round(rbytes / (reattend_us * 1e-6) / 1e9, 1),
                    "frac_of_hbm": round(rbytes / (reattend_us * 1e-6) / 1e9 / hbm, 4)}
    # ---- SnapKV prefill scoring of every layer over the current cache (one launch per
    # layer), graph of L layers; FLOPs = QK^T of the observation queries once
    prefill_score = None
    if cache.cfg.obs_window:
        QO = torch.stack([inp.obs_q(l, OBS_WINDOW) for l in range(L)])
        gp = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gp):
            for l in range(L):
                cache.prefill_score(l, QO[l])
        for _ in range(2):
            gp.replay()
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record()
        replay_in_flight(lambda i: gp, args.attend_reps)
        p1.record()
        torch.cuda.synchronize()
        assert cache.get_status() == 0, cache.last_error()
        ps_us = p0.elapsed_time(p1) * 1e3 / (args.attend_reps * L)
        qk_flops = 2.0 * OBS_WINDOW * Hq * entries * D
        peak_tf, tf_kind = bf16_peak()
        tf = qk_flops / (ps_us * 1e-6) / 1e12
        prefill_score = {"n_obs": OBS_WINDOW, "layer_us": round(ps_us, 3), "launches_per_layer": 1,
                         "qk_flops_per_layer": int(qk_flops), "tflops": round(tf, 1),
                         "tflops_executed": round(2 * tf, 1), "peak_tflops": peak_tf, "peak_source": tf_kind,
                         "frac": round(tf / peak_tf, 4), "frac_executed": round(2 * tf / peak_tf, 4),
                         "k_bytes_per_layer_pass": int(entries * kv_bytes_per_entry(wl) // 2)}
    traffic = None                      # DRAM bytes per launch measured by ncu, this workload only
    if wl0.name == "e4m3-b16-ctx32768-window4096":
        traffic = profiled_traffic(["attention_scored_kv_gb300/csrc/attend_tc.cu",
                                    "attention_scored_kv_gb300/csrc/kvs_internal.cuh"],
                                   "attend_tc_e4m3_b16_ctx32768_w4096.md")

    # ---- end to end through the binding with host buffers.  Every step copies its Q/K/V
    # in from pinned host memory and its outputs and kept ids back, inside the timed
    # region.  The copies run on a second stream with double-buffered device buffers, as
    # a serving loop would: step i+2's inputs go in and step i's results come out while
    # step i+1 computes (events order each copy against the steps that use its buffer).
    NE = min(NI, 64)
    pin = lambda x: x.cpu().pin_memory()
    Qh, Kh, Vh = pin(Q[:NE]), pin(K[:NE]), pin(V[:NE])
    Qd = [torch.empty_like(Q[0]) for _ in range(2)]
    Kd = [torch.empty_like(K[0]) for _ in range(2)]
    Vd = [torch.empty_like(V[0]) for _ in range(2)]
    OUTd = [torch.empty_like(OUT) for _ in range(2)]
    IDSd = [torch.empty_like(keep_ids) for _ in range(2)]
    CNTd = [torch.empty_like(keep_cnt) for _ in range(2)]
    OUTh = [torch.empty(OUT.shape, dtype=OUT.dtype).pin_memory() for _ in range(2)]
    IDSh = [torch.empty(keep_ids.shape, dtype=torch.int32).pin_memory() for _ in range(2)]
    CNTh = [torch.empty(keep_cnt.shape, dtype=torch.int32).pin_memory() for _ in range(2)]
    h2d = Qd[0].numel() * Qd[0].element_size() + 2 * Kd[0].numel() * Kd[0].element_size()
    d2h = OUT.numel() * 4 + keep_ids.numel() * 4 + keep_cnt.numel() * 4

    egraphs = []
    for par in range(2):
        Qd[par].copy_(Qh[par])
        Kd[par].copy_(Kh[par])
        Vd[par].copy_(Vh[par])
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(0, Qd[par], Kd[par], Vd[par], OUTd[par], IDSd[par], CNTd[par])
        egraphs.append(g)
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]

    def put_inputs(i):                     # on the copy stream, into buffer i % 2
        par = i % 2
        with torch.cuda.stream(copy):
            Qd[par].copy_(Qh[i % NE], non_blocking=True)
            Kd[par].copy_(Kh[i % NE], non_blocking=True)
            Vd[par].copy_(Vh[i % NE], non_blocking=True)
            in_ready[par].record(copy)

    def run_e2e(n):
        put_inputs(0)
        put_inputs(1)
        for i in range(n):
            par = i % 2
            comp.wait_event(in_ready[par])
            if i >= 2:
                comp.wait_event(out_read[par])     # step i-2's outputs have been read back
            egraphs[par].replay()
            done[par].record(comp)
            with torch.cuda.stream(copy):
                copy.wait_event(done[par])
                OUTh[par].copy_(OUTd[par], non_blocking=True)
                IDSh[par].copy_(IDSd[par], non_blocking=True)
                CNTh[par].copy_(CNTd[par], non_blocking=True)
                out_read[par].record(copy)
            if i + 2 < n:
                put_inputs(i + 2)
        comp.wait_stream(copy)                # the last results are on the host

    run_e2e(min(args.warmup, NE) + 2)
    torch.cuda.synchronize()
    barrier(world)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    c0.record(comp)
    copy.wait_stream(comp)                    # the copies start inside the timed region
    run_e2e(args.e2e_steps)
    c1.record(comp)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    barrier(world)
    e2e_ms = max_over_ranks(max(c0.elapsed_time(c1), wall * 1e3), world, dev)
    assert cache.get_status() == 0, cache.last_error()
    e2e_value = world * args.e2e_steps / (e2e_ms / 1e3)

    result = {
        "metric": METRIC, "value": round(steps_per_s, 2), "unit": "decode steps/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3" if wl.kv_format == "e4m3" else wl.kv_format,
        "data": "synthetic (seeded N(0,1) inputs, no dataset or weights)",
        "config": {
            "workload": wl0.name, "batch": B, "context": wl0.context if not wl0.context_range else list(wl0.context_range),
            "window": wl0.window, "h2o_budget_tokens": wl0.h2o_budget_tokens, "layers": L, "q_heads": Hq,
            "kv_heads": Hkv, "head_dim": D, "kv_format": wl.kv_format,
            "compute": "K/V decoded to f16 (E4M3) or kept bf16, mma.sync tensor cores, fp32 accumulate; fp64 score tables",
            "l2": "inputs larger than L2: each step scans %.1f MB of KV (10 layers), L2 is 129 MB" % (
                L * bytes_per_launch / 1e6),
            "graph": "one CUDA graph per step (%d distinct step inputs cycled)" % NI,
            "loop": "at most %d steps in flight: step i is enqueued once step i-%d has finished" % (
                IN_FLIGHT, IN_FLIGHT),
            "parallelism": "replicas x%d (independent sequences per GPU)" % world,
            "prefill_s": round(prefill_s, 2),
        },
        "kv_scan_gbs": round(achieved, 1),
        "kv_scan_frac_of_hbm": round(achieved / hbm, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "traffic": traffic, "peak_source": peak_kind,
                     "kernel": "attend_tc_kernel", "launch_us": round(attend_us, 3),
                     "algorithmic_bytes_per_launch": int(bytes_per_launch)},
        "e2e": {"value": round(e2e_value, 2), "unit": "decode steps/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": args.e2e_steps},
        "unbounded_queue": {"value": round(world * args.steps / (ums / 1e3), 2), "unit": "decode steps/s",
                            "ms_per_step": round(ums / args.steps, 5), "steps": args.steps},
        "reattend": reattend,
        "prefill_score": prefill_score,
        "gpu_launches": int(per_step_launches * args.steps),
        "clocks": clocks,
    }
    return result, wl0


# --------------------------------------------------------------------------- CPU (oracle)
def oracle_sample(wl, steps_budget, seconds_cap=None, layers_per_step=None):
    """Time the float64 oracle on one sequence of the workload at its resident size.

    Returns (seconds per full-batch decode step, description, cores)."""
    from oracle.cache import OracleKV
    cores = len(os.sched_getaffinity(0))
    n_res = wl.window if wl.window else (wl.h2o_budget_tokens if wl.h2o_budget_tokens else wl.max_context)
    o = OracleKV(num_layers=wl.num_layers, num_q_heads=wl.num_q_heads, num_kv_heads=wl.num_kv_heads,
                 head_dim=wl.head_dim, num_seqs=1, max_positions=n_res + steps_budget + 4, kv_format=wl.kv_format,
                 window=wl.window)
    inp = workloads.Inputs(workloads.scaled_down(wl.name, name=wl.name, context=n_res, context_range=None,
                                                 batch=1, steps=steps_budget + 4), device="cpu")
    for l in range(wl.num_layers):
        k, v = inp.prefill_kv(l, 0)
        o.append(l, 0, workloads.as_f64(k), workloads.as_f64(v))
    return o, inp, cores, n_res


def run_cpu_baseline(wl, steps):
    o, inp, cores, n_res = oracle_sample(wl, steps)
    t0 = time.perf_counter()
    for t in range(steps):
        for l in range(wl.num_layers):
            k, v = inp.step_kv(l, t)
            o.append(l, 0, workloads.as_f64(k[0]), workloads.as_f64(v[0]))
            o.attend(l, 0, workloads.as_f64(inp.step_q(l, t)[0]))
        o.accumulate()
        o.select(0, wl.keep_k(n_res // 16 + 1))
    dt = (time.perf_counter() - t0) / steps          # one sequence, one step
    value = 1.0 / (dt * wl.batch)                     # full batch: batch x that
    # the KV bytes the sampled step scans (every layer, n_res entries) over its time
    kv_gbs = n_res * kv_bytes_per_entry(wl) * wl.num_layers / dt / 1e9
    return {"value": round(value, 5), "unit": "decode steps/s", "cores": cores, "kind": "oracle",
            "kv_gbs_equivalent": round(kv_gbs, 4),
            "sample": "%d decode steps of 1 of %d sequences (%d layers, %d resident entries each, float64 numpy); "
                      "the batch step is extrapolated as %d x the per-sequence step" % (
                          steps, wl.batch, wl.num_layers, n_res, wl.batch)}


def run_reference(args, world, rank):
    """The oracle as the reference program: each step a bounded sample of the workload
    (one layer of one sequence: append + attend over the resident entries, plus the
    sequence's accumulate/select once per layer sweep), extrapolated to the batch."""
    if rank != 0:
        return None
    wl = workloads.get(args.workload)
    total = args.warmup + args.steps
    o, inp, cores, n_res = oracle_sample(wl, total // wl.num_layers + 2)
    times = []
    t_sweep = 0
    for i in range(total):
        l = i % wl.num_layers
        step = i // wl.num_layers
        k, v = inp.step_kv(l, step)
        t0 = time.perf_counter()
        o.append(l, 0, workloads.as_f64(k[0]), workloads.as_f64(v[0]))
        o.attend(l, 0, workloads.as_f64(inp.step_q(l, step)[0]))
        if l == wl.num_layers - 1:
            o.accumulate()
            o.select(0, wl.keep_k(n_res // 16 + 1))
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    per_layer_seq = sum(times) / len(times)
    factor = wl.num_layers * wl.batch                # samples in one decode step of the workload
    step_s = per_layer_seq * factor
    value = 1.0 / step_s
    sample = ("each timed step: one layer of one sequence (append + attend over %d entries; the sequence's "
              "accumulate + select on every %d-th); value = 1 / (mean sample time x %d layers x %d sequences)" % (
                  n_res, wl.num_layers, wl.num_layers, wl.batch))
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "decode steps/s", "n_gpus": world,
        # steps and ms_per_step describe what was timed (one layer of one sequence per
        # step); the workload step is extrapolation_factor such samples
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_layer_seq * 1e3, 3),
        "timed_s": round(sum(times), 3), "extrapolation_factor": factor,
        "ms_per_workload_step_extrapolated": round(step_s * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) inputs)",
        "config": {"workload": wl.name, "batch": wl.batch, "layers": wl.num_layers, "window": wl.window,
                   "kv_format": wl.kv_format},
        "cpu_baseline": {"value": round(value, 5), "unit": "decode steps/s", "cores": cores, "kind": "oracle",
                         "kv_gbs_equivalent": round(n_res * kv_bytes_per_entry(wl) / per_layer_seq / 1e9, 4),
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "decode steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        res = run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res))
        return
    res, wl0 = run_ours(args, world, rank, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = run_cpu_baseline(wl0, args.cpu_steps)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
