#!/usr/bin/env python
"""Benchmark: absorbed MLA decode tokens/s on one B300, with the latent-cache
stream's roofline fraction.

A step is one decode step of one MLA layer for every sequence of the workload:
cache append of the new token(s) -> absorbed decode (fold, split-K attention,
merge) -> W_UV up-projection, all through the C ABI.  Default workload: the
DeepSeek-V3-shaped decode (hidden 7168, 128 heads, d_h 128, d_c 512, d_r 64,
batch 64, 4096 cached rows + 1 new token per sequence, bf16, seed 2).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica of the workload (weak scaling; the path has no exchange step).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode tokens/s (1 B300) and latent-cache HBM GB/s as % of roofline"
UNIT = "tokens/s"
DOMINANT_KERNEL_SOURCES = ["head_latent_attention_25_b300/csrc/mla_decode_tc.cu",
                           "head_latent_attention_25_b300/csrc/tc_ptx.cuh",
                           "head_latent_attention_25_b300/csrc/mla_common.cuh"]
DOMINANT_KERNEL_NAME = "split_tc_kernel"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=1000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="v3_b64_l4096",
                   help="a named workload or one sweep point (v3_sweep_b<batch>_l<context>)")
    p.add_argument("--num-splits", type=int, default=0)
    p.add_argument("--sweep", action="store_true", help="one line per sweep point (not the contract line)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true",
                   help="time eager launches only (default: the step captured once into a CUDA graph)")
    p.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    p.add_argument("--no-from-h", action="store_true",
                   help="skip the companion measurement of the step with the query computed from h")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d["bf16_tflops_sustained"], "measured"
    except Exception:
        return 6400.0, 1800.0, 1400.0, "fallback"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """SM clock and clock-event (throttle) reasons of one GPU, read through NVML by a
    host thread every ~2 ms and kept with their wall times, so that even a timed region
    of a few milliseconds holds samples.  Read-only: no setting of the GPU is touched.
    When NVML cannot be used the reason is kept in ``error`` and reported."""
    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40), ("hw_power_brake_slowdown", 0x80),
               ("sw_thermal_slowdown", 0x20), ("sw_power_cap", 0x4))

    def __init__(self, uuid: str, period_s: float = 0.002):
        import threading
        self.rows, self.error, self.period = [], None, period_s
        self._stop = threading.Event()
        self._thread = None
        self.source = "nvml"
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nv = pynvml
            self._h = pynvml.nvmlDeviceGetHandleByUUID(uuid)
            self._max = float(pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM))
            target = self._run
        except Exception as e:                     # no NVML binding: nvidia-smi in a loop
            self.error = f"nvml unavailable ({type(e).__name__}); nvidia-smi every 20 ms"
            self.source, self.period, self._uuid = "nvidia-smi", 0.02, uuid
            target = self._run_smi
        self._thread = threading.Thread(target=target, daemon=True)
        self._thread.start()

    def _run_smi(self):
        import subprocess
        fields = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.active"]
        try:
            proc = subprocess.Popen(["nvidia-smi", "-i", self._uuid, "--query-gpu=" + ",".join(fields),
                                     "--format=csv,noheader,nounits", "-lms", "20"],
                                    stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
        except Exception as e:
            self.error = f"nvidia-smi failed: {type(e).__name__}: {e}"
            return
        while not self._stop.is_set():
            line = proc.stdout.readline()
            if not line:
                self.error = "nvidia-smi ended: " + (proc.stderr.read() or "")[:200]
                break
            parts = [x.strip() for x in line.split(",")]
            try:
                self.rows.append((time.time(), float(parts[0]), float(parts[1]), int(parts[2], 16)))
            except (ValueError, IndexError):
                continue
        proc.terminate()
        try:
            proc.wait(timeout=5)
        except Exception:
            proc.kill()

    def _run(self):
        nv, h = self._nv, self._h
        while not self._stop.is_set():
            try:
                t = time.time()
                sm = float(nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM))
                r = int(nv.nvmlDeviceGetCurrentClocksEventReasons(h))
                self.rows.append((t, sm, self._max, r))
            except Exception as e:
                self.error = f"nvml read failed: {type(e).__name__}: {e}"
                return
            time.sleep(self.period)

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        return self.rows

    def summary(self, windows):
        """Median SM clock and the union of active reasons over the samples taken inside
        the given (t0, t1) wall-time windows."""
        sel = [r for r in self.rows if any(t0 <= r[0] <= t1 for t0, t1 in windows)]
        span = sum(t1 - t0 for t0, t1 in windows)
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window_s": span, "source": self.source, "error": self.error or "no sample in the window"}
        reasons = sorted({n for r in sel for n, bit in self.REASONS if r[3] & bit})
        return {"sm_mhz": statistics.median(r[1] for r in sel), "sm_max_mhz": max(r[2] for r in sel),
                "reasons": reasons, "samples": len(sel), "window_s": span,
                "source": f"{self.source} every {self.period * 1e3:.0f} ms during the timed loops"}


# ---------------------------------------------------------------- evidence from ncu
def kernel_source_hash():
    h = hashlib.sha256()
    for p in DOMINANT_KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def ncu_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary,
    or None when there is none or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{DOMINANT_KERNEL_NAME}_{workload}.txt")
    if not os.path.exists(path):
        return None
    kv = {}
    for line in open(path):
        if ":" in line:
            k, v = line.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_source_sha256") != kernel_source_hash():
        return None
    try:
        return int(float(kv["dram_bytes_per_launch"]))
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------- CPU oracle timing
def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


def cpu_baseline(wl, budget_s: float):
    """Explicit (K/V materialising) oracle over whole sequences until the budget is spent."""
    import mla_inputs
    from oracle import oracle_sequence
    weights, h, queries = mla_inputs.make_all(wl)
    lens = mla_inputs.context_lengths(wl)
    t0 = time.perf_counter()
    n = 0
    while n < wl.batch:
        oracle_sequence(wl, weights, h, queries, n, lens[n])
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
            "sample": f"{n} of {wl.batch} sequences of {wl.name}, all {wl.n_heads} heads, whole step "
                      f"(append + explicit decode + W_UV), fp64, {dt:.1f} s"}


# ---------------------------------------------------------------- workload facts
def workload_facts(wl, lens):
    rows = sum(n + wl.n_new for n in lens)
    row_bytes = (wl.d_c + wl.d_r) * (2 if wl.dtype == "bf16" else 4)
    flops_per_row = 2 * wl.n_heads * ((wl.d_c + wl.d_r) + wl.d_c)
    return rows, rows * row_bytes, rows * flops_per_row


L2_BYTES = 126 * 2 ** 20
NOMINAL_HBM_GBS = 8000.0             # "about 8 TB/s", the nominal HBM3e figure


def step_footprint(wl, lens):
    """Bytes a step reads from memory: the attended cache rows plus the weights."""
    el = 2 if wl.dtype == "bf16" else 4
    _, cache_bytes, _ = workload_facts(wl, lens)
    weights = ((wl.d_c + wl.d_r) * wl.hidden + 2 * wl.n_heads * wl.d_h * wl.d_c) * el
    return cache_bytes + weights


def l2_note(wl, lens):
    mb = step_footprint(wl, lens) / 1e6
    if step_footprint(wl, lens) > L2_BYTES:
        return f"inputs larger than L2 ({mb:.0f} MB of cache rows and weights per step); no flush"
    return (f"inputs fit in L2 ({mb:.1f} MB of cache rows and weights per step); no flush, "
            f"so repeated steps read them from L2")


def config_of(wl, lens, extra=None):
    c = {"workload": wl.name, "batch": wl.batch, "n_heads": wl.n_heads, "d_h": wl.d_h, "d_c": wl.d_c,
         "d_r": wl.d_r, "hidden": wl.hidden, "context_rows": (lens[0] if wl.ragged is None else
                                                               [int(min(lens)), int(max(lens))]),
         "new_tokens_per_seq": wl.n_new, "seed": wl.seed, "l2": l2_note(wl, lens)}
    if extra:
        c.update(extra)
    return c


# ---------------------------------------------------------------- our arm
# ---------------------------------------------------------------- multi-rank timing
def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time (every rank gets it).  Replicas only: the ranks run
    independent copies of the workload and exchange nothing but this number."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_throughput(units_per_rank: int, world: int, steps: int, ms_max: float) -> float:
    """Whole-job units per second: every rank's units over the slowest rank's time."""
    return units_per_rank * world * steps / (ms_max / 1e3)


# Workloads whose step is also measured with the query computed on the GPU from the new
# token's h (c_q = W_DQ h, q_C = W_UQ c_q, q_R = W_QR c_q) instead of given q_C, q_R.
FROM_H = {"v3_b64_l4096": "v3_b64_l4096_from_h"}


def time_from_h(args, name):
    """Graph-replay time of the h -> o step of workload ``name`` (mean of K replays)."""
    import torch
    import mla_inputs
    from head_latent_attention_25_b300 import runner
    wl = mla_inputs.WORKLOADS[name]
    lens = mla_inputs.context_lengths(wl)
    st = runner.from_workload(wl, ctx_lens=lens, num_splits=args.num_splits)
    g = st.capture()
    for _ in range(args.warmup):
        g.replay()
    stream = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(args.steps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0
    ms = a.elapsed_time(b) / args.steps
    el = 2 if wl.dtype == "bf16" else 4
    q_weights = (wl.d_q * wl.hidden + wl.n_heads * (wl.d_h + wl.d_r) * wl.d_q) * el
    out = {"workload": name, "ms_per_step": ms, "value": wl.batch / (ms / 1e3), "unit": UNIT,
           "query_weight_bytes": q_weights,
           "path": "c_q = W_DQ h, [q_C; q_R] = [W_UQ; W_QR] c_q, then the same step (graph replay)"}
    del st, g
    torch.cuda.empty_cache()
    return out


def time_fp8_decode(args, name):
    """The decode (fold, attention, merge) of the same batch and lengths over an fp8 cache
    (E4M3 codes with power-of-two group scales, bf16 rotary part; seeded random codes) beside
    the same decode over a bf16 cache (the workload's rows): mean of K launches each."""
    import torch
    import mla_inputs
    from head_latent_attention_25_b300 import (fp8_row_bytes, make_dims, mla_decode_absorbed,
                                               mla_decode_absorbed_fp8, mla_decode_workspace_size, runner,
                                               MLA_BF16)
    wl = mla_inputs.WORKLOADS[name]
    st = runner.from_workload(wl, num_splits=args.num_splits)
    st.step()
    torch.cuda.synchronize()
    rows = st.total_rows
    rb = fp8_row_bytes(wl.d_c, wl.d_r)
    g = torch.Generator(device="cuda").manual_seed(wl.seed)
    cache8 = torch.empty(rows, rb, dtype=torch.uint8, device="cuda")
    codes = torch.randint(0, 0x7E, (rows, wl.d_c), dtype=torch.uint8, device="cuda", generator=g)
    signs = torch.randint(0, 2, (rows, wl.d_c), dtype=torch.uint8, device="cuda", generator=g) * 128
    cache8[:, :wl.d_c] = codes | signs
    cache8[:, wl.d_c:wl.d_c + 4 * (wl.d_c // 128)].view(torch.float32)[:] = 2.0 ** -14
    cache8[:, wl.d_c + 4 * (wl.d_c // 128):].view(torch.bfloat16)[:] = st.cache[:rows, wl.d_c:]
    dims = st.dims
    ws_bytes = mla_decode_workspace_size(dims, MLA_BF16, st.batch, st.max_seq_len, args.num_splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    o8 = torch.empty_like(st.o_lat)
    lse8 = torch.empty(st.batch, wl.n_heads, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps

    def fp8():
        mla_decode_absorbed_fp8(dims, st.batch, st.q_c, st.q_r, st.w["w_uk"], cache8, rows, st.row_off,
                                st.seq_len, st.max_seq_len, args.num_splits, ws, ws_bytes, o8, lse8, st.dev_status)

    ms8, ms16 = timed(fp8), timed(st.decode)
    assert int(st.dev_status.item()) == 0
    out = {"workload": wl.name, "fp8_decode_ms": ms8, "bf16_decode_ms": ms16, "fp8_cache_bytes": rows * rb,
           "bf16_cache_bytes": rows * (wl.d_c + wl.d_r) * 2,
           "note": "fold + attention + merge; fp8 rows: E4M3 latent with power-of-two group scales, "
                   "bf16 rotary part; codes turned into bf16 tiles in shared memory"}
    del st
    torch.cuda.empty_cache()
    return out


def time_output_forms(args, name):
    """The layer output after the step, u = W_O [o_1; ...; o_n_h], timed two ways (mean of
    K launches each, CUDA events): two-step (W_UV per head, then W_O) and with W_UV merged
    into W_O (W_OV applied to the latent output)."""
    import dataclasses
    import torch
    import mla_inputs
    from head_latent_attention_25_b300 import runner
    wl = dataclasses.replace(mla_inputs.WORKLOADS[name], name=name + "_out", w_o=True)
    st = runner.from_workload(wl, num_splits=args.num_splits)
    st.step()
    st.merge_output_weights()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / args.steps

    def two_step():
        st.project_out()
        st.project_output()

    ms_two, ms_merged = timed(two_step), timed(st.project_output_merged)
    assert int(st.dev_status.item()) == 0
    el = 2 if wl.dtype == "bf16" else 4
    w_two = wl.n_heads * wl.d_h * (wl.d_c + wl.hidden) * el
    w_merged = wl.n_heads * wl.d_c * wl.hidden * el
    out = {"workload": wl.name, "two_step_ms": ms_two, "merged_ms": ms_merged,
           "two_step_weight_bytes": w_two, "merged_weight_bytes": w_merged,
           "two_step_gbs": w_two / (ms_two / 1e3) / 1e9, "merged_gbs": w_merged / (ms_merged / 1e3) / 1e9}
    del st
    torch.cuda.empty_cache()
    return out


def run_ours(args, wl, rank, world):
    import torch
    import torch.distributed as dist
    import mla_inputs
    from head_latent_attention_25_b300 import runner, mla_copy_from_host, mla_launch_count, mla_profile_events

    dev = torch.cuda.current_device()
    lens = mla_inputs.context_lengths(wl)
    st = runner.from_workload(wl, ctx_lens=lens, num_splits=args.num_splits)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()


    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = str(dev)
    sampler = ClockSampler(uuid) if rank == 0 else None

    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    assert int(st.dev_status.item()) == 0, "device status set during warm-up"
    windows = []                        # wall-time windows of the timed loops (clock record)

    K = args.steps
    ev_split = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for a, b in ev_split:               # torch creates the CUDA event on its first record
        a.record(stream)
        b.record(stream)
    t_beg, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    n0 = mla_launch_count()
    wall0 = time.time()
    t_beg.record(stream)
    for i in range(K):
        mla_profile_events(*ev_split[i])
        st.step()
    t_end.record(stream)
    torch.cuda.synchronize()
    windows.append((wall0, time.time()))
    barrier(world)
    mla_profile_events(None, None)
    launches = mla_launch_count() - n0
    ms_eager = max_over_ranks(t_beg.elapsed_time(t_end), world)
    split_times = [a.elapsed_time(b) for a, b in ev_split]
    split_ms = statistics.mean(split_times)
    assert int(st.dev_status.item()) == 0

    # the same step captured once into a CUDA graph and replayed K times (the kernels
    # and their arguments are identical; only the host launch path differs)
    ms_graph = None
    g = None
    replay_ms = []
    if not args.no_graph:
        g = st.capture()
        for _ in range(args.warmup):
            g.replay()
        g_beg, g_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        wall0 = time.time()
        g_beg.record(stream)
        for _ in range(K):
            g.replay()
        g_end.record(stream)
        torch.cuda.synchronize()
        windows.append((wall0, time.time()))
        barrier(world)
        assert int(st.dev_status.item()) == 0
        ms_graph = max_over_ranks(g_beg.elapsed_time(g_end), world)
        # per-replay durations for the median: at least 50 replays and at least 0.5 s,
        # each bracketed by events recorded between consecutive replays
        n_med = max(50, K, int(0.5 / max(ms_graph / K / 1e3, 1e-6)) + 1)
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_med + 1)]
        torch.cuda.synchronize()
        wall0 = time.time()
        evs[0].record(stream)
        for i in range(n_med):
            g.replay()
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        windows.append((wall0, time.time()))
        replay_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(n_med)]
        assert int(st.dev_status.item()) == 0
    clocks = None
    if sampler:
        sampler.stop()
        clocks = sampler.summary(windows)
    ms = ms_graph if ms_graph is not None else ms_eager

    # end to end: every step's inputs come from pinned host memory and its result goes back
    # to pinned host memory, as in a serving loop: the copies run on two further streams (one
    # per direction) through double-buffered device staging, so step k+1's inputs and step
    # k-1's result move while step k computes; every step still carries its own copies.
    # h, q_c and q_r are views of one contiguous device buffer (st.inputs): one copy each
    # way; a workload that projects its query from h moves only h.  The host-to-device move is
    # the library's mla_copy_from_host (a kernel reading the pinned host buffer over the bus:
    # a 4 MB copy-engine transfer ran at ~11 GB/s on these hosts, the kernel at ~48 GB/s) or
    # the copy engine, whichever the warm-up times faster (below); results come back with
    # cudaMemcpyAsync.  With graphs, each staging
    # slot has a graph of its own (staged inputs in, the step, result out), and the stream
    # and copy calls go straight to the CUDA runtime when its Python binding is present, so
    # the host issues a handful of calls per step.
    dev_in = st.h.view(-1) if wl.query_from_h else st.inputs
    in_host = dev_in.cpu().pin_memory()
    h2d = in_host.numel() * in_host.element_size()
    d2h = st.out.numel() * st.out.element_size()
    NS = 2
    copy_stream = torch.cuda.Stream()                    # host -> device
    back_stream = torch.cuda.Stream()                    # device -> host (the other copy engine)
    stage_in = [torch.empty_like(dev_in) for _ in range(NS)]
    stage_out = [torch.empty_like(st.out) for _ in range(NS)]
    out_host = [torch.empty(st.out.shape, dtype=st.out.dtype).pin_memory() for _ in range(NS)]
    ev_in = [torch.cuda.Event() for _ in range(NS)]      # inputs of the slot are on the device
    ev_used = [torch.cuda.Event() for _ in range(NS)]    # the step of the slot has run
    ev_out = [torch.cuda.Event() for _ in range(NS)]     # the slot's result is on the host
    for e in ev_in + ev_used + ev_out:                   # torch creates the CUDA event on its first record
        e.record(stream)
    used = [False] * NS
    transport = ["kernel"]                               # chosen below: "kernel" or "copy_engine"

    def slot_body(sl, s):
        dev_in.copy_(stage_in[sl])
        if wl.query_from_h:
            st.x_q.copy_(st.h[:, -1, :])
        st.step(s)
        stage_out[sl].copy_(st.out)

    gs = None
    if g is not None:
        gs = []
        cs = torch.cuda.Stream()
        cs.wait_stream(stream)
        for sl in range(NS):
            gg = torch.cuda.CUDAGraph()
            with torch.cuda.stream(cs):
                slot_body(sl, cs)                         # warm-up outside capture
            torch.cuda.synchronize()
            with torch.cuda.graph(gg, stream=cs):
                slot_body(sl, cs)
            gs.append(gg)
        torch.cuda.synchronize()
    try:
        from cuda.bindings import runtime as rt
        D2H = rt.cudaMemcpyKind.cudaMemcpyDeviceToHost
        S, C, R = stream.cuda_stream, copy_stream.cuda_stream, back_stream.cuda_stream
        e_in = [e.cuda_event for e in ev_in]
        e_used = [e.cuda_event for e in ev_used]
        e_out = [e.cuda_event for e in ev_out]

        def ck(r):
            if r[0] != rt.cudaError_t.cudaSuccess:
                raise RuntimeError(f"CUDA runtime call failed in the end-to-end loop: {r[0]}")

        H2D = rt.cudaMemcpyKind.cudaMemcpyHostToDevice

        def h2d_copy(k):
            sl = k % NS
            if used[sl]:
                ck(rt.cudaStreamWaitEvent(C, e_used[sl], 0))          # step k-NS has read this slot
            if transport[0] == "kernel":
                mla_copy_from_host(stage_in[sl], in_host, h2d, C)
            else:
                ck(rt.cudaMemcpyAsync(stage_in[sl].data_ptr(), in_host.data_ptr(), h2d, H2D, C))
            ck(rt.cudaEventRecord(e_in[sl], C))

        def compute(k):
            sl = k % NS
            ck(rt.cudaStreamWaitEvent(S, e_in[sl], 0))
            if used[sl]:
                ck(rt.cudaStreamWaitEvent(S, e_out[sl], 0))           # step k-NS's result has left the slot
            if gs is not None:
                gs[sl].replay()
            else:
                slot_body(sl, stream)
            ck(rt.cudaEventRecord(e_used[sl], S))
            used[sl] = True

        def d2h_copy(k):
            sl = k % NS
            ck(rt.cudaStreamWaitEvent(R, e_used[sl], 0))
            ck(rt.cudaMemcpyAsync(out_host[sl].data_ptr(), stage_out[sl].data_ptr(), d2h, D2H, R))
            ck(rt.cudaEventRecord(e_out[sl], R))
        e2e_calls = "CUDA runtime binding"
    except ImportError:
        def h2d_copy(k):
            sl = k % NS
            with torch.cuda.stream(copy_stream):
                if used[sl]:
                    copy_stream.wait_event(ev_used[sl])
                if transport[0] == "kernel":
                    mla_copy_from_host(stage_in[sl], in_host, h2d, copy_stream)
                else:
                    stage_in[sl].copy_(in_host, non_blocking=True)
                ev_in[sl].record(copy_stream)

        def compute(k):
            sl = k % NS
            stream.wait_event(ev_in[sl])
            if used[sl]:
                stream.wait_event(ev_out[sl])
            if gs is not None:
                gs[sl].replay()
            else:
                slot_body(sl, stream)
            ev_used[sl].record(stream)
            used[sl] = True

        def d2h_copy(k):
            sl = k % NS
            with torch.cuda.stream(back_stream):
                back_stream.wait_event(ev_used[sl])
                out_host[sl].copy_(stage_out[sl], non_blocking=True)
                ev_out[sl].record(back_stream)
        e2e_calls = "torch stream calls"

    def e2e_run(n):
        copy_stream.wait_stream(stream)
        back_stream.wait_stream(stream)
        h2d_copy(0)
        for k in range(n):
            if k + 1 < n:
                h2d_copy(k + 1)
            compute(k)
            d2h_copy(k)
        stream.wait_stream(copy_stream)
        stream.wait_stream(back_stream)                  # the last result is on the host

    # Transport of the inputs: the host-read kernel moves them faster but needs SMs, which it
    # then takes from the step while it runs beside it; the copy engine needs none but has a
    # large fixed cost per copy on these hosts.  The warm-up times both and keeps the faster.
    def e2e_time(n):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        e2e_run(n)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    tried = {}
    for t in ("kernel", "copy_engine"):
        transport[0] = t
        e2e_run(args.warmup)
        tried[t] = e2e_time(max(args.warmup, 3))
    transport[0] = min(tried, key=tried.get)
    e2e_run(args.warmup)
    e_beg, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    e_beg.record(stream)
    e2e_run(K)
    e_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e_beg.elapsed_time(e_end), world)
    assert int(st.dev_status.item()) == 0
    assert torch.equal(out_host[(K - 1) % NS].to(st.out.device), st.out)

    if rank != 0:
        return None
    rows, cache_bytes, flops = workload_facts(wl, lens)
    hbm, tf_burst, tf_sus, src = peaks()
    split_s = split_ms / 1e3
    gbs = cache_bytes / split_s / 1e9
    tfs = flops / split_s / 1e12
    value = job_throughput(wl.batch, world, K, ms)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic (seeded N(0,0.02) weights and cache)",
        "config": config_of(wl, lens, {"parallelism": "replicas" if world > 1 else "single_gpu",
                                       "num_splits": args.num_splits or "auto",
                                       "launch": "cuda_graph" if ms_graph is not None else "eager"}),
        "ms_per_step_eager": ms_eager / K,
        "ms_per_step_median": statistics.median(replay_ms) if replay_ms else None,
        "ms_per_step_replays": len(replay_ms),
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "traffic": ncu_traffic(wl.name), "kernel": DOMINANT_KERNEL_NAME,
                     "peak_source": f"{src} copy bandwidth",
                     "frac_of_nominal": gbs / NOMINAL_HBM_GBS, "nominal_peak": NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": cache_bytes, "kernel_ms": split_ms,
                     "kernel_ms_median": statistics.median(split_times)},
        "roofline_tensor": {"achieved": tfs, "unit": "TFLOP/s", "peak_burst": tf_burst,
                            "peak_sustained": tf_sus, "frac_burst": tfs / tf_burst,
                            "frac_sustained": tfs / tf_sus, "algorithmic_flops_per_launch": flops},
        "cache_gbs_step": cache_bytes / (ms / K / 1e3) / 1e9,
        "e2e": {"value": job_throughput(wl.batch, world, K, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "launch": "cuda_graph" if g is not None else "eager",
                "copies": "inputs and results on two further streams (one per direction), double-buffered "
                          "staging, overlapped with compute; host-to-device by mla_copy_from_host (a kernel "
                          "reading the pinned host buffer) or the copy engine, whichever the warm-up timed "
                          "faster; device-to-host by cudaMemcpyAsync; one graph per staging slot; " + e2e_calls,
                "h2d_transport": transport[0], "warmup_ms": tried},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if wl.name in FROM_H and not args.no_from_h and not args.no_graph:
        line["h_to_o"] = time_from_h(args, FROM_H[wl.name])
        line["output_projection"] = time_output_forms(args, wl.name)
        line["fp8_cache"] = time_fp8_decode(args, wl.name)
        # the decode alone (fold, attention, merge) beside the whole layer step of `value`
        dec_ms = line["fp8_cache"]["bf16_decode_ms"]
        line["decode_only"] = {"ms_per_step": dec_ms, "value": wl.batch * world / (dec_ms / 1e3), "unit": UNIT,
                               "launch": "eager launches, mean of K"}
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_budget)
    return line


# ---------------------------------------------------------------- reference arm
def run_reference(args, wl):
    """The oracle as it stands, timed on the host cores: each step decodes one sequence
    over a subset of heads sized so the whole run stays within a few minutes."""
    import mla_inputs
    from oracle import oracle_sequence
    weights, h, queries = mla_inputs.make_all(wl)
    lens = mla_inputs.context_lengths(wl)
    t = time.perf_counter()
    oracle_sequence(wl, weights, h, queries, 0, lens[0], heads=list(range(min(4, wl.n_heads))))
    per_head = (time.perf_counter() - t) / min(4, wl.n_heads)
    budget_per_step = 150.0 / max(1, args.steps + args.warmup)
    n_heads = max(1, min(wl.n_heads, int(budget_per_step / max(per_head, 1e-9))))
    heads = list(range(n_heads))
    for i in range(args.warmup):
        b = i % wl.batch
        oracle_sequence(wl, weights, h, queries, b, lens[b], heads=heads)
    t0 = time.perf_counter()
    for i in range(args.steps):
        b = i % wl.batch
        oracle_sequence(wl, weights, h, queries, b, lens[b], heads=heads)
    dt = time.perf_counter() - t0
    value = args.steps * (n_heads / wl.n_heads) / dt
    sample = (f"each step: one sequence of {wl.name} ({n_heads} of {wl.n_heads} heads, "
              f"counted as {n_heads}/{wl.n_heads} token), append + explicit decode + W_UV, fp64")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,0.02) weights and cache)", "config": config_of(wl, lens),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def named_workloads():
    """Every workload --workload accepts: the named ones and each point of the sweep."""
    import mla_inputs
    return dict(mla_inputs.WORKLOADS, **{w.name: w for w in mla_inputs.sweep_workloads()})


def main():
    args = parse()
    import mla_inputs
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    named = named_workloads()
    if args.workload not in named:
        raise SystemExit(f"unknown workload {args.workload!r}; known: {', '.join(named)}")
    wl = named[args.workload]
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, wl)), flush=True)
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    if args.sweep:
        for w in mla_inputs.sweep_workloads():
            line = run_ours(args, w, rank, world)
            if line:
                print(json.dumps(line), flush=True)
            torch.cuda.empty_cache()
    else:
        line = run_ours(args, wl, rank, world)
        if line:
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
