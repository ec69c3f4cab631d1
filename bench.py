#!/usr/bin/env python3
"""Benchmark of the paged KV-pool attention hot path on GB300.

A step is one decode step of the Llama-3-8B-shaped workload, the largest
decode configuration (32 layers, 200 real requests padded with 56 CUDA-Graph
padding requests to batch 256, H_q 32, H_kv 8, head_dim 128, page_size 1,
contexts log-uniform in [1024, 8192], pool 1.2x the live tokens): per layer,
store_kv of the 256 new tokens and split-KV decode attention, in one
minisgl_store_decode_attn call (partial kernel, which also stores the new
rows, + LSE merge kernel); the same step as two calls (minisgl_store_kv, then
minisgl_decode_attn) is reported beside it.  The metric is paged
decode-attention HBM GB/s (algorithmic bytes / time) with the step's tokens/s
(200 real tokens per step) beside it.  Secondary objects: the Qwen3-0.6B
28-layer step, the long 64-row-page layer, tiny-decode latency, store_kv of an
8192-token extend batch, extend (chunked prefill) TFLOP/s on the radix-shared
workload, fused RoPE + store_kv, a mixed chunk + decode batch, shared-prefix
(cascade) decode, and programmatic dependent launch on/off.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference]

Under torchrun (N > 1) each rank runs its own copy of the workload (data
parallel over requests, no collective on the data path): weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

L2_BYTES = 129 * 2 ** 20


# --------------------------------------------------------------------------- #
# algorithmic work
# --------------------------------------------------------------------------- #
def decode_layer_bytes(case) -> int:
    """Bytes one decode-attention call must move at minimum: each context
    token's K and V row for every KV head (the padding requests all read one
    dummy row, counted once), every page-table entry read, the queries, the
    outputs and seq_lens."""
    Hkv, d, Hq = case.num_kv_heads, case.head_dim, case.num_q_heads
    ctx = int(case.seq_lens[:case.num_real].sum())
    entries = int(case.seq_lens.sum())
    dummy = int(case.batch - case.num_real) > 0
    kv_rows = ctx + (1 if dummy else 0)
    return (kv_rows * 2 * Hkv * d * 2 + entries * 4 + case.batch * Hq * d * 2 * 2 + case.batch * 4)


def store_layer_bytes(case) -> int:
    """store_kv: read k and v rows, write them into the pool, read out_loc."""
    return case.batch * (2 * 2 * case.num_kv_heads * case.head_dim * 2 + 4)


def cascade_layer_bytes(case) -> int:
    """Shared-prefix decode reading the shared rows once: the prefix K/V and
    its page-table entries once, each request's private rows and entries,
    the queries, outputs and seq_lens."""
    Hkv, d, Hq = case.num_kv_heads, case.head_dim, case.num_q_heads
    P = case.shared_len
    own = int((case.seq_lens - P).clamp(min=0).sum())
    return ((P + own) * (2 * Hkv * d * 2 + 4) + case.batch * Hq * d * 2 * 2 + case.batch * 4)


def rope_store_bytes(case) -> int:
    """Fused RoPE + store_kv over all extend batches: per token, q read and
    written, k and v read and written to the pool, one cos/sin row, the
    position and out_loc: 4 d (H_q + 2 H_kv + 1) + 8 bytes."""
    d, Hq, Hkv = case.head_dim, case.num_q_heads, case.num_kv_heads
    return int(sum(case.extend_lens)) * (4 * d * (Hq + 2 * Hkv + 1) + 8)


def extend_flops(case) -> float:
    """Causal-visible FLOPs: 4 d H_q (E C + E(E+1)/2) per request chunk."""
    f = 0.0
    d, Hq = case.head_dim, case.num_q_heads
    for b in case.batches:
        for C, E in zip(b.cached_lens.tolist(), b.extend_lens.tolist()):
            f += 4.0 * d * Hq * (E * C + E * (E + 1) / 2)
    return f


# --------------------------------------------------------------------------- #
# peaks, clocks, ncu traffic
# --------------------------------------------------------------------------- #
def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"]),
                "bf16_tflops_sustained": float(j.get("bf16_tflops_sustained", j["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            ident = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            ident = None
        self.ident = ident

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                   "-lms", "200"]
            if self.ident:
                cmd += ["-i", self.ident]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def profile_traffic(kernel_file: str, summary_name: str):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    summary is missing or was taken on a different version of the kernel source."""
    path = os.path.join(ROOT, "profiles", summary_name)
    src = os.path.join(ROOT, "paged_kv_cache_row_gb300", "csrc", kernel_file)
    try:
        text = open(path).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != digest:
        return None
    return float(m.group(1))


# --------------------------------------------------------------------------- #
# distributed plumbing
# --------------------------------------------------------------------------- #
def dist_setup(n_gpus: int, backend: str = ""):
    """Rank setup from the torchrun environment.  One process per GPU with
    NCCL on a GPU machine; the gloo backend (CPU) serves the multi-process tests.
    The data path has no collective: every rank runs its own batch."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group("gloo")
    elif backend == "nccl":
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's time: the job finishes when every rank has."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units all ranks processed (each rank the same
    amount: weak scaling) over the slowest rank's time, per second."""
    return world * units_per_rank / (ms_max * 1e-3)


# --------------------------------------------------------------------------- #
# the oracle on the host cores (CPU baseline and the reference arm)
# --------------------------------------------------------------------------- #
def oracle_decode_sample(case, pool_t, k_new, v_new, q, layers, reqs):
    """Prepare host inputs for oracle decode of `reqs` on `layers` (store_kv of
    their new rows, then decode).  Returns (callable, algorithmic bytes)."""
    import numpy as np
    import oracle
    orc = oracle.get()
    W = case.page_table.shape[1]
    rows = torch.cat([case.page_table[r, :int(case.seq_lens[r])] for r in reqs]).long()
    uniq = torch.unique(rows)
    idx = uniq.to(pool_t.device)

    def u16(t):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()

    pos = {int(x): i for i, x in enumerate(uniq.tolist())}
    pt = torch.zeros((len(reqs), W), dtype=torch.int32)
    sl = torch.zeros(len(reqs), dtype=torch.int32)
    for i, r in enumerate(reqs):
        n = int(case.seq_lens[r])
        sl[i] = n
        pt[i, :n] = torch.tensor([pos[int(x)] for x in case.page_table[r, :n].tolist()],
                                 dtype=torch.int32)
    loc = torch.tensor([pos[int(case.out_loc[r])] for r in reqs], dtype=torch.int32)
    per_layer = []
    for l in layers:
        hk, hv = u16(pool_t[0, l].index_select(0, idx)), u16(pool_t[1, l].index_select(0, idx))
        per_layer.append((hk, hv, k_new[l][reqs].cpu(), v_new[l][reqs].cpu(), q[l][reqs].cpu()))
    Hkv, d, Hq = case.num_kv_heads, case.head_dim, case.num_q_heads
    ctx = int(sl.sum())
    nbytes = len(layers) * (ctx * (2 * Hkv * d * 2 + 4) + len(reqs) * (Hq * d * 4 + 4)
                            + len(reqs) * (2 * 2 * Hkv * d * 2 + 4))

    def run():
        # store_kv rewrites the same rows with the same values on every run
        for hk, hv, kn, vn, qq in per_layer:
            orc.store_kv(hk, hv, kn, vn, loc)
            orc.decode(qq, hk, hv, pt, sl, case.sm_scale)

    return run, nbytes


def cpu_cores_used() -> int:
    return 1  # the oracle is single-threaded C


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine()


def oracle_all_cores(case, pool_t, k_new, v_new, q, budget_s=10.0):
    """The same oracle on every host core: the batch's requests are dealt
    round-robin to one thread per core, each thread calling the oracle on its
    own requests (ctypes releases the GIL, so the C calls run in parallel).
    Returns (GB/s, threads, sample text)."""
    from concurrent.futures import ThreadPoolExecutor
    cores = len(os.sched_getaffinity(0))
    B = case.batch
    groups = [list(range(i, B, cores)) for i in range(min(cores, B))]
    lay = sorted({0, case.num_layers - 1})
    runs = [oracle_decode_sample(case, pool_t, k_new, v_new, q, lay, g) for g in groups]
    nbytes = sum(b for _, b in runs)
    with ThreadPoolExecutor(len(runs)) as ex:
        t0 = time.perf_counter()
        n = 0
        while True:
            list(ex.map(lambda rb: rb[0](), runs))
            n += 1
            if time.perf_counter() - t0 > budget_s or n >= 200:
                break
        dt = time.perf_counter() - t0
    sample = (f"store_kv + decode of all {B} requests on layers {lay}, one thread per core "
              f"({len(runs)} threads), repeated {n}x, {dt:.1f} s, fp64 C")
    return nbytes * n / dt / 1e9, len(runs), sample


# --------------------------------------------------------------------------- #
# GPU arm
# --------------------------------------------------------------------------- #
def ev_time(fn, reps, stream, before=None):
    """Mean duration in ms of `fn` over `reps` calls, each bracketed by CUDA
    events on the launching stream; `before` (an L2 flush) runs outside the
    events before every call."""
    evs = []
    for _ in range(reps):
        if before is not None:
            before()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in evs)


def graph_ms(fn, n, replays, stream):
    """Device time in ms per call of `fn`: n calls captured in one CUDA graph,
    the graph replayed `replays` times after 3 untimed replays, so no host
    time sits between the launches."""
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        for _ in range(n):
            fn()
    for _ in range(3):
        gr.replay()
    ms = ev_time(gr.replay, replays, stream) / n
    del gr
    return ms


def input_wait_schedule(L: int) -> dict:
    """Layers before which the e2e step's compute stream waits for input
    copies: {layer: last layer whose inputs the wait covers}, at layers 0, 1,
    2, 4, 8, ... (each wait covers the inputs of the layers up to about twice
    as far), so every layer's inputs are covered by the time it runs."""
    sched, w = {0: 0}, 1
    while w < L:
        sched[w] = min(L - 1, 2 * w + 1)
        w *= 2
    return sched


def headline_case(layers: int):
    """The Llama-3-8B decode workload with its pool at 1.2x the live tokens,
    or 1.05x when the device has too little free memory for that (the pool of
    32 layers at 1.2x is about 108 GB)."""
    free, _ = torch.cuda.mem_get_info()
    case = workloads.decode_llama3_8b(num_layers=layers)
    if workloads.decode_pool_bytes(case) + (8 << 30) > free:
        case = workloads.decode_llama3_8b(num_layers=layers, pool_factor=1.05)
        case.pool_factor = 1.05
    else:
        case.pool_factor = 1.2
    return case


def decode_step_fn(mk, case, pool, k_new, v_new, q, pt, sl, loc, outs, ws, fused=True):
    """One decode step over all layers: per layer store_kv of the step's new
    rows and split-KV decode + LSE merge, fused into one call or as two."""
    L = case.num_layers

    def step():
        for l in range(L):
            if fused:
                mk.minisgl_store_decode_attn(pool, l, k_new[l], v_new[l], loc, q[l], pt, sl,
                                             case.sm_scale, out=outs[l], workspace=ws)
            else:
                mk.minisgl_store_kv(pool, l, k_new[l], v_new[l], loc)
                mk.minisgl_decode_attn(pool, l, q[l], pt, sl, case.sm_scale, out=outs[l], workspace=ws)
    return step


def time_steps(step, steps, warmup, stream, world):
    """Device time per step over exactly `steps` steps after `warmup`, with a
    barrier and a synchronize on both sides, max over ranks."""
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(e0.elapsed_time(e1) / steps, world)


def secondary_decode_step(mk, args, dev, stream, peaks, case):
    """A whole multi-layer decode step of another workload (fused calls)."""
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, dev)
    pool = mk.KVPool(pool_t, case.page_size)
    pt, sl, loc = case.page_table.to(dev), case.seq_lens.to(dev), case.out_loc.to(dev)
    ws = mk.decode_workspace(case.batch, case.num_q_heads, pool)
    outs = torch.empty((case.num_layers,) + tuple(q.shape[1:]), dtype=torch.bfloat16, device=dev)
    step = decode_step_fn(mk, case, pool, k_new, v_new, q, pt, sl, loc, outs, ws)
    ms = time_steps(step, max(5, args.steps // 4), args.warmup, stream, 1)
    mk.minisgl_debug_set_pdl(False)
    ms_off = time_steps(step, max(5, args.steps // 4), args.warmup, stream, 1)
    mk.minisgl_debug_set_pdl(True)
    ms_on = time_steps(step, max(5, args.steps // 4), args.warmup, stream, 1)
    layer_b = decode_layer_bytes(case) + store_layer_bytes(case)
    gbs = case.num_layers * layer_b / (ms * 1e-3) / 1e9
    res = {"workload": case.name, "layers": case.num_layers, "batch": case.batch,
           "real_requests": case.num_real, "H_q": case.num_q_heads, "H_kv": case.num_kv_heads,
           "page_size": case.page_size, "context_tokens": int(case.seq_lens[:case.num_real].sum()),
           "call": "minisgl_store_decode_attn per layer", "ms_per_step": round(ms, 4),
           "achieved_gbs": round(gbs, 1), "frac_of_hbm": round(gbs / peaks["hbm_gbs"], 4),
           "tokens_per_s": round(case.num_real / (ms * 1e-3), 1),
           "pdl_ab": {"ms_per_step_pdl_off": round(ms_off, 4), "ms_per_step_pdl_on": round(ms_on, 4),
                      "gain": round(ms_off / ms_on - 1.0, 4)},
           "l2": "inputs larger than L2 (%.2f GB of K/V per layer)" % (layer_b / 1e9)}
    del pool_t, k_new, v_new, q, outs
    torch.cuda.empty_cache()
    return res


def bench_tiny(mk, args, dev, stream):
    """Tiny decode (batch 4, GQA 4, d 64): latency of one store + decode."""
    tc = workloads.decode_tiny()
    tpool_t, tk, tv, tq = workloads.make_decode_values(tc, dev)
    tpool = mk.KVPool(tpool_t)
    tpt, tsl, tloc = tc.page_table.to(dev), tc.seq_lens.to(dev), tc.out_loc.to(dev)
    tws = mk.decode_workspace(tc.batch, tc.num_q_heads, tpool)
    tout = torch.empty_like(tq[0])

    def t_fused():
        mk.minisgl_store_decode_attn(tpool, 0, tk[0], tv[0], tloc, tq[0], tpt, tsl, tc.sm_scale,
                                     out=tout, workspace=tws)

    def t_two():
        mk.minisgl_store_kv(tpool, 0, tk[0], tv[0], tloc)
        mk.minisgl_decode_attn(tpool, 0, tq[0], tpt, tsl, tc.sm_scale, out=tout, workspace=tws)

    reps = max(50, args.steps)
    for fn in (t_fused, t_two):
        for _ in range(args.warmup):
            fn()
    torch.cuda.synchronize()

    def graph_us(fn, n=20):
        return graph_ms(fn, n, 20, stream) * 1e3

    return {"workload": tc.name, "batch": tc.batch, "context_tokens": int(tc.seq_lens.sum()),
            "us_store_decode_fused": round(graph_us(t_fused), 2),
            "us_store_kv_then_decode": round(graph_us(t_two), 2),
            "timing": "device time per call: 20 calls captured in a CUDA graph, replayed 20x",
            "us_per_python_call_fused": round(ev_time(t_fused, reps, stream) * 1e3, 2),
            "us_per_python_call_two": round(ev_time(t_two, reps, stream) * 1e3, 2),
            "python_call_note": "one call at a time through the Python binding: host-bound",
            "note": "latency bound: the whole pool (4 MB) stays in L2"}


def bench_store_kv_at_scale(mk, args, dev, stream, peaks):
    """store_kv of 8192-token batches (the chunked-prefill budget; 67 MB moved
    per launch) in steady state: eight batches with disjoint rows and their
    own k/v are stored one after the other, so each launch reads and writes
    memory the previous seven have pushed out of the L2 (536 MB in all)."""
    rot = workloads.store_rotation()
    Hkv, d = rot.num_kv_heads, rot.head_dim
    pool_t = workloads.make_pool(1, rot.num_rows, Hkv, d, 0.5, rot.seed, dev)
    pool = mk.KVPool(pool_t)
    g = torch.Generator(device=dev).manual_seed(rot.seed * 104729 + 7)
    n = int(rot.out_locs[0].numel())
    ks = [torch.empty((n, Hkv, d), dtype=torch.bfloat16, device=dev).normal_(0, 0.5, generator=g)
          for _ in rot.out_locs]
    vs = [torch.empty((n, Hkv, d), dtype=torch.bfloat16, device=dev).normal_(0, 0.5, generator=g)
          for _ in rot.out_locs]
    locs = [l.to(dev) for l in rot.out_locs]

    def rotation():
        for k, v, l in zip(ks, vs, locs):
            mk.minisgl_store_kv(pool, 0, k, v, l)

    for _ in range(args.warmup):
        rotation()
    reps = max(5, args.steps // 4)
    nb = len(locs)
    # device time: two rotations (16 launches) captured in a CUDA graph and
    # replayed, so the launches run back to back as in a captured model step;
    # one Python call per launch is also timed, for context (a 67 MB store
    # takes about as long on the device as the binding takes on the host)
    ms = graph_ms(rotation, 2, reps, stream) / nb
    eager_ms = ev_time(lambda: [rotation() for _ in range(reps)], 1, stream) / (reps * nb)
    s_b = n * (2 * 2 * Hkv * d * 2 + 4)
    # context: a plain device copy of the same bytes (k and v of a batch into a
    # contiguous buffer), in the same rotation, by torch, timed the same way
    cdst = [torch.empty((2, n, Hkv, d), dtype=torch.bfloat16, device=dev) for _ in locs]

    def copy_rotation():
        for k, v, c in zip(ks, vs, cdst):
            c[0].copy_(k)
            c[1].copy_(v)

    for _ in range(args.warmup):
        copy_rotation()
    c_ms = graph_ms(copy_rotation, 2, reps, stream) / nb
    res = {"workload": rot.name, "tokens": n, "algorithmic_bytes": s_b,
           "ms_per_launch": round(ms, 5), "achieved_gbs": round(s_b / (ms * 1e-3) / 1e9, 1),
           "frac_of_hbm": round(s_b / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
           "traffic": profile_traffic("store_kv.cu", "store_kv_extend_batch.md"),
           "launches_timed": 2 * reps * nb,
           "timing": "device time: 2 rotations (16 launches) captured in a CUDA graph, replayed",
           "eager_python_calls": {"ms_per_launch": round(eager_ms, 5),
                                  "gbs": round(s_b / (eager_ms * 1e-3) / 1e9, 1),
                                  "note": "one Python binding call per launch: the host sets the pace"},
           "same_size_copy": {"ms": round(c_ms, 5), "gbs": round(s_b / (c_ms * 1e-3) / 1e9, 1),
                              "what": "torch copy of the same k and v bytes into contiguous buffers, "
                                      "same rotation (two copy kernels per batch), same CUDA-graph timing",
                              "store_kv_relative": round(c_ms / ms, 4)},
           "l2": "8 batches with disjoint rows stored in turn: 536 MB per rotation, larger than L2"}
    del pool_t, ks, vs, cdst
    torch.cuda.empty_cache()
    return res


def bench_extend(mk, args, dev, stream, peaks, flush):
    """store_kv + extend per chunked-prefill batch of the radix-shared
    workload (TFLOP/s of causal-visible FLOPs), and fused RoPE + store_kv
    over the same batches."""
    ecase = workloads.extend_radix_shared()
    epool_t, per_batch = workloads.make_extend_values(ecase, dev)
    epool = mk.KVPool(epool_t)
    eargs = [(b.page_table.to(dev), b.cached_lens.to(dev), b.extend_lens.to(dev),
              b.q_offsets.to(dev), b.out_loc.to(dev)) for b in ecase.batches]
    eouts = [torch.empty_like(qq) for _, _, qq in per_batch]

    def estep():
        for (k, v, qq), (ept, ecl, eel, eqo, eloc), eo in zip(per_batch, eargs, eouts):
            mk.minisgl_store_kv(epool, 0, k, v, eloc)
            mk.minisgl_extend_attn(epool, 0, qq, ept, ecl, eel, eqo, ecase.sm_scale, out=eo)

    for _ in range(args.warmup):
        estep()
    torch.cuda.synchronize()
    eks = max(5, args.steps // 10)
    xev = []
    for _ in range(eks):
        for (k, v, qq), (ept, ecl, eel, eqo, eloc), eo in zip(per_batch, eargs, eouts):
            flush()  # q, out and the batch's rows (~170 MB) would partly stay in L2
            mk.minisgl_store_kv(epool, 0, k, v, eloc)
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            mk.minisgl_extend_attn(epool, 0, qq, ept, ecl, eel, eqo, ecase.sm_scale, out=eo)
            b_.record(stream)
            xev.append((a, b_))
    torch.cuda.synchronize()
    ext_ms_per_pass = sum(a.elapsed_time(b_) for a, b_ in xev) / eks
    fl = extend_flops(ecase)
    tf = fl / (ext_ms_per_pass * 1e-3) / 1e12
    launch_fl = fl / len(ecase.batches)
    launch_ms = ext_ms_per_pass / len(ecase.batches)
    ext = {
        "workload": ecase.name, "metric": "extend-attn TFLOP/s (causal-visible FLOPs)",
        "value": round(tf, 2), "unit": "TFLOP/s", "ms_per_pass": round(ext_ms_per_pass, 4),
        "batches": len(ecase.batches), "tokens": int(sum(ecase.extend_lens)),
        "tokens_per_s": round(sum(ecase.extend_lens) / (ext_ms_per_pass * 1e-3), 1),
        "l2": "flushed (256 MB write) before each batch's store_kv + timed extend call",
        "roofline": {"bound": "tensor", "achieved": round(launch_fl / (launch_ms * 1e-3) / 1e12, 2),
                     "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": round(launch_fl / (launch_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                     "traffic": profile_traffic("extend.cu", "extend_radix_shared.md"),
                     "peak_source": peaks["source"] + " bf16 dense burst"},
    }
    # the same batches through the shared-prefix (cascade) extend call
    P = int(ecase.prefix_rows.numel())
    Tmax = max(b.total_tokens for b in ecase.batches)
    cws = torch.zeros(mk.minisgl_cascade_extend_workspace_bytes(Tmax, ecase.num_q_heads, ecase.head_dim),
                      dtype=torch.uint8, device=dev)

    def cstep():
        for (k, v, qq), (ept, ecl, eel, eqo, eloc), eo in zip(per_batch, eargs, eouts):
            mk.minisgl_store_kv(epool, 0, k, v, eloc)
            mk.minisgl_cascade_extend_attn(epool, 0, qq, ept, ecl, eel, eqo, P, ecase.sm_scale, out=eo,
                                           workspace=cws)

    for _ in range(args.warmup):
        cstep()
    torch.cuda.synchronize()
    cev = []
    for _ in range(eks):
        for (k, v, qq), (ept, ecl, eel, eqo, eloc), eo in zip(per_batch, eargs, eouts):
            flush()
            mk.minisgl_store_kv(epool, 0, k, v, eloc)
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            mk.minisgl_cascade_extend_attn(epool, 0, qq, ept, ecl, eel, eqo, P, ecase.sm_scale, out=eo,
                                           workspace=cws)
            b_.record(stream)
            cev.append((a, b_))
    torch.cuda.synchronize()
    c_ms = sum(a.elapsed_time(b_) for a, b_ in cev) / eks
    ext["cascade_extend"] = {
        "call": "minisgl_cascade_extend_attn (prefix pass of all new tokens over the shared rows, "
                "then each request's own rows with the prefix partial folded in)",
        "shared_len": P, "value": round(fl / (c_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
        "ms_per_pass": round(c_ms, 4), "relative_to_extend": round(ext_ms_per_pass / c_ms, 4),
        "faster": "cascade extend" if c_ms < ext_ms_per_pass else "extend",
        "l2": "flushed (256 MB write) before each batch's store_kv + timed call"}
    del cws
    # fused RoPE + store_kv over the same batches (the step before attention)
    max_pos = max(int((b.cached_lens + b.extend_lens).max()) for b in ecase.batches)
    table = workloads.rope_cos_sin_cache(ecase.head_dim, max_pos).to(dev)
    epos = [workloads.extend_positions(b).to(dev) for b in ecase.batches]
    rq = [qq.clone() for _, _, qq in per_batch]

    def rstep():
        for (k, v, _), qq, pp, (_, _, _, _, eloc) in zip(per_batch, rq, epos, eargs):
            mk.minisgl_rope_store_kv(epool, 0, qq, k, v, pp, table, eloc)

    for _ in range(args.warmup):
        rstep()
    r_ms = ev_time(rstep, eks, stream)
    r_bytes = rope_store_bytes(ecase)
    rope = {"workload": ecase.name + " (all batches)", "ms_per_pass": round(r_ms, 4),
            "tokens": int(sum(ecase.extend_lens)),
            "achieved_gbs": round(r_bytes / (r_ms * 1e-3) / 1e9, 1),
            "frac_of_hbm": round(r_bytes / (r_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "algorithmic_bytes_per_pass": r_bytes,
            "l2": "inputs larger than L2 (%.0f MB per pass)" % (r_bytes / 1e6)}
    del epool_t, per_batch, rq, eouts
    torch.cuda.empty_cache()
    return ext, rope


def bench_mixed(mk, args, dev, stream, flush):
    """A mixed batch (chunked prefill + 64 decode requests): one extend
    launch over all requests against extend over the chunk requests followed
    by store_decode_attn over the decode requests."""
    mc = workloads.mixed_chunk_decode()
    mb = mc.batches[0]
    mpool_t, mper = workloads.make_extend_values(mc, dev)
    mpool = mk.KVPool(mpool_t)
    mk_, mv_, mq_ = mper[0]
    nd = mc.num_decode
    nb = len(mb.req_ids) - nd
    Tc = int(mb.q_offsets[nb])
    m_pt, m_cl, m_el, m_qo, m_loc = (mb.page_table.to(dev), mb.cached_lens.to(dev), mb.extend_lens.to(dev),
                                     mb.q_offsets.to(dev), mb.out_loc.to(dev))
    mout = torch.empty_like(mq_)
    c_pt, c_cl, c_el, c_qo = m_pt[:nb], m_cl[:nb], m_el[:nb], m_qo[:nb + 1]
    d_pt, d_sl, d_loc = m_pt[nb:], (m_cl[nb:] + 1).contiguous(), m_loc[Tc:]
    dws = mk.decode_workspace(nd, mc.num_q_heads, mpool)

    def mixed_one():
        mk.minisgl_store_kv(mpool, 0, mk_, mv_, m_loc)
        mk.minisgl_extend_attn(mpool, 0, mq_, m_pt, m_cl, m_el, m_qo, mc.sm_scale, out=mout)

    def mixed_split():
        mk.minisgl_store_kv(mpool, 0, mk_[:Tc], mv_[:Tc], m_loc[:Tc])
        mk.minisgl_extend_attn(mpool, 0, mq_[:Tc], c_pt, c_cl, c_el, c_qo, mc.sm_scale, out=mout[:Tc])
        mk.minisgl_store_decode_attn(mpool, 0, mk_[Tc:], mv_[Tc:], d_loc, mq_[Tc:], d_pt, d_sl,
                                     mc.sm_scale, out=mout[Tc:], workspace=dws)

    for fn in (mixed_one, mixed_split):
        for _ in range(args.warmup):
            fn()
    reps = max(5, args.steps // 10)
    m1 = ev_time(mixed_one, reps, stream, before=flush)
    m2 = ev_time(mixed_split, reps, stream, before=flush)
    res = {"workload": mc.name, "chunk_tokens": Tc, "decode_requests": nd,
           "ms_one_extend_launch": round(m1, 4), "ms_extend_then_store_decode": round(m2, 4),
           "faster": "one extend launch" if m1 < m2 else "extend + store_decode_attn",
           "calls_one": "store_kv + extend_attn over all requests",
           "calls_split": "store_kv + extend_attn over the chunk requests, then store_decode_attn "
                          "over the decode requests",
           "l2": "flushed (256 MB write) before every timed pass"}
    del mpool_t, mper, mout
    torch.cuda.empty_cache()
    return res


def bench_cascade(mk, args, dev, stream, peaks, flush):
    """Shared-prefix (cascade) decode against plain decode on radix-shared
    batches with a 4096-, a 1024- and a 256-token prefix."""
    casc = []
    for sc in (workloads.decode_shared_prefix_qwen3(),
               workloads.decode_shared_prefix_qwen3(prefix_len=1024),
               workloads.decode_shared_prefix_qwen3(prefix_len=256)):
        spool_t, sk, sv, sq = workloads.make_decode_values(sc, dev)
        spool = mk.KVPool(spool_t)
        spt, ssl, sloc = sc.page_table.to(dev), sc.seq_lens.to(dev), sc.out_loc.to(dev)
        mk.minisgl_store_kv(spool, 0, sk[0], sv[0], sloc)
        sout = torch.empty_like(sq[0])
        runs = {
            "cascade": lambda: mk.minisgl_cascade_decode_attn(spool, 0, sq[0], spt, ssl, sc.shared_len,
                                                              sc.sm_scale, out=sout),
            "plain": lambda: mk.minisgl_decode_attn(spool, 0, sq[0], spt, ssl, sc.sm_scale, out=sout),
        }
        t_ms = {}
        for nm, fn in runs.items():
            for _ in range(args.warmup):
                fn()
            t_ms[nm] = ev_time(fn, max(10, args.steps // 10), stream, before=flush)
        plain_b = decode_layer_bytes(sc)
        casc_b = cascade_layer_bytes(sc)
        casc.append({"workload": sc.name, "shared_len": sc.shared_len,
                     "ms_cascade": round(t_ms["cascade"], 5),
                     "ms_plain_decode": round(t_ms["plain"], 5),
                     "speedup": round(t_ms["plain"] / t_ms["cascade"], 3),
                     "algorithmic_bytes_cascade": casc_b, "algorithmic_bytes_plain": plain_b,
                     "achieved_gbs_cascade": round(casc_b / (t_ms["cascade"] * 1e-3) / 1e9, 1),
                     "frac_of_hbm_cascade": round(casc_b / (t_ms["cascade"] * 1e-3) / 1e9
                                                  / peaks["hbm_gbs"], 4),
                     "l2": "flushed (256 MB write) before every timed call"})
        del spool_t, sk, sv, sq
        torch.cuda.empty_cache()
    return casc


PARTS = ("qwen3_step", "long_page64", "tiny", "store_kv", "extend", "mixed", "cascade")


def secondary_objects(mk, args, dev, stream, peaks, st_ms=None, B=None, st_b=None, parts=PARTS):
    extras = {}
    flush_buf = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
    flush = flush_buf.zero_
    if "qwen3_step" in parts:
        extras["qwen3_0p6b_step"] = secondary_decode_step(mk, args, dev, stream, peaks,
                                                          workloads.decode_qwen3_0p6b())
    if "long_page64" in parts:
        extras["long_page64_layer"] = secondary_decode_step(mk, args, dev, stream, peaks,
                                                            workloads.decode_long_page64())
    if "tiny" in parts:
        extras["tiny_decode_latency"] = bench_tiny(mk, args, dev, stream)
    if "store_kv" in parts:
        extras["store_kv"] = bench_store_kv_at_scale(mk, args, dev, stream, peaks)
        if st_ms is not None:
            extras["store_kv"]["headline_layer_store"] = {
                "tokens": B, "ms_per_launch": round(st_ms, 5),
                "achieved_gbs": round(st_b / (st_ms * 1e-3) / 1e9, 1),
                "note": "one row per request: launch-latency bound"}
    if "extend" in parts:
        extras["extend"], extras["rope_store_kv"] = bench_extend(mk, args, dev, stream, peaks, flush)
    if "mixed" in parts:
        extras["mixed_batch"] = bench_mixed(mk, args, dev, stream, flush)
    if "cascade" in parts:
        extras["cascade_decode"] = bench_cascade(mk, args, dev, stream, peaks, flush)
    del flush_buf
    torch.cuda.empty_cache()
    return extras


def run_part(args):
    """One secondary object alone (for profiler captures on a small footprint)."""
    import paged_kv_cache_row_gb300 as mk
    from paged_kv_cache_row_gb300 import build as mkbuild
    mkbuild.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    out = secondary_objects(mk, args, dev, torch.cuda.current_stream(), measured_peaks(),
                            parts=(args.part,))
    print(json.dumps({"part": args.part, **out}), flush=True)



def run_gpu(args, world, rank, local):
    import paged_kv_cache_row_gb300 as mk
    from paged_kv_cache_row_gb300 import build as mkbuild
    if rank == 0:
        mkbuild.build()
    barrier(world)
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = measured_peaks()
    stream = torch.cuda.current_stream()

    # ================= headline: Llama-3-8B decode step, 32 layers ================= #
    case = headline_case(args.layers)
    L, B, Hq, Hkv, d = case.num_layers, case.batch, case.num_q_heads, case.num_kv_heads, case.head_dim
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, dev)
    pool = mk.KVPool(pool_t, case.page_size)
    pt, sl, loc = case.page_table.to(dev), case.seq_lens.to(dev), case.out_loc.to(dev)
    ws = mk.decode_workspace(B, Hq, pool)
    outs = torch.empty((L, B, Hq, d), dtype=torch.bfloat16, device=dev)
    step = decode_step_fn(mk, case, pool, k_new, v_new, q, pt, sl, loc, outs, ws, fused=True)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- timed region: exactly K steps ----
    clocks = ClockSampler(dev.index) if rank == 0 else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop() if clocks else None
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)

    dec_b = decode_layer_bytes(case)
    st_b = store_layer_bytes(case)
    step_bytes = L * (dec_b + st_b)
    value = job_rate(step_bytes, world, ms) / 1e9
    tokens_s = job_rate(case.num_real, world, ms)

    # ---- the same step as two calls per layer: store_kv, then decode_attn ----
    two_step = decode_step_fn(mk, case, pool, k_new, v_new, q, pt, sl, loc, outs, ws, fused=False)
    fms = time_steps(two_step, args.steps, args.warmup, stream, world)

    # ---- programmatic dependent launch off, then on again (same process, same order) ----
    pdl_ab = None
    if not args.no_extend:
        ab_steps = max(5, args.steps // 2)
        mk.minisgl_debug_set_pdl(False)
        ms_off = time_steps(step, ab_steps, args.warmup, stream, world)
        mk.minisgl_debug_set_pdl(True)
        ms_on = time_steps(step, ab_steps, args.warmup, stream, world)
        pdl_ab = {"workload": case.name, "steps": ab_steps,
                  "ms_per_step_pdl_off": round(ms_off, 4), "ms_per_step_pdl_on": round(ms_on, 4),
                  "ms_per_step_pdl_on_timed_region": round(ms, 4),
                  "gain": round(ms_off / ms_on - 1.0, 4),
                  "switch": "minisgl_debug_set_pdl (launch attribute on/off, same library)"}

    # ---- per-call durations of the dominant call, CUDA events on the launch stream ----
    n_rep = max(3, min(args.steps, 20))
    ev = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(n_rep * L)]
    i = 0
    for _ in range(n_rep):
        for l in range(L):
            a, b_, c, d_ = ev[i]
            a.record(stream)
            mk.minisgl_store_kv(pool, l, k_new[l], v_new[l], loc)
            b_.record(stream)
            mk.minisgl_decode_attn(pool, l, q[l], pt, sl, case.sm_scale, out=outs[l], workspace=ws)
            c.record(stream)
            mk.minisgl_store_decode_attn(pool, l, k_new[l], v_new[l], loc, q[l], pt, sl, case.sm_scale,
                                         out=outs[l], workspace=ws)
            d_.record(stream)
            i += 1
    torch.cuda.synchronize()
    dec_ms = statistics.mean(b_.elapsed_time(c) for _, b_, c, _ in ev)
    st_ms = statistics.mean(a.elapsed_time(b_) for a, b_, _, _ in ev)
    fused_ms = statistics.mean(c.elapsed_time(d_) for _, _, c, d_ in ev)
    # the call's average duration over the timed region (steps x layers calls,
    # each the partial kernel with the fused store plus the merge kernel)
    call_ms = ms / L
    achieved = (dec_b + st_b) / (call_ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    traffic = profile_traffic("decode.cu", "decode_llama3_8b.md")

    # ---- e2e: the same step through the C ABI with host buffers ----
    pin = lambda t: t.cpu().pin_memory()
    h_in = [pin(k_new), pin(v_new), pin(q), pin(case.page_table), pin(case.seq_lens), pin(case.out_loc)]
    d_in = [torch.empty_like(t, device=dev) for t in h_in]
    h_out = torch.empty(outs.shape, dtype=outs.dtype).pin_memory()
    bi = sum(t.numel() * t.element_size() for t in h_in)
    bo = h_out.numel() * h_out.element_size()

    # Copies run on their own streams so they overlap the layers: the page
    # table, seq_lens and out_loc go first, then each layer's k, v and q, and
    # each layer's output comes back as soon as that layer is done.  The
    # compute stream waits for the inputs only before layers 0, 1, 2, 4, 8,
    # 16, ..., each time for those of the layers up to about twice as far
    # (an event wait between two calls ends the programmatic launch overlap
    # of the second with the first, and the copies run far ahead of the
    # layers).  The compute stream waits for the last output copy, so the
    # timed region holds all of them.
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    meta_ev = torch.cuda.Event()
    in_ev = [torch.cuda.Event() for _ in range(L)]
    out_ev = [torch.cuda.Event() for _ in range(L)]
    in_wait = input_wait_schedule(L)

    def e2e_step():
        h2d.wait_stream(stream)  # the previous step is done with the device inputs
        with torch.cuda.stream(h2d):
            for i in (3, 4, 5):
                d_in[i].copy_(h_in[i], non_blocking=True)
            meta_ev.record(h2d)
            for l in range(L):
                for i in (0, 1, 2):
                    d_in[i][l].copy_(h_in[i][l], non_blocking=True)
                in_ev[l].record(h2d)
        stream.wait_event(meta_ev)
        for l in range(L):
            if l in in_wait:
                stream.wait_event(in_ev[in_wait[l]])
            mk.minisgl_store_decode_attn(pool, l, d_in[0][l], d_in[1][l], d_in[5], d_in[2][l], d_in[3],
                                         d_in[4], case.sm_scale, out=outs[l], workspace=ws)
            out_ev[l].record(stream)
        with torch.cuda.stream(d2h):
            for l in range(L):
                d2h.wait_event(out_ev[l])
                h_out[l].copy_(outs[l], non_blocking=True)
        stream.wait_stream(d2h)

    e2e_ms = time_steps(e2e_step, max(3, args.steps // 4), 2, stream, world)
    e2e_value = job_rate(step_bytes, world, e2e_ms) / 1e9

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        reqs = list(range(0, case.num_real, 25))
        lay = sorted({0, L - 1})  # the first and the last layer
        run, nbytes = oracle_decode_sample(case, pool_t, k_new, v_new, q, lay, reqs)
        t0 = time.perf_counter()
        n = 0
        while True:
            run()
            n += 1
            if time.perf_counter() - t0 > 10.0 or n >= 200:
                break
        dt = time.perf_counter() - t0
        cpu = {"value": round(nbytes * n / dt / 1e9, 4), "unit": "GB/s", "cores": cpu_cores_used(),
               "kind": "oracle", "cpu_model": cpu_model(),
               "host_cores_available": len(os.sched_getaffinity(0)),
               "sample": f"store_kv + decode of requests {reqs} (of {case.num_real} real) on layers "
                         f"{lay} (every layer has the same lengths, so the rate holds for all {L}), "
                         f"repeated {n}x, {dt:.1f} s, single-threaded fp64 C"}
        ac_v, ac_threads, ac_sample = oracle_all_cores(case, pool_t, k_new, v_new, q)
        cpu["all_cores"] = {"value": round(ac_v, 4), "unit": "GB/s", "cores": ac_threads,
                            "kind": "oracle", "sample": ac_sample}

    head_cfg = {"workload": case.name, "layers": L, "batch": B, "real_requests": case.num_real,
                "H_q": Hq, "H_kv": Hkv, "head_dim": d, "page_size": case.page_size,
                "context_tokens": int(case.seq_lens[:case.num_real].sum()),
                "pool_rows_per_layer": case.num_rows, "pool_factor": case.pool_factor,
                "pool_gb": round(workloads.decode_pool_bytes(case) / 1e9, 1),
                "l2": "inputs larger than L2: each layer reads %.2f GB of K/V, a step %.1f GB"
                      % (dec_b / 1e9, step_bytes / 1e9),
                "parallelism": f"dp{world} (independent batches per GPU)"}
    del pool_t, k_new, v_new, q, outs, h_in, d_in, h_out, ws
    torch.cuda.empty_cache()

    # ================= secondary objects (not part of the headline) ================= #
    extras = {} if args.no_extend else secondary_objects(mk, args, dev, stream, peaks, st_ms, B, st_b)

    gpu_launches = args.steps * L * 2  # per layer: decode partial (with the store) + LSE merge
    line = {
        "metric": "paged decode-attn HBM GB/s (algorithmic bytes, store_kv + decode per layer) "
                  "& tokens/s",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_per_s": round(tokens_s, 1),
        "config": head_cfg,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "store_decode_attn call (split-KV partial kernel with the fused "
                               "store, then the LSE merge kernel), one layer",
                     "algorithmic_bytes_per_launch": dec_b + st_b, "ms_per_launch": round(call_ms, 5),
                     "ms_per_launch_how": "timed region / (steps x layers): the call's average duration "
                                          "inside the step, CUDA events on the launch stream",
                     "isolated_call": {"ms": round(fused_ms, 5),
                                       "achieved_gbs": round((dec_b + st_b) / (fused_ms * 1e-3) / 1e9, 1),
                                       "how": "each call bracketed by its own events (launch latency "
                                              "not hidden by the previous call)"},
                     "decode_attn_call_alone": {"ms": round(dec_ms, 5),
                                                "achieved_gbs": round(dec_b / (dec_ms * 1e-3) / 1e9, 1)},
                     "step_frac": round(value / world / peak, 4),
                     "peak_source": peaks["source"] + " hbm copy"},
        "two_call_step": {"ms_per_step": round(fms, 4),
                          "value": round(job_rate(step_bytes, world, fms) / 1e9, 2), "unit": "GB/s",
                          "frac_of_hbm": round(job_rate(step_bytes, world, fms) / 1e9 / world / peak, 4)},
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "ms_per_step": round(e2e_ms, 4),
                "tokens_per_s": round(job_rate(case.num_real, world, e2e_ms), 1),
                "copies": "pinned host buffers; per-layer H2D and D2H on two copy streams, "
                          "overlapped with the layers, inside the timed region"},
        "gpu_launches": gpu_launches,
        "pdl_ab": pdl_ab,
        "cpu_baseline": cpu,
    }
    line.update(extras)
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# reference arm: the oracle on the host cores
# --------------------------------------------------------------------------- #
def run_reference(args, world, rank):
    if rank != 0:
        return
    case = workloads.decode_llama3_8b(num_layers=1)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, dev)
    reqs = [0, 67, 134]
    run, nbytes = oracle_decode_sample(case, pool_t, k_new, v_new, q, [0], reqs)
    del pool_t
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    sample = (f"each step: store_kv + decode of requests {reqs} of the {case.name} batch on "
              f"layer 0 ({nbytes / 1e6:.1f} MB algorithmic), single-threaded fp64 C oracle")
    line = {
        "impl": "reference",
        "metric": "paged decode-attn HBM GB/s (algorithmic bytes, store_kv + decode per layer) "
                  "& tokens/s",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": case.name, "layers": 32, "batch": case.batch,
                   "real_requests": case.num_real, "sample_requests": reqs,
                   "parallelism": "single CPU thread"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_cores_used(),
                         "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--layers", type=int, default=32,
                    help="layers of the headline decode workload (32 = the full model; fewer only "
                         "for profiler captures that must stay small)")
    ap.add_argument("--no-extend", action="store_true",
                    help="time the headline decode step only (no secondary workloads)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--part", choices=PARTS, default=None,
                    help="run one secondary object alone and print it (profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    if args.part:
        run_part(args)
        return
    world, rank, local = dist_setup(args.gpus)
    run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
