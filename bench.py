#!/usr/bin/env python3
"""Benchmark of the paged KV-pool attention hot path on GB300.

A step is one decode step of the Qwen3-0.6B-shaped workload (28 layers,
batch 64, H_q 16, H_kv 8, head_dim 128, page_size 1, contexts U[512,4096]):
per layer, store_kv of the 64 new tokens and split-KV decode attention, in
one minisgl_store_decode_attn call (partial kernel, which also stores the new
rows, + LSE merge kernel); the same step as two calls (minisgl_store_kv, then
minisgl_decode_attn) is reported beside it.  The metric is paged decode-attention
HBM GB/s (algorithmic bytes / time) with tokens/s beside it; the extend
(chunked-prefill) kernel is measured on the radix-shared extend workload in
TFLOP/s as a second object.

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
def run_gpu(args, world, rank, local):
    import paged_kv_cache_row_gb300 as mk
    from paged_kv_cache_row_gb300 import build as mkbuild
    if rank == 0:
        mkbuild.build()
    barrier(world)
    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = measured_peaks()

    case = workloads.decode_qwen3_0p6b(num_layers=args.layers)
    L, B, Hq, Hkv, d = case.num_layers, case.batch, case.num_q_heads, case.num_kv_heads, case.head_dim
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, dev)
    pool = mk.KVPool(pool_t, case.page_size)
    pt, sl, loc = case.page_table.to(dev), case.seq_lens.to(dev), case.out_loc.to(dev)
    ws = mk.decode_workspace(B, Hq, pool)
    outs = torch.empty((L, B, Hq, d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def step(kk=k_new, vv=v_new, qq=q, ptab=pt, seq=sl, oloc=loc):
        # per layer: store_kv of the 64 new rows fused into split-KV decode + LSE merge
        for l in range(L):
            mk.minisgl_store_decode_attn(pool, l, kk[l], vv[l], oloc, qq[l], ptab, seq, case.sm_scale,
                                         out=outs[l], workspace=ws)

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
    ms_local = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms_local, world)

    dec_b = decode_layer_bytes(case)
    st_b = store_layer_bytes(case)
    step_bytes = L * (dec_b + st_b)
    value = job_rate(step_bytes, world, ms) / 1e9
    tokens_s = job_rate(case.num_real, world, ms)

    # ---- the same step as two calls per layer: store_kv, then decode_attn ----
    def fstep():
        for l in range(L):
            mk.minisgl_store_kv(pool, l, k_new[l], v_new[l], loc)
            mk.minisgl_decode_attn(pool, l, q[l], pt, sl, case.sm_scale, out=outs[l], workspace=ws)

    for _ in range(args.warmup):
        fstep()
    torch.cuda.synchronize()
    barrier(world)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        fstep()
    g1.record(stream)
    torch.cuda.synchronize()
    fms = max_over_ranks(g0.elapsed_time(g1) / args.steps, world)

    # ---- per-call durations of the dominant call, CUDA events on the launch stream ----
    n_rep = max(3, min(args.steps, 50))
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
    achieved = (dec_b + st_b) / (fused_ms * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    traffic = profile_traffic("decode.cu", "decode_qwen3_0p6b.md")

    # ---- the other decode workloads, one layer each: per-call GB/s and tokens/s ----
    others = None
    if not args.no_extend:
        others = []
        for oc in (workloads.decode_llama3_8b(num_layers=1), workloads.decode_long_page64()):
            opool_t, ok_, ov_, oq = workloads.make_decode_values(oc, dev)
            opool = mk.KVPool(opool_t, oc.page_size)
            opt, osl, oloc = oc.page_table.to(dev), oc.seq_lens.to(dev), oc.out_loc.to(dev)
            ows = mk.decode_workspace(oc.batch, oc.num_q_heads, opool)
            oout = torch.empty_like(oq[0])

            def ostep_fused():
                mk.minisgl_store_decode_attn(opool, 0, ok_[0], ov_[0], oloc, oq[0], opt, osl, oc.sm_scale,
                                             out=oout, workspace=ows)

            def ostep_two():
                mk.minisgl_store_kv(opool, 0, ok_[0], ov_[0], oloc)
                mk.minisgl_decode_attn(opool, 0, oq[0], opt, osl, oc.sm_scale, out=oout, workspace=ows)

            def otime(fn):
                for _ in range(args.warmup):
                    fn()
                torch.cuda.synchronize()
                oev = []
                for _ in range(max(10, args.steps // 10)):
                    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    fn()
                    b_.record(stream)
                    oev.append((a, b_))
                torch.cuda.synchronize()
                return statistics.mean(a.elapsed_time(b_) for a, b_ in oev)

            oms = otime(ostep_fused)
            oms_two = otime(ostep_two)
            ob = decode_layer_bytes(oc) + store_layer_bytes(oc)
            others.append({"workload": oc.name, "batch": oc.batch, "real_requests": oc.num_real,
                           "H_q": oc.num_q_heads, "H_kv": oc.num_kv_heads, "page_size": oc.page_size,
                           "context_tokens": int(oc.seq_lens[:oc.num_real].sum()),
                           "call": "minisgl_store_decode_attn",
                           "ms_per_layer": round(oms, 5),
                           "two_call_ms_per_layer": round(oms_two, 5),
                           "achieved_gbs": round(ob / (oms * 1e-3) / 1e9, 1),
                           "frac_of_hbm": round(ob / (oms * 1e-3) / 1e9 / peak, 4),
                           "tokens_per_s_per_layer": round(oc.num_real / (oms * 1e-3), 1),
                           "l2": "inputs larger than L2 (%.1f GB of K/V per call)" % (ob / 1e9)})
            del opool_t, ok_, ov_, oq

    # ---- shared-prefix (cascade) decode vs plain decode on one radix-shared batch ----
    casc = None
    if not args.no_extend:
        sc = workloads.decode_shared_prefix_qwen3()
        spool_t, sk, sv, sq = workloads.make_decode_values(sc, dev)
        spool = mk.KVPool(spool_t)
        spt, ssl, sloc = sc.page_table.to(dev), sc.seq_lens.to(dev), sc.out_loc.to(dev)
        mk.minisgl_store_kv(spool, 0, sk[0], sv[0], sloc)
        sout = torch.empty_like(sq[0])
        flush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
        runs = {
            "cascade": lambda: mk.minisgl_cascade_decode_attn(spool, 0, sq[0], spt, ssl, sc.shared_len,
                                                              sc.sm_scale, out=sout),
            "plain": lambda: mk.minisgl_decode_attn(spool, 0, sq[0], spt, ssl, sc.sm_scale, out=sout),
        }
        t_ms = {}
        for nm, fn in runs.items():
            for _ in range(args.warmup):
                fn()
            torch.cuda.synchronize()
            evs = []
            for _ in range(max(10, args.steps // 10)):
                flush.zero_()  # the 4096-row prefix (33 MB) would otherwise stay in L2
                a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b_.record(stream)
                evs.append((a, b_))
            torch.cuda.synchronize()
            t_ms[nm] = statistics.mean(a.elapsed_time(b_) for a, b_ in evs)
        plain_b = decode_layer_bytes(sc)
        casc_b = cascade_layer_bytes(sc)
        casc = {"workload": sc.name, "ms_cascade": round(t_ms["cascade"], 5),
                "ms_plain_decode": round(t_ms["plain"], 5),
                "speedup": round(t_ms["plain"] / t_ms["cascade"], 3),
                "algorithmic_bytes_cascade": casc_b, "algorithmic_bytes_plain": plain_b,
                "achieved_gbs_cascade": round(casc_b / (t_ms["cascade"] * 1e-3) / 1e9, 1),
                "l2": "flushed (256 MB write) before every timed call"}
        del spool_t, sk, sv, sq, flush

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
    # compute stream waits for the last copy, so the timed region holds all of
    # them.
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    meta_ev = torch.cuda.Event()
    in_ev = [torch.cuda.Event() for _ in range(L)]
    out_ev = [torch.cuda.Event() for _ in range(L)]

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
            stream.wait_event(in_ev[l])
            mk.minisgl_store_decode_attn(pool, l, d_in[0][l], d_in[1][l], d_in[5], d_in[2][l], d_in[3],
                                         d_in[4], case.sm_scale, out=outs[l], workspace=ws)
            out_ev[l].record(stream)
        with torch.cuda.stream(d2h):
            for l in range(L):
                d2h.wait_event(out_ev[l])
                h_out[l].copy_(outs[l], non_blocking=True)
        stream.wait_stream(d2h)

    e2e_steps = max(3, args.steps // 4)
    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1) / e2e_steps, world)
    e2e_value = job_rate(step_bytes, world, e2e_ms) / 1e9

    # ---- extend: radix-shared chunked prefill, store_kv + extend per batch ----
    ext = None
    rope = None
    if not args.no_extend:
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
        eflush = torch.empty(256 * 2 ** 20, dtype=torch.uint8, device=dev)
        for _ in range(eks):
            for (k, v, qq), (ept, ecl, eel, eqo, eloc), eo in zip(per_batch, eargs, eouts):
                eflush.zero_()  # q, out and the batch's rows (~170 MB) would partly stay in L2
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
            "l2": "flushed (256 MB write) before each batch's store_kv + timed extend call",
            "roofline": {"bound": "tensor", "achieved": round(launch_fl / (launch_ms * 1e-3) / 1e12, 2),
                         "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": round(launch_fl / (launch_ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
                         "traffic": profile_traffic("extend.cu", "extend_radix_shared.md"),
                         "peak_source": peaks["source"] + " bf16 dense burst"},
        }
        # ---- fused RoPE + store_kv over the same batches (the step before attention) ----
        max_pos = max(int((b.cached_lens + b.extend_lens).max()) for b in ecase.batches)
        table = workloads.rope_cos_sin_cache(ecase.head_dim, max_pos).to(dev)
        epos = [workloads.extend_positions(b).to(dev) for b in ecase.batches]
        rq = [qq.clone() for _, _, qq in per_batch]

        def rstep():
            for (k, v, _), qq, pp, (_, _, _, _, eloc) in zip(per_batch, rq, epos, eargs):
                mk.minisgl_rope_store_kv(epool, 0, qq, k, v, pp, table, eloc)

        for _ in range(args.warmup):
            rstep()
        torch.cuda.synchronize()
        rev = []
        for _ in range(eks):
            a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            rstep()
            b_.record(stream)
            rev.append((a, b_))
        torch.cuda.synchronize()
        r_ms = statistics.mean(a.elapsed_time(b_) for a, b_ in rev)
        r_bytes = rope_store_bytes(ecase)
        rope = {"workload": ecase.name + " (all batches)", "ms_per_pass": round(r_ms, 4),
                "tokens": int(sum(ecase.extend_lens)),
                "achieved_gbs": round(r_bytes / (r_ms * 1e-3) / 1e9, 1),
                "frac_of_hbm": round(r_bytes / (r_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                "algorithmic_bytes_per_pass": r_bytes,
                "l2": "inputs larger than L2 (%.0f MB per pass)" % (r_bytes / 1e6)}
        del epool_t, per_batch, rq, eflush

    # ---- CPU baseline: the oracle on a bounded sample (rank 0, N = 1) ----
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        reqs = list(range(0, B, 8))
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
               "kind": "oracle",
               "sample": f"store_kv + decode of requests {reqs} (of {B}) on layers {lay} "
                         f"(every layer has the same lengths, so the rate holds for all {L}), "
                         f"repeated {n}x, {dt:.1f} s, single-threaded fp64 C"}
        ac_v, ac_threads, ac_sample = oracle_all_cores(case, pool_t, k_new, v_new, q)
        cpu["all_cores"] = {"value": round(ac_v, 4), "unit": "GB/s", "cores": ac_threads,
                            "kind": "oracle", "sample": ac_sample}

    gpu_launches = args.steps * L * 2  # per layer: decode partial (with the store) + LSE merge
    line = {
        "metric": "paged decode-attn HBM GB/s (algorithmic bytes, store_kv + decode per layer)",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "tokens_per_s": round(tokens_s, 1),
        "config": {"workload": case.name, "layers": L, "batch": B, "H_q": Hq, "H_kv": Hkv,
                   "head_dim": d, "page_size": case.page_size,
                   "context_tokens": int(case.seq_lens.sum()),
                   "l2": "inputs larger than L2: each layer reads %.0f MB of K/V, a step %.1f GB"
                         % (dec_b / 1e6, step_bytes / 1e9),
                   "parallelism": f"dp{world} (independent batches per GPU)"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "store_decode_attn call (split-KV partial kernel with the fused "
                               "store, then the LSE merge kernel)",
                     "algorithmic_bytes_per_launch": dec_b + st_b, "ms_per_launch": round(fused_ms, 5),
                     "decode_attn_call_alone": {"ms": round(dec_ms, 5),
                                                "achieved_gbs": round(dec_b / (dec_ms * 1e-3) / 1e9, 1)},
                     "peak_source": peaks["source"] + " hbm copy"},
        "two_call_step": {"ms_per_step": round(fms, 4),
                                    "value": round(job_rate(step_bytes, world, fms) / 1e9, 2),
                                    "unit": "GB/s",
                                    "frac_of_hbm": round(job_rate(step_bytes, world, fms) / 1e9 / peak, 4)},
        "store_kv": {"ms_per_launch": round(st_ms, 5),
                     "achieved_gbs": round(st_b / (st_ms * 1e-3) / 1e9, 1)},
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": bi,
                "d2h_bytes_per_step": bo, "ms_per_step": round(e2e_ms, 4),
                "copies": "pinned host buffers; per-layer H2D and D2H on two copy streams, "
                          "overlapped with the layers, inside the timed region"},
        "gpu_launches": gpu_launches,
        "extend": ext,
        "rope_store_kv": rope,
        "cascade_decode": casc,
        "decode_other_workloads": others,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- #
# reference arm: the oracle on the host cores
# --------------------------------------------------------------------------- #
def run_reference(args, world, rank):
    if rank != 0:
        return
    case = workloads.decode_qwen3_0p6b()
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    pool_t, k_new, v_new, q = workloads.make_decode_values(case, dev)
    reqs = [0, 21, 42]
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
        "metric": "paged decode-attn HBM GB/s (algorithmic bytes, store_kv + decode per layer)",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": case.name, "layers": case.num_layers, "batch": case.batch,
                   "sample_requests": reqs, "parallelism": "single CPU thread"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cpu_cores_used(),
                         "kind": "oracle", "sample": sample},
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
    ap.add_argument("--layers", type=int, default=28,
                    help="layers of the decode workload (28 = the full model; fewer only for "
                         "profiler captures that must stay small)")
    ap.add_argument("--no-extend", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        run_reference(args, world, rank)
        return
    world, rank, local = dist_setup(args.gpus)
    run_gpu(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
