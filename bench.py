"""Benchmark: OTT decode-step attention on one GB300 (or N, one process each).

A step is one pass of the whole hot path for one new token of every sequence:
ott_append (the token enters the fp16 ring; every G tokens the flush packs a
group into 2-bit blocks) followed by ott_decode_attn (split-K attention over
blocks, ring and pool, plus the combine). The default workload is the
Llama-2-7B-shaped layer at batch 32 with a 4096-token prefill, G=128, R=32,
P=32. `value` is decode tokens/s (batch x steps / time); the JSON line also
carries the decode kernel's achieved GB/s against the measured HBM peak.

Multi-GPU (torchrun): every rank runs an independent shard of a larger batch
(weak scaling); no collective touches the data path, only the barrier and
the max-over-ranks of the timing.

    python bench.py [--steps K] [--warmup W] [--workload NAME] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_kv_cache_ott_gb300 import metrics, synth  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
METRIC = "OTT decode-attn GB/s (% of HBM peak) and decode tokens/s at B=32, 4K ctx"
E2E_START = ("caches rebuilt from the same prompts and advanced by the same warm-up steps: the e2e steps take "
             "the device-timed steps' inputs at the same context lengths")
E2E_ZERO_COPY_MAX = 512 * 1024   # step inputs at or above this travel by copy, below it by ott_step_host
DECODE_SRC = os.path.join(ROOT, "bit_kv_cache_ott_gb300", "csrc", "ott_decode.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def shard(w, rank: int, world: int):
    """Weak scaling: rank r runs its own batch of sequences (a different seed)."""
    return w.with_(seed=w.seed + 7919 * rank) if world > 1 else w


def max_over_ranks(x: float, device=None) -> float:
    """The slowest rank's time: every rank contributes, all receive the max."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(B: int, steps: int, world: int, ms: float) -> float:
    """Whole-job throughput: every rank decodes B tokens per step."""
    return B * steps * world / (ms * 1e-3)


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def decode_src_hash() -> str:
    with open(DECODE_SRC, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(workload: str):
    """dram bytes per decode launch from a committed ncu capture, if it was
    taken on the current decode kernel source (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
    except Exception:
        return None
    if t.get("decode_src_sha256_16") != decode_src_hash():
        return None
    return t.get("per_launch_bytes", {}).get(workload)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ oracle arm

def synth_T(w) -> str:
    return f"{w.len_lo}..{w.L}" if w.ragged else f"{w.L}"


def step_bytes(w, Ts) -> int:
    """Algorithmic bytes of one decode call with sequence b at Ts[b] tokens."""
    if w.topk > 0:
        return sum(metrics.topk_bytes(t, 1, w.Hq, w.Hkv, w.d, w.G, w.R, w.P, w.topk) for t in Ts)
    if len(set(Ts)) == 1:
        return metrics.decode_bytes(Ts[0], len(Ts), w.Hq, w.Hkv, w.d, w.G, w.R, w.P)
    return sum(metrics.decode_bytes(t, 1, w.Hq, w.Hkv, w.d, w.G, w.R, w.P) for t in Ts)


def decode_call(c, w, q, out, stream):
    """The workload's decode entry point: full, or Top-K sparse."""
    if w.topk > 0:
        return c.decode_attn_topk(q, w.topk, out, stream=stream)
    return c.decode_attn(q, out, stream)


def oracle_decode(orc, w, q):
    return orc.decode_topk(q, w.topk) if w.topk > 0 else orc.decode(q)


def cold_of(w):
    """The cold-pool capacity of a workload, or None (displaced tokens written back)."""
    return w.cold if w.cold >= 0 else None


def cold_quant_bytes(c) -> int:
    """Cold-pool policy: bytes of a cache's quantized blocks and cold pool as
    the device holds them now (their sizes depend on the data)."""
    bc, nc = c.cold_sizes()
    return sum(metrics.cold_unit_bytes(bc[u], nc[u], c.d) for u in range(len(nc)))


def _oracle_prefill(orc, w, lens):
    K, V = synth.prefill_kv(w)
    if w.ragged:
        orc.prefill_lens(K, V, lens)
    else:
        orc.prefill(K, V)


def oracle_rate(w, steps: int, warmup: int, units_sample: int):
    """The CPU oracle (single thread) on a sample of the workload's units:
    prefill, then `warmup` untimed and `steps` timed decode steps (append +
    decode of every query head of the sampled units). Returns decode tokens/s
    scaled to the full workload, and a description of the sample."""
    from oracle.oracle import OracleCache
    Bs = max(1, min(w.B, units_sample // w.Hkv))
    ws = w.with_(B=Bs)
    orc = OracleCache(ws.B, ws.Hq, ws.Hkv, ws.d, ws.G, ws.R, ws.P, cold=cold_of(ws))
    lens = synth.seq_lens(w)
    _oracle_prefill(orc, ws, lens[:Bs])
    inputs = [synth.step_kvq(ws, s) for s in range(warmup + steps)]
    for s in range(warmup):
        k, v, q = inputs[s]
        orc.append(k, v)
        oracle_decode(orc, ws, q)
    t0 = time.perf_counter()
    for s in range(warmup, warmup + steps):
        k, v, q = inputs[s]
        orc.append(k, v)
        oracle_decode(orc, ws, q)
    dt = time.perf_counter() - t0
    # scaled to the whole workload by algorithmic bytes (= by units when all lengths are equal)
    frac = step_bytes(ws, lens[:Bs]) / step_bytes(w, lens)
    per_step_full = dt / steps / frac
    rate = w.B / (per_step_full * w.layers)   # tokens/s: each token passes every layer
    sample = (f"{Bs} of {w.B} sequences ({Bs * w.Hkv} of {w.B * w.Hkv} (sequence, kv head) units), "
              f"{steps} timed decode steps after {warmup} warm-up, T={synth_T(w)}+; one layer; scaled by bytes")
    return rate, dt, sample


_WORKER_BARRIER = None


def _oracle_worker_init(barrier):
    global _WORKER_BARRIER
    _WORKER_BARRIER = barrier


def _oracle_worker(task):
    """One host process of the all-cores baseline: the oracle on its own
    slice of (sequence, kv head) units, timed after every worker has
    prefilled (so that the timed regions run concurrently)."""
    name, hk, seed, steps, warmup, length = task
    from oracle.oracle import OracleCache
    w = synth.WORKLOADS[name]
    g = w.Hq // w.Hkv
    ws = w.with_(B=1, Hkv=hk, Hq=g * hk, seed=seed)
    orc = OracleCache(1, ws.Hq, ws.Hkv, ws.d, ws.G, ws.R, ws.P, cold=cold_of(ws))
    _oracle_prefill(orc, ws, [length])
    inputs = [synth.step_kvq(ws, s) for s in range(warmup + steps)]
    for s in range(warmup):
        k, v, q = inputs[s]
        orc.append(k, v)
        oracle_decode(orc, ws, q)
    _WORKER_BARRIER.wait()
    t0 = time.perf_counter()
    for s in range(warmup, warmup + steps):
        k, v, q = inputs[s]
        orc.append(k, v)
        oracle_decode(orc, ws, q)
    return time.perf_counter() - t0


def oracle_rate_cores(w, steps: int, warmup: int, units_per_proc: int):
    """The CPU oracle on every host core this process may use: one spawned
    process per core, each on its own units (one sequence, up to
    `units_per_proc` kv heads, its own seed), timed concurrently. Returns
    decode tokens/s scaled to the full workload, the slowest worker's time,
    a description of the sample and the process count."""
    import multiprocessing as mp
    ncore = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    U = w.B * w.Hkv
    hk = max(1, min(w.Hkv, units_per_proc))
    nproc = max(1, min(ncore, (U + hk - 1) // hk))
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(nproc)
    lens = synth.seq_lens(w)
    tasks = [(w.name, hk, w.seed + 7919 * (i + 1), steps, warmup, lens[i % w.B]) for i in range(nproc)]
    with ctx.Pool(nproc, initializer=_oracle_worker_init, initargs=(barrier,)) as pool:
        # a worker that cannot start would stall the barrier: bound the wait
        dts = pool.map_async(_oracle_worker, tasks).get(timeout=900)
    dt = max(dts)
    units = nproc * hk
    # scaled to the whole workload by algorithmic bytes (= by units when all lengths are equal)
    w1 = w.with_(Hkv=hk, Hq=(w.Hq // w.Hkv) * hk)
    sampled = sum(step_bytes(w1, [lens[i % w.B]]) for i in range(nproc))
    per_step_full = dt / steps * step_bytes(w, lens) / sampled
    rate = w.B / (per_step_full * w.layers)
    sample = (f"{nproc} processes x {hk} (sequence, kv head) units ({units} of {U}), {steps} timed decode steps "
              f"after {warmup} warm-up, timed concurrently, T={synth_T(w)}+; one layer; scaled by bytes")
    return rate, dt, sample, nproc


def run_reference(args, w):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    rate, dt, sample, nproc = oracle_rate_cores(w, args.steps, args.warmup, args.oracle_units_per_core)
    # ms_per_step is the measured time of one step of the sampled work (what
    # this run actually did); value is that rate scaled to the whole workload
    # by algorithmic bytes, with the factor stated in `extrapolation`
    sampled_ms = 1e3 * dt / args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sampled_ms,
        "extrapolation": {"sampled_ms_per_step": sampled_ms,
                          "full_workload_ms_per_step": (1e3 * w.B / rate) if rate > 0 else None,
                          "scale_factor": ((1e3 * w.B / rate) / sampled_ms) if rate > 0 and sampled_ms > 0 else None,
                          "basis": "algorithmic bytes of the sampled units against the whole workload; "
                                   "value is decode tokens/s of the whole workload at the sampled rate"},
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)",
        "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "L": w.L,
                   "G": w.G, "R": w.R, "P": w.P, "layers": w.layers},
        "cpu_baseline": {"value": rate, "unit": "tokens/s", "cores": nproc, "kind": "oracle", "sample": sample},
        "e2e": {"value": rate, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

def copy_peak(ott, dev, stream, gib: int = 2, reps: int = 10):
    """HBM bandwidth of a plain streaming copy (the library's ott_hbm_copy),
    measured in this process: `gib` GiB read and as many written per call,
    best of `reps` event-timed calls after 3 warm-up calls."""
    n = gib << 28   # float32 elements
    src = torch.empty(n, dtype=torch.float32, device=dev).fill_(1.0)
    dst = torch.empty_like(src)
    for _ in range(3):
        ott.hbm_copy(dst, src, stream)
    best = None
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        ott.hbm_copy(dst, src, stream)
        b.record(stream)
        b.synchronize()
        t = a.elapsed_time(b)
        best = t if best is None else min(best, t)
    nbytes = 2 * n * 4
    del src, dst
    torch.cuda.empty_cache()
    return {"gbs": nbytes / (best * 1e-3) / 1e9, "bytes_per_call": nbytes, "kernel": "ott_hbm_copy",
            "method": f"{gib} GiB read + {gib} GiB written per call, best of {reps} CUDA-event-timed calls"}


def prefill_launches(w, lens, sm_count: int) -> int:
    """Kernel launches of one layer's prefill, as the library issues them: a
    prompt of two or more groups takes the parallel pass (group keys, pool
    scan, every block at once; with P = 0 the blocks alone), except under the
    cold-pool policy, and in a ragged batch (one pass per sequence) only when
    fewer (sequence, kv head) units flush than the GPU has SMs; otherwise the
    flushes run group by group (one launch per group for all units that have
    it). Then the residual tokens are copied (one launch, or one per sequence
    of a ragged batch)."""
    nfs = [metrics.flush_count(L, w.G, w.R) for L in lens]
    few = w.B * w.Hkv < sm_count

    def par_cost(nu, nf):
        # group keys, pool scan (plus its carry pass when the scan is cut
        # into chunks), every block; with P = 0 the blocks alone
        if w.P == 0:
            return 1
        chunks = max(1, min(32, -(-nf // 32), -(-2 * sm_count // nu)))
        return 3 + (chunks > 1)

    if not w.ragged:
        nf = nfs[0]
        return (par_cost(w.B * w.Hkv, nf) if (nf >= 2 and w.cold < 0) else nf) + 1
    par = [nf >= 2 and w.cold < 0 and few for nf in nfs]
    serial = max([nf for nf, p in zip(nfs, par) if not p], default=0)
    return sum(par_cost(w.Hkv, nf) for nf, p in zip(nfs, par) if p) + serial + len(lens)


def measure_prefill(ott, w, wr, dev, stream, reps: int = 3):
    """One layer's prefill from K, V already on the device: CUDA events on
    the launch stream around ott_prefill (ott_prefill_lens for a ragged
    batch) into a fresh cache, median of `reps` after one warm-up call. The
    inputs (K and V of every prompt token) are larger than L2."""
    lens = synth.seq_lens(wr)
    K, V = synth.prefill_kv(wr, layer=0, device=str(dev))
    times = []
    for r in range(reps + 1):
        pool = None
        if w.paged:
            pool = sum(metrics.flush_count(t, w.G, w.R) for t in lens) * w.Hkv + 1
        c = ott.OTTCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P, max_tokens=w.L + 8, ragged=w.ragged,
                         cold=cold_of(w), pool_blocks=pool)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        if w.ragged:
            c.prefill_lens(K, V, lens, stream)
        else:
            c.prefill(K, V, stream)
        b.record(stream)
        b.synchronize()
        c.check_device()
        if r > 0:
            times.append(a.elapsed_time(b))
        c.close()
    del K, V
    torch.cuda.empty_cache()
    ms = statistics.median(times)
    nbytes = sum(metrics.prefill_bytes_per_unit(L, w.d, w.G, w.R, w.P) for L in lens) * w.Hkv
    return {"ms": ms, "tokens": sum(lens), "tokens_per_s": sum(lens) / (ms * 1e-3),
            "algorithmic_bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "launches": prefill_launches(w, lens, torch.cuda.get_device_properties(dev).multi_processor_count),
            "reps": reps,
            "timing": "CUDA events around the prefill call into a fresh cache, median of "
                      f"{reps} after one warm-up; bytes: every prompt token read once (K and V), "
                      "blocks with token indices, final pool and fp16 residual written"}


def run_ours(args, w):
    import bit_kv_cache_ott_gb300 as ott

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ott.load()

    def barrier():
        if ws > 1:
            torch.distributed.barrier()

    # weak scaling: rank r holds its own shard of B sequences
    wr = shard(w, rank, ws)
    K_steps, W_steps = args.steps, args.warmup
    # e2e: by default the same steps as the timed region, on caches rebuilt
    # from the same prompts (so at the same context lengths)
    E_steps = K_steps if args.e2e_steps < 0 else args.e2e_steps
    total_steps = W_steps + max(K_steps, E_steps) + w.G + 2   # + the flush probe
    lens = synth.seq_lens(wr)

    def build_caches():
        cs = []
        for layer in range(w.layers):
            pool = None
            if w.paged:   # the blocks the run fills, from one pool
                pool = sum(metrics.flush_count(t + total_steps, w.G, w.R) for t in lens) * w.Hkv + 1
            c = ott.OTTCache(w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P, max_tokens=w.L + total_steps, ragged=w.ragged,
                             cold=cold_of(w), pool_blocks=pool)
            K, V = synth.prefill_kv(wr, layer=layer, device=str(dev))
            if w.ragged:
                c.prefill_lens(K, V, lens)
            else:
                c.prefill(K, V)
            del K, V
            cs.append(c)
        torch.cuda.synchronize()
        return cs

    caches = build_caches()

    # step inputs (drawn on the host with the CPU generator, staged on the device)
    n_distinct = min(total_steps, 64)
    host = [synth.step_kvq(wr, s) for s in range(n_distinct)]
    dev_in = [tuple(t.to(dev) for t in x) for x in host]
    stream = torch.cuda.current_stream()
    out = torch.empty(w.B, w.Hq, w.d, dtype=torch.float16, device=dev)

    def step(s):
        k, v, q = dev_in[s % n_distinct]
        for c in caches:
            c.append(k, v, stream)
            decode_call(c, w, q, out, stream)

    def flush_due_next(Ts):
        """Does the next append make some sequence flush?"""
        return any((t + 1 - w.R) % w.G == 0 and t + 1 >= w.G + w.R for t in Ts)

    # caches that fit in about twice the L2 would be read from L2 by repeated
    # calls: a buffer larger than L2 is written between the timed calls, then
    # a second one is read, so that the written lines reach DRAM there and not
    # as write-backs inside the next timed call
    cache_total = caches[0].device_bytes() * w.layers
    l2_flush = cache_total < 2 * L2_BYTES
    l2_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if l2_flush else None
    l2_rd = torch.zeros(64, 2 * L2_BYTES // 256, dtype=torch.float32, device=dev) if l2_flush else None
    l2_sink = torch.empty(64, dtype=torch.float32, device=dev) if l2_flush else None

    def flush_l2(s):
        if l2_buf is not None:
            l2_buf.fill_(float(s))
            torch.sum(l2_rd, dim=1, out=l2_sink)

    for s in range(W_steps):
        step(s)
    torch.cuda.synchronize()

    # the HBM copy peak of this GPU, measured in this run (2 GiB read + 2 GiB written)
    peak_run = None
    if not args.no_copy_peak:
        peak_run = copy_peak(ott, dev, stream)

    # timed region: K whole steps (append, with its flush when one is due,
    # then the decode call), with no event inside the loop; with an L2 flush,
    # each step is bracketed by events and the flush writes fall outside
    Ts = [caches[0].seq_counts(b)[0] for b in range(w.B)]
    T0 = max(Ts)
    cold = w.cold >= 0
    flush_steps = 0
    step_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(K_steps if l2_flush else 0)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        torch.cuda.synchronize()
        e0.record(stream)
        for s in range(K_steps):
            flush_steps += int(flush_due_next(Ts))
            Ts = [t + 1 for t in Ts]
            if l2_flush:
                flush_l2(s)
                step_events[s][0].record(stream)
            step(W_steps + s)
            if l2_flush:
                step_events[s][1].record(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
    ms = sum(a.elapsed_time(b) for a, b in step_events) if l2_flush else e0.elapsed_time(e1)
    flushes = flush_steps * w.layers
    # append + decode + combine (+ the Top-K bounds and pick), plus flushes
    launches = K_steps * w.layers * (5 if w.topk > 0 else 3) + flushes
    ms = max_over_ranks(ms, dev)
    s_next = W_steps + K_steps

    # One flush cycle (G steps) after the timed region:
    #  * the flush: every append is bracketed by its own events, and the
    #    append that flushes is compared with the median plain append. The
    #    flush runs once every G steps for a batch of equal lengths, so K
    #    timed steps rarely hold their share of it; `value` charges it at its
    #    rate, one flush per G steps. A ragged batch flushes its sequences at
    #    different steps, so its timed steps already hold their share.
    #  * the roofline: at 8 points spread over the cycle (the decode call's
    #    bytes fall as the fp16 residual empties at a flush), 8 decode calls
    #    back to back between one pair of events; with an L2 flush between
    #    calls, each call has its own events. Bytes and time are summed over
    #    every timed call.
    n_pts, per_pt = 8, 8
    pt_every = max(1, w.G // n_pts)
    app_ev, app_due, dec_groups = [], [], []
    for i in range(w.G):
        k, v, q = dev_in[s_next % n_distinct]
        due = flush_due_next(Ts)
        Ts = [t + 1 for t in Ts]
        ea = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        ea[0].record(stream)
        for c in caches:
            c.append(k, v, stream)
        ea[1].record(stream)
        app_ev.append(ea)
        app_due.append(due)
        s_next += 1
        if i % pt_every == 0 and len(dec_groups) < n_pts:
            evs = []
            if l2_flush:
                for j in range(per_pt):
                    flush_l2(j)
                    ed = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    ed[0].record(stream)
                    for c in caches:
                        decode_call(c, w, q, out, stream)
                    ed[1].record(stream)
                    evs.append(ed)
            else:
                ed = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                ed[0].record(stream)
                for j in range(per_pt):
                    for c in caches:
                        decode_call(c, w, q, out, stream)
                ed[1].record(stream)
                evs.append(ed)
            call_bytes = (step_bytes(w, list(Ts)) * w.layers if not cold else
                          sum(metrics.hot_bytes(Ts[0], w.B, w.Hq, w.Hkv, w.d, w.G, w.R, w.P) + cold_quant_bytes(c)
                              for c in caches))
            dec_groups.append((evs, call_bytes))
    torch.cuda.synchronize()
    n_dec = n_pts * per_pt
    dec_ms = sum(a_.elapsed_time(b_) for evs, _ in dec_groups for a_, b_ in evs)
    dec_bytes_list = [cb for _, cb in dec_groups for _ in range(per_pt)]
    dec_call_bytes = sum(dec_bytes_list) / n_dec
    flush_us = None
    if not w.ragged:
        adt = [a_.elapsed_time(b_) for a_, b_ in app_ev]
        plain = [t for t, d in zip(adt, app_due) if not d]
        with_flush = [t for t, d in zip(adt, app_due) if d]
        if plain and with_flush:
            flush_us = max(0.0, 1e3 * (statistics.mean(with_flush) - statistics.median(plain)))
    ms_amortized = ms
    if flush_us is not None:
        ms_amortized = ms + (K_steps / w.G - flush_steps) * flush_us * 1e-3

    for c in caches:
        c.check_device()
    cache_bytes = caches[0].device_bytes() * w.layers

    value = job_tokens_per_s(w.B, K_steps, ws, ms_amortized)
    n_launch = n_dec * w.layers
    achieved = dec_call_bytes * n_dec / (dec_ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()

    # end to end through the public API with host buffers (pinned), per step.
    # Copy path: k, v, q host->device, append, decode, out device->host. Two buffer sets:
    # the copy stream brings in step s+1's inputs and reads back step s's
    # output while step s's kernels run, as a serving loop would drive the API.
    e2e = None
    if E_steps > 0:
        # the e2e run starts from the prompts again and takes the same warm-up
        # steps (device-resident inputs, untimed): its timed steps then see the
        # same inputs, context lengths and flushes as the device-timed region
        for c in caches:
            c.close()
        caches = build_caches()
        for s in range(W_steps):
            step(s)
        torch.cuda.synchronize()
    # Feeding the kernels from pinned host memory (ott_step_host) keeps the
    # launch chain but puts host-memory latency on each step's critical path;
    # it pays for small inputs. Steps with large inputs copy them on a second
    # stream a step ahead instead.
    in_step_bytes = sum(t.numel() * t.element_size() for t in host[0])
    # (caches that fit in L2 are timed step by step with L2 flushed in between,
    # which a copy stream running a step ahead cannot be)
    copy_stream_e2e = in_step_bytes >= E2E_ZERO_COPY_MAX and not l2_flush
    if E_steps > 0 and copy_stream_e2e:
        # each step's k, v and q travel in one pinned buffer (one copy per step)
        shapes = [tuple(t.shape) for t in host[0]]
        sizes = [t.numel() for t in host[0]]
        pin = [torch.cat([t.reshape(-1) for t in x]).pin_memory() for x in host]
        nb = 2
        flat = [torch.empty(sum(sizes), dtype=torch.float16, device=dev) for _ in range(nb)]
        din = [tuple(f.narrow(0, o, n).view(sh) for o, n, sh in zip((0, sizes[0], sizes[0] + sizes[1]), sizes, shapes))
               for f in flat]
        douts = [torch.empty_like(out) for _ in range(nb)]
        out_h = [torch.empty(w.B, w.Hq, w.d, dtype=torch.float16).pin_memory() for _ in range(nb)]
        cstream = torch.cuda.Stream(device=dev)
        copied = [torch.cuda.Event() for _ in range(nb)]     # a buffer's inputs have landed
        computed = [torch.cuda.Event() for _ in range(nb)]   # the step that used a buffer is done
        drained = [torch.cuda.Event() for _ in range(nb)]    # a buffer's output has been read back

        def h2d(s):
            b = s % nb
            with torch.cuda.stream(cstream):
                if s >= nb:
                    cstream.wait_event(computed[b])
                flat[b].copy_(pin[(W_steps + s) % n_distinct], non_blocking=True)
                copied[b].record(cstream)

        torch.cuda.synchronize()
        barrier()
        x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        x0.record(stream)
        cstream.wait_stream(stream)
        h2d(0)
        for s in range(E_steps):
            b = s % nb
            if s + 1 < E_steps:
                h2d(s + 1)
            stream.wait_event(copied[b])
            if s >= nb:
                stream.wait_event(drained[b])
            dk, dv, dq = din[b]
            for c in caches:
                c.append(dk, dv, stream)
                decode_call(c, w, dq, douts[b], stream)
            computed[b].record(stream)
            with torch.cuda.stream(cstream):
                cstream.wait_event(computed[b])
                out_h[b].copy_(douts[b], non_blocking=True)
                drained[b].record(cstream)
        stream.wait_stream(cstream)
        x1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = max_over_ranks(x0.elapsed_time(x1), dev)
        e2e = {"value": job_tokens_per_s(w.B, E_steps, ws, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": int(pin[0].numel() * pin[0].element_size()),
               "d2h_bytes_per_step": int(out_h[0].numel() * out_h[0].element_size()), "steps": E_steps,
               "copies": "k, v, q in one pinned host buffer per step, double-buffered on a second stream",
               "start": E2E_START}

    # ott_step_host appends k, v and decodes q (full or Top-K) straight from
    # pinned host memory (the append kernel reads them; the combine writes out
    # back to pinned host memory), so the step stays one chain of kernels.
    if E_steps > 0 and not copy_stream_e2e:
        shapes = [tuple(t.shape) for t in host[0]]
        sizes = [t.numel() for t in host[0]]
        pin = [torch.cat([t.reshape(-1) for t in x]).pin_memory() for x in host]
        offs = (0, sizes[0], sizes[0] + sizes[1])
        views = [tuple(p_.narrow(0, o, n).view(sh) for o, n, sh in zip(offs, sizes, shapes)) for p_ in pin]
        out_h = [torch.empty(w.B, w.Hq, w.d, dtype=torch.float16).pin_memory() for _ in range(2)]
        # with an L2 flush, each step has its own events and the flush falls outside
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(E_steps if l2_flush else 1)]
        torch.cuda.synchronize()
        barrier()
        if not l2_flush:
            ev[0][0].record(stream)
        for s in range(E_steps):
            kh, vh, qh = views[(W_steps + s) % n_distinct]
            if l2_flush:
                flush_l2(s)
                ev[s][0].record(stream)
            for c in caches:
                c.step_host(kh, vh, qh, out_h[s % 2], w.topk, stream)
            if l2_flush:
                ev[s][1].record(stream)
        if not l2_flush:
            ev[0][1].record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = max_over_ranks(sum(a_.elapsed_time(b_) for a_, b_ in ev), dev)
        in_bytes = int(pin[0].numel() * pin[0].element_size())
        out_bytes = int(out_h[0].numel() * out_h[0].element_size())
        e2e = {"value": job_tokens_per_s(w.B, E_steps, ws, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": in_bytes * w.layers, "d2h_bytes_per_step": out_bytes * w.layers,
               "steps": E_steps,
               "copies": "ott_step_host per layer: k, v and q read by the append kernel from one pinned host "
                         "buffer per step, out written by the combine into pinned host memory (two, alternating)",
               "start": E2E_START,
               "l2": "flushed between steps (each step timed on its own)" if l2_flush else "no flush needed"}

    # the prefill of one layer's cache (the parallel pass), timed on its own
    pf = None
    if not args.no_prefill:
        pf = measure_prefill(ott, w, wr, dev, stream)
        pf_ms = max_over_ranks(pf["ms"], dev)
        pf.update(ms=pf_ms, tokens_per_s=ws * pf["tokens"] / (pf_ms * 1e-3),
                  gbs=ws * pf["algorithmic_bytes"] / (pf_ms * 1e-3) / 1e9, n_gpus=ws)
        pf["frac_of_hbm_peak"] = pf["gbs"] / ws / hbm_peak()[0]

    # one decode-time flush (every unit packs one group): its bytes against its time
    flush_roof = None
    if flush_us:
        nf_now = metrics.flush_count(T0, w.G, w.R)
        # one flush of every unit of every layer (each layer has its own cache)
        fb = w.layers * w.B * w.Hkv * metrics.flush_bytes_per_unit(nf_now, w.d, w.G, w.P)
        flush_roof = {"kernel": "k_flush (one group of every unit, every layer)", "algorithmic_bytes": fb,
                      "achieved_gbs": fb / (flush_us * 1e-6) / 1e9,
                      "frac_of_hbm_peak": fb / (flush_us * 1e-6) / 1e9 / hbm_peak()[0],
                      "timing": "CUDA events around each append of one flush cycle: the appends that flush "
                                "minus the median of those that do not"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        rate1, dt1, sample1 = oracle_rate(w, args.oracle_steps, 1, args.oracle_units)
        rate, dt, sample, nproc = oracle_rate_cores(w, args.oracle_steps, 1, args.oracle_units_per_core)
        cpu = {"value": rate, "unit": "tokens/s", "cores": nproc, "kind": "oracle", "sample": sample,
               "seconds": round(dt, 2),
               "one_core": {"value": rate1, "cores": 1, "sample": sample1, "seconds": round(dt1, 2)}}

    if rank == 0:
        fp16_bytes = sum(metrics.fp16_cache_bytes(t, 1, w.Hkv, w.d) for t in synth.seq_lens(wr)) * w.layers
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws, "steps": K_steps,
            "warmup": W_steps, "ms_per_step": ms_amortized / K_steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp16 storage, fp32 accumulation", "data": "synthetic (seeded)",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "L": w.L,
                       "G": w.G, "R": w.R, "P": w.P, "layers": w.layers, "T_start": T0,
                       **({"topk": w.topk, "topk_bytes": "bound pass over every non-empty block's scale/zero "
                           "header, plus the K smallest non-empty blocks (a lower bound)"} if w.topk > 0 else {}),
                       **({"paged": "blocks from one pool of the blocks the run fills, through a block table"}
                          if w.paged else {}),
                       **({"cold": w.cold, "cold_bytes": "block and cold-pool sizes read from the device "
                           "after the decode timing cycle"} if w.cold >= 0 else {}),
                       **({"ragged_lens": {"min": min(lens), "max": max(lens),
                                           "mean": round(sum(lens) / len(lens), 1)}} if w.ragged else {}),
                       "l2": (f"cache {cache_bytes / 1e6:.0f} MB, L2 {L2_BYTES / 1e6:.0f} MB: a "
                              f"{2 * L2_BYTES / 1e6:.0f} MB buffer is written, then another read, between timed "
                              f"calls (outside the timing)"
                              if l2_flush else
                              f"cache {cache_bytes / 1e6:.0f} MB > 2 x L2 {L2_BYTES / 1e6:.0f} MB, no flush needed"),
                       "parallelism": f"weak-scaled shards x{ws}" if ws > 1 else "1 GPU"},
            "ms_per_step_measured": ms / K_steps,
            "prefill": pf,
            "flush": {"us_per_flush": flush_us, "flush_steps_in_timed_region": flush_steps, "roofline": flush_roof,
                      "charged": (f"one flush per {w.G} steps: {K_steps / w.G:.3f} flushes for {K_steps} steps, "
                                  f"{flush_steps} timed" if flush_us is not None else
                                  "ragged batch: its timed steps hold their own flushes")},
            "decode_gbs": achieved, "decode_pct_of_hbm_peak": 100.0 * achieved / peak,
            "decode_us_per_launch": 1e3 * dec_ms / n_launch,
            "decode_calls_timed": n_dec,
            "flushes_in_timed_region": flushes,
            "bytes_per_decoded_token": dec_call_bytes / w.B,
            "cache_bytes": cache_bytes, "fp16_cache_bytes": fp16_bytes,
            "peak_same_run": peak_run,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": f"hbm_gbs of {peak_kind}",
                         "frac_same_run": (achieved / peak_run["gbs"]) if peak_run else None,
                         "pct_of_nominal_8000": 100.0 * achieved / 8000.0,
                         "kernel": ("k_topk_bounds + k_topk_pick + k_decode + k_combine (ott_decode_attn_topk)" if w.topk > 0
                                    else "k_decode + k_combine (ott_decode_attn)"),
                         "timing": (f"{n_dec} decode calls at 8 points of one flush cycle after the timed steps, "
                                    f"{per_pt} back to back per point between CUDA events on the launch stream"
                                    + (" (each call with its own events, L2 flushed between calls)" if l2_flush else "")
                                    + "; bytes of each call by its point's token counts"),
                         "algorithmic_bytes_per_launch": dec_call_bytes / w.layers,
                         "traffic": recorded_traffic(w.name)},
            "clocks": clk.summary(),
            "gpu_launches": launches,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    for c in caches:
        c.close()
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--e2e-steps", type=int, default=-1, help="steps of the e2e run (default: --steps)")
    ap.add_argument("--workload", default=synth.HEADLINE, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--oracle-units", type=int, default=64)
    ap.add_argument("--oracle-steps", type=int, default=24)
    ap.add_argument("--oracle-units-per-core", type=int, default=8)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-copy-peak", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
