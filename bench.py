"""Benchmark of the fused single-pass mHC step (n = 4 streams, d = 5120) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: the projection weights are split into
their three bf16 planes (mhc_pack_weights) and the fused kernel (mhc_fused_step_packed) reads
X and F once and writes X', y, p, u, C. The workload is the prefill batch B=4, T=8192
(N = 32,768 tokens, 3.4 GB of streams per step, far larger than L2), seeded synthetic inputs.

Tokens are independent, so N GPUs run N independent batches (weak scaling, the default; no
collective on the data path); the printed value is all ranks' tokens over the slowest rank's time.
--scaling strong splits one batch into contiguous token shards, one per rank, and reports the
batch's tokens over the slowest rank's time.

--impl reference times the CPU oracle (the only reference this method has) on a bounded sample
of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused mHC step tokens/s at n=4,d=5120; % of HBM roofline (1×GB300)"
WORKLOAD = "prefill32k"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0}
STREAM_BYTES_PER_TOKEN = (2 * 4 + 2) * 5120 * 2      # (2n+2) d bf16: read X, F; write X', y
SMALL_BYTES_PER_TOKEN = 16 + 16 + 64 + 16 + 16 + 64  # p,u,C previous in; p,u,C out (fp32)


def algorithmic_bytes(N: int, d: int = 5120) -> int:
    """Bytes one fused launch must move: the streams and small per-token vectors, plus the packed
    weights and the gain once."""
    return N * (STREAM_BYTES_PER_TOKEN + SMALL_BYTES_PER_TOKEN) + 640 * d + d * 4


L2_BYTES = 129 << 20


def percentile(sorted_ms, q):
    """The q-th percentile of an ascending list, by linear interpolation between ranks."""
    if not sorted_ms:
        return None
    pos = (len(sorted_ms) - 1) * q / 100.0
    lo = int(pos)
    hi = min(lo + 1, len(sorted_ms) - 1)
    return sorted_ms[lo] + (sorted_ms[hi] - sorted_ms[lo]) * (pos - lo)


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return json.load(fh), "measured"
    except Exception:
        return PEAKS_FALLBACK, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("fused.cu", "ptx.cuh", "mix_math.cuh", "hc_arith.cuh", "layout.cuh"):
        with open(os.path.join(ROOT, "stream_residual_fusion_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(N: int):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary, scaled to N
    tokens; None when the summary was taken on different kernel source."""
    path = os.path.join(ROOT, "profiles", "fused_step_prefill_ncu.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel source hash:\s*`?([0-9a-f]{16})", text)
    m_bpt = re.search(r"dram bytes per token:\s*([0-9.]+)", text)
    if not m_hash or not m_bpt or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_bpt.group(1)) * N


# ---------------------------------------------------------------------------------------------
# clocks during the timed region


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []
        self.proc = None
        self.t_on = self.t_off = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def mark_on(self):
        self.t_on = time.time()

    def mark_off(self):
        self.t_off = time.time()

    def stop(self):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        inside = [r for t, r in self.rows if self.t_on is not None and self.t_on <= t <= self.t_off]
        rows = inside or [r for _, r in self.rows][-3:]
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for name, v in zip(names, r[5:9]):
                    if v.lower() == "active":
                        reasons.add(name)
            except (ValueError, IndexError):
                continue
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "in_timed_region": bool(inside)}


# ---------------------------------------------------------------------------------------------
# CPU oracle leg (reported baseline; also the reference arm)


def _oracle_chunk(args):
    seed, lo, hi = args[:3]
    workload = args[3] if len(args) > 3 else WORKLOAD
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import oracle as O
    from stream_residual_fusion_gb300 import synth
    w = synth.WORKLOADS[workload]
    inp = synth.make_inputs(hi - lo, 4, w.d, seed=seed, scale_uniform=w.scale_uniform,
                            x_stream_std=w.x_stream_std, outlier_frac=w.outlier_frac)
    a = O.inputs_to_f64(inp)
    t0 = time.perf_counter()
    O.fused_step(a["X"], a["F"], a["pre"], a["post"], a["comb"], a["W"], a["scale"], a["base"],
                 a["gain"])
    return hi - lo, time.perf_counter() - t0


def oracle_throughput(tokens_per_worker: int = 256):
    """The oracle, as it stands, on a bounded sample of the workload: one spawned single-threaded
    process per host core, each on its own slice of tokens. Returns (tokens/s, cores, sample)."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    env_keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in env_keys}
    for k in env_keys:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        jobs = [(7000 + i, 0, tokens_per_worker) for i in range(cores)]
        t0 = time.perf_counter()
        with ctx.Pool(cores) as pool:
            res = pool.map(_oracle_chunk, jobs)
        wall = time.perf_counter() - t0
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    toks = sum(r[0] for r in res)
    busy = max(r[1] for r in res)
    sample = (f"{toks} tokens of the B=4,T=8192 recipe (n=4, d=5120), {cores} spawned "
              f"single-threaded processes x {tokens_per_worker} tokens; slowest worker {busy:.1f} s "
              f"(wall {wall:.1f} s incl. start-up)")
    return toks / busy, cores, sample


def oracle_rate(workload: str, tokens: int, workers: int, chunk: int = 2048):
    """Tokens/s of the oracle on `tokens` tokens of `workload`, cut into chunks of at most
    `chunk` tokens spread over `workers` spawned single-threaded processes; the time is the
    slowest worker's busy time (start-up excluded)."""
    import multiprocessing as mp
    env_keys = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in env_keys}
    os.environ.update({k: "1" for k in env_keys})
    try:
        per = -(-tokens // workers)
        jobs = []
        for w_ in range(workers):
            n = min(per, tokens - w_ * per)
            if n > 0:
                jobs.append([(8000 + w_ * 97 + c, 0, min(chunk, n - c), workload)
                             for c in range(0, n, chunk)])
        with mp.get_context("spawn").Pool(len(jobs)) as pool:
            res = pool.map(_oracle_jobs, jobs)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return sum(r[0] for r in res) / max(r[1] for r in res)


def _oracle_jobs(jobs):
    toks = busy = 0.0
    for j in jobs:
        t, b = _oracle_chunk(j)
        toks += t
        busy += b
    return toks, busy


def run_table(args):
    """Per workload: the oracle on all host cores and on one core (median of 3 runs after one
    warm-up, a bounded sample of tokens), and the fused kernel's p50 on the GPU (>= 100 launches,
    >= 20 for the largest; L2 flushed between launches where the streams fit in it). One JSON
    line per workload."""
    import torch
    from stream_residual_fusion_gb300 import mhc, synth
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else None
    for name, w in synth.WORKLOADS.items():
        row = {"workload": name, "config": w.name, "N": w.N, "cores": cores}
        for label, workers, cap in (("all_cores", cores, args.table_tokens),
                                    ("one_core", 1, max(8, args.table_tokens // 8))):
            n = min(w.N, cap)
            oracle_rate(name, min(n, 8), 1)                       # warm-up
            rates = [oracle_rate(name, n, workers) for _ in range(3)]
            row[f"oracle_{label}_tok_s"] = statistics.median(rates)
            row[f"oracle_{label}_sample_tokens"] = n
        if dev is not None:
            inp = synth.make_workload(w, seed=3000, device=dev)
            inp.pop("outliers", None)
            Wp = mhc.pack_weights(inp["W"])
            scratch = torch.empty(mhc.step_scratch_bytes(w.d), dtype=torch.uint8, device=dev)
            out = mhc.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], None,
                                 inp["scale"], inp["base"], inp["gain"], W_packed=Wp,
                                 scratch=scratch)
            flush = (torch.empty(256 << 20, dtype=torch.uint8, device=dev)
                     if fits_in_l2(w.N) else None)
            reps = 20 if w.N >= 100000 else 100
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(reps + 10)]
            for i, (a, b) in enumerate(ev):
                if flush is not None:
                    flush.fill_(1)
                a.record()
                mhc.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], None,
                               inp["scale"], inp["base"], inp["gain"], W_packed=Wp,
                               scratch=scratch, out=out)
                b.record()
            torch.cuda.synchronize()
            ms = sorted(a.elapsed_time(b) for a, b in ev[10:])
            row.update(path=("cluster" if mhc.step_path(w.N, w.d) == mhc.PATH_CLUSTER else "persistent"),
                       gpu_launches=reps, gpu_p50_ms=percentile(ms, 50), gpu_p95_ms=percentile(ms, 95),
                       gpu_p99_ms=percentile(ms, 99),
                       gpu_tok_s=w.N / (percentile(ms, 50) / 1e3),
                       frac_measured=algorithmic_bytes(w.N, w.d) / (percentile(ms, 50) / 1e3) / 1e9 / peak,
                       frac_nominal=algorithmic_bytes(w.N, w.d) / (percentile(ms, 50) / 1e3) / 1e9 / 8000.0,
                       peak_kind=peak_kind, l2=("flushed" if flush is not None else "inputs > L2"))
            del inp, out, Wp, scratch, flush
            torch.cuda.empty_cache()
        print(json.dumps(row), flush=True)
    return 0


def fits_in_l2(n_tokens: int) -> bool:
    """A step's streams (read and written) fit in twice L2: such workloads flush L2 before every
    timed launch, larger ones are timed back to back."""
    return n_tokens * STREAM_BYTES_PER_TOKEN < 2 * L2_BYTES


def workload_config(w, n_total: int, n_rank: int) -> dict:
    """The workload both arms report (the reference arm's oracle runs a bounded sample of it,
    described in its cpu_baseline.sample)."""
    return {"workload": f"{w.name} (N={n_total}), n=4, d={w.d}", "B": w.B, "T": w.T, "n": 4,
            "d": w.d, "tokens_per_rank": n_rank, "sinkhorn_iters": 20,
            "comb_reading": "code: X'_k = u_k F + sum_j C_jk X_j",
            "l2": (f"inputs larger than L2 ({n_rank * 51200 / 1e9:.2f} GB of streams read per step)"
                   if not fits_in_l2(n_rank) else
                   "inputs smaller than L2: a 256 MB write flushes L2 before every timed step, "
                   "outside the step's own events, whose mean is ms_per_step")}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    per = max(8, int(os.environ.get("MHC_REF_TOKENS_PER_WORKER", "24")))
    values = []
    sample = cores = None
    for _ in range(args.warmup):
        oracle_throughput(tokens_per_worker=8)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        v, cores, sample = oracle_throughput(tokens_per_worker=per)
        values.append(v)
    wall = time.perf_counter() - t0
    value = statistics.median(values)
    from stream_residual_fusion_gb300 import synth
    w = synth.WORKLOADS[WORKLOAD]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * wall / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, w.N, w.N),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------------------------
# the GPU arm


def run_ours(args):
    global WORKLOAD
    WORKLOAD = args.workload
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from stream_residual_fusion_gb300 import mhc, synth
    from stream_residual_fusion_gb300.dist import (max_over_ranks, slice_tokens,
                                                   strong_scaling_throughput, token_shard,
                                                   weak_scaling_throughput)
    w = synth.WORKLOADS[WORKLOAD]
    N_total, d = w.N, w.d
    strong = args.scaling == "strong"
    # weak: every rank steps its own batch of the workload; strong: one batch, each rank its
    # contiguous token shard (the same batch on every rank: one seed)
    inp = synth.make_workload(w, seed=3000 if strong else 3000 + rank, device=dev)
    inp.pop("outliers", None)
    if strong:
        lo, hi = token_shard(N_total, rank, world)
        inp.update({k: v.clone() for k, v in slice_tokens(inp, lo, hi).items()})
    N = inp["X"].shape[0]                    # tokens this rank steps
    torch.cuda.synchronize()

    out = {"Xp": torch.empty_like(inp["X"]), "y": torch.empty(N, d, dtype=torch.bfloat16, device=dev),
           "pre": torch.empty(N, 4, device=dev), "post": torch.empty(N, 4, device=dev),
           "comb": torch.empty(N, 4, 4, device=dev)}
    Wp = torch.empty(mhc.packed_weights_bytes(d), dtype=torch.uint8, device=dev)
    scratch = torch.empty(mhc.step_scratch_bytes(d), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    # launch-shape flags (default: the library's automatic choice)
    shape_flags = ((mhc.split_flag(args.split) if args.split else 0) |
                   (mhc.tile_flag(args.tile) if args.tile else 0) |
                   {"auto": 0, "persistent": mhc.PATH_PERSISTENT, "cluster": mhc.PATH_CLUSTER}[args.path])
    path = "cluster" if mhc.step_path(N, d, shape_flags) == mhc.PATH_CLUSTER else "persistent"
    kernel_name = "cluster_step_kernel" if path == "cluster" else "step_kernel<true>"
    if args.prepacked:
        mhc.pack_weights(inp["W"], out=Wp, stream=stream)

    def step(ev_a=None, ev_b=None):
        if not args.prepacked:
            mhc.pack_weights(inp["W"], out=Wp, stream=stream)                # launch 1
        if ev_a is not None:
            ev_a.record(stream)
        mhc.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], None,
                       inp["scale"], inp["base"], inp["gain"], W_packed=Wp, scratch=scratch,
                       out=out, stream=stream, flags=shape_flags)            # launch 2
        if ev_b is not None:
            ev_b.record(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if mhc.get_status() != mhc.MHC_OK:
        raise RuntimeError("device-side wait gave up during warm-up")
    graph = None
    if args.graph:
        # the whole step (packing + fused launch) replayed from a CUDA graph; the per-kernel
        # events are recorded outside it, around each replay
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        captured_stream = stream
        stream = side
        with torch.cuda.graph(graph, stream=side):
            step()
        stream = captured_stream
        torch.cuda.synchronize()

    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    clocks = ClockSampler(visible[local].strip() if local < len(visible) else local)
    clocks.start()
    time.sleep(0.3)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    # Workloads whose streams fit in L2: a 256 MB write flushes it before every timed step,
    # outside events that bracket the whole step, and the step time is the mean of those.
    flush = (torch.empty(256 << 20, dtype=torch.uint8, device=dev)
             if fits_in_l2(N) else None)
    st = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_on()
    t_start.record(stream)
    for i in range(K):
        if flush is not None:
            # one pair of events per step (nested pairs add their own cost to the outer one);
            # the fused launch alone is timed in the percentile pass below, flushed the same way
            flush.fill_(1)
            st[i][0].record(stream)
            if graph is None:
                step()
            else:
                graph.replay()
            st[i][1].record(stream)
        elif graph is None:
            step(*ev[i])
        else:
            ev[i][0].record(stream)
            graph.replay()
            ev[i][1].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    total_ms = t_start.elapsed_time(t_end)
    fused_ms = [a.elapsed_time(b) for a, b in ev] if flush is None else None
    step_ms = [a.elapsed_time(b) for a, b in st] if flush is not None else None

    # percentile pass, after the headline timing: PCT_LAUNCHES more steps, the fused launch of
    # each bracketed by its own events; L2 is flushed between launches when the workload's
    # streams fit in it
    pct_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.pct_launches)]
    for a, b in pct_ev:
        if flush is not None:
            flush.fill_(1)
        if graph is None:
            step(a, b)
        else:
            a.record(stream)
            graph.replay()
            b.record(stream)
    torch.cuda.synchronize()
    clocks.mark_off()
    pct_ms = sorted(a.elapsed_time(b) for a, b in pct_ev)
    if fused_ms is None:
        fused_ms = pct_ms
    if world > 1:
        dist.barrier()
    clocks.stop()
    status = mhc.get_status()

    # the slowest rank's time: the whole timed region over K, or with L2 flushed between steps
    # the mean of the per-step events
    ms_per_step = max_over_ranks(statistics.mean(step_ms) if flush is not None else total_ms / K,
                                 device=dev)

    def throughput(seconds):
        return (strong_scaling_throughput(N_total, seconds) if strong
                else weak_scaling_throughput(N, world, seconds))
    value = throughput(ms_per_step / 1e3)

    # ------------------------------------------------------------------ end to end, host buffers
    e2e = None
    if not args.no_e2e:
        e2e_steps = max(2, min(5, K))
        host = {k: inp[k].to("cpu").pin_memory() for k in ("X", "F", "pre", "post", "comb")}
        host_out = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory() for k, v in out.items()}
        h2d = sum(v.numel() * v.element_size() for v in host.values())
        d2h = sum(v.numel() * v.element_size() for v in host_out.values())
        chunk = mhc.default_chunk_tokens(N)
        staging = torch.empty(mhc.host_staging_bytes(d, chunk), dtype=torch.uint8, device=dev)

        def e2e_step():
            # host tensors in, host tensors out: chunked copies overlap the fused step
            mhc.fused_step_host(host["X"], host["F"], host["pre"], host["post"], host["comb"],
                                inp["W"], inp["scale"], inp["base"], inp["gain"], out=host_out,
                                staging=staging, chunk_tokens=chunk, stream=stream)

        e2e_step()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        a.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        te = max_over_ranks(a.elapsed_time(b) / e2e_steps, device=dev)
        e2e = {"value": throughput(te / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": te, "steps": e2e_steps,
               "call": f"mhc_fused_step_host (pinned host tensors, {chunk}-token chunks)"}
        del host, host_out, staging

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks, peak_kind = measured_peaks()
    fused_avg = statistics.mean(fused_ms)
    achieved = algorithmic_bytes(N, d) / (fused_avg / 1e3) / 1e9
    peak = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    # the committed DRAM counts are the persistent kernel's: none for the cluster kernel's line
    traffic = ncu_traffic(N) if path == "persistent" else None
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": args.scaling, "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(w, N_total, N),
        "launch": {"step": (("CUDA-graph replay of " if args.graph else "") +
                            ("mhc_fused_step_packed (weights packed once, before timing)"
                             if args.prepacked else "mhc_pack_weights + mhc_fused_step_packed")),
                   "path": path,
                   "launch_shape": dict(zip(("split", "tile", "groups"),
                                            mhc.step_config(N, d, shape_flags)[:3]))},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
                     "frac_of_nominal_8000": achieved / 8000.0,
                     "kernel": (f"{kernel_name} (fused), timed with the packing as one graph replay"
                                if args.graph and not args.prepacked else f"{kernel_name} (fused)"),
                     "kernel_ms_avg": fused_avg,
                     "kernel_timed_over": ("the timed steps" if flush is None else
                                           "the percentile pass (L2 flushed before each launch)"),
                     "algorithmic_bytes_per_launch": algorithmic_bytes(N, d)},
        "kernel_percentiles": {
            "launches": len(pct_ms), "p50_ms": percentile(pct_ms, 50),
            "p95_ms": percentile(pct_ms, 95), "p99_ms": percentile(pct_ms, 99),
            "min_ms": pct_ms[0], "max_ms": pct_ms[-1],
            "how": ("CUDA events around each fused launch of a separate pass of "
                    f"{len(pct_ms)} steps after the timed region" +
                    ("; L2 flushed (256 MB write) between launches" if flush is not None else
                     "; inputs larger than L2"))},
        "clocks": dict(clocks.summary(),
                       window="the timed steps and the percentile pass right after them"),
        "e2e": e2e,
        "gpu_launches": (1 if args.prepacked else 2) * K,
        "status": "ok" if status == mhc.MHC_OK else "device wait gave up",
        "gpu": torch.cuda.get_device_name(dev),
        "torch": torch.__version__,
    }
    if world == 1 and not args.no_cpu_baseline:
        v, cores, sample = oracle_throughput()
        line["cpu_baseline"] = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


# bytes per token each kernel of the unfused form must move (d = 5120, n = 4, no m output)
UNFUSED_BYTES_PER_TOKEN = {
    "hc_post": 4 * 5120 * 2 + 5120 * 2 + 16 + 64 + 4 * 5120 * 2,   # read X, F, u, C; write X'
    "mixes": 4 * 5120 * 2 + 96,                                      # read X'; write p, u, C
    "hc_pre": 4 * 5120 * 2 + 16 + 5120 * 2,                          # read X', p; write y_hat
    "rmsnorm": 5120 * 2 + 5120 * 2,                                  # read y_hat; write y
}


def run_unfused(args):
    """The unfused GPU form of the same step: hc_post, hc_mixes (+ split and Sinkhorn), hc_pre and
    RMSNorm as four launches that pass X' and y_hat through HBM, timed per kernel beside the fused
    step on the same inputs (one GPU)."""
    import torch
    from stream_residual_fusion_gb300 import mhc, synth
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    N, d = w.N, w.d
    inp = synth.make_workload(w, seed=3000, device=dev)
    inp.pop("outliers", None)
    stream = torch.cuda.current_stream(dev)
    Xp = torch.empty_like(inp["X"])
    yhat = torch.empty(N, d, dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(yhat)
    mx = {"pre": torch.empty(N, 4, device=dev), "post": torch.empty(N, 4, device=dev),
          "comb": torch.empty(N, 4, 4, device=dev)}
    ws = torch.empty(mhc.workspace_bytes(d), dtype=torch.uint8, device=dev)
    out = {"Xp": torch.empty_like(inp["X"]), "y": torch.empty_like(yhat),
           "pre": torch.empty(N, 4, device=dev), "post": torch.empty(N, 4, device=dev),
           "comb": torch.empty(N, 4, 4, device=dev)}
    Wp = torch.empty(mhc.packed_weights_bytes(d), dtype=torch.uint8, device=dev)
    scratch = torch.empty(mhc.step_scratch_bytes(d), dtype=torch.uint8, device=dev)
    names = list(UNFUSED_BYTES_PER_TOKEN)

    def unfused(ev=None):
        rec = (lambda i: ev[i].record(stream)) if ev else (lambda i: None)
        rec(0)
        mhc.hc_post(inp["X"], inp["F"], inp["post"], inp["comb"], out=Xp, stream=stream)
        rec(1)
        mhc.mixes(Xp, inp["W"], inp["scale"], inp["base"], with_mixes=False, workspace=ws,
                  out=mx, stream=stream)
        rec(2)
        mhc.hc_pre(Xp, inp["pre"], out=yhat, stream=stream)
        rec(3)
        mhc.rmsnorm(yhat, inp["gain"], 1e-6, out=y, stream=stream)
        rec(4)

    def fused(ev=None):
        mhc.pack_weights(inp["W"], out=Wp, stream=stream)
        if ev:
            ev[0].record(stream)
        mhc.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], None,
                       inp["scale"], inp["base"], inp["gain"], W_packed=Wp, scratch=scratch,
                       out=out, stream=stream)
        if ev:
            ev[1].record(stream)

    for _ in range(max(3, args.warmup)):
        unfused()
        fused()
    torch.cuda.synchronize()
    K = args.steps
    T = lambda: torch.cuda.Event(enable_timing=True)
    evu = [[T() for _ in range(5)] for _ in range(K)]
    evf = [[T() for _ in range(2)] for _ in range(K)]
    for i in range(K):                      # interleaved, so both see the same clocks
        unfused(evu[i])
        fused(evf[i])
    torch.cuda.synchronize()
    if mhc.get_status() != mhc.MHC_OK:
        raise RuntimeError("device-side wait gave up")
    same = bool(torch.equal(Xp, out["Xp"]))
    per = {nm: statistics.median(e[j].elapsed_time(e[j + 1]) for e in evu)
           for j, nm in enumerate(names)}
    total = statistics.median(e[0].elapsed_time(e[4]) for e in evu)
    fused_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evf)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    kernels = {}
    for nm in names:
        b = N * UNFUSED_BYTES_PER_TOKEN[nm]
        kernels[nm] = {"ms_p50": per[nm], "algorithmic_bytes": b,
                       "gbs": b / (per[nm] / 1e3) / 1e9, "frac": b / (per[nm] / 1e3) / 1e9 / peak}
    unf_bytes = N * sum(UNFUSED_BYTES_PER_TOKEN.values())
    line = {
        "metric": "unfused four-kernel mHC step tokens/s at n=4,d=5120 (beside the fused step)",
        "form": "unfused", "value": N / (total / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": K, "warmup": args.warmup, "ms_per_step": total, "higher_is_better": True,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{w.name} (N={N}), n=4, d={d}", "sinkhorn_iters": 20},
        "kernels": kernels,
        "unfused_algorithmic_bytes_per_token": sum(UNFUSED_BYTES_PER_TOKEN.values()),
        "fused_algorithmic_bytes_per_token": STREAM_BYTES_PER_TOKEN + SMALL_BYTES_PER_TOKEN,
        "unfused_ms_p50": total, "fused_ms_p50": fused_ms, "fused_speedup": total / fused_ms,
        "unfused_bytes_per_launch_sum": unf_bytes, "peak_gbs": peak, "peak_kind": peak_kind,
        "x_prime_identical": same, "gpu_launches": K * 6,
    }
    print(json.dumps(line), flush=True)
    return 0


# bytes per token of the step with MXFP8 y (d = 5120, n = 4): read X, F and the previous tuple;
# write X', the E4M3 codes of y, its E8M0 block scales and p, u, C
MXFP8_BYTES_PER_TOKEN = 5 * 5120 * 2 + 96 + 4 * 5120 * 2 + 5120 + 5120 // 32 + 96


def run_mxfp8(args):
    """The fused step with y written as MXFP8 (codes + block scales), timed beside the bf16-y
    step on the same inputs (one GPU), each against its own algorithmic bytes."""
    import torch
    from stream_residual_fusion_gb300 import mhc, synth
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    N, d = w.N, w.d
    inp = synth.make_workload(w, seed=3000, device=dev)
    inp.pop("outliers", None)
    stream = torch.cuda.current_stream(dev)
    Wp = mhc.pack_weights(inp["W"], stream=stream)
    scratch = torch.empty(mhc.step_scratch_bytes(d), dtype=torch.uint8, device=dev)
    small = lambda: {"pre": torch.empty(N, 4, device=dev), "post": torch.empty(N, 4, device=dev),
                     "comb": torch.empty(N, 4, 4, device=dev), "Xp": torch.empty_like(inp["X"])}
    out_bf, out_mx = small(), small()
    out_bf["y"] = torch.empty(N, d, dtype=torch.bfloat16, device=dev)
    out_mx["y_codes"] = torch.empty(N, d, dtype=torch.uint8, device=dev)
    out_mx["y_scale"] = torch.empty(N, d // 32, dtype=torch.uint8, device=dev)
    args_in = (inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"])
    tail = (inp["scale"], inp["base"], inp["gain"])

    def bf16_step():
        mhc.fused_step(*args_in, None, *tail, W_packed=Wp, scratch=scratch, out=out_bf,
                       stream=stream)

    def mx_step():
        mhc.fused_step_mxfp8(*args_in, Wp, *tail, scratch=scratch, out=out_mx, stream=stream)

    for _ in range(max(3, args.warmup)):
        bf16_step()
        mx_step()
    torch.cuda.synchronize()
    K = args.steps
    T = lambda: torch.cuda.Event(enable_timing=True)
    ev = [[T() for _ in range(3)] for _ in range(K)]
    for i in range(K):                      # interleaved, so both see the same clocks
        ev[i][0].record(stream)
        bf16_step()
        ev[i][1].record(stream)
        mx_step()
        ev[i][2].record(stream)
    torch.cuda.synchronize()
    if mhc.get_status() != mhc.MHC_OK:
        raise RuntimeError("device-side wait gave up")
    bf_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    mx_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    mx_bytes = N * MXFP8_BYTES_PER_TOKEN + 640 * d + d * 4
    bf_bytes = algorithmic_bytes(N, d)
    line = {
        "metric": "fused mHC step tokens/s at n=4,d=5120 with MXFP8 y (beside the bf16-y step)",
        "form": "mxfp8", "value": N / (mx_ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": K, "warmup": args.warmup, "ms_per_step": mx_ms, "higher_is_better": True,
        "dtype": "bf16 streams, e4m3/e8m0 y", "data": "synthetic",
        "config": {"workload": f"{w.name} (N={N}), n=4, d={d}", "sinkhorn_iters": 20},
        "mxfp8_algorithmic_bytes_per_token": MXFP8_BYTES_PER_TOKEN,
        "mxfp8_ms_p50": mx_ms, "mxfp8_frac": mx_bytes / (mx_ms / 1e3) / 1e9 / peak,
        "bf16_ms_p50": bf_ms, "bf16_frac": bf_bytes / (bf_ms / 1e3) / 1e9 / peak,
        "speedup_vs_bf16_y": bf_ms / mx_ms, "peak_gbs": peak, "peak_kind": peak_kind,
        "x_prime_identical": bool(torch.equal(out_bf["Xp"], out_mx["Xp"])),
        "gpu_launches": K * 2,
    }
    print(json.dumps(line), flush=True)
    return 0


# bytes per token of the backward (d = 5120, n = 4). Algorithmic, the least a single pass must
# move: read X, F, gXp, gy and the small per-token inputs (p, u, C of the previous step, m, and
# the gradients of p, u, C); write gX, gF and the gradients of the previous p, u, C.
BACKWARD_BYTES_PER_TOKEN = (4 + 1 + 4 + 1) * 5120 * 2 + (4 + 1) * 5120 * 2 + 96 + 96 + 96 + 96
# What the five kernels move: the token pass and the weight pass each read X' and gy again.
BACKWARD_DESIGN_BYTES_PER_TOKEN = BACKWARD_BYTES_PER_TOKEN + 2 * (4 * 5120 * 2 + 5120 * 2)


def run_backward(args):
    """mhc_fused_step_backward on the workload (default B=4, T=8192): the gradients of every
    input and parameter of the step from seeded gradients of its outputs, timed with CUDA events
    per call (inputs larger than L2), against the backward's algorithmic bytes."""
    import torch
    from stream_residual_fusion_gb300 import mhc, synth
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    w = synth.WORKLOADS[args.workload]
    N, d = w.N, w.d
    inp = synth.make_workload(w, seed=3000, device=dev)
    inp.pop("outliers", None)
    up = synth.make_upstream(N, 4, d, seed=3001, device=dev)
    stream = torch.cuda.current_stream(dev)
    fw = mhc.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"],
                        inp["scale"], inp["base"], inp["gain"], with_mixes=True, stream=stream)
    ws = torch.empty(mhc.backward_workspace_bytes(N, d), dtype=torch.uint8, device=dev)
    out = {}

    def step():
        return mhc.fused_step_backward(inp["X"], inp["F"], fw["Xp"], fw["mixes"], inp["pre"],
                                       inp["post"], inp["comb"], inp["W"], inp["scale"],
                                       inp["base"], inp["gain"], up["gXp"], up["gy"], up["gpre"],
                                       up["gpost"], up["gcomb"], out=out or None, workspace=ws,
                                       stream=stream)
    out.update(step())
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    K = args.steps
    T = lambda: torch.cuda.Event(enable_timing=True)
    ev = [(T(), T()) for _ in range(K)]
    visible = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
    clk = ClockSampler(visible[dev.index].strip() if dev.index < len(visible) else dev.index)
    clk.start()
    time.sleep(0.3)
    clk.mark_on()
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    clk.mark_off()
    clk.stop()
    if mhc.get_status() != mhc.MHC_OK:
        raise RuntimeError("device-side wait gave up")
    ms = sorted(a.elapsed_time(b) for a, b in ev)
    p50 = percentile(ms, 50)
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", PEAKS_FALLBACK["hbm_gbs"]))
    alg = N * BACKWARD_BYTES_PER_TOKEN + 2 * (24 * 4 * d * 4) + 2 * d * 4
    design = N * BACKWARD_DESIGN_BYTES_PER_TOKEN + 2 * (24 * 4 * d * 4) + 2 * d * 4
    line = {
        "metric": "backward of the fused mHC step tokens/s at n=4,d=5120; % of HBM roofline",
        "form": "backward", "value": N / (p50 / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": K, "warmup": args.warmup, "ms_per_step": p50, "higher_is_better": True,
        "dtype": "bf16 streams, fp32 parameters and gradients of parameters", "data": "synthetic",
        "config": {"workload": f"{w.name} (N={N}), n=4, d={d}", "sinkhorn_iters": 20,
                   "l2": "inputs larger than L2"},
        "roofline": {"bound": "hbm", "achieved": alg / (p50 / 1e3) / 1e9, "peak": peak,
                     "unit": "GB/s", "frac": alg / (p50 / 1e3) / 1e9 / peak, "traffic": None,
                     "peak_kind": peak_kind,
                     "algorithmic_bytes_per_launch": alg,
                     "what": "the whole call (six launches) against the single-pass bytes"},
        "design_bytes_per_launch": design,
        "design_frac": design / (p50 / 1e3) / 1e9 / peak,
        "ms_p50": p50, "ms_p95": percentile(ms, 95), "ms_p99": percentile(ms, 99),
        "clocks": clk.summary(), "gpu_launches": K * 6,
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--table", action="store_true",
                    help="per-workload table: the oracle on all host cores and on one core beside "
                         "the fused kernel's GPU p50")
    ap.add_argument("--table-tokens", type=int, default=2048,
                    help="oracle sample per run for --table (one core: an eighth of it)")
    ap.add_argument("--scaling", choices=("weak", "strong"), default="weak",
                    help="weak: every rank steps a whole batch; strong: one batch split into "
                         "contiguous token shards over the ranks")
    ap.add_argument("--pct-launches", type=int, default=200,
                    help="launches of the percentile pass after the timed region (>= 100)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="time CUDA-graph replays of the step (no host submission cost; for small workloads)")
    ap.add_argument("--form", choices=("fused", "unfused", "mxfp8", "backward"), default="fused",
                    help="unfused: time the four-kernel form beside the fused step; mxfp8: the "
                         "step with MXFP8 y beside the bf16-y step; backward: the gradients of "
                         "the step (one GPU each)")
    ap.add_argument("--prepacked", action="store_true",
                    help="pack the weights once before timing (as a decode loop does); the step is "
                         "then the fused launch alone")
    ap.add_argument("--split", type=int, default=0,
                    help="force the CTAs per tile (MHC_SPLIT flags); 0 = automatic")
    ap.add_argument("--tile", type=int, default=0,
                    help="force the tokens per tile (MHC_TILE flags); 0 = automatic")
    ap.add_argument("--path", choices=("auto", "persistent", "cluster"), default="auto",
                    help="kernel of the fused step (MHC_PATH flags): the library's choice, the "
                         "persistent kernel, or the cluster kernel (one cluster per 40 tokens)")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="synthetic workload (default: the B=4,T=8192 prefill; others are for profiling)")
    args = ap.parse_args()
    args.pct_launches = max(100, args.pct_launches)
    if args.impl == "reference":
        return run_reference(args)
    if args.table:
        return run_table(args)
    if args.form == "unfused":
        return run_unfused(args)
    if args.form == "mxfp8":
        return run_mxfp8(args)
    if args.form == "backward":
        return run_backward(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
