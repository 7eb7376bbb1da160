"""Whole-batch parity at the large workloads: every token of a GPU step against the CPU oracle,
in chunks, on a pool of spawned processes (one per host core).

The main process copies one chunk at a time of the step's inputs and outputs from the GPU (bf16
as raw 16-bit words, fp32 as is) and hands it to a worker; at most two chunks per worker are in
flight, so host memory holds a few hundred MB whatever the batch. A worker runs the oracle on
its chunk's inputs and applies the comparison rules of tests/parity.py to the chunk's outputs;
it returns None or the first failure. The pool is started with `spawn`: the workers never touch
CUDA and do not inherit the parent's CUDA context.
"""
from __future__ import annotations

import os
import threading

import numpy as np

PER_TOKEN_IN = ("X", "F", "pre", "post", "comb")
PER_TOKEN_OUT = ("Xp", "y", "y_codes", "y_scale", "pre", "post", "comb", "mixes")
PARAMS = ("W", "scale", "base", "gain")

_params = None


def _bf16_bits_to_f64(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _to_host(t):
    """A CUDA (or CPU) tensor as a numpy array: bf16 as uint16 bit patterns, others as is."""
    import torch
    t = t.detach().to("cpu")
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


_BLAS_ENV = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _init_worker(params):
    global _params
    _params = params


def _widen(a):
    return _bf16_bits_to_f64(a) if a.dtype == np.uint16 else np.asarray(a, dtype=np.float64)


def check_chunk(task):
    """Worker: oracle on one chunk, compared with the GPU's outputs for it. Returns (lo, hi,
    None) or (lo, hi, failure text)."""
    import oracle as O
    from tests import parity as P
    lo, hi, ins, outs, kw = task
    a = {k: _widen(v) for k, v in ins.items()}
    p = {k: np.asarray(v, dtype=np.float64) for k, v in _params.items()}
    ref = O.fused_step(a["X"], a["F"], a["pre"], a["post"], a["comb"], p["W"], p["scale"],
                       p["base"], p["gain"], **kw)
    got = {k: (v if k in ("y_codes", "y_scale") else _widen(v)) for k, v in outs.items()}
    try:
        P.assert_exact(got["Xp"], ref["Xp"], "X'")
        if "y" in got:
            P.assert_bf16_within(got["y"], ref["y"])
        if "y_codes" in got:                          # y as MXFP8: codes and block scales
            P.check_mxfp8(got["y_codes"], got["y_scale"], ref["y"])
        for k in ("pre", "post", "comb"):
            P.assert_abs(got[k], ref[k], P.TOL_PUC, k)
        if "mixes" in got:
            P.assert_mixes(got["mixes"], ref["mixes"])
    except AssertionError as e:
        return lo, hi, f"tokens [{lo}, {hi}): {e}"
    return lo, hi, None


def full_parity(inp: dict, out: dict, *, chunk: int = 512, workers: int | None = None,
                oracle_kw: dict | None = None, timeout_s: float = 900.0) -> int:
    """Compare every token of `out` (the GPU step's outputs, CUDA tensors; y as bf16 `y`, or as
    MXFP8 `y_codes` and `y_scale`) with the oracle on `inp` (the step's inputs). Raises
    AssertionError naming the first failing chunk; returns the number of tokens compared. A pool
    that does not finish within `timeout_s` (a worker that died at start-up, for example) fails
    the comparison instead of waiting forever."""
    import multiprocessing as mp
    N = inp["X"].shape[0]
    if workers is None:
        workers = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    workers = max(1, min(workers, -(-N // chunk)))
    params = {k: _to_host(inp[k]) for k in PARAMS}
    outs_keys = [k for k in PER_TOKEN_OUT if k in out and out[k] is not None]
    ctx = mp.get_context("spawn")
    failures = []
    compared = 0
    gate = threading.BoundedSemaphore(2 * workers)

    def done(res):
        nonlocal compared
        lo, hi, err = res
        compared += hi - lo
        if err is not None:
            failures.append((lo, err))
        gate.release()

    def fail(exc):
        failures.append((-1, f"worker raised {exc!r}"))
        gate.release()

    # one BLAS thread per worker: the spawned children take the environment at start-up
    saved = {k: os.environ.get(k) for k in _BLAS_ENV}
    os.environ.update({k: "1" for k in _BLAS_ENV})
    try:
        pool = ctx.Pool(workers, initializer=_init_worker, initargs=(params,))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    import time
    deadline = time.monotonic() + timeout_s
    with pool:
        pending = []
        for lo in range(0, N, chunk):
            hi = min(N, lo + chunk)
            if not gate.acquire(timeout=max(1.0, deadline - time.monotonic())):
                raise AssertionError(f"oracle pool made no progress within {timeout_s:.0f} s")
            ins = {k: _to_host(inp[k][lo:hi]) for k in PER_TOKEN_IN}
            outs = {k: _to_host(out[k][lo:hi]) for k in outs_keys}
            pending.append(pool.apply_async(check_chunk, ((lo, hi, ins, outs, oracle_kw or {}),),
                                            callback=done, error_callback=fail))
        for r in pending:
            r.wait(max(1.0, deadline - time.monotonic()))
            if not r.ready():
                raise AssertionError(f"oracle pool did not finish within {timeout_s:.0f} s")
    if failures:
        failures.sort()
        raise AssertionError(f"{len(failures)} chunk(s) failed; first: {failures[0][1]}")
    assert compared == N, (compared, N)
    return compared
