"""ctypes binding of libmhc.so, the GB300 single-pass mHC step.

Argument marshalling only: every step of the computation runs in the library's CUDA kernels.
PyTorch is used for device memory and streams. If the library is missing or fails to load, the
import of the binding raises; there is no other code path.

Calls mirror the C ABI in include/mhc.h (same names without the `mhc_` prefix). Tensors must be
CUDA (fused_step_host: per-token tensors on the host), contiguous, with the dtypes the header
lists; outputs are allocated here with torch unless passed in.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# MHC_LIBRARY names another build of the same ABI (for example the bounds-checked build,
# libmhc_checked.so); the import fails if that file is missing too.
LIB_PATH = os.environ.get("MHC_LIBRARY") or os.path.join(_PKG, "libmhc.so")

MHC_OK = 0
MHC_ERR_NULL = -1
MHC_ERR_SHAPE = -2
MHC_ERR_ALIGN = -3
MHC_ERR_ALIAS = -4
MHC_ERR_CUDA = -5
MHC_ERR_TIMEOUT = -6
MHC_ERR_WORKSPACE = -7
MHC_ERR_BOUNDS = -8

COMB_ROW_DEST = 0x1
DEBUG_NEVER_ARRIVE = 0x2
DEBUG_PLANT_OOB = 0x4          # bounds-checked build only
SPLIT_SHIFT = 8
TILE_SHIFT = 16
PATH_PERSISTENT = 0x8          # the persistent (cooperative) kernel
PATH_CLUSTER = 0x10            # the cluster kernel (one thread-block cluster per 40 tokens)

N_STREAMS = 4
MIX = (2 + N_STREAMS) * N_STREAMS


class MhcError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {lib.mhc_strerror(code).decode()} ({code})")


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_F = ctypes.c_float
_U = ctypes.c_uint
_SZ = ctypes.c_size_t

# name -> (restype, argtypes); the signatures of include/mhc.h
SIGNATURES = {
    "mhc_packed_weights_bytes": (_SZ, [_I, _I]),
    "mhc_workspace_bytes": (_SZ, [_I, _I]),
    "mhc_packed_block_columns": (_I, []),
    "mhc_fused_step": (_I, [_P] * 15 + [_I64, _I, _I, _I, _F, _F, _U, _P, _SZ, _P]),
    "mhc_fused_step_packed": (_I, [_P] * 15 + [_I64, _I, _I, _I, _F, _F, _U, _P, _SZ, _P]),
    "mhc_fused_step_mxfp8": (_I, [_P] * 16 + [_I64, _I, _I, _I, _F, _F, _U, _P, _SZ, _P]),
    "mhc_step_scratch_bytes": (_SZ, [_I, _I]),
    "mhc_fused_step_backward": (_I, [_P] * 25 + [_I64, _I, _I, _I, _F, _F, _U, _P, _SZ, _P]),
    "mhc_backward_workspace_bytes": (_SZ, [_I64, _I, _I]),
    "mhc_fused_step_noalloc": (_I, [_P] * 15 + [_I64, _I, _I, _I, _F, _F, _U, _P]),
    "mhc_noalloc_scratch_bytes": (_SZ, []),
    "mhc_fused_step_host": (_I, [_P] * 15 + [_I64, _I, _I, _I, _F, _F, _U, _P, _SZ, _I64, _P]),
    "mhc_host_staging_bytes": (_SZ, [_I, _I, _I64, _I]),
    "mhc_host_chunks": (_I64, [_I64, _I64, ctypes.POINTER(_I64), _I64]),
    "mhc_mixes": (_I, [_P] * 8 + [_I64, _I, _I, _I, _F, _F, _U, _P, _SZ, _P]),
    "mhc_sinkhorn": (_I, [_P] * 6 + [_I64, _I, _I, _F, _P]),
    "mhc_rmsnorm": (_I, [_P] * 3 + [_I64, _I, _F, _P]),
    "mhc_hc_post": (_I, [_P] * 5 + [_I64, _I, _I, _U, _P]),
    "mhc_hc_pre": (_I, [_P] * 3 + [_I64, _I, _I, _P]),
    "mhc_pack_weights": (_I, [_P, _P, _I, _I, _P]),
    "mhc_get_status": (_I, [_P]),
    "mhc_strerror": (ctypes.c_char_p, [_I]),
    "mhc_set_trace": (_I, [_P, _I64]),
    "mhc_step_config": (_I, [_I64, _I, _I, _U, ctypes.POINTER(_I), ctypes.POINTER(_I),
                             ctypes.POINTER(_I)]),
    "mhc_step_path": (_I, [_I64, _I, _I, _U]),
    "mhc_version": (_I, []),
    "mhc_checked_build": (_I, []),
}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libmhc.so not built at {path}; run __graft_entry__.build()")
    handle = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


lib = load_library()


# ---------------------------------------------------------------------------------------------
# helpers

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(rc: int, where: str):
    if rc != MHC_OK:
        raise MhcError(rc, where)


def _need(t, dtype, name, device="cuda"):
    if not isinstance(t, torch.Tensor) or t.device.type != device:
        raise TypeError(f"{name} must be a {device} tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def split_flag(split: int) -> int:
    """Flag bits that force the number of CTAs splitting the width (1, 2, 4, 8, 16 or 32; 0 =
    automatic)."""
    if split == 0:
        return 0
    if split < 1 or split & (split - 1):
        raise ValueError("split must be a power of two")
    return (split.bit_length() & 0xF) << SPLIT_SHIFT


def tile_flag(tokens: int) -> int:
    """Flag bits that force the tokens per tile (a multiple of 8, 8..128)."""
    return ((tokens // 8) & 0x1F) << TILE_SHIFT


def workspace_bytes(d: int, n: int = N_STREAMS) -> int:
    return int(lib.mhc_workspace_bytes(n, d))


def packed_weights_bytes(d: int, n: int = N_STREAMS) -> int:
    return int(lib.mhc_packed_weights_bytes(n, d))


def step_scratch_bytes(d: int, n: int = N_STREAMS) -> int:
    return int(lib.mhc_step_scratch_bytes(n, d))


# ---------------------------------------------------------------------------------------------
# the calls

def pack_weights(W, out=None, stream=None):
    _need(W, torch.float32, "W")
    n = N_STREAMS
    d = W.shape[1] // n
    if out is None:
        out = torch.empty(packed_weights_bytes(d, n), dtype=torch.uint8, device=W.device)
    _check(lib.mhc_pack_weights(_ptr(W), _ptr(out), n, d, _stream(stream)), "mhc_pack_weights")
    return out


def _step_outputs(X, out, with_mixes):
    N, n, d = X.shape
    dev = X.device
    pin = dev.type == "cpu"                    # host outputs of fused_step_host: page-locked
    out = dict(out or {})

    def need(key, shape, dtype):               # allocate only what the caller did not pass
        if key not in out:
            out[key] = torch.empty(shape, dtype=dtype, device=dev, pin_memory=pin)
    need("Xp", X.shape, torch.bfloat16)
    need("y", (N, d), torch.bfloat16)
    need("pre", (N, n), torch.float32)
    need("post", (N, n), torch.float32)
    need("comb", (N, n, n), torch.float32)
    if with_mixes:
        need("mixes", (N, MIX), torch.float32)
    return out


def fused_step(X, F, pre_prev, post_prev, comb_prev, W, scale, base, gain, *, iters=20,
               hc_eps=1e-6, norm_eps=1e-6, flags=0, with_mixes=False, out=None, workspace=None,
               W_packed=None, scratch=None, stream=None):
    """One fused single-pass mHC step (mhc_fused_step, or mhc_fused_step_packed when
    `W_packed` is given; then `scratch` is its step scratch). Returns dict with Xp, y, pre,
    post, comb (and mixes)."""
    _need(X, torch.bfloat16, "X")
    _need(F, torch.bfloat16, "F")
    for t, nm in ((pre_prev, "pre_prev"), (post_prev, "post_prev"), (comb_prev, "comb_prev"),
                  (scale, "scale"), (base, "base"), (gain, "gain")):
        _need(t, torch.float32, nm)
    N, n, d = X.shape
    o = _step_outputs(X, out, with_mixes)
    common_out = [_ptr(o["Xp"]), _ptr(o["y"]), _ptr(o["pre"]), _ptr(o["post"]), _ptr(o["comb"]),
                  _ptr(o.get("mixes"))]
    if W_packed is not None:
        _need(W_packed, torch.uint8, "W_packed")
        if scratch is None:
            scratch = torch.empty(step_scratch_bytes(d, n), dtype=torch.uint8, device=X.device)
        rc = lib.mhc_fused_step_packed(
            _ptr(X), _ptr(F), _ptr(pre_prev), _ptr(post_prev), _ptr(comb_prev), _ptr(W_packed),
            _ptr(scale), _ptr(base), _ptr(gain), *common_out, N, n, d, iters, hc_eps, norm_eps,
            flags, _ptr(scratch), scratch.numel(), _stream(stream))
        _check(rc, "mhc_fused_step_packed")
    else:
        _need(W, torch.float32, "W")
        if workspace is None:
            workspace = torch.empty(workspace_bytes(d, n), dtype=torch.uint8, device=X.device)
        rc = lib.mhc_fused_step(
            _ptr(X), _ptr(F), _ptr(pre_prev), _ptr(post_prev), _ptr(comb_prev), _ptr(W),
            _ptr(scale), _ptr(base), _ptr(gain), *common_out, N, n, d, iters, hc_eps, norm_eps,
            flags, _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
        _check(rc, "mhc_fused_step")
    return o


MX_BLOCK = 32   # features per MXFP8 block (one E8M0 scale each)


def fused_step_mxfp8(X, F, pre_prev, post_prev, comb_prev, W_packed, scale, base, gain, *,
                     iters=20, hc_eps=1e-6, norm_eps=1e-6, flags=0, with_mixes=False, out=None,
                     scratch=None, stream=None):
    """mhc_fused_step_mxfp8: the fused step with y written as MXFP8 (E4M3 codes `y_codes`
    uint8 [N, d] and E8M0 block scales `y_scale` uint8 [N, d/32]) instead of bf16 y. Returns
    dict with Xp, y_codes, y_scale, pre, post, comb (and mixes)."""
    _need(X, torch.bfloat16, "X")
    _need(F, torch.bfloat16, "F")
    _need(W_packed, torch.uint8, "W_packed")
    for t, nm in ((pre_prev, "pre_prev"), (post_prev, "post_prev"), (comb_prev, "comb_prev"),
                  (scale, "scale"), (base, "base"), (gain, "gain")):
        _need(t, torch.float32, nm)
    N, n, d = X.shape
    o = dict(out or {})
    if "y_codes" not in o:
        o["y_codes"] = torch.empty(N, d, dtype=torch.uint8, device=X.device)
    if "y_scale" not in o:
        o["y_scale"] = torch.empty(N, d // MX_BLOCK, dtype=torch.uint8, device=X.device)
    o["y"] = o["y_codes"]                        # _step_outputs fills the rest, not y
    o = _step_outputs(X, o, with_mixes)
    del o["y"]
    if scratch is None:
        scratch = torch.empty(step_scratch_bytes(d, n), dtype=torch.uint8, device=X.device)
    rc = lib.mhc_fused_step_mxfp8(
        _ptr(X), _ptr(F), _ptr(pre_prev), _ptr(post_prev), _ptr(comb_prev), _ptr(W_packed),
        _ptr(scale), _ptr(base), _ptr(gain), _ptr(o["Xp"]), _ptr(o["y_codes"]), _ptr(o["y_scale"]),
        _ptr(o["pre"]), _ptr(o["post"]), _ptr(o["comb"]), _ptr(o.get("mixes")), N, n, d, iters,
        hc_eps, norm_eps, flags, _ptr(scratch), scratch.numel(), _stream(stream))
    _check(rc, "mhc_fused_step_mxfp8")
    return o


def backward_workspace_bytes(N: int, d: int, n: int = N_STREAMS) -> int:
    return int(lib.mhc_backward_workspace_bytes(N, n, d))


def fused_step_backward(X, F, Xp, mixes, pre_prev, post_prev, comb_prev, W, scale, base, gain,
                        gXp, gy, gpre, gpost, gcomb, *, iters=20, hc_eps=1e-6, norm_eps=1e-6,
                        flags=0, out=None, workspace=None, stream=None):
    """mhc_fused_step_backward: gradients of the fused step. Xp and mixes are the forward's X'
    and m outputs; gXp, gy, gpre, gpost, gcomb the gradients of its outputs. Returns dict with
    gX, gF (bf16), gpre_prev, gpost_prev, gcomb_prev, gW, gbase, gscale, ggain (fp32)."""
    for t, nm in ((X, "X"), (F, "F"), (Xp, "Xp"), (gXp, "gXp"), (gy, "gy")):
        _need(t, torch.bfloat16, nm)
    for t, nm in ((mixes, "mixes"), (pre_prev, "pre_prev"), (post_prev, "post_prev"),
                  (comb_prev, "comb_prev"), (W, "W"), (scale, "scale"), (base, "base"),
                  (gain, "gain"), (gpre, "gpre"), (gpost, "gpost"), (gcomb, "gcomb")):
        _need(t, torch.float32, nm)
    N, n, d = X.shape
    dev = X.device
    o = dict(out or {})

    def need(key, shape, dtype):
        if key not in o:
            o[key] = torch.empty(shape, dtype=dtype, device=dev)
    need("gX", (N, n, d), torch.bfloat16)
    need("gF", (N, d), torch.bfloat16)
    need("gpre_prev", (N, n), torch.float32)
    need("gpost_prev", (N, n), torch.float32)
    need("gcomb_prev", (N, n, n), torch.float32)
    need("gW", tuple(W.shape), torch.float32)
    need("gbase", tuple(base.shape), torch.float32)
    need("gscale", (3,), torch.float32)
    need("ggain", (d,), torch.float32)
    if workspace is None:
        workspace = torch.empty(max(1, backward_workspace_bytes(N, d, n)), dtype=torch.uint8,
                                device=dev)
    rc = lib.mhc_fused_step_backward(
        _ptr(X), _ptr(F), _ptr(Xp), _ptr(mixes), _ptr(pre_prev), _ptr(post_prev), _ptr(comb_prev),
        _ptr(W), _ptr(scale), _ptr(base), _ptr(gain), _ptr(gXp), _ptr(gy), _ptr(gpre),
        _ptr(gpost), _ptr(gcomb), _ptr(o["gX"]), _ptr(o["gF"]), _ptr(o["gpre_prev"]),
        _ptr(o["gpost_prev"]), _ptr(o["gcomb_prev"]), _ptr(o["gW"]), _ptr(o["gbase"]),
        _ptr(o["gscale"]), _ptr(o["ggain"]), N, n, d, iters, hc_eps, norm_eps, flags,
        _ptr(workspace), workspace.numel(), _stream(stream))
    _check(rc, "mhc_fused_step_backward")
    return o


def fused_step_noalloc(X, F, pre_prev, post_prev, comb_prev, W, scale, base, gain, *, iters=20,
                       hc_eps=1e-6, norm_eps=1e-6, flags=0, with_mixes=False, out=None,
                       stream=None):
    """mhc_fused_step_noalloc: the fused step with the library's fixed per-device scratch, for
    callers that cannot allocate device memory when the step runs. Only the outputs are
    allocated here (pass `out` to allocate nothing)."""
    _need(X, torch.bfloat16, "X")
    _need(F, torch.bfloat16, "F")
    for t, nm in ((pre_prev, "pre_prev"), (post_prev, "post_prev"), (comb_prev, "comb_prev"),
                  (W, "W"), (scale, "scale"), (base, "base"), (gain, "gain")):
        _need(t, torch.float32, nm)
    N, n, d = X.shape
    o = _step_outputs(X, out, with_mixes)
    rc = lib.mhc_fused_step_noalloc(
        _ptr(X), _ptr(F), _ptr(pre_prev), _ptr(post_prev), _ptr(comb_prev), _ptr(W), _ptr(scale),
        _ptr(base), _ptr(gain), _ptr(o["Xp"]), _ptr(o["y"]), _ptr(o["pre"]), _ptr(o["post"]),
        _ptr(o["comb"]), _ptr(o.get("mixes")), N, n, d, iters, hc_eps, norm_eps, flags,
        _stream(stream))
    _check(rc, "mhc_fused_step_noalloc")
    return o


def host_staging_bytes(d: int, chunk_tokens: int, with_mixes: bool = False,
                       n: int = N_STREAMS) -> int:
    return int(lib.mhc_host_staging_bytes(n, d, chunk_tokens, int(with_mixes)))


def host_chunks(N: int, chunk_tokens: int) -> list[int]:
    """Token counts of the chunks fused_step_host cuts N tokens into."""
    k = int(lib.mhc_host_chunks(N, chunk_tokens, None, 0))
    if k < 0:
        raise MhcError(k, "mhc_host_chunks")
    buf = (_I64 * max(k, 1))()
    lib.mhc_host_chunks(N, chunk_tokens, buf, k)
    return list(buf[:k])


def default_chunk_tokens(N: int) -> int:
    """About 16 chunks, a multiple of 128 tokens, between 1024 and 8192 (N if smaller)."""
    return max(1, min(N, max(1024, min(8192, -(-N // 16 // 128) * 128))))


def fused_step_host(X, F, pre_prev, post_prev, comb_prev, W, scale, base, gain, *, iters=20,
                    hc_eps=1e-6, norm_eps=1e-6, flags=0, with_mixes=False, out=None,
                    staging=None, chunk_tokens=None, stream=None):
    """mhc_fused_step_host: the fused step on HOST tensors (X, F, pre/post/comb_prev and the
    outputs on the CPU, pinned for overlap), parameters W, scale, base, gain on the GPU. The
    outputs are complete once `stream` has been synchronised."""
    _need(X, torch.bfloat16, "X", "cpu")
    _need(F, torch.bfloat16, "F", "cpu")
    for t, nm in ((pre_prev, "pre_prev"), (post_prev, "post_prev"), (comb_prev, "comb_prev")):
        _need(t, torch.float32, nm, "cpu")
    for t, nm in ((W, "W"), (scale, "scale"), (base, "base"), (gain, "gain")):
        _need(t, torch.float32, nm)
    N, n, d = X.shape
    chunk = int(chunk_tokens or default_chunk_tokens(N))
    o = _step_outputs(X, out, with_mixes)
    if staging is None:
        staging = torch.empty(host_staging_bytes(d, chunk, with_mixes, n), dtype=torch.uint8,
                              device=W.device)
    rc = lib.mhc_fused_step_host(
        _ptr(X), _ptr(F), _ptr(pre_prev), _ptr(post_prev), _ptr(comb_prev), _ptr(W), _ptr(scale),
        _ptr(base), _ptr(gain), _ptr(o["Xp"]), _ptr(o["y"]), _ptr(o["pre"]), _ptr(o["post"]),
        _ptr(o["comb"]), _ptr(o.get("mixes")), N, n, d, iters, hc_eps, norm_eps, flags,
        _ptr(staging), staging.numel(), chunk, _stream(stream))
    _check(rc, "mhc_fused_step_host")
    return o


def mixes(X, W, scale, base, *, iters=20, hc_eps=1e-6, norm_eps=1e-6, flags=0, with_mixes=True,
          workspace=None, out=None, stream=None):
    """hc_mixes alone (mhc_mixes). Returns dict with pre, post, comb (and mixes)."""
    _need(X, torch.bfloat16, "X")
    for t, nm in ((W, "W"), (scale, "scale"), (base, "base")):
        _need(t, torch.float32, nm)
    N, n, d = X.shape
    dev = X.device
    o = dict(out or {})
    shapes = {"pre": (N, n), "post": (N, n), "comb": (N, n, n)}
    if with_mixes:
        shapes["mixes"] = (N, MIX)
    for key, shape in shapes.items():        # allocate only what the caller did not pass
        if key not in o:
            o[key] = torch.empty(shape, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(workspace_bytes(d, n), dtype=torch.uint8, device=dev)
    rc = lib.mhc_mixes(_ptr(X), _ptr(W), _ptr(scale), _ptr(base), _ptr(o.get("mixes")),
                       _ptr(o["pre"]), _ptr(o["post"]), _ptr(o["comb"]), N, n, d, iters, hc_eps,
                       norm_eps, flags, _ptr(workspace),
                       workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "mhc_mixes")
    return o


def sinkhorn(mixes_, scale, base, *, iters=20, hc_eps=1e-6, stream=None):
    """Split + Sinkhorn alone (mhc_sinkhorn). Returns dict with pre, post, comb."""
    for t, nm in ((mixes_, "mixes"), (scale, "scale"), (base, "base")):
        _need(t, torch.float32, nm)
    N = mixes_.shape[0]
    n = N_STREAMS
    dev = mixes_.device
    o = {"pre": torch.empty(N, n, dtype=torch.float32, device=dev),
         "post": torch.empty(N, n, dtype=torch.float32, device=dev),
         "comb": torch.empty(N, n, n, dtype=torch.float32, device=dev)}
    rc = lib.mhc_sinkhorn(_ptr(mixes_), _ptr(scale), _ptr(base), _ptr(o["pre"]), _ptr(o["post"]),
                          _ptr(o["comb"]), N, n, iters, hc_eps, _stream(stream))
    _check(rc, "mhc_sinkhorn")
    return o


def rmsnorm(x, gain, eps=1e-6, out=None, stream=None):
    _need(x, torch.bfloat16, "x")
    _need(gain, torch.float32, "gain")
    N, d = x.shape
    y = torch.empty_like(x) if out is None else out
    _check(lib.mhc_rmsnorm(_ptr(x), _ptr(gain), _ptr(y), N, d, eps, _stream(stream)), "mhc_rmsnorm")
    return y


def hc_post(X, F, post, comb, flags=0, out=None, stream=None):
    _need(X, torch.bfloat16, "X")
    _need(F, torch.bfloat16, "F")
    N, n, d = X.shape
    Xo = torch.empty_like(X) if out is None else out
    _check(lib.mhc_hc_post(_ptr(X), _ptr(F), _ptr(post), _ptr(comb), _ptr(Xo), N, n, d, flags,
                           _stream(stream)), "mhc_hc_post")
    return Xo


def hc_pre(Xp, pre, out=None, stream=None):
    _need(Xp, torch.bfloat16, "Xp")
    _need(pre, torch.float32, "pre")
    N, n, d = Xp.shape
    y = torch.empty(N, d, dtype=torch.bfloat16, device=Xp.device) if out is None else out
    _check(lib.mhc_hc_pre(_ptr(Xp), _ptr(pre), _ptr(y), N, n, d, _stream(stream)), "mhc_hc_pre")
    return y


def step_config(N: int, d: int, flags: int = 0, n: int = N_STREAMS):
    """(split, tokens per tile, groups) of the fused step for N tokens on the current device."""
    sp, tt, gr = _I(0), _I(0), _I(0)
    _check(lib.mhc_step_config(N, n, d, flags, ctypes.byref(sp), ctypes.byref(tt), ctypes.byref(gr)),
           "mhc_step_config")
    return sp.value, tt.value, gr.value


def step_path(N: int, d: int, flags: int = 0, n: int = N_STREAMS) -> int:
    """PATH_PERSISTENT or PATH_CLUSTER: the kernel the fused step runs for N tokens on the
    current device."""
    r = lib.mhc_step_path(N, n, d, flags)
    if r < 0:
        _check(r, "mhc_step_path")
    return r


def set_trace(buffer=None):
    """Record per-CTA phase timestamps of later fused launches into `buffer` (a CUDA int64
    tensor of 8 entries per CTA), or turn tracing off with None."""
    if buffer is None:
        _check(lib.mhc_set_trace(None, 0), "mhc_set_trace")
    else:
        _check(lib.mhc_set_trace(_ptr(buffer), buffer.numel() * buffer.element_size()),
               "mhc_set_trace")


def get_status(stream=None) -> int:
    """Synchronise the stream; MHC_OK, MHC_ERR_BOUNDS (checked build) or MHC_ERR_TIMEOUT (then
    cleared)."""
    return int(lib.mhc_get_status(_stream(stream)))
