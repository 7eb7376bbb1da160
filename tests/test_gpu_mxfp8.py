"""Parity of the fused step with MXFP8 y (mhc_fused_step_mxfp8) with the CPU oracle: X', p, u, C
and the mix numbers bit-identical to the bf16-y step; the E8M0 scales and E4M3 codes against the
oracle's encoding of its bf16 y (oracle.mx), and, as a property of the kernel, equal to a library
MXFP8 cast of the kernel's own bf16 y; over several tiles with a ragged tail, the width splits,
short tiles, an all-zero token, power-of-two rescaling and every token of the benchmark
workload."""
import numpy as np
import pytest
import torch

from tests.oracle_pool import full_parity
from tests.parity import check_mxfp8, check_step, oracle_step, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def M():
    from stream_residual_fusion_gb300 import build
    build.build()
    import stream_residual_fusion_gb300.mhc as m
    return m


@pytest.fixture(scope="module")
def synth():
    from stream_residual_fusion_gb300 import synth as s
    return s


def _both(M, inp, flags=0):
    """The bf16-y step on the persistent kernel (the kernel the MXFP8 form runs) and the MXFP8
    form."""
    Wp = M.pack_weights(inp["W"])
    args = (inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"])
    tail = (inp["scale"], inp["base"], inp["gain"])
    bf = M.fused_step(*args, None, *tail, W_packed=Wp, flags=flags | M.PATH_PERSISTENT,
                      with_mixes=True)
    q = M.fused_step_mxfp8(*args, Wp, *tail, flags=flags, with_mixes=True)
    assert M.get_status() == M.MHC_OK
    return bf, q


def _same_as_cast(q, y):
    """The codes and scales equal an MXFP8 encoding of the bf16 y by torch ops: block scale from
    the largest magnitude's exponent, then a saturated float8_e4m3fn cast of y / X."""
    N, d = y.shape
    a = y.float().abs().reshape(N, d // 32, 32).amax(dim=2)
    e = torch.where(a > 0, torch.floor(torch.log2(a)), torch.full_like(a, -127.0))
    code = torch.clamp(e - 8 + 127, 0, 254)
    assert torch.equal(q["y_scale"].float(), code)
    X = torch.exp2(code - 127).repeat_interleave(32, dim=1)
    cast = torch.clamp(y.float() / X, -448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(q["y_codes"], cast)


@pytest.mark.parametrize("N,d,split,tile", [
    (1, 256, 0, 0),
    (300, 5120, 0, 0),       # 3 tiles, ragged last one
    (300, 5120, 16, 0),
    (160, 4096, 32, 0),
    (300, 1024, 4, 0),
    (330, 1024, 0, 40),      # 40-token tiles: rows 40..127 idle
    (130, 640, 1, 0),        # widest slice
])
def test_mxfp8_parity(M, synth, N, d, split, tile):
    inp = synth.make_inputs(N, 4, d, seed=6000 + N + d, device=DEV, scale_uniform=True,
                            x_stream_std=True)
    flags = M.split_flag(split) | (M.tile_flag(tile) if tile else 0)
    bf, q = _both(M, inp, flags)
    for k in ("Xp", "pre", "post", "comb", "mixes"):
        assert torch.equal(bf[k], q[k]), k
    _same_as_cast(q, bf["y"])
    ref = oracle_step(inp)
    check_step(bf, ref)
    check_mxfp8(q["y_codes"].cpu().numpy(), q["y_scale"].cpu().numpy(), ref["y"])


def test_mxfp8_comb_row_dest_in_place_no_mixes(M, synth):
    """The other comb reading, X' written over X, and no m output: X', p, u, C equal the bf16
    step's, the codes equal the cast of its y."""
    N, d = 257, 5120
    inp = synth.make_inputs(N, 4, d, seed=6200, device=DEV, scale_uniform=True)
    inp["comb"] = torch.rand(N, 4, 4, device=DEV)      # not symmetric: the readings differ
    Wp = M.pack_weights(inp["W"])
    tail = (inp["scale"], inp["base"], inp["gain"])
    bf = M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], None, *tail,
                      W_packed=Wp, flags=M.COMB_ROW_DEST | M.PATH_PERSISTENT)
    X = inp["X"].clone()
    q = M.fused_step_mxfp8(X, inp["F"], inp["pre"], inp["post"], inp["comb"], Wp, *tail,
                           flags=M.COMB_ROW_DEST, out={"Xp": X})
    assert M.get_status() == M.MHC_OK
    assert q["Xp"].data_ptr() == X.data_ptr() and "mixes" not in q
    for k in ("Xp", "pre", "post", "comb"):
        assert torch.equal(bf[k], q[k]), k
    _same_as_cast(q, bf["y"])
    ref = oracle_step(inp, comb_row_dest=True)
    check_mxfp8(q["y_codes"].cpu().numpy(), q["y_scale"].cpu().numpy(), ref["y"])


def test_mxfp8_zero_and_wide_range_tokens(M, synth):
    """A token whose streams and sublayer output are all zero gets scale code 0 and zero codes;
    tokens scaled by 2^-40 and 2^30 keep their codes and move their scales by -40 and +30."""
    N, d = 200, 2048
    inp = synth.make_inputs(N, 4, d, seed=6100, device=DEV, scale_uniform=True)
    inp["X"][7] = 0
    inp["F"][7] = 0
    bf, q = _both(M, inp)
    _same_as_cast(q, bf["y"])
    ref = oracle_step(inp)
    check_mxfp8(q["y_codes"].cpu().numpy(), q["y_scale"].cpu().numpy(), ref["y"])
    assert (q["y_scale"][7] == 0).all() and (q["y_codes"][7] == 0).all()
    # gain scaled by a power of two scales y exactly: codes unchanged, scales shifted
    for shift in (-40, 30):
        inp2 = dict(inp, gain=inp["gain"] * 2.0 ** shift)
        _, q2 = _both(M, inp2)
        nz = q["y_scale"].long() > 0
        assert torch.equal(q2["y_codes"][nz.repeat_interleave(32, dim=1)],
                           q["y_codes"][nz.repeat_interleave(32, dim=1)])
        assert torch.equal(q2["y_scale"].long()[nz], q["y_scale"].long()[nz] + shift)


def test_mxfp8_workload_full(M, synth):
    """The B=4, T=8192 workload: every token equal to the cast of the kernel's bf16 y and, in
    chunks on a process pool, against the oracle; no NaN code."""
    w = synth.WORKLOADS["prefill32k"]
    inp = synth.make_workload(w, seed=1, device=DEV)
    inp.pop("outliers", None)
    Wp = M.pack_weights(inp["W"])
    q = M.fused_step_mxfp8(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], Wp,
                           inp["scale"], inp["base"], inp["gain"])
    bf = M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], None,
                      inp["scale"], inp["base"], inp["gain"], W_packed=Wp, flags=M.PATH_PERSISTENT)
    assert M.get_status() == M.MHC_OK
    _same_as_cast(q, bf["y"])                           # every token
    del bf
    codes = q["y_codes"]
    assert not ((codes & 0x7F) == 0x7F).any()          # no NaN codes
    assert (q["y_scale"] <= 254).all()
    assert full_parity(inp, q) == w.N                 # every token against the oracle
