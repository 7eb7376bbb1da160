"""The bounds-checked build (libmhc_checked.so, MHC_CHECKED=1): every copy, store and exchange
access of the fused step tests its index first, skips a failing one and reports MHC_ERR_BOUNDS.

  * On valid inputs no check fires: parity with the oracle across launch shapes, ragged tails
    and both y forms, with sentinel padding around every output left untouched.
  * With MHC_DEBUG_PLANT_OOB (accepted by the bounds-checked library only) one finisher row and
    one MXFP8 scale row of the first CTA get an index N rows past the end: the checks skip those stores, the
    status reports MHC_ERR_BOUNDS, the padding (larger than N rows, so even an unchecked store
    would have stayed inside this test's own buffer) is untouched, and every other output
    matches the regular build.
"""
import importlib.util
import os

import pytest
import torch

from tests.parity import check_step, oracle_step

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def M():
    from stream_residual_fusion_gb300 import build
    build.build()
    import stream_residual_fusion_gb300.mhc as m
    return m


@pytest.fixture(scope="module")
def MC(M):
    """A second instance of the binding, loaded on the checked build."""
    from stream_residual_fusion_gb300 import build
    path = build.build(checked=True)
    saved = os.environ.get("MHC_LIBRARY")
    os.environ["MHC_LIBRARY"] = path
    try:
        spec = importlib.util.spec_from_file_location("mhc_checked_binding", M.__file__)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
    finally:
        if saved is None:
            os.environ.pop("MHC_LIBRARY", None)
        else:
            os.environ["MHC_LIBRARY"] = saved
    assert mod.lib.mhc_checked_build() == 1 and M.lib.mhc_checked_build() == 0
    return mod


@pytest.fixture(scope="module")
def synth():
    from stream_residual_fusion_gb300 import synth as s
    return s


def _padded_outputs(N, d, mx, pad_after):
    rows = {"Xp": ((4, d), torch.bfloat16), "pre": ((4,), torch.float32),
            "post": ((4,), torch.float32), "comb": ((4, 4), torch.float32),
            "mixes": ((24,), torch.float32)}
    if mx:
        rows.update(y_codes=((d,), torch.uint8), y_scale=((d // 32,), torch.uint8))
    else:
        rows["y"] = ((d,), torch.bfloat16)
    full, view = {}, {}
    for k, (shape, dt) in rows.items():
        full[k] = torch.empty((2 + N + pad_after, *shape), dtype=dt, device=DEV)
        full[k].view(torch.uint8).fill_(SENTINEL)
        view[k] = full[k][2:2 + N]
    return full, view


def _padding_untouched(full, N):
    for k, f in full.items():
        b = f.view(torch.uint8).reshape(f.shape[0], -1)
        assert bool((b[:2] == SENTINEL).all()) and bool((b[2 + N:] == SENTINEL).all()), k


def _step(mod, inp, Wp, mx, flags, out):
    args = (inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"])
    tail = (inp["scale"], inp["base"], inp["gain"])
    if mx:
        return mod.fused_step_mxfp8(*args, Wp, *tail, flags=flags, with_mixes=True, out=out)
    return mod.fused_step(*args, None, *tail, W_packed=Wp, flags=flags, with_mixes=True, out=out)


def test_plant_flag_refused_by_the_regular_build(M, synth):
    inp = synth.make_inputs(8, 4, 256, seed=1, device=DEV)
    with pytest.raises(M.MhcError) as e:
        M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"],
                     inp["scale"], inp["base"], inp["gain"], flags=M.DEBUG_PLANT_OOB)
    assert e.value.code == M.MHC_ERR_SHAPE


@pytest.mark.parametrize("mx", [False, True], ids=["bf16_y", "mxfp8_y"])
@pytest.mark.parametrize("N,d,split,tile", [
    (1, 5120, 0, 0), (300, 5120, 0, 0), (300, 5120, 32, 64), (257, 1024, 4, 0),
    (300, 512, 1, 8), (4097, 5120, 0, 0),
])
def test_checked_build_parity_no_check_fires(M, MC, synth, mx, N, d, split, tile):
    inp = synth.make_inputs(N, 4, d, seed=900 + N + d + split, device=DEV, scale_uniform=True,
                            x_stream_std=True)
    inp.pop("outliers", None)
    flags = (MC.split_flag(split) if split else 0) | (MC.tile_flag(tile) if tile else 0)
    Wp = M.pack_weights(inp["W"])
    full, view = _padded_outputs(N, d, mx, 256)
    got = _step(MC, inp, Wp, mx, flags, view)
    assert MC.get_status() == MC.MHC_OK
    _padding_untouched(full, N)
    ref = _step(M, inp, Wp, mx, flags, None)        # the regular build on the same inputs
    assert M.get_status() == M.MHC_OK
    for k in view:
        assert torch.equal(got[k], ref[k]), k
    if not mx:
        check_step(got, oracle_step(inp))


@pytest.mark.parametrize("mx", [False, True], ids=["bf16_y", "mxfp8_y"])
@pytest.mark.parametrize("N,split,tile", [(300, 0, 0), (300, 32, 64), (200, 32, 0)])
def test_planted_out_of_range_rows_are_caught(M, MC, synth, mx, N, split, tile):
    d = 5120
    inp = synth.make_inputs(N, 4, d, seed=950 + N + split, device=DEV, scale_uniform=True)
    inp.pop("outliers", None)
    flags = (MC.split_flag(split) if split else 0) | (MC.tile_flag(tile) if tile else 0)
    Wp = M.pack_weights(inp["W"])
    full, view = _padded_outputs(N, d, mx, 2 * N + 128)
    got = _step(MC, inp, Wp, mx, flags | MC.DEBUG_PLANT_OOB, view)
    assert MC.get_status() == MC.MHC_ERR_BOUNDS
    assert MC.get_status() == MC.MHC_OK                  # read once, then cleared
    _padding_untouched(full, N)
    ref = _step(M, inp, Wp, mx, flags, None)
    assert M.get_status() == M.MHC_OK
    # the first token's finisher row was skipped (still sentinel); every other row is written
    for k in ("pre", "post", "comb", "mixes"):
        row0 = got[k][0].view(torch.uint8)
        assert bool((row0 == SENTINEL).all()), k
        assert torch.equal(got[k][1:], ref[k][1:]), k
    assert torch.equal(got["Xp"], ref["Xp"])
    if mx:
        assert torch.equal(got["y_codes"], ref["y_codes"])
        differ = got["y_scale"] != ref["y_scale"]
        assert 1 <= int(differ.sum()) <= 2                   # the planted scale store(s) only
        assert bool((got["y_scale"][differ] == SENTINEL).all())
    else:
        assert torch.equal(got["y"], ref["y"])


@pytest.mark.parametrize("N,d", [(100, 5120), (41, 1024)])
def test_cluster_kernel_checked_build(M, MC, synth, N, d):
    """The cluster kernel (MHC_PATH_CLUSTER) in the bounds-checked build: no check fires on a
    regular call and the results equal the regular build's; the planted out-of-range row of the
    first token's finisher store is caught and skipped, every other row written."""
    inp = synth.make_inputs(N, 4, d, seed=970 + N, device=DEV, scale_uniform=True)
    inp.pop("outliers", None)
    Wp = M.pack_weights(inp["W"])
    flags = MC.PATH_CLUSTER
    full, view = _padded_outputs(N, d, False, 2 * N + 64)
    got = _step(MC, inp, Wp, False, flags, view)
    assert MC.get_status() == MC.MHC_OK
    _padding_untouched(full, N)
    ref = _step(M, inp, Wp, False, flags, None)
    assert M.get_status() == M.MHC_OK
    for k in view:
        assert torch.equal(got[k], ref[k]), k
    check_step(got, oracle_step(inp))
    full, view = _padded_outputs(N, d, False, 2 * N + 64)
    got = _step(MC, inp, Wp, False, flags | MC.DEBUG_PLANT_OOB, view)
    assert MC.get_status() == MC.MHC_ERR_BOUNDS
    _padding_untouched(full, N)
    for k in ("pre", "post", "comb", "mixes"):
        assert bool((got[k][0].view(torch.uint8) == SENTINEL).all()), k
        assert torch.equal(got[k][1:], ref[k][1:]), k
    assert torch.equal(got["Xp"], ref["Xp"]) and torch.equal(got["y"], ref["y"])
