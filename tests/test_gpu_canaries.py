"""Out-of-range writes: every output of the fused step sits inside a larger buffer filled with a
sentinel byte, with padding rows before and after the N rows the call is given; after the step
the padding must be untouched, and every input unchanged. Ragged token counts (one token, one
past a tile, several tiles with a ragged tail, one short of the full B=4, T=8192 batch) for the
bf16-y and the MXFP8-y entry points, in the automatic launch shape and in a wide-group and a
short-tile shape."""
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"
SENTINEL = 0xA5
PAD_BEFORE = 3          # rows
PAD_AFTER = 256         # rows: two full tiles past the end


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


def _padded(N, row_shape, dtype):
    """A [PAD_BEFORE + N + PAD_AFTER, *row_shape] buffer of sentinel bytes and the view of its N
    middle rows (contiguous, 16-byte aligned: every row here is a multiple of 16 bytes)."""
    full = torch.empty((PAD_BEFORE + N + PAD_AFTER, *row_shape), dtype=dtype, device=DEV)
    full.view(torch.uint8).fill_(SENTINEL)
    view = full[PAD_BEFORE:PAD_BEFORE + N]
    assert view.is_contiguous() and view.data_ptr() % 16 == 0
    return full, view


def _untouched(full, N, name):
    b = full.view(torch.uint8).reshape(full.shape[0], -1)
    before, after = b[:PAD_BEFORE], b[PAD_BEFORE + N:]
    for part, where in ((before, "before"), (after, "after")):
        bad = part != SENTINEL
        if bad.any():
            row = int(bad.any(dim=1).nonzero()[0])
            raise AssertionError(f"{name}: padding {where} the output changed (row {row} of "
                                 f"that padding, {int(bad.sum())} bytes)")


def _outputs(N, d, mx):
    rows = {"Xp": ((4, d), torch.bfloat16), "pre": ((4,), torch.float32),
            "post": ((4,), torch.float32), "comb": ((4, 4), torch.float32),
            "mixes": ((24,), torch.float32)}
    if mx:
        rows["y_codes"] = ((d,), torch.uint8)
        rows["y_scale"] = ((d // 32,), torch.uint8)
    else:
        rows["y"] = ((d,), torch.bfloat16)
    full, view = {}, {}
    for k, (shape, dt) in rows.items():
        full[k], view[k] = _padded(N, shape, dt)
    return full, view


@pytest.mark.parametrize("mx", [False, True], ids=["bf16_y", "mxfp8_y"])
@pytest.mark.parametrize("N,split,tile", [
    (1, 0, 0), (129, 0, 0), (300, 0, 0), (300, 32, 0), (300, 8, 40), (32767, 0, 0),
])
def test_no_write_outside_the_outputs(M, synth, mx, N, split, tile):
    d = 5120
    inp = synth.make_inputs(N, 4, d, seed=500 + N + split, device=DEV, scale_uniform=True)
    inp.pop("outliers", None)
    before = {k: v.clone() for k, v in inp.items()}
    flags = (M.split_flag(split) if split else 0) | (M.tile_flag(tile) if tile else 0)
    Wp = M.pack_weights(inp["W"])
    full, view = _outputs(N, d, mx)
    args = (inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], None if not mx else Wp,
            inp["scale"], inp["base"], inp["gain"])
    if mx:
        got = M.fused_step_mxfp8(*args, flags=flags, with_mixes=True, out=view)
    else:
        got = M.fused_step(*args, W_packed=Wp, flags=flags, with_mixes=True, out=view)
    assert M.get_status() == M.MHC_OK
    for k, v in view.items():
        assert got[k].data_ptr() == v.data_ptr(), k
        _untouched(full[k], N, k)
    for k, v in before.items():
        assert torch.equal(inp[k], v), f"input {k} changed"
    # the N rows themselves were written: no row of the small outputs is still all sentinel
    for k in ("pre", "post", "comb", "mixes"):
        left = (view[k].view(torch.uint8).reshape(N, -1) == SENTINEL).all(dim=1)
        assert not left.any(), f"{k}: row {int(left.nonzero()[0])} never written"
