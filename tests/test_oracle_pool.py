"""The chunked whole-batch comparison (tests/oracle_pool.py) on the CPU: outputs the oracle
itself produced pass, and one planted difference in any output fails, naming its chunk."""
import numpy as np
import pytest
import torch

import oracle as O
from stream_residual_fusion_gb300 import synth
from tests.oracle_pool import full_parity


def _oracle_outputs(inp):
    a = O.inputs_to_f64(inp)
    r = O.fused_step(a["X"], a["F"], a["pre"], a["post"], a["comb"], a["W"], a["scale"],
                     a["base"], a["gain"])
    out = {k: torch.from_numpy(r[k]).to(torch.bfloat16) for k in ("Xp", "y")}
    out.update({k: torch.from_numpy(r[k]).float() for k in ("pre", "post", "comb", "mixes")})
    return out


@pytest.fixture(scope="module")
def case():
    inp = synth.make_inputs(70, 4, 256, seed=5, scale_uniform=True, x_stream_std=True)
    inp.pop("outliers", None)
    return inp, _oracle_outputs(inp)


def test_full_parity_accepts_the_oracle_itself(case):
    inp, out = case
    assert full_parity(inp, out, chunk=16, workers=3) == 70


@pytest.mark.parametrize("key,token", [("Xp", 37), ("y", 69), ("comb", 0), ("mixes", 50)])
def test_full_parity_names_the_chunk_with_a_planted_difference(case, key, token):
    inp, out = case
    bad = {k: v.clone() for k, v in out.items()}
    if key in ("Xp", "y"):
        flat = bad[key][token].view(-1)
        flat[3] = flat[3] * 1.5 + 1.0                 # far beyond any tolerance
    else:
        bad[key][token].view(-1)[2] += 1e-3
    lo = token // 16 * 16
    with pytest.raises(AssertionError, match=rf"tokens \[{lo}, {min(70, lo + 16)}\)"):
        full_parity(inp, bad, chunk=16, workers=3)


def test_full_parity_mxfp8_outputs():
    """y as MXFP8: the oracle's own encoding of its y passes; a changed scale code fails."""
    from oracle import mx
    inp = synth.make_inputs(40, 4, 256, seed=6)
    inp.pop("outliers", None)
    out = _oracle_outputs(inp)
    codes, scales = mx.mxfp8_quantize(out.pop("y").double().numpy())
    out["y_codes"] = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    out["y_scale"] = torch.from_numpy(np.ascontiguousarray(scales, dtype=np.uint8))
    assert full_parity(inp, out, chunk=16, workers=2) == 40
    out["y_scale"][33, 1] += 3
    with pytest.raises(AssertionError, match=r"tokens \[32, 40\)"):
        full_parity(inp, out, chunk=16, workers=2)
