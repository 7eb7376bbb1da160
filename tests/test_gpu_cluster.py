"""The cluster kernel of the fused step (one thread-block cluster per 40-token tile, partial sums
through distributed shared memory; MHC_PATH_CLUSTER) against the CPU oracle: every chunk count
per CTA (1..10), both cluster sizes, ragged and tiny batches, launches with more clusters than the
GPU runs at once, both readings of comb, the iteration counts, outliers with a tiny eps, in
place, its X' equal to the persistent kernel's, output canaries, the bounded-wait status path,
the automatic choice of path, and CUDA-graph capture."""
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
def synth():
    from stream_residual_fusion_gb300 import synth as s
    return s


def _run(M, inp, flags=0, **kw):
    return M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"],
                        inp["scale"], inp["base"], inp["gain"], with_mixes=True, flags=flags, **kw)


CASES = [
    # N, d, cluster size (0 = automatic for the width)
    (1, 5120, 0),            # one token: 39 idle rows
    (7, 5120, 0),
    (40, 5120, 0),           # one full tile, 10 chunks per CTA
    (41, 5120, 0),           # a second tile of one token
    (256, 5120, 0),          # the decode batch: 7 clusters, the last of 16 tokens
    (300, 5120, 0),          # 8 clusters: more than a GB300 runs at once
    (1000, 2048, 0),         # 25 clusters of 4 chunks
    (64, 512, 0),            # one chunk per CTA
    (100, 1536, 0),          # 3 chunks: the last accumulation group holds one chunk
    (50, 4608, 0),           # 9 chunks
    (200, 2560, 8),          # 8-CTA clusters, 10 chunks each
    (70, 256, 8),            # 8-CTA clusters, one chunk (the narrowest width)
    (90, 1024, 8),
]


@pytest.mark.parametrize("N,d,cl", CASES)
def test_cluster_parity(M, synth, N, d, cl):
    inp = synth.make_inputs(N, 4, d, seed=7000 + N + d + cl, device=DEV, scale_uniform=True,
                            x_stream_std=True)
    flags = M.PATH_CLUSTER | (M.split_flag(cl) if cl else 0)
    assert M.step_path(N, d, flags) == M.PATH_CLUSTER
    out = _run(M, inp, flags)
    assert M.get_status() == M.MHC_OK
    check_step(out, oracle_step(inp))


@pytest.mark.parametrize("N,d", [(256, 5120), (45, 1024)])
def test_cluster_matches_persistent_kernel(M, synth, N, d):
    """X' of the two kernels is the same bit for bit (per-element arithmetic); the mixes and
    the coefficients agree to float32 summation order."""
    inp = synth.make_inputs(N, 4, d, seed=7100 + N, device=DEV, scale_uniform=True)
    a = _run(M, inp, M.PATH_CLUSTER)
    b = _run(M, inp, M.PATH_PERSISTENT)
    assert M.get_status() == M.MHC_OK
    assert torch.equal(a["Xp"], b["Xp"])
    ya, yb = a["y"].float(), b["y"].float()
    ulp = torch.ldexp(torch.ones_like(yb), torch.frexp(yb.abs())[1] - 8)
    assert bool(((ya - yb).abs() <= ulp).all())
    for k in ("pre", "post", "comb"):
        assert float((a[k] - b[k]).abs().max()) <= 1e-5, k
    rel = ((a["mixes"] - b["mixes"]).abs().amax(1) / b["mixes"].abs().amax(1)).max()
    assert float(rel) <= 1e-5


def test_cluster_comb_row_dest_iterations_and_outliers(M, synth):
    inp = synth.make_inputs(96, 4, 5120, seed=7200, device=DEV, outlier_frac=0.05)
    out = _run(M, inp, M.PATH_CLUSTER | M.COMB_ROW_DEST, norm_eps=1e-20, hc_eps=1e-6)
    check_step(out, oracle_step(inp, norm_eps=1e-20, comb_row_dest=True))
    for iters in (1, 2, 7):
        out = _run(M, inp, M.PATH_CLUSTER, iters=iters)
        check_step(out, oracle_step(inp, iters=iters))


def test_cluster_in_place(M, synth):
    inp = synth.make_inputs(40, 4, 5120, seed=7300, device=DEV)
    ref = oracle_step(inp)
    X = inp["X"].clone()
    out = M.fused_step(X, inp["F"], inp["pre"], inp["post"], inp["comb"], inp["W"], inp["scale"],
                       inp["base"], inp["gain"], with_mixes=True, flags=M.PATH_CLUSTER, out={"Xp": X})
    assert out["Xp"].data_ptr() == X.data_ptr()
    check_step(out, ref)


@pytest.mark.parametrize("N", [1, 31, 129, 300])
def test_cluster_outputs_stay_in_bounds(M, synth, N):
    """Every output in a buffer with two sentinel rows before it and 64 after: nothing outside
    the N rows changes."""
    d = 5120
    inp = synth.make_inputs(N, 4, d, seed=7400 + N, device=DEV)
    rows = {"Xp": ((4, d), torch.bfloat16), "y": ((d,), torch.bfloat16), "pre": ((4,), torch.float32),
            "post": ((4,), torch.float32), "comb": ((4, 4), torch.float32),
            "mixes": ((24,), torch.float32)}
    full, view = {}, {}
    for k, (shape, dt) in rows.items():
        full[k] = torch.empty((2 + N + 64, *shape), dtype=dt, device=DEV)
        full[k].view(torch.uint8).fill_(SENTINEL)
        view[k] = full[k][2:2 + N]
    Wp = M.pack_weights(inp["W"])
    out = M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], None, inp["scale"],
                       inp["base"], inp["gain"], W_packed=Wp, with_mixes=True, flags=M.PATH_CLUSTER,
                       out=view)
    assert M.get_status() == M.MHC_OK
    for k, f in full.items():
        b = f.view(torch.uint8).reshape(f.shape[0], -1)
        assert bool((b[:2] == SENTINEL).all()) and bool((b[2 + N:] == SENTINEL).all()), k
    check_step(out, oracle_step(inp))


def test_cluster_bounded_wait_reports_timeout(M, synth):
    inp = synth.make_inputs(40, 4, 512, seed=7500, device=DEV)
    out = _run(M, inp, M.PATH_CLUSTER | M.DEBUG_NEVER_ARRIVE)
    assert M.get_status() == M.MHC_ERR_TIMEOUT
    check_step(out, oracle_step(inp))
    out = _run(M, inp, M.PATH_CLUSTER)
    assert M.get_status() == M.MHC_OK
    check_step(out, oracle_step(inp))


def test_automatic_path(M):
    """The cluster kernel while every tile's cluster runs at once, the persistent kernel beyond,
    and always the persistent kernel with explicit shape flags or for widths no cluster fits."""
    split, tile, groups = M.step_config(256, 5120)
    if M.step_path(256, 5120) == M.PATH_CLUSTER:
        assert (split, tile, groups) == (16, 40, 7)
    assert M.step_path(32768, 5120) == M.PATH_PERSISTENT
    assert M.step_path(256, 5120, M.split_flag(32)) == M.PATH_PERSISTENT
    assert M.step_path(256, 5120, M.PATH_PERSISTENT) == M.PATH_PERSISTENT
    assert M.step_path(8, 6144) == M.PATH_PERSISTENT            # 12 chunks per CTA: too wide
    assert M.step_path(5000, 5120, M.PATH_CLUSTER) == M.PATH_CLUSTER


@pytest.mark.parametrize("path", ["cluster", "persistent"])
def test_decode_step_in_cuda_graph(M, synth, path):
    """The packed decode step captures into a CUDA graph on either path; replays with new inputs
    copied into the captured buffers give the eager results."""
    N, d = 256, 5120
    flags = M.PATH_CLUSTER if path == "cluster" else M.PATH_PERSISTENT
    inp = synth.make_inputs(N, 4, d, seed=7600, device=DEV)
    Wp = M.pack_weights(inp["W"])
    scratch = torch.empty(M.step_scratch_bytes(d), dtype=torch.uint8, device=DEV)
    out = {"Xp": torch.empty_like(inp["X"]), "y": torch.empty(N, d, dtype=torch.bfloat16, device=DEV),
           "pre": torch.empty(N, 4, device=DEV), "post": torch.empty(N, 4, device=DEV),
           "comb": torch.empty(N, 4, 4, device=DEV)}

    def step():
        M.fused_step(inp["X"], inp["F"], inp["pre"], inp["post"], inp["comb"], None, inp["scale"],
                     inp["base"], inp["gain"], W_packed=Wp, scratch=scratch, out=out, flags=flags)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    for seed in (7601, 7602):
        new = synth.make_inputs(N, 4, d, seed=seed, device=DEV)
        for k in ("X", "F", "pre", "post", "comb"):
            inp[k].copy_(new[k])
        g.replay()
        torch.cuda.synchronize()
        assert M.get_status() == M.MHC_OK
        got = {k: v.clone() for k, v in out.items()}
        step()
        torch.cuda.synchronize()
        for k in got:
            assert torch.equal(got[k], out[k]), k
        ref = oracle_step({k: v for k, v in inp.items()})
        check_step(got, ref, with_mixes=False)
