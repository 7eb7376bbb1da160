"""Host-side pieces of bench.py (no GPU): the algorithmic byte counts it reports, checked against
the oracle's pinned traffic counts, the lookup of the committed ncu traffic summary, and which
workloads are timed with L2 flushed."""
import pytest

import bench
import oracle as O


def test_algorithmic_bytes_match_the_traffic_counts():
    # the oracle counts bf16 elements per token (pinned by tests/golden/traffic.txt)
    fused = 2 * O.traffic_per_token(O.fused_traffic_steps(4, 5120))
    unfused = 2 * O.traffic_per_token(O.unfused_traffic_steps(4, 5120))
    assert bench.STREAM_BYTES_PER_TOKEN == fused == 102400
    # previous p, u, C in and new p, u, C out: 2 x (16 + 16 + 64) bytes
    assert bench.SMALL_BYTES_PER_TOKEN == 192
    assert bench.algorithmic_bytes(32768) == 32768 * 102592 + 640 * 5120 + 4 * 5120
    # the unfused chain: twice the stream traffic, the same small vectors
    assert sum(bench.UNFUSED_BYTES_PER_TOKEN.values()) == unfused + 192 == 204992
    # MXFP8 y: y's 10,240 bf16 bytes become 5,120 code bytes and 160 scale bytes
    assert bench.MXFP8_BYTES_PER_TOKEN == 102592 - 10240 + 5120 + 160 == 97632


def test_ncu_traffic_lookup(tmp_path, monkeypatch):
    """The bench takes DRAM bytes per token from the committed summary only when it names the
    current kernel sources."""
    current = bench.kernel_source_hash()
    prof = tmp_path / "profiles"
    prof.mkdir()
    summary = prof / "fused_step_prefill_ncu.md"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda: current)
    summary.write_text(f"kernel source hash: `{current}`\n\ndram bytes per token: 100000\n")
    assert bench.ncu_traffic(10) == 1_000_000
    summary.write_text("kernel source hash: `0123456789abcdef`\n\ndram bytes per token: 100000\n")
    assert bench.ncu_traffic(10) is None
    summary.unlink()
    assert bench.ncu_traffic(10) is None


def test_percentile_interpolates_between_ranks():
    xs = [float(i) for i in range(1, 201)]            # 200 launches: 1.0 .. 200.0 ms
    assert bench.percentile(xs, 50) == pytest.approx(100.5)
    assert bench.percentile(xs, 99) == pytest.approx(198.01)
    assert bench.percentile(xs, 0) == 1.0 and bench.percentile(xs, 100) == 200.0
    assert bench.percentile([3.0], 95) == 3.0 and bench.percentile([], 50) is None


def test_small_workloads_are_timed_with_l2_flushed():
    """The two batches whose streams fit in L2 (8 and 256 tokens) flush it before every timed
    step and say so in config.l2; the prefill batches are larger than L2 and say that."""
    from stream_residual_fusion_gb300 import synth
    flushed = {name: bench.fits_in_l2(w.N) for name, w in synth.WORKLOADS.items()}
    assert flushed == {"tiny": True, "decode256": True, "prefill4k": False, "prefill32k": False,
                       "prefill128k": False}
    for name, w in synth.WORKLOADS.items():
        l2 = bench.workload_config(w, w.N, w.N)["l2"]
        assert l2.startswith("inputs smaller than L2: a 256 MB write flushes L2") == flushed[name], name
        assert l2.startswith("inputs larger than L2") == (not flushed[name]), name
