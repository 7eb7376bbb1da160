"""CPU oracle for the single-pass mHC step -- TEST INFRASTRUCTURE, not part of the product.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference leg may import this
package. The CUDA library never links, loads or calls it, and it shares no code with the CUDA path.

Pages followed (cited by title and section throughout):
  * "DeepSeek V4.1 · Stream weights for the feed-forward" -- sections "Why", "All 5 steps",
    "Parameters" (table "Exact per-instance accounting") and "Code" (excerpts of Block.__init__,
    hc_mixes / hc_pre / hc_post, and the hc_split_sinkhorn TileLang kernel).
  * "DeepSeek V4.1 · MoE RMSNorm" -- the RMSNorm formula block and "Code" (RMSNorm, Block.forward).
  * "2A · Single-Pass mHC" -- section 3 "Giải pháp" (Sinkhorn rounds) and section 4 "Profiling"
    (the [[3,1],[1,1]] hand check and the 1e-6 float64 criterion).

mx.py holds the MXFP8 encoding of y (a format the pages leave open; the reading taken is stated
there). backward.py holds the gradients of the step (the pages define no backward pass; the
reading taken -- reverse-mode differentiation of the forward code with the bf16 casts passed
straight through -- is stated there).

Every function is pinned by tests under tests/ (tests/test_oracle_*.py); nothing here is
"parity unpinned".
"""
from .mhc import (  # noqa: F401
    bf16_round, fl32, hc_post, hc_pre, hc_mixes_scores, hc_split, sinkhorn, sinkhorn_plain,
    hc_mixes, rmsnorm, fused_step, parameter_counts, traffic_per_token, unfused_traffic_steps,
    fused_traffic_steps, inputs_to_f64,
)
