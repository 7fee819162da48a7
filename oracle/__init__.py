"""CPU oracle for the DSpark draft-head round (TEST INFRASTRUCTURE).

A plain float64 numpy statement of what the hot path computes, written from the
method's pages and pinned by tests/ against closed forms, brute force and
published known-answer vectors.  Only tests/, __graft_entry__.smoke() and
bench.py's CPU-baseline leg may import it.  It shares no code with the CUDA
library and never imports it.
"""
from . import philox  # noqa: F401
from .dspark import (  # noqa: F401
    BREAK, FIXED_K, UNCONSTRAINED, base_logits, confidence_label, draft_round,
    fused_draft, global_order, markov_draft, rnn_draft, round_bf16, schedule, schedule_async,
    survival,
    expected_calibration_error, sts_fit, theta_curve, theta_of_lengths, verify,
)
