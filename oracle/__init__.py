"""Float64 CPU oracle of the speculative-sampling verification step.

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and
bench.py's CPU-baseline leg, never by the product path.
"""
from .spec_oracle import (  # noqa: F401
    BOUNDARY_EPS, Z_FLOOR, STAT_KEYS, widen, row_is_valid, softmax_t, inverse_cdf, draw_candidates, verify_row,
    draw_boundary_probability, accept_boundary_probability,
    greedy_row, stats_position, topk_threshold, topp_threshold, apply_threshold, verify_sample, verify_greedy, accept_stats, sample_rows, exact_joint,
    expected_tokens, walltime_improvement, operations_factor, optimal_gamma, alpha_from_beta,
)
