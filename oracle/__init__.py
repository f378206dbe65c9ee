"""fp64 CPU oracle of the speculative-sampling verification step.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.
"""

from .spec_sampling import (  # noqa: F401
    OracleResult,
    SampleResult,
    GreedyResult,
    NucleusResult,
    STATUS_EMPTY_ROW,
    STATUS_NONFINITE,
    STATUS_OK,
    STATUS_TOKEN_RANGE,
    STATUS_UNIFORM_RANGE,
    acceptance_thresholds,
    draft_sample,
    first_rejection,
    inverse_cdf,
    residual_weights,
    temperature_softmax,
    verify,
    verify_greedy,
    verify_topk,
    topk_mask,
    topp_mask,
    verify_topp,
    verify_inputs,
    LMHeadStats,
    lm_head_stats,
)
