"""Seeded synthetic inputs for the speculative-sampling verification step.

This package only draws random numbers in the shapes and distributions of the
workloads; it holds none of the verification arithmetic (no normalisation, no
acceptance ratio, no residual). Both the fp64 oracle and the CUDA library are
fed from here, and neither imports the other.
"""

from .configs import (LMHEAD_WORKLOADS, SWEEP_K, SWEEP_NOISE, WORKLOADS, LMHeadWorkload, Workload,
                      get_workload, sweep_workload)
from .generate import (DTYPES, make_batch, make_inputs, make_lmhead_inputs, make_sequence,
                       make_topk_inputs, make_topp_inputs, topk_draft_tokens, topp_draft_tokens)

__all__ = [
    "WORKLOADS",
    "SWEEP_K",
    "SWEEP_NOISE",
    "Workload",
    "sweep_workload",
    "get_workload",
    "make_inputs",
    "make_batch",
    "make_lmhead_inputs",
    "LMHeadWorkload",
    "LMHEAD_WORKLOADS",
    "make_sequence",
    "make_topk_inputs",
    "topk_draft_tokens",
    "make_topp_inputs",
    "topp_draft_tokens",
    "DTYPES",
]
