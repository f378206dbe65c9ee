"""The scoring step's projection fused with the row statistics
(sv_lmhead_stats, tcgen05 tensor cores) against the fp64 oracle.

Tolerance: the kernel accumulates the D products of a logit in fp32, the
oracle in fp64. Each logit may differ by 2^-20 times the sum of the absolute
products, sum_d |h_d w_vd| (sixteen units of fp32 rounding on the magnitude
that the accumulation passes through); the row maximum and the log-sum-exp of
l/T may differ by the row's largest such bound over T, plus 1e-6 relative for
the fp32 exponentials of the on-chip reduction."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import speculative_sampling_verification_gb300 as sv
from synthetic import LMHEAD_WORKLOADS, make_lmhead_inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv.load_library(build=True)


def check(inp, T, rm, lse, at):
    h = inp["hidden"].cpu().to(torch.float64).numpy()
    w = inp["weight"].cpu().to(torch.float64).numpy()
    tok = inp["tokens"].cpu().numpy()
    ref = oracle.lm_head_stats(h, w, T, tok)
    bound = np.abs(h) @ np.abs(w).T * 2.0 ** -20          # per logit
    row_b = bound.max(axis=1) / np.float32(T)
    rm, lse, at = rm.cpu().numpy(), lse.cpu().numpy(), at.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(rm - ref.row_max) <= row_b), np.max(np.abs(rm - ref.row_max) - row_b)
    assert np.all(np.abs(lse - ref.lse) <= row_b + 1e-6 * np.abs(ref.lse)), \
        np.max(np.abs(lse - ref.lse) - row_b)
    has = (tok >= 0) & (tok < w.shape[0])
    assert np.all(np.isnan(at[~has]))
    n = np.nonzero(has)[0]
    assert np.all(np.abs(at[n] - ref.at[n]) <= bound[n, tok[n]]), \
        np.max(np.abs(at[n] - ref.at[n]) - bound[n, tok[n]])


SHAPES = [(1, 64, 256), (37, 128, 1000), (128, 256, 4097), (200, 1000, 2051), (300, 512, 513),
          (129, 8, 300), (256, 4096, 1536)]


@pytest.mark.parametrize("N,D,V", SHAPES)
@pytest.mark.parametrize("T", [1.0, 0.8])
def test_lmhead_stats_match_the_oracle(N, D, V, T):
    inp = make_lmhead_inputs(N, D, V, logit_std=3.0, seed=N + D + V, device=DEV)
    ws = torch.empty(sv.sv_lmhead_workspace_size(N, D, V), dtype=torch.uint8, device=DEV)
    rm, lse, at = sv.lmhead_stats(inp["hidden"], inp["weight"], inp["tokens"], T, workspace=ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) == 0
    check(inp, T, rm, lse, at)


def test_lmhead_out_of_range_tokens_and_large_logits():
    N, D, V = 64, 256, 777
    inp = make_lmhead_inputs(N, D, V, logit_std=40.0, seed=5, device=DEV)
    inp["tokens"][1] = V
    inp["tokens"][2] = V - 1
    inp["tokens"][3] = 0
    rm, lse, at = sv.lmhead_stats(inp["hidden"], inp["weight"], inp["tokens"], 0.5)
    torch.cuda.synchronize()
    check(inp, 0.5, rm, lse, at)
    assert np.isnan(at[1].item()) and not np.isnan(at[2].item())


def test_lmhead_nonfinite_row_is_reported():
    N, D, V = 40, 128, 600
    inp = make_lmhead_inputs(N, D, V, seed=9, device=DEV)
    inp["hidden"][7, 3] = float("nan")
    ws = torch.empty(sv.sv_lmhead_workspace_size(N, D, V), dtype=torch.uint8, device=DEV)
    rm, lse, at = sv.lmhead_stats(inp["hidden"], inp["weight"], inp["tokens"], 1.0, workspace=ws)
    torch.cuda.synchronize()
    assert sv.sv_read_device_status(ws) & 32
    assert np.isnan(lse[7].item()) and np.isnan(rm[7].item())
    ok = torch.ones(N, dtype=torch.bool)
    ok[7] = False
    assert torch.isfinite(lse.cpu()[ok]).all()


def test_lmhead_full_workload_sampled_rows():
    """The 576 x 8192 x 128256 workload in one call; the oracle checks a sample
    of rows (the tolerance does not depend on the sample)."""
    w = LMHEAD_WORKLOADS["lmhead-c3"]
    inp = make_lmhead_inputs(w.N, w.D, w.V, logit_std=w.logit_std, seed=w.seed, device=DEV)
    rm, lse, at = sv.lmhead_stats(inp["hidden"], inp["weight"], inp["tokens"], w.temperature)
    torch.cuda.synchronize()
    rows = torch.tensor([0, 1, 127, 128, 300, 511, 575])
    sub = {"hidden": inp["hidden"][rows.to(DEV)], "weight": inp["weight"],
           "tokens": inp["tokens"][rows.to(DEV)]}
    check(sub, w.temperature, rm[rows.to(DEV)], lse[rows.to(DEV)], at[rows.to(DEV)])
