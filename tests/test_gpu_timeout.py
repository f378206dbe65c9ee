"""Failure detection without a GPU fault: a draw CTA of the fused kernel
waits for a flag that nothing sets (the plans' release is withheld by a test
hook); its bounded wait runs out, the call reports SV_DEV_TIMEOUT, and the
context stays usable for the next, correct call."""

from __future__ import annotations

import time

import pytest
import torch

import oracle
import speculative_sampling_verification_gb300 as sv
from synthetic import get_workload, make_inputs
from tests import _parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def test_withheld_plans_time_out_and_the_context_survives():
    w = get_workload("c1")
    inp = make_inputs(w, step=7)
    args = [inp[k].to(DEV) for k in ("target", "draft", "tokens", "uniforms")]
    ws = sv.new_workspace(w.B, w.K, w.V, sv.SV_F32, DEV)
    out = torch.full((w.B, w.K + 1), 12345, dtype=torch.int32, device=DEV)
    nacc = torch.empty(w.B, dtype=torch.int32, device=DEV)
    sv.sv_force_path(2)
    try:
        sv.sv_test_withhold_plans(True)
        t0 = time.perf_counter()
        assert sv.spec_verify(*args, inp["temperature"], out, nacc, ws) == 0
        status = sv.sv_read_device_status(ws)
        waited = time.perf_counter() - t0
        assert status & 256, status            # SV_DEV_TIMEOUT
        assert 0.15 < waited < 5.0, waited     # the 200 ms limit, not a hang
        # The draw never ran: its position holds -1 (not a stale value), the
        # accepted prefix and the padding are in place.
        o, n = out.cpu().numpy()[0], int(nacc.cpu().numpy()[0])
        assert 0 <= n <= w.K, n
        assert o[n] == -1, o
        assert (o[:n] == inp["tokens"].numpy()[0, :n]).all(), o
        assert (o[n + 1:] == -1).all(), o
        sv.sv_test_withhold_plans(False)
        assert sv.spec_verify(*args, inp["temperature"], out, nacc, ws) == 0
        assert sv.sv_read_device_status(ws) == 0
        ref = oracle.verify_inputs(inp)
        _parity.compare(out.cpu().numpy(), nacc.cpu().numpy(), ref,
                        inp["tokens"].numpy()).assert_ok()
    finally:
        sv.sv_test_withhold_plans(False)
        sv.sv_force_path(0)
