"""Whole-batch parity against the fp64 oracle (tests/parity_at_scale.py) at a
bounded size: every sequence of every step of the 8x4x32000, 64x8x128256 and
256x4x256000 workloads and of the 20 acceptance-sweep cells, verified on the
GPU and by the oracle on the host cores. The full-size run (at least 1e5
decisions per workload) is the module's command line."""

from __future__ import annotations

import pytest

from tests import parity_at_scale

pytestmark = pytest.mark.gpu


def test_whole_batches_match_the_oracle():
    s = parity_at_scale.run("c2,c3,c4,sweep", min_decisions=3000, min_decisions_cell=300)
    for r in s["workloads"]:
        assert r["unexcused_differences"] == 0, r
        assert r["device_status"] == 0, r
        assert not any(r["intermediates"]["over_tolerance"].values()), r
        assert r["decisions"] >= (3000 if "sweep" not in r["workload"] else 300), r
    t = s["totals"]
    # the excused-difference bar over all decisions (one allowed below 1e5 decisions)
    assert t["excused_differences"] <= max(1, parity_at_scale.MAX_EXCUSED_RATE
                                           * t["decisions"]), t


@pytest.mark.parametrize("op", ["topk", "topp", "greedy", "sample"])
def test_other_paths_over_whole_batches_match_the_oracle(op):
    """The filtered verifications, greedy mode and the draft sampler over whole
    batches of the 8x4x32000 workload."""
    s = parity_at_scale.run("c2", min_decisions=2000, op=op)
    for r in s["workloads"]:
        assert r["unexcused_differences"] == 0, r
        assert r["decisions"] >= 2000, r
        if op == "topp":
            assert r["cut_unexcused_rows"] == 0, r
    t = s["totals"]
    assert t["excused_differences"] <= max(1, parity_at_scale.MAX_EXCUSED_RATE
                                           * t["decisions"]), t
