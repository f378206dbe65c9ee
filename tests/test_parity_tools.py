"""The comparison rules of tests/parity_at_scale.py for greedy mode and the
draft sampler, on hand-made oracle results: identical outputs pass, a draw that
differs within the margin of its CDF ends is tolerated and counted, any other
difference is a failure, and failed rows must draw -1."""

from __future__ import annotations

import numpy as np

import oracle
from tests import _parity, parity_at_scale as pas


def _sample_ref(tokens, status, margin):
    n = len(tokens)
    return oracle.SampleResult(tokens=np.asarray(tokens, np.int64), status=np.asarray(status, np.int64),
                               sample_margin=np.asarray(margin, float), sample_prob=np.full(n, 0.5),
                               lse=np.zeros(n))


def test_sample_identical_draws_pass_and_count():
    ref = _sample_ref([3, 7, -1], [0, 0, 32], [0.1, 5e-7, np.nan])
    rep = pas.compare_sample(np.array([3, 7, -1]), ref)
    assert (rep.sequences, rep.decisions, rep.near_threshold, rep.excused) == (3, 2, 1, 0)
    assert not rep.failures


def test_sample_difference_within_the_margin_is_tolerated():
    ref = _sample_ref([3, 7], [0, 0], [0.1, 0.5 * _parity.MARGIN])
    rep = pas.compare_sample(np.array([3, 8]), ref)
    assert rep.excused == 1 and not rep.failures


def test_sample_difference_outside_the_margin_fails():
    ref = _sample_ref([3, 7], [0, 0], [0.1, 2 * _parity.MARGIN])
    rep = pas.compare_sample(np.array([3, 8]), ref)
    assert rep.excused == 0 and len(rep.failures) == 1


def test_sample_failed_row_must_draw_minus_one():
    ref = _sample_ref([3, -1], [0, 32], [0.1, np.nan])
    assert len(pas.compare_sample(np.array([3, 5]), ref).failures) == 1
    assert not pas.compare_sample(np.array([3, -1]), ref).failures


def _greedy_ref(out, nacc, status):
    out = np.asarray(out, np.int64)
    return oracle.GreedyResult(out_tokens=out, n_accepted=np.asarray(nacc, np.int64),
                               status=np.asarray(status, np.int64), argmax=out.copy())


def test_greedy_identical_passes_and_counts_comparisons():
    ref = _greedy_ref([[1, 2, -1], [-1, -1, -1]], [1, -1], [0, 32])
    rep = pas.compare_greedy(ref.out_tokens.copy(), ref.n_accepted.copy(), ref)
    assert rep.decisions == 2 and not rep.failures


def test_greedy_any_difference_fails():
    ref = _greedy_ref([[1, 2, -1], [4, 5, 6]], [1, 2], [0, 0])
    out = ref.out_tokens.copy()
    out[1, 2] = 9
    assert len(pas.compare_greedy(out, ref.n_accepted.copy(), ref).failures) == 1
    nacc = ref.n_accepted.copy()
    nacc[0] = 0
    assert len(pas.compare_greedy(ref.out_tokens.copy(), nacc, ref).failures) == 1
