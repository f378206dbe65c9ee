"""The fp64 oracle against its pins (CPU only)."""

import numpy as np
import pytest

import oracle
from tests import _pins


def test_golden_hand_cases():
    _pins.pin_golden(oracle)


def test_theorem1_exact_law_equals_q():
    _pins.pin_theorem1(oracle)


def test_sequential_application_recovers_q_at_each_position():
    _pins.pin_sequential(oracle)


def test_chi_square_million_trials_v8():
    _pins.pin_chi_square(oracle, trials=1_000_000, V=8)


def test_chi_square_million_trials_v64():
    _pins.pin_chi_square(oracle, trials=1_000_000, V=64, seed=4, chunk=100_000)


def test_expected_accepted_length():
    _pins.pin_expected_length(oracle)


def test_library_special_cases():
    _pins.pin_library_special_cases(oracle)


def test_invariants():
    _pins.pin_invariants(oracle)


def test_failure_statuses():
    _pins.pin_failures(oracle)


def test_bf16_inputs_widen_exactly():
    torch = pytest.importorskip("torch")
    from synthetic import make_inputs
    from synthetic.configs import shrink, WORKLOADS

    w = shrink(WORKLOADS["c3"], B=2, V=4096)
    inp = make_inputs(w)
    r = oracle.verify_inputs(inp)
    t64 = inp["target"].to(torch.float64).numpy()
    # every bf16 value round-trips through fp64 unchanged
    assert np.array_equal(torch.from_numpy(t64).to(torch.bfloat16).view(torch.int16).numpy(),
                          inp["target"].view(torch.int16).numpy())
    assert (r.status == 0).all()
    assert ((r.n_accepted >= 0) & (r.n_accepted <= w.K)).all()


def test_temperature_is_widened_from_fp32():
    """The step takes T as fp32 (U6): 0.6 means fp32(0.6) = 0.60000002384..."""
    rng = np.random.default_rng(2)
    tl = rng.normal(0, 2.0, (1, 2, 9))
    dl = tl[:, :1] + rng.normal(0, 1.0, (1, 1, 9))
    tok = np.array([[3]])
    uni = np.array([[0.99, 0.5, 0.5]])
    r = oracle.verify(tl, dl, tok, uni, 0.6)
    from scipy.special import logsumexp

    T32 = float(np.float32(0.6))
    np.testing.assert_allclose(r.lse[0, 0], logsumexp(tl[0, 0] / T32), rtol=1e-14)
    assert abs(r.lse[0, 0] - logsumexp(tl[0, 0] / 0.6)) > 1e-9


def test_rejects_bad_temperature_and_shapes():
    tl = np.zeros((1, 2, 4))
    dl = np.zeros((1, 1, 4))
    with pytest.raises(ValueError):
        oracle.verify(tl, dl, np.zeros((1, 1)), np.zeros((1, 3)), 0.0)
    with pytest.raises(ValueError):
        oracle.verify(tl, dl, np.zeros((1, 1)), np.zeros((1, 3)), float("nan"))
    with pytest.raises(ValueError):
        oracle.verify(tl, dl, np.zeros((1, 2)), np.zeros((1, 3)), 1.0)


def test_draft_sampler_hand_cases():
    _pins.pin_draft_golden(oracle)


def test_draft_sampler_law_is_softmax():
    _pins.pin_draft_law(oracle)


def test_draft_sampler_failures():
    _pins.pin_draft_failures(oracle)


def test_draft_sampler_is_the_bonus_draw():
    _pins.pin_draft_matches_bonus(oracle)


def test_greedy_hand_cases():
    _pins.pin_greedy_golden(oracle)


def test_greedy_is_the_zero_temperature_limit():
    _pins.pin_greedy_is_zero_temperature(oracle)


def test_greedy_failures():
    _pins.pin_greedy_failures(oracle)


def test_topk_mask_hand_cases():
    _pins.pin_topk_mask_cases(oracle)


def test_topk_with_k_at_least_v_is_verify():
    _pins.pin_topk_full_is_verify(oracle)


def test_topk_with_k_one_is_greedy():
    _pins.pin_topk_one_is_greedy(oracle)


def test_topk_first_token_law_is_filtered_q():
    _pins.pin_topk_law(oracle)


def test_topk_hand_case_filters_the_draft_too():
    _pins.pin_topk_hand_case(oracle)


def test_topp_mask_hand_cases():
    _pins.pin_topp_mask_cases(oracle)


def test_topp_against_subset_enumeration():
    _pins.pin_topp_brute_force(oracle)


def test_topp_hand_case_filters_both_rows():
    _pins.pin_topp_hand_case(oracle)


def test_topp_one_is_verify():
    _pins.pin_topp_one_is_verify(oracle)


def test_topp_tiny_is_top1():
    _pins.pin_topp_tiny_is_top1(oracle)


def test_topp_first_token_law_is_filtered_q():
    _pins.pin_topp_law(oracle)


def test_topk_against_the_ranking_definition():
    _pins.pin_topk_order_property(oracle)


def test_lm_head_hand_cases():
    _pins.pin_lm_head_golden(oracle)


def test_lm_head_against_loops_and_scipy():
    _pins.pin_lm_head_brute_force(oracle)


def test_lm_head_invariances():
    _pins.pin_lm_head_invariances(oracle)
