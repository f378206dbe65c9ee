"""Mutation check of the pins: each plausible mistake, planted in a private
copy of the oracle's source on the CPU, must make at least one fast pin fail.
The real oracle is never modified."""

import importlib.util
import os
import sys
import types

import pytest

from tests import _pins

ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                          "oracle", "spec_sampling.py")

MUTATIONS = [
    ("residual sign flipped",
     "w = np.maximum(0.0, q_row - p_row)", "w = np.maximum(0.0, p_row - q_row)"),
    ("residual clamp dropped",
     "w = np.maximum(0.0, q_row - p_row)", "w = np.abs(q_row - p_row)"),
    ("ratio transposed",
     "ratio = q_at / np.where(p_at > 0, p_at, 1.0)", "ratio = p_at / np.where(q_at > 0, q_at, 1.0)"),
    ("non-strict acceptance",
     "accept = u_acc < thr", "accept = u_acc <= thr"),
    ("bonus drawn with the residual uniform",
     "uniforms[:, K], uniforms[:, K + 1])", "uniforms[:, K], uniforms[:, K])"),
    ("bonus drawn from target row K-1",
     "q_row = q[rows, j]", "q_row = q[rows, np.minimum(j, K - 1)]"),
    ("zero-residual fallback dropped",
     "w = np.where(fallback[..., None], q_row, w)", "w = w"),
    ("non-strict inverse CDF",
     "above = C > target[:, None]", "above = C >= target[:, None]"),
    ("temperature multiplies",
     "z = logits / np.float64(temperature)", "z = logits * np.float64(temperature)"),
    ("scan stops at first acceptance",
     "np.argmin(accept, axis=1)", "np.argmax(accept, axis=1)"),
    ("accepted prefix not copied",
     "out[b, : j[b]] = tokens[b, : j[b]]", "out[b, : j[b]] = idx[b]"),
    ("margin takes the farther end",
     "np.minimum(u - lo, hi - u)", "np.maximum(u - lo, hi - u)"),
    ("draft row index off by one",
     "p_row = p[rows, np.minimum(j, K - 1)]", "p_row = p[rows, np.minimum(j + 1, K - 1)]"),
    ("acceptance uses the wrong uniform",
     "u_acc = uniforms[:, :K]", "u_acc = uniforms[:, 1:K + 1]"),
    ("q(x)=0 accepts",
     "np.where(q_at > 0, 1.0, 0.0)", "np.where(q_at > 0, 1.0, 1.0)"),
    ("sampler ignores the temperature",
     "p, lse, status = temperature_softmax(logits, T)", "p, lse, status = temperature_softmax(logits, 1.0)"),
    ("sampler accepts bad uniforms",
     "status = status | np.where(u_ok, 0, STATUS_UNIFORM_RANGE)", "status = status"),
    ("sampler reports failed rows' draws",
     "return SampleResult(np.where(failed, -1, idx), status,", "return SampleResult(idx, status,"),
    ("greedy ties go to the largest id",
     "am = np.argmax(np.where(np.isnan(target), -np.inf, target), axis=-1)",
     "am = V - 1 - np.argmax(np.where(np.isnan(target), -np.inf, target)[..., ::-1], axis=-1)"),
    ("greedy emits the draft token at the mismatch",
     "out[b, j[b]] = am[b, j[b]]", "out[b, j[b]] = tokens[b, min(j[b], K - 1)]"),
    ("greedy compares with the next row's argmax",
     "match = tokens == am[:, :K]", "match = tokens == am[:, 1:]"),
    ("top-k ties go to the larger id",
     "order = np.argsort(-(row + 0.0), kind=\"stable\")",
     "order = (V - 1 - np.argsort(-(row[::-1] + 0.0), kind=\"stable\"))"),
    ("top-k keeps one too many",
     "keep = order[:k]", "keep = order[:k + 1]"),
    ("top-k filters the target only",
     "return verify(topk_mask(target, top_k), topk_mask(draft, top_k), tokens, uniforms,",
     "return verify(topk_mask(target, top_k), draft, tokens, uniforms,"),
    ("nucleus cut is strict (> p)",
     "reach = np.nonzero(c >= top_p)[0]", "reach = np.nonzero(c > top_p)[0]"),
    ("nucleus keeps one entry too few",
     "out[r, order[n:]] = -np.inf", "out[r, order[n - 1:]] = -np.inf"),
    ("nucleus ties go to the larger id",
     "order = np.argsort(-(flat[r] + 0.0), kind=\"stable\")",
     "order = (V - 1 - np.argsort(-(flat[r][::-1] + 0.0), kind=\"stable\"))"),
    ("nucleus cut before the temperature",
     "q, _, st = temperature_softmax(flat, temperature)", "q, _, st = temperature_softmax(flat, 1.0)"),
    ("lm-head gathers a neighbouring column",
     "at[ok] = logits[np.arange(N)[ok], tok[ok]]", "at[ok] = logits[np.arange(N)[ok], tok[ok] - 1]"),
    ("lm-head statistics ignore the temperature",
     "    z = logits / T\n    m = np.max(z, axis=-1)", "    z = logits\n    m = np.max(z, axis=-1)"),
    ("lm-head maximum over the whole batch",
     "    m = np.max(z, axis=-1)\n    lse", "    m = np.max(z) + 0 * z[:, 0]\n    lse"),
    ("lm-head gathers z instead of l",
     "at[ok] = logits[np.arange(N)[ok], tok[ok]]", "at[ok] = z[np.arange(N)[ok], tok[ok]]"),
    ("lm-head weight used untransposed (square shapes hide it)",
     "logits = np.matmul(h, w.T)", "logits = np.matmul(h, w.reshape(w.shape[1], w.shape[0]))"),
    ("nucleus filters the target only",
     "res = verify(tm, dm, tokens, uniforms, temperature)", "res = verify(tm, draft, tokens, uniforms, temperature)"),
]


def _mutant(old: str, new: str) -> types.ModuleType:
    src = open(ORACLE_SRC).read()
    assert src.count(old) >= 1, old
    src = src.replace(old, new)
    name = "oracle_mutant"
    spec = importlib.util.spec_from_loader(name, loader=None)
    mod = importlib.util.module_from_spec(spec)
    sys.modules[name] = mod
    try:
        exec(compile(src, ORACLE_SRC + " (mutant)", "exec"), mod.__dict__)
    finally:
        del sys.modules[name]
    return mod


@pytest.mark.parametrize("label,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(label, old, new):
    mod = _mutant(old, new)
    caught = []
    for pin in _pins.FAST_PINS:
        try:
            pin(mod)
        except Exception as e:  # AssertionError or a crash both count as caught
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"no pin caught: {label}"


def test_unmutated_copy_passes_all_fast_pins():
    mod = _mutant("import numpy as np", "import numpy as np")
    for pin in _pins.FAST_PINS:
        pin(mod)
