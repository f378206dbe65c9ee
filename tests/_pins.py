"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Each pin takes the oracle module as an argument so that the same checks can be
run against deliberately broken copies of it (tests/test_oracle_mutations.py):
a plausible mistake anywhere in the oracle must make at least one pin fail.

None of these checks re-types the oracle's own formulas. They use
* the hand-worked cases in tests/golden/hand_cases.json;
* Theorem 1 of "Accelerating Large Language Model Decoding with Speculative
  Sampling" (Supplementary Materials, Proofs; card §4.2): the emitted token of
  one step is distributed exactly as q. The oracle is treated as a black box
  whose output is piecewise constant in each uniform; the breakpoints are
  located by bisection and the law is integrated exactly;
* the acceptance probability sum_x min(p(x), q(x)) from the same proof;
* library routines (scipy softmax / logsumexp, numpy searchsorted) for the
  special cases that reduce to them;
* invariants (1..K+1 emitted tokens, accepted prefix equals the drafts,
  exact temperature rescaling).
"""

from __future__ import annotations

import json
import os

import numpy as np
from scipy.special import logsumexp, softmax
from scipy.stats import chi2

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
GOLDEN = os.path.join(GOLDEN_DIR, "hand_cases.json")


# ---------------------------------------------------------------- helpers

def probs_to_logits(probs) -> np.ndarray:
    """ln(prob) rounded to fp32 (zero probability -> -inf), widened back to fp64."""
    p = np.asarray(probs, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(p).astype(np.float32).astype(np.float64)


def load_golden():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def run_fixed_rows(O, tl, dl, tokens, uniforms, T):
    """Run the oracle on n sequences that share the rows tl [K+1,V], dl [K,V]."""
    n = len(tokens)
    tl_b = np.broadcast_to(tl, (n,) + tl.shape)
    dl_b = np.broadcast_to(dl, (n,) + dl.shape)
    return O.verify(tl_b, dl_b, np.asarray(tokens), np.asarray(uniforms, dtype=np.float64), T)


def sup_true(pred, n, iters=64):
    """For n monotone predicates (true on [0, a), false on [a, 1]) return each a.
    A predicate already true at 1 gives 1; one false at 0 gives 0."""
    lo = np.zeros(n)
    hi = np.ones(n)
    t_hi = pred(hi.copy())
    t_lo = pred(lo.copy())
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        t = pred(mid)
        lo = np.where(t, mid, lo)
        hi = np.where(t, hi, mid)
    return np.where(t_hi, 1.0, np.where(t_lo, hi, 0.0))


def accept_measure(O, tl, dl, pos, prefix, T):
    """Lebesgue measure of {u_pos : draft x at position `pos` is accepted}, for
    every candidate x, with the drafts before `pos` fixed to `prefix` and
    accepted (their uniforms are 0). Returns an array over x."""
    K = dl.shape[0]
    V = tl.shape[1]
    xs = np.arange(V)

    def pred(u):
        toks = np.zeros((V, K), dtype=np.int64)
        toks[:, :pos] = prefix
        toks[:, pos] = xs
        uni = np.zeros((V, K + 2))
        uni[:, pos] = u
        uni[:, pos + 1:K] = 1.0   # later drafts, if any, are rejected; irrelevant here
        r = run_fixed_rows(O, tl, dl, toks, uni, T)
        return r.n_accepted > pos

    return sup_true(pred, V)


def draw_measure(O, tl, dl, pos, prefix, T, slot, rejected_token=None):
    """Measure of {u_slot : emitted token at `pos` == y} for every y.

    With `rejected_token` set, draft x = rejected_token sits at `pos` and its
    test is forced to fail (u_pos = 1.0, rejecting whenever the threshold is
    at most 1), so the residual draw is measured; without it, all K drafts
    are the prefix and accepted, so the bonus draw is measured."""
    K = dl.shape[0]
    V = tl.shape[1]
    ys = np.arange(V)

    def pred(u):
        toks = np.zeros((V, K), dtype=np.int64)
        uni = np.zeros((V, K + 2))
        toks[:, :pos] = prefix
        if rejected_token is not None:
            toks[:, pos] = rejected_token
            uni[:, pos] = 1.0
        uni[:, slot] = u
        r = run_fixed_rows(O, tl, dl, toks, uni, T)
        return r.out_tokens[:, pos] <= ys

    F = sup_true(pred, V)
    return np.diff(np.concatenate([[0.0], F]))


def step_law(O, tl, dl, pos, prefix, T):
    """Exact law of the token emitted at position `pos`, given that the drafts
    in `prefix` were accepted: sum_x p(x) [a(x) 1{y=x} + (1-a(x)) m_x(y)]."""
    K = dl.shape[0]
    V = tl.shape[1]
    p = softmax(dl[pos] / T)
    a = accept_measure(O, tl, dl, pos, prefix, T)
    law = p * a
    for x in range(V):
        if p[x] == 0.0 or a[x] == 1.0:
            continue
        m = draw_measure(O, tl, dl, pos, prefix, T, slot=K, rejected_token=x)
        law = law + p[x] * (1.0 - a[x]) * m
    return law, a, p


# ---------------------------------------------------------------- pins

def pin_golden(O):
    """Hand-worked cases (tests/golden/hand_cases.json)."""
    for c in load_golden():
        tl = probs_to_logits(c["target_probs"])[None]
        dl = probs_to_logits(c["draft_probs"])[None]
        tok = np.array([c["tokens"]])
        uni = np.array([c["uniforms"]], dtype=np.float32).astype(np.float64)
        r = O.verify(tl, dl, tok, uni, 1.0)
        name = c["name"]
        assert r.status[0] == 0, name
        assert list(r.out_tokens[0]) == c["expected_out"], (name, r.out_tokens[0])
        assert r.n_accepted[0] == c["expected_n_accepted"], name
        assert bool(r.residual_fallback[0]) == c["expected_fallback"], name
        np.testing.assert_allclose(r.thresholds[0], c["expected_thresholds"], atol=1e-6,
                                   err_msg=name)
        exp_r = np.array([float(v) for v in c["expected_ratios"]])
        np.testing.assert_allclose(r.ratios[0], exp_r, rtol=1e-6, err_msg=name)
        # Logits are ln(prob) at T = 1, so each row's maximum is the log of its
        # largest probability (the probabilities of a row sum to one).
        rows = list(c["target_probs"]) + list(c["draft_probs"])
        np.testing.assert_allclose(r.row_max[0], [np.log(max(pr)) for pr in rows], atol=1e-6,
                                   err_msg=name)
        exp_m = np.array([np.nan if v is None else v for v in c["expected_accept_margins"]])
        np.testing.assert_allclose(r.accept_margin[0], exp_m, atol=1e-6, err_msg=name)
        np.testing.assert_allclose(r.sample_margin[0], c["expected_sample_margin"], atol=1e-6,
                                   err_msg=name)
        np.testing.assert_allclose(r.sample_prob[0], c["expected_sample_prob"], atol=1e-6,
                                   err_msg=name)


def theorem1_cases():
    rng = np.random.default_rng(7)
    V = 8
    base_t = rng.normal(0, 2.0, (2, V))
    base_d = base_t[:1] + rng.normal(0, 1.5, (1, V))
    masked_t = base_t.copy()
    masked_t[0, 3] = -np.inf           # q(3) = 0
    masked_d = base_d.copy()
    masked_d[0, 5] = -np.inf           # p(5) = 0: never drafted
    far_d = rng.normal(0, 3.0, (1, V))
    return [
        ("random", base_t, base_d, 1.0),
        ("temperature-0.6875", base_t, base_d, 0.6875),
        ("temperature-1.875", base_t, base_d, 1.875),
        ("masked", masked_t, masked_d, 1.0),
        ("q-equals-p", base_t, base_t[:1].copy(), 1.0),
        ("far-draft", base_t, far_d, 1.0),
    ]


def pin_theorem1(O):
    """Theorem 1: one step emits x with probability exactly q(x) (to 1e-12),
    and the acceptance probability is sum_x min(p(x), q(x))."""
    for name, tl, dl, T in theorem1_cases():
        law, a, p = step_law(O, tl, dl, 0, np.zeros(0, dtype=np.int64), T)
        q = softmax(tl[0] / T)
        np.testing.assert_allclose(law, q, rtol=0, atol=1e-12, err_msg=name)
        assert abs(np.sum(p * a) - np.sum(np.minimum(p, q))) < 1e-12, name


def pin_sequential(O):
    """Applying the rule position after position recovers the target
    distribution at each position (card, §4.2): K=2, V=4, exact."""
    rng = np.random.default_rng(11)
    V, K, T = 4, 2, 1.0
    tl = rng.normal(0, 1.5, (K + 1, V))
    dl = tl[:K] + rng.normal(0, 1.0, (K, V))
    q = softmax(tl / T, axis=-1)
    law0, _, _ = step_law(O, tl, dl, 0, np.zeros(0, dtype=np.int64), T)
    np.testing.assert_allclose(law0, q[0], atol=1e-12)
    for x0 in range(V):
        law1, _, _ = step_law(O, tl, dl, 1, np.array([x0]), T)
        np.testing.assert_allclose(law1, q[1], atol=1e-12, err_msg=f"x0={x0}")
    # both drafts accepted: the bonus draw at position K follows q_K
    for prefix in ([0, 1], [3, 2]):
        m = draw_measure(O, tl, dl, K, np.array(prefix), T, slot=K + 1)
        np.testing.assert_allclose(m, q[K], atol=1e-12, err_msg=f"bonus {prefix}")


def pin_chi_square(O, trials=1_000_000, V=8, seed=3, chunk=200_000):
    """Seeded trials of one step (K=1): the first emitted token against q, and
    the bonus token (when the draft is accepted) against q_1; Pearson chi^2
    p-values above 1e-3. Drafts are drawn by Gumbel-max, so no softmax of
    the oracle's is used to make them."""
    rng = np.random.default_rng(seed)
    tl = rng.normal(0, 2.0, (2, V))
    dl = tl[:1] + rng.normal(0, 1.0, (1, V))
    T = 1.0
    counts0 = np.zeros(V)
    counts1 = np.zeros(V)
    n_acc = 0
    for s in range(0, trials, chunk):
        n = min(chunk, trials - s)
        g = rng.gumbel(size=(n, V))
        toks = np.argmax(dl[0] / T + g, axis=1)[:, None]
        uni = rng.random((n, 3)).astype(np.float32).astype(np.float64)
        r = run_fixed_rows(O, tl, dl, toks, uni, T)
        counts0 += np.bincount(r.out_tokens[:, 0], minlength=V)
        acc = r.n_accepted == 1
        counts1 += np.bincount(r.out_tokens[acc, 1], minlength=V)
        n_acc += int(acc.sum())
    q = softmax(tl / T, axis=-1)
    p = softmax(dl / T, axis=-1)
    for counts, qq, n in ((counts0, q[0], trials), (counts1, q[1], n_acc)):
        exp = n * qq
        stat = np.sum((counts - exp) ** 2 / exp)
        pval = chi2.sf(stat, V - 1)
        assert pval > 1e-3, (stat, pval)
    # acceptance rate against sum min(p, q) (binomial, 5 sigma)
    beta = np.sum(np.minimum(p[0], q[0]))
    sd = np.sqrt(beta * (1 - beta) / trials)
    assert abs(n_acc / trials - beta) < 5 * sd, (n_acc / trials, beta)


def pin_expected_length(O, n=200_000, seed=5):
    """Mean accepted count over independent positions: E[n] = sum_k prod_{t<k} beta_t,
    beta_t = sum_x min(p_t, q_t); Monte Carlo within 5 standard errors."""
    rng = np.random.default_rng(seed)
    V, K, T = 16, 4, 1.0
    tl = rng.normal(0, 2.0, (K + 1, V))
    dl = tl[:K] + rng.normal(0, 0.8, (K, V))
    q = softmax(tl / T, axis=-1)
    p = softmax(dl / T, axis=-1)
    beta = np.sum(np.minimum(p, q[:K]), axis=-1)
    expect = sum(np.prod(beta[:k]) for k in range(1, K + 1))
    g = rng.gumbel(size=(n, K, V))
    toks = np.argmax(dl[None] / T + g, axis=-1)
    uni = rng.random((n, K + 2))
    r = run_fixed_rows(O, tl, dl, toks, uni, T)
    mean = r.n_accepted.mean()
    se = r.n_accepted.std() / np.sqrt(n)
    assert abs(mean - expect) < 5 * se, (mean, expect, se)


def pin_library_special_cases(O):
    """(i) the log-sum-exp of every row against scipy's logsumexp in fp64;
    (ii) p == q: every draft is accepted and the bonus token equals
    numpy.searchsorted over the CDF of q_K (side='right')."""
    rng = np.random.default_rng(13)
    B, K, V, T = 5, 3, 257, 0.9375
    tl = rng.normal(0, 3.0, (B, K + 1, V))
    tl[0, 1, :100] = -np.inf
    dl = tl[:, :K] + rng.normal(0, 0.5, (B, K, V))
    toks = rng.integers(0, V, (B, K))
    uni = rng.random((B, K + 2))
    r = O.verify(tl, dl, toks, uni, T)
    ref = np.concatenate([logsumexp(tl / T, axis=-1), logsumexp(dl / T, axis=-1)], axis=1)
    np.testing.assert_allclose(r.lse, ref, rtol=1e-12)

    same = tl[:, :K].copy()
    toks2 = np.argmax(same / T + rng.gumbel(size=same.shape), axis=-1)
    uni2 = rng.random((B, K + 2)) * 0.999
    r2 = O.verify(tl, same, toks2, uni2, T)
    assert (r2.n_accepted == K).all()
    for b in range(B):
        qk = softmax(tl[b, K] / T)
        cdf = np.cumsum(qk)
        want = int(np.searchsorted(cdf, uni2[b, K + 1] * cdf[-1], side="right"))
        assert r2.out_tokens[b, K] == want
        assert list(r2.out_tokens[b, :K]) == list(toks2[b])


def pin_invariants(O):
    """Emission count in [1, K+1], accepted prefix equals the drafts, the
    sampled token has positive weight in the distribution it came from, -1
    padding, and exact invariance under (l, T) -> (2l, 2T)."""
    rng = np.random.default_rng(17)
    for K, V, noise in ((1, 50, 0.3), (4, 300, 1.0), (7, 33, 2.5)):
        B, T = 64, 1.0
        tl = rng.normal(0, 2.0, (B, K + 1, V))
        dl = tl[:, :K] + rng.normal(0, noise, (B, K, V))
        toks = np.argmax(dl / T + rng.gumbel(size=dl.shape), axis=-1)
        uni = rng.random((B, K + 2))
        r = O.verify(tl, dl, toks, uni, T)
        q = softmax(tl / T, axis=-1)
        p = softmax(dl / T, axis=-1)
        assert (r.status == 0).all()
        n = r.n_accepted
        assert ((n >= 0) & (n <= K)).all()
        for b in range(B):
            j = n[b]
            assert list(r.out_tokens[b, :j]) == list(toks[b, :j])
            assert (r.out_tokens[b, j + 1:] == -1).all()
            y = r.out_tokens[b, j]
            if j < K and not r.residual_fallback[b]:
                assert q[b, j, y] > p[b, j, y]
            else:
                assert q[b, j, y] > 0
        r2 = O.verify(2.0 * tl, 2.0 * dl, toks, uni, 2.0 * T)
        assert (r2.out_tokens == r.out_tokens).all()
        assert (r2.n_accepted == r.n_accepted).all()


def pin_failures(O):
    """Failed sequences: -1 outputs with the right status bit; others untouched."""
    rng = np.random.default_rng(19)
    B, K, V = 6, 2, 20
    tl = rng.normal(0, 1.0, (B, K + 1, V))
    dl = tl[:, :K] + rng.normal(0, 0.5, (B, K, V))
    toks = rng.integers(0, V, (B, K))
    uni = rng.random((B, K + 2))
    tl[1, 2, 4] = np.nan
    dl[2, 0, :] = -np.inf
    toks[3, 1] = V
    uni[4, 3] = 1.5
    tl[5, 0, 0] = np.inf
    r = O.verify(tl, dl, toks, uni, 1.0)
    assert r.status[0] == 0 and r.n_accepted[0] >= 0
    assert r.status[1] == O.STATUS_NONFINITE
    assert r.status[2] == O.STATUS_EMPTY_ROW
    assert r.status[3] == O.STATUS_TOKEN_RANGE
    assert r.status[4] == O.STATUS_UNIFORM_RANGE
    assert r.status[5] == O.STATUS_NONFINITE
    for b in range(1, B):
        assert (r.out_tokens[b] == -1).all() and r.n_accepted[b] == -1


# ---------------------------------------------------------------- draft-side sampler pins

def load_draft_golden():
    with open(os.path.join(GOLDEN_DIR, "draft_sample_cases.json")) as f:
        return json.load(f)["cases"]


def _golden_logits(vals):
    return np.array([[-np.inf if v == "-inf" else float(v) for v in vals]])


def pin_draft_golden(O):
    """Hand-worked draws (tests/golden/draft_sample_cases.json)."""
    for c in load_draft_golden():
        r = O.draft_sample(_golden_logits(c["logits"]), np.array([c["u"]]), c["temperature"])
        name = c["name"]
        assert r.status[0] == 0, name
        assert r.tokens[0] == c["token"], (name, r.tokens[0])
        np.testing.assert_allclose(r.sample_prob[0], c["prob"], atol=1e-12, err_msg=name)
        np.testing.assert_allclose(r.sample_margin[0], c["margin"], atol=1e-12, err_msg=name)


def pin_draft_law(O, n=200_000, V=16, seed=11):
    """The sampler's law is softmax(l / T): chi-square of seeded draws against
    scipy's softmax (a different routine from the oracle's)."""
    from scipy import stats

    rng = np.random.default_rng(seed)
    logits = rng.normal(0.0, 2.0, size=V)
    T = 0.7
    u = rng.random(n)
    r = O.draft_sample(np.repeat(logits[None], n, axis=0), u, T)
    assert (r.status == 0).all()
    counts = np.bincount(r.tokens, minlength=V)
    expect = softmax(logits / np.float32(T).astype(np.float64)) * n
    keep = expect > 5
    obs, exp = counts[keep], expect[keep]
    if (~keep).any():  # lump the rare tokens into one bin
        obs, exp = np.append(obs, counts[~keep].sum()), np.append(exp, expect[~keep].sum())
    assert stats.chisquare(obs, exp * obs.sum() / exp.sum()).pvalue > 1e-4


def pin_draft_failures(O):
    """U12 for the sampler: each bad row fails alone with its status bit."""
    good = np.zeros(6)
    rows = np.stack([good, good, good, good, good, good])
    rows[1, 2] = np.nan
    rows[2, 4] = np.inf
    rows[3, :] = -np.inf
    u = np.array([0.3, 0.3, 0.3, 0.3, np.nan, 1.5])
    r = O.draft_sample(rows, u, 1.0)
    assert r.status[0] == 0 and r.tokens[0] == 1   # C_0 = 1/6 <= 0.3 < C_1 = 1/3
    assert r.status[1] == O.STATUS_NONFINITE and r.tokens[1] == -1
    assert r.status[2] == O.STATUS_NONFINITE and r.tokens[2] == -1
    assert r.status[3] == O.STATUS_EMPTY_ROW and r.tokens[3] == -1
    assert r.status[4] == O.STATUS_UNIFORM_RANGE and r.tokens[4] == -1
    assert r.status[5] == O.STATUS_UNIFORM_RANGE and r.tokens[5] == -1
    r = O.draft_sample(np.zeros((1, 3)), np.array([-0.1]), 1.0)
    assert r.status[0] == O.STATUS_UNIFORM_RANGE


def pin_draft_matches_bonus(O):
    """When every draft is accepted, the verifier's bonus draw (Algorithm 2
    step 4) is the sampler applied to target row K with uniform u[K+1]."""
    rng = np.random.default_rng(13)
    B, K, V = 6, 3, 40
    tl = rng.normal(0, 1.5, size=(B, K + 1, V))
    dl = tl[:, :K].copy()                      # p == q on every drafted row: all accept
    tok = rng.integers(0, V, size=(B, K))
    uni = rng.random((B, K + 2))
    r = O.verify(tl, dl, tok, uni, 0.9)
    assert (r.n_accepted == K).all()
    s = O.draft_sample(tl[:, K], uni[:, K + 1], 0.9)
    assert (r.out_tokens[:, K] == s.tokens).all()


# ---------------------------------------------------------------- greedy-mode pins

def pin_greedy_golden(O):
    """Hand-worked greedy cases (tests/golden/greedy_cases.json)."""
    with open(os.path.join(GOLDEN_DIR, "greedy_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        tl = np.array([[[-np.inf if v == "-inf" else float(v) for v in row] for row in c["target"]]])
        r = O.verify_greedy(tl, np.array([c["tokens"]]))
        assert r.status[0] == 0, c["name"]
        assert list(r.out_tokens[0]) == c["out"], (c["name"], r.out_tokens[0])
        assert r.n_accepted[0] == c["n_accepted"], c["name"]


def pin_greedy_is_zero_temperature(O, B=64, K=4, V=50, seed=17):
    """Greedy mode is the general rule on one-hot distributions: with logits
    spaced at least 1 apart and T = 1e-3, softmax(l/T) is one-hot in fp64, and
    verify must give exactly verify_greedy's outputs for any drafts."""
    rng = np.random.default_rng(seed)
    tl = np.stack([np.stack([rng.permutation(V) for _ in range(K + 1)]) for _ in range(B)]).astype(float)
    dl = np.stack([np.stack([rng.permutation(V) for _ in range(K)]) for _ in range(B)]).astype(float)
    am_q = tl.argmax(-1)
    am_p = dl.argmax(-1)
    # drafts: mostly the draft argmax, sometimes the target argmax, sometimes random
    pick = rng.random((B, K))
    tok = np.where(pick < 0.5, am_p, np.where(pick < 0.8, am_q[:, :K], rng.integers(0, V, (B, K))))
    uni = rng.random((B, K + 2)) * 0.999
    r = O.verify(tl, dl, tok, uni, 1e-3)
    g = O.verify_greedy(tl, tok)
    assert (r.status == 0).all() and (g.status == 0).all()
    assert (r.out_tokens == g.out_tokens).all() and (r.n_accepted == g.n_accepted).all()
    assert (g.n_accepted < K).any() and (g.n_accepted == K).any()


def pin_greedy_failures(O):
    """U12 for greedy mode: each bad sequence fails alone."""
    rng = np.random.default_rng(19)
    B, K, V = 5, 2, 16
    tl = rng.normal(size=(B, K + 1, V))
    tok = rng.integers(0, V, size=(B, K))
    tl[1, 2, 3] = np.nan
    tl[2, 0, 0] = np.inf
    tl[3, 1, :] = -np.inf
    tok[4, 1] = V
    r = O.verify_greedy(tl, tok)
    assert list(r.status) == [0, O.STATUS_NONFINITE, O.STATUS_NONFINITE, O.STATUS_EMPTY_ROW,
                              O.STATUS_TOKEN_RANGE]
    for b in range(1, B):
        assert (r.out_tokens[b] == -1).all() and r.n_accepted[b] == -1
    assert 0 <= r.n_accepted[0] <= K and (r.out_tokens[0, : r.n_accepted[0] + 1] >= 0).all()


# ---------------------------------------------------------------- top-k pins

def pin_topk_mask_cases(O):
    """Hand-checked masks (U16): ties to the smaller id, -0 equal to +0,
    -inf entries last, k >= V keeps the row."""
    ni = -np.inf
    cases = [
        ([3.0, 1.0, 3.0, 2.0, -0.0, 0.0], 3, [3.0, ni, 3.0, 2.0, ni, ni]),
        ([1.0, 2.0, 2.0, 2.0], 2, [ni, 2.0, 2.0, ni]),
        ([-0.0, 0.0, -1.0], 1, [-0.0, ni, ni]),
        ([0.0, -0.0, -1.0], 1, [0.0, ni, ni]),
        ([ni, 5.0, ni, 4.0], 3, [ni, 5.0, ni, 4.0]),          # a -inf entry fills the third slot
        ([1.0, 2.0, 3.0], 3, [1.0, 2.0, 3.0]),
        ([1.0, 2.0, 3.0], 7, [1.0, 2.0, 3.0]),
    ]
    for row, k, want in cases:
        got = O.topk_mask(np.array([row]), k)[0]
        assert np.array_equal(got, np.array(want)), (row, k, got)


def pin_topk_order_property(O):
    """Against the definition, without sorting: on random tie-heavy rows
    (finite, -0 mixed with +0) the mask keeps exactly min(k, V) entries, and
    no removed entry outranks a kept one (a larger logit, or an equal logit
    and a smaller id)."""
    rng = np.random.default_rng(53)
    for trial in range(300):
        V = int(rng.integers(1, 12))
        row = rng.integers(-2, 3, V).astype(float)
        row[(row == 0) & (rng.random(V) < 0.5)] = -0.0
        k = int(rng.integers(1, V + 3))
        masked = O.topk_mask(row[None], k)[0]
        keep = np.isfinite(masked)
        assert keep.sum() == min(k, V), (row, k, masked)
        assert (masked[keep] == row[keep]).all()
        for i in np.nonzero(keep)[0]:
            for j in np.nonzero(~keep)[0]:
                assert row[i] > row[j] or (row[i] == row[j] and i < j), (row, k, masked)


def pin_topk_hand_case(O):
    """Worked by hand: V = 3, K = 1, k = 2, T = 1. Target probabilities
    .5, .3, .2 keep ids 0, 1 -> q = .625, .375, 0; draft .2, .3, .5 keep ids
    2, 1 -> p = 0, .375, .625. The draft x~ = 2 has q(2) = 0: rejected. The
    residual (q - p)_+ = .625, 0, 0 draws id 0 for any uniform (had p not
    been filtered, (q - p)_+ = .425, .075, 0 would draw id 1 at u = .9)."""
    tl = np.log(np.array([[[0.5, 0.3, 0.2], [0.4, 0.4, 0.2]]]))
    dl = np.log(np.array([[[0.2, 0.3, 0.5]]]))
    r = O.verify_topk(tl, dl, np.array([[2]]), np.array([[0.5, 0.9, 0.5]]), 1.0, 2)
    assert r.status[0] == 0
    assert list(r.out_tokens[0]) == [0, -1] and r.n_accepted[0] == 0, r.out_tokens
    np.testing.assert_allclose(r.thresholds[0], [0.0])
    np.testing.assert_allclose(r.sample_prob[0], 1.0)


def pin_topk_full_is_verify(O):
    """k >= V is no filter: verify_topk equals verify."""
    rng = np.random.default_rng(23)
    B, K, V = 16, 3, 30
    tl, dl = rng.normal(0, 2, (B, K + 1, V)), rng.normal(0, 2, (B, K, V))
    tok, uni = rng.integers(0, V, (B, K)), rng.random((B, K + 2))
    a, b = O.verify(tl, dl, tok, uni, 0.8), O.verify_topk(tl, dl, tok, uni, 0.8, V)
    assert (a.out_tokens == b.out_tokens).all() and (a.n_accepted == b.n_accepted).all()
    np.testing.assert_array_equal(a.thresholds, b.thresholds)


def pin_topk_one_is_greedy(O):
    """k = 1 leaves one-hot distributions at each row's first argmax, on which
    the general rule is the greedy rule (U15), for any drafts and T."""
    rng = np.random.default_rng(29)
    B, K, V = 64, 4, 20
    tl = np.round(rng.normal(0, 1.5, (B, K + 1, V)), 1)    # rounded: ties occur
    dl = np.round(rng.normal(0, 1.5, (B, K, V)), 1)
    pick = rng.random((B, K))
    tok = np.where(pick < 0.5, dl.argmax(-1), np.where(pick < 0.8, tl[:, :K].argmax(-1),
                                                       rng.integers(0, V, (B, K))))
    uni = rng.random((B, K + 2)) * 0.999
    r = O.verify_topk(tl, dl, tok, uni, 1.3, 1)
    g = O.verify_greedy(tl, tok)
    assert (r.out_tokens == g.out_tokens).all() and (r.n_accepted == g.n_accepted).all()


def pin_topk_law(O, n=200_000, V=12, k=5, seed=31):
    """Theorem 1 under the transform: the first emitted token is distributed as
    the top-k filtered q; chi-square against scipy's softmax of the kept
    logits, with the draft drawn from the filtered p by inverse CDF."""
    from scipy import stats

    rng = np.random.default_rng(seed)
    tl = rng.normal(0, 1.0, (1, 2, V))
    dl = rng.normal(0, 1.0, (1, 1, V))
    T = 0.9
    keep_q = np.argsort(-tl[0, 0], kind="stable")[:k]
    keep_p = np.argsort(-dl[0, 0], kind="stable")[:k]
    pf = np.zeros(V)
    pf[keep_p] = softmax(dl[0, 0, keep_p] / T)
    toks = np.minimum(np.searchsorted(np.cumsum(pf), rng.random(n), side="right"), V - 1)
    r = O.verify_topk(np.repeat(tl, n, 0), np.repeat(dl, n, 0), toks[:, None],
                      rng.random((n, 3)), T, k)
    first = r.out_tokens[:, 0]
    counts = np.bincount(first, minlength=V)
    assert counts[np.setdiff1d(np.arange(V), keep_q)].sum() == 0
    expect = softmax(tl[0, 0, keep_q] / T) * n
    assert stats.chisquare(counts[keep_q], expect * counts[keep_q].sum() / expect.sum()).pvalue > 1e-4


def pin_topp_mask_cases(O):
    """Hand-checked nucleus masks (U17): probabilities .5/.3/.15/.05 keep 1,
    2, 3, 4 entries at p = .4/.7/.9/.99; equal logits go to the smaller id
    (-0 equal to +0); the order is by logit, not by id; -inf entries are
    never needed; the temperature is applied before the cut."""
    ni = -np.inf
    lg = np.log([0.5, 0.3, 0.15, 0.05])
    for p, n in ((0.4, 1), (0.7, 2), (0.9, 3), (0.99, 4), (1.0, 4)):
        m, k, _ = O.topp_mask(lg[None], 1.0, p)
        assert k[0] == n and np.isfinite(m[0]).sum() == n and np.isfinite(m[0, :n]).all(), (p, m)
    m, k, _ = O.topp_mask(np.zeros((1, 4)), 1.0, 0.3)        # .25 each: two needed
    assert list(np.isfinite(m[0])) == [True, True, False, False]
    # .25 each is exact in fp64, so the cumulative sums hit p = .25 and .5
    # exactly: reaching p is enough
    assert O.topp_mask(np.zeros((1, 4)), 1.0, 0.25)[1][0] == 1
    assert O.topp_mask(np.zeros((1, 4)), 1.0, 0.5)[1][0] == 2
    m, _, _ = O.topp_mask(np.array([[-0.0, 0.0, -5.0]]), 1.0, 0.3)
    assert list(np.isfinite(m[0])) == [True, False, False]
    m, _, _ = O.topp_mask(np.array([[1.0, 3.0, 2.0]]), 1.0, 0.8)   # .665 + .245 >= .8
    assert list(np.isfinite(m[0])) == [False, True, True]
    m, _, _ = O.topp_mask(np.array([[ni, 0.0, 0.0, ni]]), 1.0, 0.9)
    assert list(np.isfinite(m[0])) == [False, True, True, False]
    lt = np.log([[0.5, 0.3, 0.2]])
    # T = 1: .5 + .3 = .8 < .85 needs all three; T = .5: .658 + .237 >= .85
    assert O.topp_mask(lt, 1.0, 0.85)[1][0] == 3 and O.topp_mask(lt, 0.5, 0.85)[1][0] == 2


def pin_topp_brute_force(O):
    """Against an enumeration of subsets on tiny rows: the kept set has the
    smallest size among all subsets whose mass reaches p, the largest mass
    among subsets of that size, and nothing removed outranks anything kept
    (larger logit, or equal logit and smaller id)."""
    import itertools

    rng = np.random.default_rng(37)
    for trial in range(120):
        V = int(rng.integers(2, 7))
        row = np.round(rng.normal(0, 1.2, V), 1)
        T = float(rng.choice([0.5, 1.0, 1.7]))
        p = float(rng.choice([0.2, 0.5, 0.75, 0.9, 0.97]))
        q = softmax(row / T)
        masked, kept, _ = O.topp_mask(row[None], T, p)
        keep = np.isfinite(masked[0])
        size = None
        for s in range(1, V + 1):
            best = max(q[list(c)].sum() for c in itertools.combinations(range(V), s))
            if best >= p - 1e-12:
                size = s
                break
        assert size is not None and keep.sum() == size == kept[0], (row, T, p, keep)
        best = max(q[list(c)].sum() for c in itertools.combinations(range(V), size))
        assert abs(q[keep].sum() - best) < 1e-12
        for i in np.nonzero(keep)[0]:
            for j in np.nonzero(~keep)[0]:
                assert row[i] > row[j] or (row[i] == row[j] and i < j), (row, keep)


def pin_topp_hand_case(O):
    """Worked by hand: V = 3, K = 1, T = 1, p = .7. Target row 0 .5/.3/.2 keeps
    ids 0, 1 (q = .625, .375, 0); target row 1 .2/.2/.6 keeps ids 2, 0
    (q = .25, 0, .75); the draft .1/.3/.6 keeps ids 2, 1 (p = 0, 1/3, 2/3).
    Sequence A drafts id 1: q/p = 1.125, accepted; the bonus at u = .3 over
    .25, 0, .75 is id 2 (unfiltered it would be id 1). Sequence B drafts id 2:
    q = 0, rejected; the residual .625, 1/24, 0 at u = .9 is id 0 (with an
    unfiltered draft, .525, .075, 0 would give id 1)."""
    tl = np.log(np.array([[[0.5, 0.3, 0.2], [0.2, 0.2, 0.6]]] * 2))
    dl = np.log(np.array([[[0.1, 0.3, 0.6]]] * 2))
    uni = np.array([[0.5, 0.5, 0.3], [0.5, 0.9, 0.5]])
    n = O.verify_topp(tl, dl, np.array([[1], [2]]), uni, 1.0, 0.7)
    r = n.result
    assert (r.status == 0).all()
    assert list(r.out_tokens[0]) == [1, 2] and r.n_accepted[0] == 1, r.out_tokens
    assert list(r.out_tokens[1]) == [0, -1] and r.n_accepted[1] == 0, r.out_tokens
    np.testing.assert_allclose(r.thresholds[:, 0], [1.0, 0.0])
    assert n.kept.tolist() == [[2, 2, 2], [2, 2, 2]]


def pin_topp_one_is_verify(O):
    """top_p = 1 is no filter: verify_topp equals verify."""
    rng = np.random.default_rng(41)
    B, K, V = 16, 3, 30
    tl, dl = rng.normal(0, 2, (B, K + 1, V)), rng.normal(0, 2, (B, K, V))
    tok, uni = rng.integers(0, V, (B, K)), rng.random((B, K + 2))
    a, b = O.verify(tl, dl, tok, uni, 0.8), O.verify_topp(tl, dl, tok, uni, 0.8, 1.0).result
    assert (a.out_tokens == b.out_tokens).all() and (a.n_accepted == b.n_accepted).all()
    np.testing.assert_array_equal(a.thresholds, b.thresholds)


def pin_topp_tiny_is_top1(O):
    """A nucleus smaller than every row's largest probability keeps one entry
    per row, the first argmax: verify_topp equals verify_topk with k = 1."""
    rng = np.random.default_rng(43)
    B, K, V = 32, 3, 25
    tl = np.round(rng.normal(0, 1.5, (B, K + 1, V)), 1)
    dl = np.round(rng.normal(0, 1.5, (B, K, V)), 1)
    tok, uni = rng.integers(0, V, (B, K)), rng.random((B, K + 2)) * 0.999
    a, b = O.verify_topk(tl, dl, tok, uni, 1.1, 1), O.verify_topp(tl, dl, tok, uni, 1.1, 1e-9).result
    assert (a.out_tokens == b.out_tokens).all() and (a.n_accepted == b.n_accepted).all()


def pin_topp_law(O, n=200_000, V=12, p=0.8, seed=47):
    """Theorem 1 under the nucleus transform: the first emitted token is
    distributed as the filtered q; chi-square against the renormalised
    top entries of q, with the draft drawn from the filtered p."""
    from scipy import stats

    rng = np.random.default_rng(seed)
    tl = rng.normal(0, 1.0, (1, 2, V))
    dl = rng.normal(0, 1.0, (1, 1, V))
    T = 0.9

    def nucleus(row):
        q = softmax(row / T)
        order = np.argsort(-q, kind="stable")
        n_keep = int(np.searchsorted(np.cumsum(q[order]), p)) + 1
        keep = order[:n_keep]
        f = np.zeros(V)
        f[keep] = q[keep] / q[keep].sum()
        return keep, f

    keep_q, fq = nucleus(tl[0, 0])
    _, fp = nucleus(dl[0, 0])
    toks = np.minimum(np.searchsorted(np.cumsum(fp), rng.random(n), side="right"), V - 1)
    r = O.verify_topp(np.repeat(tl, n, 0), np.repeat(dl, n, 0), toks[:, None],
                      rng.random((n, 3)), T, p).result
    counts = np.bincount(r.out_tokens[:, 0], minlength=V)
    assert counts[np.setdiff1d(np.arange(V), keep_q)].sum() == 0
    expect = fq[keep_q] * n
    assert stats.chisquare(counts[keep_q], expect * counts[keep_q].sum() / expect.sum()).pvalue > 1e-4


# ---------------------------------------------------------------- the scoring step (LM head)

def pin_lm_head_golden(O):
    """Hand-worked logits, row maxima, log-sum-exps and gathered logits
    (tests/golden/lm_head_cases.json)."""
    with open(os.path.join(GOLDEN_DIR, "lm_head_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        r = O.lm_head_stats(np.array(c["hidden"], dtype=np.float64),
                            np.array(c["weight"], dtype=np.float64), c["temperature"],
                            np.array(c["tokens"]))
        name = c["name"]
        assert np.array_equal(r.logits, np.array(c["expected_logits"], dtype=np.float64)), name
        np.testing.assert_allclose(r.row_max, c["expected_row_max"], rtol=0, atol=0, err_msg=name)
        np.testing.assert_allclose(r.lse, c["expected_lse"], rtol=1e-14, err_msg=name)
        exp_at = np.array([np.nan if v is None else v for v in c["expected_at"]])
        np.testing.assert_array_equal(r.at, exp_at, err_msg=name)


def pin_lm_head_brute_force(O, seed=61):
    """Integer-valued inputs: the logits against explicit loops over (n, v, d)
    (exact), the statistics against scipy's logsumexp of those logits, the
    gather against direct indexing; shapes chosen so that no two of N, D, V
    are equal."""
    rng = np.random.default_rng(seed)
    N, D, V = 3, 5, 7
    h = rng.integers(-3, 4, (N, D)).astype(np.float64)
    w = rng.integers(-3, 4, (V, D)).astype(np.float64)
    tok = np.array([6, 0, -1])
    ref = np.zeros((N, V))
    for n in range(N):
        for v in range(V):
            acc = 0.0
            for d in range(D):
                acc += h[n, d] * w[v, d]
            ref[n, v] = acc
    for T in (1.0, 0.75, 3.0):
        r = O.lm_head_stats(h, w, T, tok)
        assert np.array_equal(r.logits, ref)
        np.testing.assert_allclose(r.row_max, ref.max(axis=1) / T, rtol=0, atol=0)
        np.testing.assert_allclose(r.lse, logsumexp(ref / T, axis=1), rtol=1e-13)
        assert r.at[0] == ref[0, 6] and r.at[1] == ref[1, 0] and np.isnan(r.at[2])


def pin_lm_head_invariances(O, seed=67):
    """Exact invariances: (2h, 2T) gives the same z = l/T, so the same maxima
    and log-sum-exps, and twice the gathered logits; permuting the rows of W
    permutes the logits and leaves the statistics unchanged."""
    rng = np.random.default_rng(seed)
    N, D, V = 4, 16, 40
    h = np.round(rng.normal(0, 1, (N, D)) * 64) / 64
    w = np.round(rng.normal(0, 0.3, (V, D)) * 64) / 64
    tok = rng.integers(0, V, N)
    a = O.lm_head_stats(h, w, 0.75, tok)
    b = O.lm_head_stats(2 * h, w, 1.5, tok)
    np.testing.assert_array_equal(a.row_max, b.row_max)
    np.testing.assert_allclose(a.lse, b.lse, rtol=1e-15)
    np.testing.assert_array_equal(2 * a.at, b.at)
    perm = rng.permutation(V)
    inv = np.argsort(perm)
    c = O.lm_head_stats(h, w[perm], 0.75, inv[tok])
    np.testing.assert_array_equal(c.logits, a.logits[:, perm])
    np.testing.assert_array_equal(c.row_max, a.row_max)
    np.testing.assert_allclose(c.lse, a.lse, rtol=1e-14)
    np.testing.assert_array_equal(c.at, a.at)


FAST_PINS = (pin_golden, pin_theorem1, pin_sequential, pin_library_special_cases,
             pin_invariants, pin_failures, pin_draft_golden, pin_draft_failures,
             pin_draft_matches_bonus, pin_greedy_golden, pin_greedy_is_zero_temperature,
             pin_greedy_failures, pin_topk_mask_cases, pin_topk_hand_case,
             pin_topk_full_is_verify, pin_topk_one_is_greedy, pin_topk_order_property,
             pin_topp_mask_cases,
             pin_topp_brute_force, pin_topp_hand_case, pin_topp_one_is_verify,
             pin_topp_tiny_is_top1, pin_lm_head_golden, pin_lm_head_brute_force,
             pin_lm_head_invariances)
