"""fp64 CPU oracle of the speculative-sampling verification step.

TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers; the CUDA library neither imports nor
calls anything here, and this module shares no code with it.

What it computes, step by step, in the order and notation of
"Accelerating Large Language Model Decoding with Speculative Sampling"
(Chen et al., DeepMind), as summarised by its wikillm.com paper card (the
draft-side sampler of Algorithm 2 step 1, `draft_sample`, the greedy
variant, `verify_greedy`, and verification on top-k filtered distributions,
`verify_topk`, follow `verify`):

* q(.|...) and p(.|...) are the target and draft distributions. The decoding
  transform (temperature) is applied to both before anything else
  (card, §4.2 "Decoding transforms"; the Pitfalls item on transformed
  distributions).
* Draft token x~_t is accepted while r_t < min(1, q(x~_t)/p(x~_t)), left to
  right, the ratio evaluated at the drafted token (card, §4.2 "Modified
  rejection sampling"; Algorithm 2 step 3; Pitfalls, "Indexing in alg. 2").
* At the first rejection a replacement is drawn from the normalised residual
  (q - p)_+ = max(0, q - p) / sum max(0, q - p), and the loop stops
  (card, §4.2).
* If all K drafts are accepted, one bonus token is drawn from the (K+1)-th
  target distribution (card, Algorithm 2 step 4; Pitfalls, "Bonus-token typo").
* Each loop therefore emits between 1 and K+1 tokens (card, §4.2).

Readings taken where the pages leave a step open (each also listed in the
design notes):

* U1 uniform slots: u[:, t] (t < K) drives the acceptance test of x~_t,
  u[:, K] drives the residual draw, u[:, K+1] the bonus draw.
* U2 the acceptance test is strict, `u < min(1, q/p)`, as printed.
* U3 a categorical draw from weights w with uniform u is the inverse CDF over
  ascending token id: the smallest i with C_i > u * S, C_i = w_0 + ... + w_i
  summed in that order, S = C_{V-1}. If rounding (or u = 1) leaves no such i,
  the largest i with w_i > 0 is taken.
* U4 p(x~) = 0 with q(x~) > 0 accepts (the limit of min(1, q/p)); q(x~) = 0
  rejects.
* U5 zero residual (sum max(0, q - p) == 0): fall back to q itself, drawn with
  u[:, K] (the card's Pitfalls suggest the fallback; the paper is silent).
* U6 temperature: q = softmax(l / T) with T > 0 finite; T is given in fp32 and
  widened exactly.
* U8 n_accepted counts accepted drafts (0..K); out_tokens holds them, then the
  sampled token, then -1 padding (U9).
* U12 -inf logits are masked entries (probability 0). A sequence any of whose
  2K+1 rows holds NaN or +inf, or is entirely -inf, any of whose draft tokens
  lies outside [0, V), or any of whose K+2 uniforms is NaN or outside [0, 1],
  fails: all its outputs are -1 and its status word says why.

Inputs are widened exactly to fp64 (bf16 and fp32 both embed exactly). Every
decision also reports its margin, the distance of the uniform from the fp64
threshold it was compared with, so a caller can tell a genuine disagreement
from a decision that sits on a rounding boundary.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

STATUS_OK = 0
STATUS_TOKEN_RANGE = 16
STATUS_NONFINITE = 32
STATUS_EMPTY_ROW = 64
STATUS_UNIFORM_RANGE = 128


@dataclass
class OracleResult:
    out_tokens: np.ndarray       # [B, K+1] int64, -1 padded
    n_accepted: np.ndarray       # [B] int64, -1 for failed sequences
    status: np.ndarray           # [B] int64 status bits (0 = ok)
    thresholds: np.ndarray       # [B, K] fp64 min(1, q/p) at the drafted tokens
    accept_margin: np.ndarray    # [B, K] |u_t - thr_t| for decisions taken, NaN after
    sample_margin: np.ndarray    # [B] distance of u from the chosen CDF interval's ends
    sample_prob: np.ndarray      # [B] normalised weight of the sampled token
    residual_fallback: np.ndarray  # [B] bool, zero-residual fallback to q was used
    lse: np.ndarray              # [B, 2K+1] log-sum-exp of l/T: target rows 0..K, then draft rows 0..K-1
    row_max: np.ndarray          # [B, 2K+1] max of l/T per row, same order as lse (NaN: bad row)
    ratios: np.ndarray           # [B, K] q(x~)/p(x~) at the drafted tokens, not clamped

    def decisions(self) -> int:
        """Number of decisions taken (acceptance tests plus one draw per ok sequence)."""
        ok = self.status == 0
        return int(np.sum(np.isfinite(self.accept_margin[ok])) + np.sum(ok))


def temperature_softmax(logits: np.ndarray, temperature: float):
    """softmax(l / T) over the last axis, in fp64.

    The temperature transform of the card's §4.2 "Decoding transforms",
    applied identically to target and draft rows. Returns (probs, lse, status)
    with lse = log sum_i exp(l_i / T) and per-row status bits (NaN / +inf
    entries, or a row with every entry -inf).
    """
    z = logits / np.float64(temperature)
    nonfinite = np.isnan(z).any(axis=-1) | np.isposinf(z).any(axis=-1)
    with np.errstate(invalid="ignore"):
        m = np.max(z, axis=-1)
    empty = ~nonfinite & np.isneginf(m)
    bad = nonfinite | empty
    m_safe = np.where(bad, 0.0, m)
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        e = np.exp(z - m_safe[..., None])
        e = np.where(bad[..., None], 0.0, e)
        s = np.sum(e, axis=-1)
        s_safe = np.where(bad, 1.0, s)
        probs = e / s_safe[..., None]
        lse = np.where(bad, np.nan, m_safe + np.log(s_safe))
    status = np.where(nonfinite, STATUS_NONFINITE, 0) | np.where(empty, STATUS_EMPTY_ROW, 0)
    return probs, lse, status.astype(np.int64)


def acceptance_thresholds(q_at: np.ndarray, p_at: np.ndarray) -> np.ndarray:
    """min(1, q(x~)/p(x~)) at the drafted tokens (card, §4.2), with U4's limits."""
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = q_at / np.where(p_at > 0, p_at, 1.0)
    return np.where(p_at > 0, np.minimum(1.0, ratio), np.where(q_at > 0, 1.0, 0.0))


def acceptance_ratios(q_at: np.ndarray, p_at: np.ndarray) -> np.ndarray:
    """q(x~)/p(x~) at the drafted tokens, before the clamp at 1 (card, §4.2),
    with U4's limits: +inf where p(x~) = 0 < q(x~), 0 where q(x~) = 0."""
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = q_at / np.where(p_at > 0, p_at, 1.0)
    return np.where(p_at > 0, ratio, np.where(q_at > 0, np.inf, 0.0))


def first_rejection(u_acc: np.ndarray, thr: np.ndarray) -> np.ndarray:
    """Index of the first draft whose test `u < thr` fails, or K if none fails.

    Algorithm 2 step 3 scans t = 1..K left to right and stops at the first
    rejection; a separate count keeps the accepted length (card, Pitfalls).
    """
    accept = u_acc < thr
    K = accept.shape[1]
    return np.where(accept.all(axis=1), K, np.argmin(accept, axis=1)).astype(np.int64)


def residual_weights(q_row: np.ndarray, p_row: np.ndarray):
    """max(0, q - p) per token (card, §4.2); rows whose residual sums to zero
    fall back to q (U5). Returns (weights, fallback flags)."""
    w = np.maximum(0.0, q_row - p_row)
    fallback = ~(w > 0).any(axis=-1)
    w = np.where(fallback[..., None], q_row, w)
    return w, fallback


def inverse_cdf(w: np.ndarray, u: np.ndarray):
    """Draw one index per row from weights w (unnormalised) with uniform u (U3).

    Returns (index, margin, normalised weight of the index). The margin is
    the distance of u from the nearer end of the chosen index's interval
    [C_{i-1}/S, C_i/S) of the normalised CDF (0 when the fallback was taken).
    """
    B, V = w.shape
    C = np.cumsum(w, axis=-1)
    S = C[:, -1]
    target = u * S
    above = C > target[:, None]
    found = above.any(axis=-1)
    first = np.argmax(above, axis=-1)
    last_pos = V - 1 - np.argmax((w > 0)[:, ::-1], axis=-1)
    idx = np.where(found, first, last_pos)
    rows = np.arange(B)
    with np.errstate(invalid="ignore", divide="ignore"):   # S == 0 only on failed rows
        lo = np.where(idx > 0, C[rows, np.maximum(idx - 1, 0)], 0.0) / S
        hi = C[rows, idx] / S
        margin = np.where(found, np.minimum(u - lo, hi - u), 0.0)
        prob = w[rows, idx] / S
    return idx.astype(np.int64), margin, prob


def verify(target: np.ndarray, draft: np.ndarray, tokens: np.ndarray,
           uniforms: np.ndarray, temperature: float) -> OracleResult:
    """One verification step for a batch: target [B,K+1,V], draft [B,K,V]
    (fp64, widened exactly from the input dtype), tokens [B,K] ints,
    uniforms [B,K+2], temperature > 0."""
    target = np.asarray(target, dtype=np.float64)
    draft = np.asarray(draft, dtype=np.float64)
    tokens = np.asarray(tokens).astype(np.int64)
    uniforms = np.asarray(uniforms, dtype=np.float64)
    B, K1, V = target.shape
    K = K1 - 1
    if K < 1 or draft.shape != (B, K, V) or tokens.shape != (B, K) or uniforms.shape != (B, K + 2):
        raise ValueError("shape mismatch")
    # U6: the temperature is an fp32 argument; its fp32 value is widened exactly.
    with np.errstate(over="ignore"):
        T = float(np.float32(temperature))
    if not (np.isfinite(T) and T > 0):
        raise ValueError("temperature must be finite and > 0")

    # Temperature transform of both distributions, every row.
    q, lse_q, st_q = temperature_softmax(target, T)      # [B, K+1, V]
    p, lse_p, st_p = temperature_softmax(draft, T)       # [B, K, V]
    status = np.bitwise_or.reduce(st_q, axis=1) | np.bitwise_or.reduce(st_p, axis=1)
    tok_ok = ((tokens >= 0) & (tokens < V)).all(axis=1)
    status |= np.where(tok_ok, 0, STATUS_TOKEN_RANGE)
    u_ok = ((uniforms >= 0) & (uniforms <= 1)).all(axis=1)   # NaN compares false
    status |= np.where(u_ok, 0, STATUS_UNIFORM_RANGE)

    # Acceptance thresholds at the drafted tokens, and the left-to-right scan.
    tok = np.where((tokens >= 0) & (tokens < V), tokens, 0)
    q_at = np.take_along_axis(q[:, :K, :], tok[..., None], axis=-1)[..., 0]
    p_at = np.take_along_axis(p, tok[..., None], axis=-1)[..., 0]
    thr = acceptance_thresholds(q_at, p_at)
    ratios = acceptance_ratios(q_at, p_at)
    u_acc = uniforms[:, :K]
    j = first_rejection(u_acc, thr)
    taken = np.arange(K)[None, :] <= j[:, None]
    accept_margin = np.where(taken, np.abs(u_acc - thr), np.nan)

    # The one draw per sequence: residual at row j, or bonus from target row K.
    rows = np.arange(B)
    residual = j < K
    q_row = q[rows, j]
    p_row = p[rows, np.minimum(j, K - 1)]
    w_res, fallback = residual_weights(q_row, p_row)
    w = np.where(residual[:, None], w_res, q_row)
    u_draw = np.where(residual, uniforms[:, K], uniforms[:, K + 1])
    idx, sample_margin, sample_prob = inverse_cdf(w, u_draw)

    out = np.full((B, K + 1), -1, dtype=np.int64)
    for b in range(B):
        out[b, : j[b]] = tokens[b, : j[b]]
        out[b, j[b]] = idx[b]
    n_acc = j.copy()

    failed = status != 0
    out[failed] = -1
    n_acc[failed] = -1
    thr = np.where(failed[:, None], np.nan, thr)
    ratios = np.where(failed[:, None], np.nan, ratios)
    accept_margin = np.where(failed[:, None], np.nan, accept_margin)
    sample_margin = np.where(failed, np.nan, sample_margin)
    sample_prob = np.where(failed, np.nan, sample_prob)
    fallback = residual & fallback & ~failed
    lse = np.concatenate([lse_q, lse_p], axis=1)
    # Row maxima of l/T (the transformed logits), NaN where the row is bad.
    with np.errstate(invalid="ignore"):
        row_max = np.concatenate([np.max(target / T, axis=-1), np.max(draft / T, axis=-1)], axis=1)
    row_max = np.where(np.isfinite(lse), row_max, np.nan)
    return OracleResult(out, n_acc, status, thr, accept_margin, sample_margin, sample_prob,
                        fallback, lse, row_max, ratios)


@dataclass
class SampleResult:
    tokens: np.ndarray           # [N] int64, -1 for failed rows
    status: np.ndarray           # [N] status bits (U12), 0 = ok
    sample_margin: np.ndarray    # [N] distance of u from the chosen CDF interval's ends
    sample_prob: np.ndarray      # [N] probability of the drawn token
    lse: np.ndarray              # [N] log sum_i exp(l_i / T)


def draft_sample(logits: np.ndarray, uniforms: np.ndarray, temperature: float) -> SampleResult:
    """Draft-side sampling: one token per row, x~ ~ softmax(l / T).

    This is step 1 of the card's Algorithm 2 (the K sequential draft samples,
    one row per call here), drawn from the transformed draft distribution
    (card, §4.2 "Decoding transforms", and the Pitfalls item on transformed
    distributions: the drafts come from the same p the ratios use). The draw is
    the inverse CDF of U3 with the row's uniform; rows fail as in U12 (NaN or
    +inf entries, every entry -inf, or a uniform that is NaN or outside
    [0, 1]): token -1 and a status word saying why.

    logits [N, V] (widened exactly), uniforms [N], temperature > 0 (an fp32
    value widened exactly, U6).
    """
    logits = np.asarray(logits, dtype=np.float64)
    uniforms = np.asarray(uniforms, dtype=np.float64)
    if logits.ndim != 2 or uniforms.shape != (logits.shape[0],):
        raise ValueError("shape mismatch")
    with np.errstate(over="ignore"):
        T = float(np.float32(temperature))
    if not (np.isfinite(T) and T > 0):
        raise ValueError("temperature must be finite and > 0")
    p, lse, status = temperature_softmax(logits, T)
    u_ok = (uniforms >= 0) & (uniforms <= 1)   # NaN compares false
    status = status | np.where(u_ok, 0, STATUS_UNIFORM_RANGE)
    idx, margin, prob = inverse_cdf(p, np.where(u_ok, uniforms, 0.0))
    failed = status != 0
    return SampleResult(np.where(failed, -1, idx), status, np.where(failed, np.nan, margin),
                        np.where(failed, np.nan, prob), np.where(failed, np.nan, lse))


@dataclass
class GreedyResult:
    out_tokens: np.ndarray       # [B, K+1] int64, -1 padded
    n_accepted: np.ndarray       # [B] int64, -1 for failed sequences
    status: np.ndarray           # [B] status bits (U12), 0 = ok
    argmax: np.ndarray           # [B, K+1] target argmax of every row (-1 where failed)


def verify_greedy(target: np.ndarray, tokens: np.ndarray) -> GreedyResult:
    """Greedy-mode verification (T = 0).

    The paper reports greedy results but does not state the rule; the card's
    Pitfalls ("Greedy mode is not specified") infer it by applying the
    general rule to one-hot distributions: accept while the draft's greedy
    token equals the target's, otherwise emit the target's greedy token. U15:
    the drafted token x~_t is compared with argmax q_t (the two coincide when
    the drafts were taken greedily); ties in an argmax go to the smallest
    token id; at the first mismatch j the target's argmax q_j is emitted, and
    if all K match, argmax q_K (the bonus token of Algorithm 2 step 4). No
    uniforms and no draft logits are involved. A sequence fails as in U12
    (a target row with NaN or +inf, or entirely -inf; a token outside [0, V)).

    target [B, K+1, V] (widened exactly), tokens [B, K] ints.
    """
    target = np.asarray(target, dtype=np.float64)
    tokens = np.asarray(tokens).astype(np.int64)
    B, K1, V = target.shape
    K = K1 - 1
    if K < 1 or tokens.shape != (B, K):
        raise ValueError("shape mismatch")
    nonfinite = np.isnan(target).any(axis=-1) | np.isposinf(target).any(axis=-1)
    empty = ~nonfinite & np.isneginf(target).all(axis=-1)
    status = (np.bitwise_or.reduce(np.where(nonfinite, STATUS_NONFINITE, 0), axis=1)
              | np.bitwise_or.reduce(np.where(empty, STATUS_EMPTY_ROW, 0), axis=1))
    tok_ok = ((tokens >= 0) & (tokens < V)).all(axis=1)
    status = status | np.where(tok_ok, 0, STATUS_TOKEN_RANGE)
    with np.errstate(invalid="ignore"):
        am = np.argmax(np.where(np.isnan(target), -np.inf, target), axis=-1)   # first maximum
    match = tokens == am[:, :K]
    j = np.where(match.all(axis=1), K, np.argmin(match, axis=1))
    out = np.full((B, K + 1), -1, dtype=np.int64)
    for b in range(B):
        out[b, : j[b]] = tokens[b, : j[b]]
        out[b, j[b]] = am[b, j[b]]
    n_acc = j.astype(np.int64)
    failed = status != 0
    out[failed] = -1
    n_acc[failed] = -1
    return GreedyResult(out, n_acc, status.astype(np.int64), np.where(failed[:, None], -1, am))


def topk_mask(logits: np.ndarray, k: int) -> np.ndarray:
    """The top-k decoding transform on logits (U16): every entry outside the k
    largest of its row becomes -inf (probability 0 after the softmax), the
    rest are unchanged. Order: larger logit first, ties to the smaller token
    id (-0.0 equals +0.0). k >= V keeps every entry. Rows holding NaN are
    returned unchanged (they fail anyway, U12)."""
    logits = np.asarray(logits, dtype=np.float64)
    V = logits.shape[-1]
    if k >= V:
        return logits.copy()
    flat = logits.reshape(-1, V)
    out = np.full_like(flat, -np.inf)
    for r in range(flat.shape[0]):
        row = flat[r]
        if np.isnan(row).any():
            out[r] = row
            continue
        order = np.argsort(-(row + 0.0), kind="stable")   # descending; stable keeps id order
        keep = order[:k]
        out[r, keep] = row[keep]
    return out.reshape(logits.shape)


def verify_topk(target: np.ndarray, draft: np.ndarray, tokens: np.ndarray,
                uniforms: np.ndarray, temperature: float, top_k: int) -> OracleResult:
    """Verification on top-k filtered distributions: the card's §4.2
    "Decoding transforms" (apply top-k to both p and q first, then run the
    rejection scheme on the modified distributions) and Pitfalls ("Use the
    same transformed distributions everywhere"). Each of the 2K+1 rows keeps
    its top_k largest logits (U16, `topk_mask`); the temperature softmax of
    the kept entries, the thresholds, the residual and the draws are then
    exactly those of `verify`."""
    if top_k < 1:
        raise ValueError("top_k must be >= 1")
    return verify(topk_mask(target, top_k), topk_mask(draft, top_k), tokens, uniforms,
                  temperature)


@dataclass
class NucleusResult:
    result: OracleResult         # the verification on the filtered rows
    kept: np.ndarray             # [B, 2K+1] entries kept per row (target rows 0..K, then draft rows)
    cut_margin: np.ndarray       # [B, 2K+1] distance of top_p from the cumulative sums at the cut


def topp_mask(logits: np.ndarray, temperature: float, top_p: float):
    """The nucleus (top-p) decoding transform on logits (U17): per row,
    q = softmax(l / T) in fp64 (`temperature_softmax`); entries are ordered
    by logit, larger first, ties to the smaller token id (-0.0 equals +0.0);
    the shortest prefix of that order whose cumulative q, summed in that
    order, reaches top_p is kept, the rest become -inf. top_p >= 1 keeps the
    row; if rounding leaves the total below top_p, every entry with q > 0 is
    kept. Rows that fail (NaN, +inf, all -inf; U12) are returned unchanged.

    Returns (masked logits, kept count per row, cut margin per row): the
    margin is min(C_n - top_p, top_p - C_{n-1}) for the kept count n and the
    cumulative sums C, inf when the row is not cut."""
    logits = np.asarray(logits, dtype=np.float64)
    shape, V = logits.shape, logits.shape[-1]
    flat = logits.reshape(-1, V)
    out = flat.copy()
    kept = np.full(flat.shape[0], V, dtype=np.int64)
    margin = np.full(flat.shape[0], np.inf)
    if top_p >= 1.0:
        return out.reshape(shape), kept.reshape(shape[:-1]), margin.reshape(shape[:-1])
    q, _, st = temperature_softmax(flat, temperature)
    for r in range(flat.shape[0]):
        if st[r] != 0:
            continue
        order = np.argsort(-(flat[r] + 0.0), kind="stable")
        c = np.cumsum(q[r, order])
        reach = np.nonzero(c >= top_p)[0]
        n = int(reach[0]) + 1 if len(reach) else int((q[r] > 0).sum())
        kept[r] = n
        margin[r] = min(c[n - 1] - top_p if len(reach) else np.inf,
                        top_p - c[n - 2] if n >= 2 else np.inf)
        out[r, order[n:]] = -np.inf
    return out.reshape(shape), kept.reshape(shape[:-1]), margin.reshape(shape[:-1])


def verify_topp(target: np.ndarray, draft: np.ndarray, tokens: np.ndarray,
                uniforms: np.ndarray, temperature: float, top_p: float) -> NucleusResult:
    """Verification on nucleus filtered distributions: the card's §4.2
    "Decoding transforms" (apply the transform to both p and q, then the
    rejection scheme on the modified distributions) with the nucleus rule of
    `topp_mask` on each of the 2K+1 rows, at the same temperature as the
    verification."""
    if not (top_p > 0.0):
        raise ValueError("top_p must be > 0")
    with np.errstate(over="ignore"):
        T = float(np.float32(temperature))
        # Like the temperature (U6), top_p is an fp32 argument: its fp32 value,
        # widened exactly, is the mass the cut must reach.
        top_p = float(np.float32(top_p))
    tm, tk, tg = topp_mask(target, T, top_p)
    dm, dk, dg = topp_mask(draft, T, top_p)
    res = verify(tm, dm, tokens, uniforms, temperature)
    return NucleusResult(res, np.concatenate([tk, dk], axis=1), np.concatenate([tg, dg], axis=1))


@dataclass
class LMHeadStats:
    logits: np.ndarray           # [N, V] fp64 logits l = h W^T
    row_max: np.ndarray          # [N] max_i l_i / T
    lse: np.ndarray              # [N] log sum_i exp(l_i / T)
    at: np.ndarray               # [N] l at the row's token (NaN where none is given)


def lm_head_stats(hidden, weight, temperature, tokens=None) -> LMHeadStats:
    """The model's final projection and the statistics of its temperature
    transform, per row: the logits l = h W^T (hidden [N, D] times the
    transposed projection weight [V, D], in fp64 from exactly widened inputs),
    max_i l_i/T, log sum_i exp(l_i/T), and l at the row's token.

    This is the scoring step of Algorithm 2 step 2 (one target call scores
    the K+1 prefixes; card, §4.1 "Why it works (conditional scoring)") fused
    with the row statistics the verification needs (§4.2 "Decoding
    transforms"; the ratio at the drafted token, §4.2 "Modified rejection
    sampling"). `tokens` [N] holds a token id per row, or -1 for none; the
    temperature is an fp32 argument, widened exactly (U6)."""
    h = np.asarray(hidden, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    if h.ndim != 2 or w.ndim != 2 or h.shape[1] != w.shape[1]:
        raise ValueError("hidden [N, D] and weight [V, D] must share D")
    with np.errstate(over="ignore"):
        T = float(np.float32(temperature))
    if not (np.isfinite(T) and T > 0):
        raise ValueError("temperature must be finite and > 0")
    logits = np.matmul(h, w.T)
    z = logits / T
    m = np.max(z, axis=-1)
    lse = m + np.log(np.sum(np.exp(z - m[:, None]), axis=-1))
    N, V = logits.shape
    at = np.full(N, np.nan)
    if tokens is not None:
        tok = np.asarray(tokens).astype(np.int64)
        ok = (tok >= 0) & (tok < V)
        at[ok] = logits[np.arange(N)[ok], tok[ok]]
    return LMHeadStats(logits, m, lse, at)


def _widen(x) -> np.ndarray:
    """Exact widening of a torch tensor (bf16 / fp32 / int) or array to numpy fp64."""
    if hasattr(x, "detach"):
        import torch  # local: the oracle itself needs only numpy

        x = x.detach().cpu()
        if x.dtype in (torch.bfloat16, torch.float16, torch.float32, torch.float64):
            return x.to(torch.float64).numpy()
        return x.numpy()
    return np.asarray(x)


def verify_inputs(inputs: dict, chunk: int = 8) -> OracleResult:
    """`verify` over an input dict from the synthetic generator, `chunk`
    sequences at a time to bound memory; results are concatenated."""
    B = inputs["target"].shape[0]
    parts = []
    for s in range(0, B, chunk):
        e = min(B, s + chunk)
        parts.append(verify(_widen(inputs["target"][s:e]), _widen(inputs["draft"][s:e]),
                            _widen(inputs["tokens"][s:e]), _widen(inputs["uniforms"][s:e]),
                            inputs["temperature"]))
    if len(parts) == 1:
        return parts[0]
    return OracleResult(*[np.concatenate([getattr(p, f) for p in parts], axis=0)
                          for f in OracleResult.__dataclass_fields__])
