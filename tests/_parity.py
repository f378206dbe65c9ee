"""Comparison of the CUDA path's outputs with the fp64 oracle's.

A verification step takes a sequence of decisions: acceptance tests t = 0..j,
then one draw. Outputs must be identical; the only tolerated differences are
decisions whose uniform lies within MARGIN of the oracle's fp64 threshold
(an acceptance threshold, or an end of the drawn token's CDF interval). Those
are counted; any other difference is a failure.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

MARGIN = 1e-6
RATE_MIN_DECISIONS = 100_000


@dataclass
class ParityReport:
    sequences: int = 0
    decisions: int = 0
    excused: int = 0
    near_threshold: int = 0
    failures: list = field(default_factory=list)

    def add(self, other: "ParityReport") -> None:
        self.sequences += other.sequences
        self.decisions += other.decisions
        self.excused += other.excused
        self.near_threshold += other.near_threshold
        self.failures += other.failures

    def assert_ok(self, max_excused_rate: float | None = None) -> None:
        """No unexcused difference, and excused differences at most
        `max_excused_rate` of the decisions. Below RATE_MIN_DECISIONS decisions
        the rate cannot be resolved, so one excused difference is allowed;
        from there on the plain rate applies."""
        assert not self.failures, self.failures[:10]
        if max_excused_rate is not None and self.decisions:
            allowed = max_excused_rate * self.decisions
            if self.decisions < RATE_MIN_DECISIONS:
                allowed = max(1, allowed)
            assert self.excused <= allowed, self

    def as_dict(self) -> dict:
        return {"sequences": self.sequences, "decisions": self.decisions,
                "near_threshold": self.near_threshold, "excused_differences": self.excused,
                "unexcused_differences": len(self.failures)}


def compare(out, nacc, ref, drafts) -> ParityReport:
    out = np.asarray(out).astype(np.int64)
    nacc = np.asarray(nacc).astype(np.int64)
    drafts = np.asarray(drafts).astype(np.int64)
    B, K1 = out.shape
    K = K1 - 1
    rep = ParityReport(sequences=B, decisions=ref.decisions())
    ok = ref.status == 0
    rep.near_threshold = int(np.sum(ref.accept_margin[ok] < MARGIN) + np.sum(ref.sample_margin[ok] < MARGIN))
    for b in range(B):
        if ref.status[b] != 0:
            if not ((out[b] == -1).all() and nacc[b] == -1):
                rep.failures.append((b, "failed sequence not reported as failed", out[b], nacc[b]))
            continue
        jg = nacc[b]
        # Structural checks hold whatever the decisions were.
        if not (0 <= jg <= K):
            rep.failures.append((b, "n_accepted out of range", jg))
            continue
        if not (np.array_equal(out[b, :jg], drafts[b, :jg]) and (out[b, jg + 1:] == -1).all()
                and 0 <= out[b, jg]):
            rep.failures.append((b, "malformed output", out[b], jg))
            continue
        jo = ref.n_accepted[b]
        if jg == jo and np.array_equal(out[b], ref.out_tokens[b]):
            continue
        if jg != jo:
            t = min(jg, jo)
            m = ref.accept_margin[b, t]
            what = f"acceptance test t={t}"
        else:
            m = ref.sample_margin[b]
            what = "draw"
        if m < MARGIN:
            rep.excused += 1
        else:
            rep.failures.append((b, what, "gpu", out[b].tolist(), "oracle", ref.out_tokens[b].tolist(),
                                 "margin", float(m)))
    return rep
