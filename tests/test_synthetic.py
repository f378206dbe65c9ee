"""The seeded input generator (CPU)."""

import numpy as np
import torch

from synthetic import WORKLOADS, SWEEP_K, SWEEP_NOISE, get_workload, make_inputs, make_sequence
from synthetic.configs import shrink


def test_deterministic_and_per_sequence_seeded():
    w = shrink(WORKLOADS["c2"], B=4, V=2048)
    a = make_inputs(w, step=3)
    b = make_inputs(w, step=3)
    for k in ("target", "draft", "tokens", "uniforms"):
        assert torch.equal(a[k], b[k])
    sub = make_inputs(w, step=3, seqs=[2])
    assert torch.equal(sub["target"][0], a["target"][2])
    assert torch.equal(sub["tokens"][0], a["tokens"][2])
    c = make_inputs(w, step=4)
    assert not torch.equal(a["target"], c["target"])


def test_shapes_dtypes_ranges():
    for name in ("c1", "c3"):
        w = shrink(WORKLOADS[name], B=2, V=min(WORKLOADS[name].V, 3000))
        inp = make_inputs(w)
        assert inp["target"].shape == (2, w.K + 1, w.V)
        assert inp["draft"].shape == (2, w.K, w.V)
        assert inp["target"].dtype == (torch.bfloat16 if w.dtype == "bf16" else torch.float32)
        assert inp["tokens"].dtype == torch.int32
        assert ((inp["tokens"] >= 0) & (inp["tokens"] < w.V)).all()
        u = inp["uniforms"]
        assert u.dtype == torch.float32 and ((u >= 0) & (u < 1)).all()
        assert inp["temperature"] == w.temperature


def test_peaks_present():
    w = shrink(WORKLOADS["c3"], B=1, V=4096)
    tl, _, _, _ = make_sequence(w, 0, 0)
    # 32 boosted ids per row stand out far above N(0, 9) draws
    top = torch.topk(tl.float(), 32, dim=-1).values
    assert (top[:, -1] > 3.0).all()


def test_draft_tokens_follow_draft_softmax():
    """Gumbel-max drafts: frequencies match softmax(row/T) (chi-square on V=6)."""
    from scipy.stats import chisquare
    from synthetic.generate import gumbel_max_draw

    g = torch.Generator().manual_seed(0)
    row = torch.randn(1, 6, generator=g)
    T = 0.7
    rows = row.expand(200000, 6)
    toks = gumbel_max_draw(rows, T, g)
    counts = torch.bincount(toks.long(), minlength=6).double().numpy()
    p = torch.softmax(row[0].double() / T, 0).numpy()
    assert chisquare(counts, 200000 * p).pvalue > 1e-3


def test_sweep_cells():
    for k in SWEEP_K:
        for n in SWEEP_NOISE:
            w = get_workload(f"sweep-k{k}-n{n:g}")
            assert w.B == 32 and w.V == 151936 and w.K == k and w.draft_noise_std == n
    assert WORKLOADS["c3"].ideal_bytes_per_step() == 64 * 19 * 128256 * 2
