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


def test_make_batch_follows_the_recipe():
    """The batched generator: shapes, dtypes, value distributions, peaks,
    drafts inside the vocabulary, uniforms in [0, 1), reproducible by step."""
    from synthetic import make_batch

    w = shrink(WORKLOADS["c3"], B=3, V=20000)
    a = make_batch(w, step=5)
    b = make_batch(w, step=5)
    for k in ("target", "draft", "tokens", "uniforms"):
        assert torch.equal(a[k], b[k])
    assert not torch.equal(a["target"], make_batch(w, step=6)["target"])
    assert a["target"].shape == (3, w.K + 1, w.V) and a["target"].dtype == torch.bfloat16
    assert a["draft"].shape == (3, w.K, w.V) and a["draft"].dtype == torch.bfloat16
    assert a["tokens"].dtype == torch.int32 and ((a["tokens"] >= 0) & (a["tokens"] < w.V)).all()
    u = a["uniforms"]
    assert u.shape == (3, w.K + 2) and u.dtype == torch.float32 and ((u >= 0) & (u < 1)).all()
    t = a["target"].float()
    top = torch.topk(t, w.peaks + 1, dim=-1).values
    assert (top[..., w.peaks - 1] > 3.0).all()          # 32 boosted ids per row
    body = t[t < 6.0]
    assert abs(body.std().item() - w.target_std) < 0.2
    gap = (a["draft"].float() - t[:, : w.K]).std().item()
    assert abs(gap - w.draft_noise_std) < 0.05          # noise, plus bf16 rounding
    # the drafted token is typically among the draft row's largest logits
    d = a["draft"].float()
    at = torch.gather(d, -1, a["tokens"].long()[..., None])[..., 0]
    assert (at > torch.quantile(d[0, 0], 0.99)).float().mean() > 0.9


def test_make_batch_drafts_follow_draft_softmax():
    """Gumbel-max drafts of the batched generator follow softmax(dl/T): every
    sequence has its own row, so the law is checked through the drafted
    token's probability, whose mean under x~ ~ p is E[sum_i p_i^2]."""
    from synthetic import make_batch

    w = shrink(WORKLOADS["c1"], B=40000, K=1, V=5, target_std=1.0, draft_noise_std=0.5,
               temperature=0.8)
    a = make_batch(w, step=0)
    d = a["draft"][:, 0].double()
    p = torch.softmax(d / 0.8, dim=-1)
    chosen = torch.gather(p, -1, a["tokens"].long())[:, 0]
    # E[p(x~)] under x~ ~ p equals sum_i p_i^2 per row
    expect = (p * p).sum(-1).mean().item()
    got = chosen.mean().item()
    assert abs(got - expect) < 4 * (p * p).sum(-1).std().item() / 200 + 0.005
