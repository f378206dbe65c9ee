"""GPU parity of top-k filtered verification (spec_verify_topk) against the
fp64 oracle's verify_topk: the kept sets are an exact selection (ties to the
smaller id, -0 equal to +0), so outputs must match decision for decision,
excusing only decisions within the parity margin of the oracle's threshold."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import speculative_sampling_verification_gb300 as sv
from synthetic import WORKLOADS, make_inputs, make_topk_inputs
from synthetic.configs import Workload, shrink
from tests import _parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv.load_library(build=True)


def _to_dev(t: torch.Tensor, misalign: bool = False) -> torch.Tensor:
    if not misalign:
        return t.contiguous().to(DEV)
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
    view = flat[1:].view(t.shape)
    view.copy_(t.to(DEV))
    return view


def run_gpu(inp, top_k, misalign=False):
    B, K1, V = inp["target"].shape
    dt = sv.SV_BF16 if inp["target"].dtype == torch.bfloat16 else sv.SV_F32
    ws = torch.empty(max(256, sv.sv_topk_workspace_size(B, K1 - 1, V, dt, top_k)),
                     dtype=torch.uint8, device=DEV)
    out, nacc = sv.verify_topk(_to_dev(inp["target"], misalign), _to_dev(inp["draft"], misalign),
                               _to_dev(inp["tokens"]), _to_dev(inp["uniforms"]),
                               inp["temperature"], top_k, workspace=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), nacc.cpu().numpy(), sv.sv_read_device_status(ws)


def oracle_topk(inp, top_k):
    f64 = lambda t: t.to(torch.float64).numpy()
    return oracle.verify_topk(f64(inp["target"]), f64(inp["draft"]), inp["tokens"].numpy(),
                              inp["uniforms"].to(torch.float64).numpy(), inp["temperature"], top_k)


def parity(inp, top_k, misalign=False):
    out, nacc, status = run_gpu(inp, top_k, misalign)
    ref = oracle_topk(inp, top_k)
    rep = _parity.compare(out, nacc, ref, inp["tokens"].numpy())
    rep.assert_ok(max_excused_rate=1e-5)
    assert status == int(np.bitwise_or.reduce(ref.status)), (status, ref.status)
    return rep, ref


def _w(B, K, V, dt, seed, T=1.0, std=2.0, noise=0.7):
    return Workload("topk", B=B, K=K, V=V, dtype=dt, target_std=std, draft_noise_std=noise,
                    temperature=T, seed=seed)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("V", [7, 33, 1000, 4097, 32000])
@pytest.mark.parametrize("top_k", [1, 5, 50, 256])
@pytest.mark.parametrize("K", [1, 4])
def test_topk_grid(dt, V, top_k, K):
    if top_k >= V:
        top_k = V - 1
    w = _w(6, K, V, dt, seed=V * 7 + top_k + K, T=0.8 if K == 4 else 1.3)
    parity(make_topk_inputs(w, top_k), top_k, misalign=(V == 1000))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("top_k", [1, 3, 40, 200])
def test_ties_at_the_cut_go_to_the_smaller_id(dt, top_k):
    """Integer logits in [0, 4): every cut falls inside a run of equal values,
    so the kept set depends on the id tie-break (and -0.0 counts as +0.0)."""
    g = torch.Generator().manual_seed(top_k)
    B, K, V = 8, 3, 700
    inp = make_inputs(_w(B, K, V, dt, seed=top_k))
    inp["target"] = torch.randint(0, 4, (B, K + 1, V), generator=g).to(inp["target"].dtype)
    inp["draft"] = torch.randint(0, 4, (B, K, V), generator=g).to(inp["draft"].dtype)
    zeros = inp["target"] == 0
    flip = torch.rand(zeros.shape, generator=g) < 0.5
    inp["target"][zeros & flip] = -0.0
    inp["draft"][inp["draft"] == 0] = -0.0
    # drafts among the row maxima, some at the largest id (outside the kept set)
    am = inp["draft"].float().argmax(-1).to(torch.int32)
    last = (V - 1 - inp["draft"].float().flip(-1).argmax(-1)).to(torch.int32)
    inp["tokens"] = torch.where(torch.rand(B, K, generator=g) < 0.5, am, last)
    parity(inp, top_k)


def test_topk_one_is_greedy_like_and_topk_full_is_verify():
    inp = make_inputs(_w(10, 4, 3000, "f32", seed=5))
    rep, ref = parity(inp, 1)
    # top-1: every kept row is one-hot, the draw is its argmax
    assert (ref.status == 0).all()
    # top_k >= V is the unfiltered call
    B, K1, V = inp["target"].shape
    out, nacc, _ = run_gpu(inp, V)
    ref_full = oracle.verify_inputs(inp)
    _parity.compare(out, nacc, ref_full, inp["tokens"].numpy()).assert_ok(1e-5)


def test_failures_and_masked_rows():
    inp = make_topk_inputs(_w(8, 3, 500, "f32", seed=11), 20)
    t, d, tok, u = inp["target"], inp["draft"], inp["tokens"], inp["uniforms"]
    t[0, 1, 7] = float("nan")               # NaN: nonfinite
    d[1, 2, 300] = float("inf")             # +inf: nonfinite
    t[2, 3, :] = float("-inf")              # empty row
    t[3, 0, :490] = float("-inf")           # fewer finite entries than top_k
    d[3, 0, :495] = float("-inf")
    tok[4, 1] = 500                         # token out of range
    u[5, 2] = 1.5                           # uniform out of range
    t[6, 2, :] = -3.0                       # a constant row (all ties)
    t[7, :, :] = -float("inf")              # every target row empty
    t[7, :, 3] = 0.0
    parity(inp, 20)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_adversarial_orders_and_late_nan(dt):
    """Ascending rows make every element a new candidate (the buffer overflows
    and the row is selected exactly from memory); descending rows are decided
    by the first threshold; a NaN far into an ascending row must still fail
    its sequence."""
    B, K, V, k = 6, 2, 30011, 64
    inp = make_topk_inputs(_w(B, K, V, dt, seed=21), k)
    g = torch.Generator().manual_seed(5)
    base = torch.randn(V, generator=g).sort().values * 4
    for b in range(4):
        inp["target"][b] = base.to(inp["target"].dtype)
        inp["draft"][b] = (base + 0.3 * torch.randn(V, generator=g)).sort().values.to(inp["draft"].dtype)
    inp["target"][1] = inp["target"][1].flip(-1)
    inp["draft"][1] = inp["draft"][1].flip(-1)
    inp["target"][2, 1, V - 40] = float("nan")
    # drafts near the top of the (ascending) draft rows
    inp["tokens"][:4] = torch.randint(V - 3 * k, V, (4, K), generator=g).to(torch.int32)
    inp["tokens"][1] = torch.randint(0, 2 * k, (K,), generator=g).to(torch.int32)
    parity(inp, k)


def test_uniform_extremes_and_zero_residual():
    inp = make_topk_inputs(_w(6, 3, 400, "f32", seed=13), 16)
    u = inp["uniforms"]
    u[0, :] = 0.0
    u[1, :] = 1.0
    u[2, :3] = 0.999999
    # identical target and draft rows: every draft accepted unless u = 1, and
    # the zero residual falls back to the target row
    inp["draft"][3] = inp["target"][3, :3]
    u[3, 1] = 1.0
    parity(inp, 16)


@pytest.mark.parametrize("top_k", [1, 20, 256])
def test_small_versions_of_workloads(top_k):
    for name in ("c2", "c3", "c4"):
        w = shrink(WORKLOADS[name], B=6, V=min(WORKLOADS[name].V, 20011))
        parity(make_topk_inputs(w, top_k, step=1), top_k)


def test_full_size_128k_vocabulary_sampled():
    """64 sequences of 17 rows over a 128256-token bf16 vocabulary with peaked
    targets, top-50; the oracle checks a sample of the sequences."""
    w = WORKLOADS["c3"]
    top_k = 50
    inp = make_topk_inputs(w, top_k)
    out, nacc, status = run_gpu(inp, top_k)
    assert status == 0
    seqs = np.array([0, 9, 31, 40, 63])
    sub = {k: (v[seqs] if torch.is_tensor(v) else v) for k, v in inp.items()}
    ref = oracle_topk(sub, top_k)
    _parity.compare(out[seqs], nacc[seqs], ref, inp["tokens"].numpy()[seqs]).assert_ok(1e-5)
    assert ((nacc >= 0) & (nacc <= w.K)).all()
    # every emitted token is in the kept set of the row it was drawn from
    emitted = out[np.arange(w.B), nacc]
    for b in range(w.B):
        j = int(nacc[b])
        row = inp["target"][b, j].float()
        kth = torch.topk(row, top_k).values[-1]
        assert row[emitted[b]] >= kth


def test_empty_batch_is_a_no_op():
    ws = torch.zeros(256, dtype=torch.uint8, device=DEV)
    e = torch.empty(0, 4, 100, device=DEV)
    e3 = torch.empty(0, 3, 100, device=DEV)
    tok = torch.empty(0, 3, dtype=torch.int32, device=DEV)
    u = torch.empty(0, 5, dtype=torch.float32, device=DEV)
    out = torch.empty(0, 4, dtype=torch.int32, device=DEV)
    nacc = torch.empty(0, dtype=torch.int32, device=DEV)
    assert sv.spec_verify_topk(e, e3, tok, u, 1.0, 10, out, nacc, ws) == 0


def test_graph_capture_replay():
    inp = make_topk_inputs(_w(16, 4, 5000, "bf16", seed=3), 32)
    B, K1, V = inp["target"].shape
    args = [_to_dev(inp[k]) for k in ("target", "draft", "tokens", "uniforms")]
    ws = torch.empty(sv.sv_topk_workspace_size(B, K1 - 1, V, sv.SV_BF16, 32), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty(B, K1, dtype=torch.int32, device=DEV)
    nacc = torch.empty(B, dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert sv.spec_verify_topk(*args, inp["temperature"], 32, out, nacc, ws, stream=s) == 0
    torch.cuda.synchronize()
    first = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert sv.spec_verify_topk(*args, inp["temperature"], 32, out, nacc, ws, stream=s) == 0
    for _ in range(3):
        out.fill_(-7)
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, first)
    ref = oracle_topk(inp, 32)
    _parity.compare(out.cpu().numpy(), nacc.cpu().numpy(), ref, inp["tokens"].numpy()).assert_ok(1e-5)


def test_k256_on_a_256000_f32_vocabulary_sampled():
    """The largest k on the widest rows (f32, 256000 entries, 32 sequences of
    9 rows); the oracle checks a sample of the sequences."""
    w = shrink(WORKLOADS["c4"], B=32)
    top_k = 256
    inp = make_topk_inputs(w, top_k)
    out, nacc, status = run_gpu(inp, top_k)
    assert status == 0
    seqs = np.array([0, 13, 31])
    sub = {k: (v[seqs] if torch.is_tensor(v) else v) for k, v in inp.items()}
    _parity.compare(out[seqs], nacc[seqs], oracle_topk(sub, top_k),
                    inp["tokens"].numpy()[seqs]).assert_ok(1e-5)
    assert ((nacc >= 0) & (nacc <= w.K)).all()
