"""GPU parity of nucleus (top-p) filtered verification (spec_verify_topp)
against the fp64 oracle's verify_topp. The kept count of every row must match
the oracle's unless top_p lies within CUT_MARGIN of one of the cumulative sums
at the oracle's cut (the GPU sums float-float weights in another order);
sequences whose rows all match must then agree decision for decision, with
the usual margin for decisions on a rounding boundary."""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

import oracle
import speculative_sampling_verification_gb300 as sv
from synthetic import WORKLOADS, make_inputs, make_topp_inputs
from synthetic.configs import Workload, shrink
from tests import _parity

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
CUT_MARGIN = 1e-9


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


def run_gpu(inp, top_p, misalign=False):
    out, nacc, kept = sv.verify_topp(_to_dev(inp["target"], misalign),
                                     _to_dev(inp["draft"], misalign), _to_dev(inp["tokens"]),
                                     _to_dev(inp["uniforms"]), inp["temperature"], top_p)
    torch.cuda.synchronize()
    return out.cpu().numpy(), nacc.cpu().numpy(), kept.cpu().numpy()


def oracle_topp(inp, top_p):
    f64 = lambda t: t.to(torch.float64).numpy()
    return oracle.verify_topp(f64(inp["target"]), f64(inp["draft"]), inp["tokens"].numpy(),
                              f64(inp["uniforms"]), inp["temperature"], top_p)


def _subset(res, mask):
    return type(res)(*[getattr(res, f.name)[mask] for f in dataclasses.fields(res)])


def parity(inp, top_p, misalign=False, max_mismatched_rows=None):
    out, nacc, kept = run_gpu(inp, top_p, misalign)
    n = oracle_topp(inp, top_p)
    mism = kept != n.kept
    assert (n.cut_margin[mism] < CUT_MARGIN).all(), (
        np.argwhere(mism)[:5], kept[mism][:5], n.kept[mism][:5], n.cut_margin[mism][:5])
    if max_mismatched_rows is not None:
        assert mism.sum() <= max_mismatched_rows
    ok = ~mism.any(axis=1)
    rep = _parity.compare(out[ok], nacc[ok], _subset(n.result, ok), inp["tokens"].numpy()[ok])
    rep.assert_ok(max_excused_rate=1e-5)
    return n, kept, mism


def _w(B, K, V, dt, seed, T=1.0, std=2.0, noise=0.7):
    return Workload("topp", B=B, K=K, V=V, dtype=dt, target_std=std, draft_noise_std=noise,
                    temperature=T, seed=seed)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("V", [7, 33, 1000, 4097, 32000])
@pytest.mark.parametrize("top_p", [0.1, 0.5, 0.9, 0.99])
@pytest.mark.parametrize("K", [1, 4])
def test_topp_grid(dt, V, top_p, K):
    w = _w(6, K, V, dt, seed=V * 11 + int(top_p * 100) + K, T=0.8 if K == 4 else 1.3)
    parity(make_topp_inputs(w, top_p), top_p, misalign=(V == 1000))


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("std", [0.05, 0.5, 4.0])
def test_flat_and_peaked_rows(dt, std):
    """Flat rows keep most of the vocabulary (several histogram levels);
    peaked rows keep a handful."""
    w = _w(4, 3, 20011, dt, seed=int(std * 100), std=std)
    parity(make_topp_inputs(w, 0.9), 0.9)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("top_p", [0.05, 0.3, 0.7])
def test_ties_at_the_cut_go_to_the_smaller_id(dt, top_p):
    """Integer logits: the cut falls inside a run of equal values, resolved by
    id (and -0.0 counts as +0.0); a constant row is all ties."""
    g = torch.Generator().manual_seed(int(top_p * 100))
    B, K, V = 6, 2, 900
    inp = make_inputs(_w(B, K, V, dt, seed=5))
    inp["target"] = torch.randint(0, 3, (B, K + 1, V), generator=g).to(inp["target"].dtype)
    inp["draft"] = torch.randint(0, 3, (B, K, V), generator=g).to(inp["draft"].dtype)
    inp["target"][inp["target"] == 0] = -0.0
    inp["target"][0, 1, :] = 1.0
    inp["tokens"] = torch.randint(0, V, (B, K), generator=g).to(torch.int32)
    parity(inp, top_p)


def test_top_p_one_is_verify_and_tiny_is_top1():
    inp = make_inputs(_w(8, 4, 3000, "f32", seed=7))
    out, nacc, kept = run_gpu(inp, 1.0)
    assert (kept == 3000).all()
    _parity.compare(out, nacc, oracle.verify_inputs(inp), inp["tokens"].numpy()).assert_ok(1e-5)
    out, nacc, kept = run_gpu(inp, 1e-9)
    assert (kept == 1).all()
    f64 = lambda t: t.to(torch.float64).numpy()
    ref = oracle.verify_topk(f64(inp["target"]), f64(inp["draft"]), inp["tokens"].numpy(),
                             f64(inp["uniforms"]), inp["temperature"], 1)
    _parity.compare(out, nacc, ref, inp["tokens"].numpy()).assert_ok(1e-5)


def test_failures_and_masked_rows():
    inp = make_topp_inputs(_w(8, 3, 500, "f32", seed=11), 0.8)
    t, d, tok, u = inp["target"], inp["draft"], inp["tokens"], inp["uniforms"]
    t[0, 1, 7] = float("nan")
    d[1, 2, 300] = float("inf")
    t[2, 3, :] = float("-inf")
    t[3, 0, :490] = float("-inf")
    tok[4, 1] = 500
    u[5, 2] = 1.5
    t[6, 2, :] = -3.0
    t[7, :, :] = -float("inf")
    t[7, :, 3] = 0.0
    n, kept, _ = parity(inp, 0.8)
    fails = n.result.status != 0
    assert list(fails) == [True, True, True, False, True, True, False, False]


def test_small_versions_of_workloads():
    for name in ("c2", "c3", "c4"):
        w = shrink(WORKLOADS[name], B=6, V=min(WORKLOADS[name].V, 20011))
        for top_p in (0.5, 0.95):
            parity(make_topp_inputs(w, top_p, step=1), top_p)


@pytest.mark.parametrize("name,seqs", [("c3", [0, 17, 40, 63]), ("c4", [0, 99, 255])])
def test_full_size_sampled(name, seqs):
    """The full workload on the GPU; the oracle checks a sample."""
    w = WORKLOADS[name]
    top_p = 0.9
    inp = make_topp_inputs(w, top_p)
    out, nacc, kept = run_gpu(inp, top_p)
    seqs = np.array(seqs)
    sub = {k: (v[seqs] if torch.is_tensor(v) else v) for k, v in inp.items()}
    n = oracle_topp(sub, top_p)
    mism = kept[seqs] != n.kept
    assert (n.cut_margin[mism] < CUT_MARGIN).all()
    ok = ~mism.any(axis=1)
    _parity.compare(out[seqs][ok], nacc[seqs][ok], _subset(n.result, ok),
                    inp["tokens"].numpy()[seqs][ok]).assert_ok(1e-5)
    assert ((nacc >= 0) & (nacc <= w.K)).all()


def test_graph_capture_replay():
    inp = make_topp_inputs(_w(8, 4, 5000, "bf16", seed=3), 0.9)
    B, K1, V = inp["target"].shape
    args = [_to_dev(inp[k]) for k in ("target", "draft", "tokens", "uniforms")]
    ws = torch.empty(sv.sv_topp_workspace_size(B, K1 - 1, V, sv.SV_BF16), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty(B, K1, dtype=torch.int32, device=DEV)
    nacc = torch.empty(B, dtype=torch.int32, device=DEV)
    kept = torch.empty(B, 2 * K1 - 1, dtype=torch.int32, device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert sv.spec_verify_topp(*args, inp["temperature"], 0.9, out, nacc, ws, kept, stream=s) == 0
    torch.cuda.synchronize()
    first = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        assert sv.spec_verify_topp(*args, inp["temperature"], 0.9, out, nacc, ws, kept, stream=s) == 0
    for _ in range(3):
        out.fill_(-7)
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, first)


@pytest.mark.parametrize("top_p", [0.01, 0.999])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_top_p_extremes(top_p, dt):
    """A nucleus of one or two entries, and one that keeps nearly the whole
    mass (the cut deep in the tail, through the open last bins)."""
    w = _w(6, 3, 20011, dt, seed=int(top_p * 1000), std=1.5)
    parity(make_topp_inputs(w, top_p), top_p)


@pytest.mark.parametrize("dt,V,misalign", [("bf16", 4099, False), ("f32", 4099, False),
                                           ("f32", 40000, False), ("bf16", 140000, False),
                                           ("f32", 40000, True)])
@pytest.mark.parametrize("top_p", [0.3, 0.7])
def test_heavy_ties(dt, V, misalign, top_p):
    """Two-valued rows: more than 1024 entries share the cut's value, so the
    cut is resolved bit by bit over the key (across a cluster for the long
    rows, and with element loads for misaligned ones)."""
    g = torch.Generator().manual_seed(V + int(top_p * 10))
    B, K = 3, 2
    inp = make_inputs(_w(B, K, V, dt, seed=9))
    inp["target"] = torch.randint(0, 2, (B, K + 1, V), generator=g).to(inp["target"].dtype)
    inp["draft"] = torch.randint(0, 2, (B, K, V), generator=g).to(inp["draft"].dtype)
    inp["tokens"] = torch.randint(0, V, (B, K), generator=g).to(torch.int32)
    parity(inp, top_p, misalign=misalign)


@pytest.mark.parametrize("dt,V", [("f32", 400_003), ("bf16", 800_000)])
def test_rows_too_long_for_a_cluster(dt, V):
    """Rows beyond sixteen CTAs' shared memory take the kernel that re-reads
    the row from memory; the results are the same."""
    w = _w(2, 1, V, dt, seed=V % 1000, std=1.5)
    parity(make_topp_inputs(w, 0.9), 0.9)


@pytest.mark.parametrize("dt,V", [("bf16", 262_000), ("f32", 131_000)])
def test_eight_ctas_per_row(dt, V):
    """Rows of 512 KB: the largest cluster, eight CTAs, each holding 64 KB."""
    w = _w(2, 1, V, dt, seed=V % 997, std=1.5)
    for top_p in (0.3, 0.95):
        parity(make_topp_inputs(w, top_p), top_p)


@pytest.mark.parametrize("dt,V", [("f32", 40000), ("bf16", 100003)])
def test_misaligned_rows_on_a_cluster(dt, V):
    """Rows that are not 16-byte aligned take element loads into the cluster's
    shared memory (padded with -inf), here over two CTAs or more."""
    w = _w(3, 2, V, dt, seed=V % 991, std=2.0)
    for top_p in (0.5, 0.97):
        parity(make_topp_inputs(w, top_p), top_p, misalign=True)
