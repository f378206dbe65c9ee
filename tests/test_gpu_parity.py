"""Parity of the CUDA path (through the C ABI) with the fp64 oracle."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import speculative_sampling_verification_gb300 as sv
from synthetic import WORKLOADS, get_workload, make_inputs
from synthetic.configs import Workload, shrink
from tests import _parity, _pins

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=[1, 2], ids=["kernel_pair", "fused"])
def kernel_path(request):
    """Every test here runs on both paths: the streaming + draw kernel pair,
    and the fused kernel that the library takes for small calls."""
    sv.sv_force_path(request.param)
    yield request.param
    sv.sv_force_path(0)

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    sv.load_library(build=True)


def to_dev(t: torch.Tensor, misalign: bool = False) -> torch.Tensor:
    """Copy to the GPU; with `misalign`, place the data one element past a
    256-byte boundary so the base pointer is not 16-byte aligned."""
    if not misalign:
        return t.contiguous().to(DEV)
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
    view = flat[1:].view(t.shape)
    view.copy_(t.to(DEV))
    return view


def run_gpu(inp: dict, misalign: bool = False):
    args = [to_dev(inp["target"], misalign), to_dev(inp["draft"], misalign),
            to_dev(inp["tokens"]), to_dev(inp["uniforms"])]
    out, nacc, dbg = sv.verify(*args, inp["temperature"], debug=True)
    torch.cuda.synchronize()
    status = sv.sv_read_device_status(dbg["workspace"])
    return (out.cpu().numpy(), nacc.cpu().numpy(), status,
            {k: v.cpu().numpy() for k, v in dbg.items() if k != "workspace"})


def check_intermediates(dbg, ref, seqs=None):
    ok = ref.status == 0
    lse, thr, prob = dbg["row_lse"], dbg["thresholds"], dbg["sample_prob"]
    rmax, ratio = dbg["row_max"], dbg["ratios"]
    if seqs is not None:
        lse, thr, prob, rmax, ratio = lse[seqs], thr[seqs], prob[seqs], rmax[seqs], ratio[seqs]
    np.testing.assert_allclose(lse[ok], ref.lse[ok], rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(thr[ok], ref.thresholds[ok], rtol=1e-5, atol=1e-9)
    # the row maximum is one of the row's logits over T: equal up to fp64 rounding
    np.testing.assert_allclose(rmax[ok], ref.row_max[ok], rtol=1e-12, atol=0)
    # the ratio q/p itself, also where it exceeds 1 (the threshold is clamped there);
    # +inf (p = 0 < q) and 0 (q = 0) must match exactly
    np.testing.assert_allclose(ratio[ok], ref.ratios[ok], rtol=1e-5, atol=1e-300)
    assert np.array_equal(np.isinf(ratio[ok]), np.isinf(ref.ratios[ok]))
    # the drawn token's normalised weight comes from the float-float pass
    np.testing.assert_allclose(prob[ok], ref.sample_prob[ok], rtol=1e-8, atol=1e-15)


def parity_full(inp, misalign=False, intermediates=True):
    out, nacc, status, dbg = run_gpu(inp, misalign)
    ref = oracle.verify_inputs(inp)
    rep = _parity.compare(out, nacc, ref, inp["tokens"].numpy())
    rep.assert_ok(max_excused_rate=1e-5)
    if intermediates:
        check_intermediates(dbg, ref)
    expected_status = int(np.bitwise_or.reduce(ref.status)) if len(ref.status) else 0
    assert status == expected_status, (status, expected_status)
    return rep


def parity_sampled(w: Workload, step: int, seqs):
    """Full-size run on the GPU; the oracle checks the sampled sequences."""
    inp = make_inputs(w, step=step)
    out, nacc, status, dbg = run_gpu(inp)
    assert status == 0
    sub = {k: (v[seqs] if torch.is_tensor(v) else v) for k, v in inp.items()}
    ref = oracle.verify_inputs(sub)
    rep = _parity.compare(out[seqs], nacc[seqs], ref, inp["tokens"].numpy()[seqs])
    rep.assert_ok(max_excused_rate=1e-5)
    check_intermediates(dbg, ref, seqs)
    # properties that hold for every sequence
    assert ((nacc >= 0) & (nacc <= w.K)).all()
    return rep, nacc


# ---------------------------------------------------------------- hand-worked cases

def test_golden_hand_cases_on_gpu():
    for c in _pins.load_golden():
        tl = torch.from_numpy(_pins.probs_to_logits(c["target_probs"])).float()[None]
        dl = torch.from_numpy(_pins.probs_to_logits(c["draft_probs"])).float()[None]
        inp = {"target": tl, "draft": dl,
               "tokens": torch.tensor([c["tokens"]], dtype=torch.int32),
               "uniforms": torch.tensor([c["uniforms"]], dtype=torch.float32),
               "temperature": 1.0}
        out, nacc, status, dbg = run_gpu(inp)
        assert status == 0, c["name"]
        assert out[0].tolist() == c["expected_out"], (c["name"], out[0])
        assert int(nacc[0]) == c["expected_n_accepted"], c["name"]
        np.testing.assert_allclose(dbg["thresholds"][0], c["expected_thresholds"], atol=1e-6)
        np.testing.assert_allclose(dbg["ratios"][0], [float(v) for v in c["expected_ratios"]],
                                   rtol=1e-6)
        np.testing.assert_allclose(dbg["sample_prob"][0], c["expected_sample_prob"], atol=1e-6)


# ---------------------------------------------------------------- shape grid

GRID = [(dt, V, K, T)
        for dt in ("bf16", "f32")
        for V in (1, 2, 7, 33, 1000, 4097, 9001)
        for K in (1, 3, 8)
        for T in (0.6, 1.0)]


@pytest.mark.parametrize("dt,V,K,T", GRID)
def test_shape_grid(dt, V, K, T):
    w = Workload(f"grid-{dt}-{V}-{K}-{T}", B=6, K=K, V=V, dtype=dt, target_std=2.5,
                 draft_noise_std=0.8, temperature=T, seed=3000 + V + 7 * K)
    inp = make_inputs(w)
    parity_full(inp)
    if V * (2 if dt == "bf16" else 4) % 16 == 0 or V > 1000:
        parity_full(inp, misalign=True)


def test_k_max_64_and_v_one():
    parity_full(make_inputs(Workload("k64", B=3, K=64, V=515, dtype="bf16", target_std=1.0,
                                     draft_noise_std=0.2, temperature=1.0, seed=41)))
    parity_full(make_inputs(Workload("v1", B=4, K=5, V=1, dtype="f32", target_std=1.0,
                                     draft_noise_std=0.2, temperature=1.0, seed=42)))


def test_many_segments_and_chunks():
    # several streaming segments per row and several sampling chunks, ragged tails
    for dt, V in (("bf16", 70001), ("f32", 50003), ("bf16", 65536)):
        w = Workload("seg", B=3, K=2, V=V, dtype=dt, target_std=3.0, draft_noise_std=1.0,
                     temperature=0.9, seed=V)
        parity_full(make_inputs(w))


# ---------------------------------------------------------------- the workloads

def test_workload_c1():
    parity_full(make_inputs(WORKLOADS["c1"]))


def test_workload_c2_steps():
    total = _parity.ParityReport()
    for step in range(12):
        total.add(parity_full(make_inputs(WORKLOADS["c2"], step=step), intermediates=step < 2))
    total.assert_ok(max_excused_rate=1e-5)


def test_workload_c3_full_size_sampled():
    w = WORKLOADS["c3"]
    rng = np.random.default_rng(0)
    seqs = np.sort(rng.choice(w.B, 12, replace=False))
    parity_sampled(w, 0, seqs)


def test_workload_c4_full_size_sampled():
    w = WORKLOADS["c4"]
    seqs = np.array([0, 1, 77, 128, 200, 255])
    parity_sampled(w, 0, seqs)


@pytest.mark.parametrize("k,noise", [(1, 0.1), (4, 1.0), (16, 2.0)])
def test_sweep_cells_sampled(k, noise):
    w = get_workload(f"sweep-k{k}-n{noise:g}")
    parity_sampled(w, 0, np.array([0, 5, 31]))


def test_small_versions_of_workloads_in_full():
    for name in ("c2", "c3", "c4"):
        w = shrink(WORKLOADS[name], B=8, V=min(WORKLOADS[name].V, 20011))
        parity_full(make_inputs(w, step=1))


# ---------------------------------------------------------------- edge cases

def _base(B=5, K=3, V=64, dt="f32", seed=7):
    w = Workload("edge", B=B, K=K, V=V, dtype=dt, target_std=2.0, draft_noise_std=0.7,
                 temperature=1.0, seed=seed)
    return make_inputs(w)


def test_masked_entries_and_masked_drafts():
    inp = _base()
    t, d, tok = inp["target"], inp["draft"], inp["tokens"]
    t[0, :, :20] = float("-inf")
    d[0, :, 10:30] = float("-inf")
    # drafted token with p = 0 and q > 0 (accepts), and with q = 0 (rejects)
    tok[1, 0] = 5
    d[1, 0, 5] = float("-inf")
    tok[2, 1] = 9
    t[2, 1, 9] = float("-inf")
    tok[3, 0] = 11
    t[3, 0, 11] = float("-inf")
    d[3, 0, 11] = float("-inf")
    parity_full(inp)


def test_failures_reported_per_sequence():
    inp = _base(B=7)
    inp["target"][1, 2, 4] = float("nan")
    inp["draft"][2, 0, :] = float("-inf")
    inp["tokens"][3, 1] = 64
    inp["tokens"][4, 0] = -3
    inp["uniforms"][5, 2] = float("nan")
    inp["target"][6, 0, 0] = float("inf")
    out, nacc, status, _ = run_gpu(inp)
    ref = oracle.verify_inputs(inp)
    assert list(ref.status) == [0, 32, 64, 16, 16, 128, 32]
    assert status == (32 | 64 | 16 | 128)
    for b in range(1, 7):
        assert (out[b] == -1).all() and nacc[b] == -1
    _parity.compare(out, nacc, ref, inp["tokens"].numpy()).assert_ok()


def test_uniform_one_strictness_and_zero_residual():
    inp = _base(B=4, K=2, V=50)
    t, d, u = inp["target"], inp["draft"], inp["uniforms"]
    d[0] = t[0, :2]          # q == p: threshold 1, u = 1 rejects, residual is zero -> falls back to q
    u[0, 0] = 1.0
    u[1, :2] = 0.0           # accepted twice; bonus draw with u = 1 takes the last positive token
    u[1, 3] = 1.0
    t[1, 2, 40:] = float("-inf")
    u[2, 0] = 1.0            # u = 1 always rejects
    u[3, 2] = 0.0            # residual draw at u = 0
    u[3, 0] = 1.0
    rep = parity_full(inp)
    ref = oracle.verify_inputs(inp)
    assert ref.residual_fallback[0]
    assert ref.out_tokens[1, 2] == 39


def test_bf16_and_temperature_rescaling_is_exact():
    w = shrink(WORKLOADS["c3"], B=4, V=3001)
    inp = make_inputs(w)
    out1, nacc1, _, _ = run_gpu(inp)
    inp2 = dict(inp)
    inp2["target"] = inp["target"] * 2  # exact in bf16
    inp2["draft"] = inp["draft"] * 2
    inp2["temperature"] = inp["temperature"] * 2
    out2, nacc2, _, _ = run_gpu(inp2)
    assert np.array_equal(out1, out2) and np.array_equal(nacc1, nacc2)


def test_empty_batch_is_a_no_op():
    t = torch.empty(0, 3, 10, device=DEV)
    d = torch.empty(0, 2, 10, device=DEV)
    tok = torch.empty(0, 2, dtype=torch.int32, device=DEV)
    u = torch.empty(0, 4, device=DEV)
    out, nacc = sv.verify(t, d, tok, u, 1.0)
    assert out.shape == (0, 3) and nacc.shape == (0,)


# ---------------------------------------------------------------- API behaviour

def test_host_entry_point_matches_device_entry_point():
    w = shrink(WORKLOADS["c2"], B=8, V=32000)
    inp = make_inputs(w, step=3, pin_memory=True)
    out_d, nacc_d, _, _ = run_gpu(inp)
    B, K, V = w.B, w.K, w.V
    staging = torch.empty(sv.sv_staging_size(B, K, V, sv.SV_BF16), dtype=torch.uint8, device=DEV)
    ws = torch.empty(sv.sv_workspace_size(B, K, V, sv.SV_BF16), dtype=torch.uint8, device=DEV)
    h_out = torch.empty(B, K + 1, dtype=torch.int32).pin_memory()
    h_nacc = torch.empty(B, dtype=torch.int32).pin_memory()
    rc = sv.spec_verify_host(inp["target"], inp["draft"], inp["tokens"], inp["uniforms"],
                             inp["temperature"], h_out, h_nacc, staging, ws)
    assert rc == 0
    assert np.array_equal(h_out.numpy(), out_d) and np.array_equal(h_nacc.numpy(), nacc_d)


def test_async_host_entry_point_pipelined_over_two_lanes():
    """spec_verify_host_async on alternating (stream, staging, workspace)
    lanes: each step's outputs, read once its lane's stream is done, equal the
    device entry point's."""
    w = shrink(WORKLOADS["c2"], B=8, V=32000)
    B, K, V = w.B, w.K, w.V
    steps = [make_inputs(w, step=20 + i, pin_memory=True) for i in range(6)]
    want = [run_gpu(inp)[:2] for inp in steps]
    lanes = []
    for _ in range(2):
        lanes.append((torch.cuda.Stream(),
                      torch.empty(sv.sv_staging_size(B, K, V, sv.SV_BF16), dtype=torch.uint8, device=DEV),
                      torch.empty(sv.sv_workspace_size(B, K, V, sv.SV_BF16), dtype=torch.uint8, device=DEV),
                      torch.empty(B, K + 1, dtype=torch.int32).pin_memory(),
                      torch.empty(B, dtype=torch.int32).pin_memory()))
    got = [None] * len(steps)
    for i, inp in enumerate(steps + [None, None]):
        st, staging, ws, h_out, h_nacc = lanes[i % 2]
        if i >= 2:  # the previous step on this lane: wait, read its results
            st.synchronize()
            assert sv.sv_read_device_status(ws, st) == 0
            got[i - 2] = (h_out.numpy().copy(), h_nacc.numpy().copy())
        if inp is not None:
            assert sv.spec_verify_host_async(inp["target"], inp["draft"], inp["tokens"],
                                             inp["uniforms"], inp["temperature"], h_out, h_nacc,
                                             staging, ws, stream=st) == 0
    for (o, n), (wo, wn) in zip(got, want):
        assert np.array_equal(o, wo) and np.array_equal(n, wn)


@pytest.mark.parametrize("B,V", [(16, 50000), (24, 128256)])
def test_graph_capture_replay_and_determinism(B, V):
    # 27 MB of logits is one sequence group; 105 MB is three, whose draws run
    # on the library's second stream, forked and joined inside the capture.
    w = shrink(WORKLOADS["c3"], B=B, V=V)
    inp = make_inputs(w, step=2)
    args = [to_dev(inp[k]) for k in ("target", "draft", "tokens", "uniforms")]
    B, K = w.B, w.K
    out = torch.empty(B, K + 1, dtype=torch.int32, device=DEV)
    nacc = torch.empty(B, dtype=torch.int32, device=DEV)
    ws = sv.new_workspace(B, K, w.V, sv.SV_BF16, DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        assert sv.spec_verify(*args, inp["temperature"], out, nacc, ws) == 0  # first call: set-up
    torch.cuda.synchronize()
    ref_out, ref_nacc = out.clone(), nacc.clone()
    ref = oracle.verify_inputs(inp)
    _parity.compare(ref_out.cpu().numpy(), ref_nacc.cpu().numpy(), ref,
                    inp["tokens"].numpy()).assert_ok()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        sv.spec_verify(*args, inp["temperature"], out, nacc, ws)
    for _ in range(3):
        out.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, ref_out) and torch.equal(nacc, ref_nacc)
