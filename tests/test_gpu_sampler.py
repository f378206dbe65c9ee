"""GPU parity of the draft-side sampler (spec_draft_sample) against the fp64
oracle's draft_sample: the drawn token bit-exact except at a draw whose
uniform lies within 1e-6 of a CDF breakpoint (counted, and below 1e-5 of the
draws), the drawn token's probability within 1e-8 relative, and failed rows
reported as -1 with their status bits."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import speculative_sampling_verification_gb300 as sv
from synthetic import get_workload, make_inputs
from synthetic.configs import shrink

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=[1, 2], ids=["kernel_pair", "fused"])
def kernel_path(request):
    """Every test here runs on both paths: the streaming + draw kernel pair,
    and the fused kernel that the library takes for small calls."""
    sv.sv_force_path(request.param)
    yield request.param
    sv.sv_force_path(0)

DEV = torch.device("cuda:0")
MARGIN = 1e-6


def _to_dev(t: torch.Tensor, misalign: bool = False) -> torch.Tensor:
    if not misalign:
        return t.contiguous().to(DEV)
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
    view = flat[1:].view(t.shape)
    view.copy_(t.to(DEV))
    return view


def _compare(tokens, prob, ref, status=0):
    """Token parity with the margin rule; probability parity on ok rows."""
    tokens = np.asarray(tokens).astype(np.int64)
    ok = ref.status == 0
    assert (tokens[~ok] == -1).all(), "failed rows must draw -1"
    diff = ok & (tokens != ref.tokens)
    excused = diff & (ref.sample_margin < MARGIN)
    assert not (diff & ~excused).any(), (np.nonzero(diff & ~excused)[0][:10],
                                        tokens[diff][:10], ref.tokens[diff][:10])
    assert excused.sum() <= max(1, 1e-5 * ok.sum())
    same = ok & ~diff
    if prob is not None and same.any():
        np.testing.assert_allclose(np.asarray(prob)[same], ref.sample_prob[same], rtol=1e-8)
    assert status == int(np.bitwise_or.reduce(ref.status)) if ref.status.size else True


def _run(logits, uniforms, T, misalign=False):
    lg = _to_dev(logits, misalign)
    u = _to_dev(uniforms)
    N, V = logits.shape
    dt = sv.SV_BF16 if logits.dtype == torch.bfloat16 else sv.SV_F32
    ws = torch.empty(max(256, sv.sv_sample_workspace_size(N, V, dt)), dtype=torch.uint8, device=DEV)
    out = torch.empty(N, dtype=torch.int32, device=DEV)
    prob = torch.empty(N, dtype=torch.float64, device=DEV)
    assert sv.spec_draft_sample(lg, u, T, out, ws, prob) == 0
    torch.cuda.synchronize()
    status = sv.sv_read_device_status(ws)
    ref = oracle.draft_sample(logits.to(torch.float64).numpy(), uniforms.to(torch.float64).numpy(), T)
    return out.cpu().numpy(), prob.cpu().numpy(), status, ref


def _rows(N, V, dtype, seed, sigma=2.5):
    g = torch.Generator().manual_seed(seed)
    logits = (torch.randn(N, V, generator=g, dtype=torch.float32) * sigma).to(dtype)
    uniforms = torch.rand(N, generator=g, dtype=torch.float32)
    return logits, uniforms


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("V", [1, 7, 33, 1000, 4097, 32000])
@pytest.mark.parametrize("N", [1, 5, 64])
@pytest.mark.parametrize("T", [0.6, 1.0])
def test_sampler_grid(dtype, V, N, T):
    logits, u = _rows(N, V, dtype, seed=V * 131 + N * 7 + int(T * 10))
    out, prob, status, ref = _run(logits, u, T)
    _compare(out, prob, ref, status)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_sampler_misaligned_rows(dtype):
    logits, u = _rows(9, 3001, dtype, seed=5)
    out, prob, status, ref = _run(logits, u, 0.8, misalign=True)
    _compare(out, prob, ref, status)


@pytest.mark.parametrize("name", ["c2", "c3", "c4"])
def test_sampler_on_the_workloads_draft_rows(name):
    # Every draft row of the workload's first step, with fresh uniforms.
    w = get_workload(name)
    inp = make_inputs(w, step=3)
    logits = inp["draft"].reshape(w.B * w.K, w.V)
    g = torch.Generator().manual_seed(17)
    u = torch.rand(w.B * w.K, generator=g, dtype=torch.float32)
    out, prob, status, ref = _run(logits, u, w.temperature)
    assert status == 0
    _compare(out, prob, ref, status)


def test_sampler_masks_edges_and_failures():
    V = 2048
    logits, _ = _rows(8, V, torch.float32, seed=23)
    logits[0, ::2] = float("-inf")        # masked entries are never drawn
    logits[1, 5] = float("nan")           # fails: nonfinite
    logits[2, 7] = float("inf")           # fails: nonfinite
    logits[3, :] = float("-inf")          # fails: empty row
    logits[6, :-1] = float("-inf")        # one live token
    u = torch.tensor([0.3, 0.3, 0.3, 0.3, float("nan"), 1.5, 0.0, 1.0], dtype=torch.float32)
    out, prob, status, ref = _run(logits, u, 1.0)
    assert list(ref.status) == [0, 32, 32, 64, 128, 128, 0, 0]
    assert out[6] == V - 1 and out[0] % 2 == 1
    assert status == 32 | 64 | 128
    _compare(out, prob, ref, status)


def test_sampler_u_zero_and_one_pick_first_and_last_positive():
    logits, _ = _rows(4, 500, torch.float32, seed=29)
    logits[:, :3] = float("-inf")
    logits[:, -2:] = float("-inf")
    u = torch.tensor([0.0, 1.0, 0.0, 1.0], dtype=torch.float32)
    out, prob, status, ref = _run(logits, u, 0.7)
    assert list(out) == [3, 497, 3, 497]
    _compare(out, prob, ref, status)
