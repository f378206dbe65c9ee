"""GPU parity of greedy-mode verification (spec_verify_greedy) against the
fp64 oracle's verify_greedy: an argmax involves no rounding, so outputs must
be identical, ties included (smallest token id), and failed sequences -1."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import speculative_sampling_verification_gb300 as sv
from synthetic import get_workload, make_inputs

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _to_dev(t: torch.Tensor, misalign: bool = False) -> torch.Tensor:
    if not misalign:
        return t.contiguous().to(DEV)
    flat = torch.empty(t.numel() + 1, dtype=t.dtype, device=DEV)
    view = flat[1:].view(t.shape)
    view.copy_(t.to(DEV))
    return view


def _run(target, tokens, misalign=False):
    B, K1, V = target.shape
    dt = sv.SV_BF16 if target.dtype == torch.bfloat16 else sv.SV_F32
    ws = torch.empty(max(256, sv.sv_greedy_workspace_size(B, K1 - 1, V, dt)), dtype=torch.uint8,
                     device=DEV)
    out = torch.empty(B, K1, dtype=torch.int32, device=DEV)
    nacc = torch.empty(B, dtype=torch.int32, device=DEV)
    assert sv.spec_verify_greedy(_to_dev(target, misalign), _to_dev(tokens.to(torch.int32)), out,
                                 nacc, ws) == 0
    torch.cuda.synchronize()
    status = sv.sv_read_device_status(ws)
    ref = oracle.verify_greedy(target.to(torch.float64).numpy(), tokens.numpy())
    return out.cpu().numpy(), nacc.cpu().numpy(), status, ref


def _check(out, nacc, status, ref):
    assert (out == ref.out_tokens).all(), (np.nonzero((out != ref.out_tokens).any(1))[0][:8])
    assert (nacc == ref.n_accepted).all()
    assert status == int(np.bitwise_or.reduce(ref.status))


def _case(B, K, V, dtype, seed, tie_heavy=False):
    g = torch.Generator().manual_seed(seed)
    if tie_heavy:
        target = torch.randint(0, 4, (B, K + 1, V), generator=g).to(dtype)
    else:
        target = (torch.randn(B, K + 1, V, generator=g) * 3).to(dtype)
    am = target[:, :K].float().argmax(-1)  # a first maximum (torch does not promise which)
    pick = torch.rand(B, K, generator=g)
    rnd = torch.randint(0, V, (B, K), generator=g)
    tokens = torch.where(pick < 0.7, am, rnd).to(torch.int64)
    return target, tokens


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("V", [1, 7, 33, 1000, 4097, 32000])
@pytest.mark.parametrize("K", [1, 3, 8])
@pytest.mark.parametrize("misalign", [False, True], ids=["aligned", "misaligned"])
def test_greedy_grid(dtype, V, K, misalign):
    target, tokens = _case(6, K, V, dtype, seed=V * 31 + K)
    _check(*_run(target, tokens, misalign))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("V", [5, 300, 70000])
def test_greedy_ties_go_to_the_smallest_id(dtype, V):
    target, tokens = _case(16, 4, V, dtype, seed=V, tie_heavy=True)
    # drafts that pick the *last* maximum must be rejected where a tie exists
    last = V - 1 - target[:, :4].float().flip(-1).argmax(-1)
    tokens[:8] = last[:8]
    _check(*_run(target, tokens))


@pytest.mark.parametrize("name", ["c2", "c3", "c4"])
def test_greedy_on_the_workloads(name):
    w = get_workload(name)
    inp = make_inputs(w, step=4)
    greedy_drafts = inp["draft"].float().argmax(-1)
    for tokens in (greedy_drafts, inp["tokens"].to(torch.int64)):
        out, nacc, status, ref = _run(inp["target"], tokens)
        assert status == 0
        _check(out, nacc, status, ref)


def test_greedy_masks_and_failures():
    target, tokens = _case(7, 3, 1024, torch.float32, seed=41)
    target[0, :, ::3] = float("-inf")      # masked entries never win
    target[1, 2, 10] = float("nan")
    target[2, 0, 11] = float("inf")
    target[3, 1, :] = float("-inf")
    tokens[4, 2] = 1024
    tokens[5, 0] = -1
    target[6, :, :-1] = float("-inf")      # one live token per row: all drafts != V-1 reject at 0
    out, nacc, status, ref = _run(target, tokens)
    assert list(ref.status) == [0, 32, 32, 64, 16, 16, 0]
    assert out[6, 0] == 1023
    _check(out, nacc, status, ref)
