"""spec_verify_static, the entry point for callers that cannot allocate device
memory (it takes no workspace and uses the library's fixed scratch array
instead), against the workspace entry point on the same inputs, two calls in
a row.

Kept in a file of its own that sorts last, so that a run stopping at the
first failure has run every other test before it."""

import ctypes

import numpy as np
import pytest
import torch

import speculative_sampling_verification_gb300 as sv
from synthetic import WORKLOADS, make_inputs
from synthetic.configs import shrink

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _run_static(lib, args, temperature, B, K, V, dt):
    out = torch.full((B, K + 1), -7, dtype=torch.int32, device=DEV)
    nacc = torch.full((B,), -7, dtype=torch.int32, device=DEV)
    vp = ctypes.c_void_p
    rc = lib.spec_verify_static(vp(args[0].data_ptr()), vp(args[1].data_ptr()),
                                vp(args[2].data_ptr()), vp(args[3].data_ptr()), B, K, V, dt,
                                ctypes.c_float(temperature), vp(out.data_ptr()),
                                vp(nacc.data_ptr()),
                                vp(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return rc, out.cpu().numpy(), nacc.cpu().numpy()


def test_static_scratch_matches_workspace_entry_point_on_two_calls():
    lib = sv.load_library(build=True)
    for step, w in enumerate((WORKLOADS["c2"], shrink(WORKLOADS["c3"], B=16, V=60001))):
        dt = sv.SV_BF16 if w.dtype == "bf16" else sv.SV_F32
        for call in range(2):
            inp = make_inputs(w, step=10 * step + call)
            args = [inp[k].to(DEV) for k in ("target", "draft", "tokens", "uniforms")]
            out_ws, nacc_ws = sv.verify(*args, inp["temperature"])
            torch.cuda.synchronize()
            rc, out_st, nacc_st = _run_static(lib, args, inp["temperature"], w.B, w.K, w.V, dt)
            assert rc == 0, sv.sv_status_string(rc)
            # token ids and counts: the tests' tolerance for integer outputs is exact equality
            assert np.array_equal(out_st, out_ws.cpu().numpy())
            assert np.array_equal(nacc_st, nacc_ws.cpu().numpy())


def test_static_scratch_rejects_problems_beyond_its_size():
    lib = sv.load_library(build=True)
    B, K, V = 512, 8, 256000
    assert lib.sv_workspace_size(B, K, V, sv.SV_F32) > (8 << 20)
    vp = ctypes.c_void_p
    rc = lib.spec_verify_static(vp(16), vp(16), vp(16), vp(16), B, K, V, sv.SV_F32,
                                ctypes.c_float(1.0), vp(16), vp(16), None)
    assert rc == 8 and "scratch" in sv.sv_status_string(rc)


def test_static_scratch_inside_graph_capture_after_a_warm_up_call():
    """One call outside capture looks up the scratch address; a call captured
    into a CUDA graph then reuses it, and each replay matches the workspace
    entry point on the inputs the graph reads."""
    lib = sv.load_library(build=True)
    w = shrink(WORKLOADS["c3"], B=8, V=30001)
    dt = sv.SV_BF16 if w.dtype == "bf16" else sv.SV_F32
    inp = make_inputs(w, step=3)
    args = [inp[k].to(DEV) for k in ("target", "draft", "tokens", "uniforms")]
    out = torch.full((w.B, w.K + 1), -7, dtype=torch.int32, device=DEV)
    nacc = torch.full((w.B,), -7, dtype=torch.int32, device=DEV)
    vp = ctypes.c_void_p

    def call():
        return lib.spec_verify_static(vp(args[0].data_ptr()), vp(args[1].data_ptr()),
                                      vp(args[2].data_ptr()), vp(args[3].data_ptr()), w.B, w.K,
                                      w.V, dt, ctypes.c_float(inp["temperature"]),
                                      vp(out.data_ptr()), vp(nacc.data_ptr()),
                                      vp(torch.cuda.current_stream().cuda_stream))

    side = torch.cuda.Stream(DEV)
    with torch.cuda.stream(side):
        assert call() == 0  # the warm-up call, outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        rc = call()
    assert rc == 0, sv.sv_status_string(rc)
    for step in (4, 5):  # new inputs copied into the buffers the graph reads
        nxt = make_inputs(w, step=step)
        for a, k in zip(args, ("target", "draft", "tokens", "uniforms")):
            a.copy_(nxt[k].to(DEV))
        out.fill_(-7)
        nacc.fill_(-7)
        g.replay()
        torch.cuda.synchronize()
        out_ws, nacc_ws = sv.verify(*args, nxt["temperature"])
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), out_ws.cpu().numpy())
        assert np.array_equal(nacc.cpu().numpy(), nacc_ws.cpu().numpy())
