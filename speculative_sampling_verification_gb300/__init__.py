"""GB300 (sm_103a) verification step of speculative sampling.

A thin ctypes binding over libspecverify.so (C ABI in include/spec_verify.h).
The functions keep the C names; they only marshal torch tensors into
pointers, sizes and the current CUDA stream. Every step of the verification
runs in the library's CUDA kernels; there is no fallback of any kind, and a
missing library raises.

The operation is the modified rejection sampling of "Accelerating Large
Language Model Decoding with Speculative Sampling" (Chen et al.; wikillm.com
paper card, §4.2 and Algorithm 2).
"""

from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB, build_library

__all__ = [
    "SV_BF16", "SV_F32", "StatusError", "load_library", "sv_workspace_size", "sv_staging_size",
    "spec_verify", "spec_verify_debug", "spec_verify_profiled", "spec_verify_host",
    "sv_read_device_status",
    "sv_status_string", "sv_kernels_per_call", "sv_topp_kernels_per_call", "spec_verify_static",
    "verify",
    "sv_sample_workspace_size", "spec_draft_sample", "draft_sample",
    "sv_greedy_workspace_size", "spec_verify_greedy", "verify_greedy", "sv_force_path",
    "sv_test_withhold_plans", "sv_topk_workspace_size", "spec_verify_topk", "verify_topk",
    "sv_topp_workspace_size", "spec_verify_topp", "verify_topp", "spec_verify_host_async",
    "sv_lmhead_workspace_size", "sv_lmhead_stats", "lmhead_stats", "EXPORTED_SYMBOLS",
]

SV_BF16 = 0
SV_F32 = 1
SV_OK = 0
DEVICE_BITS = {16: "token_range", 32: "nonfinite", 64: "empty_row", 128: "uniform_range",
               256: "timeout"}

EXPORTED_SYMBOLS = (
    "sv_workspace_size", "spec_verify", "spec_verify_debug", "spec_verify_profiled",
    "sv_staging_size",
    "spec_verify_host", "sv_read_device_status", "sv_status_string", "sv_kernels_per_call",
    "spec_verify_static", "sv_sample_workspace_size", "spec_draft_sample",
    "sv_greedy_workspace_size", "spec_verify_greedy", "sv_force_path", "sv_test_withhold_plans",
    "sv_topk_workspace_size", "spec_verify_topk", "sv_topp_workspace_size", "spec_verify_topp",
    "spec_verify_host_async", "sv_lmhead_workspace_size", "sv_lmhead_stats",
    "sv_topp_kernels_per_call",
)

_lib = None


class StatusError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {sv_status_string(code)} (code {code})")


def load_library(path: str | None = None, build: bool = False) -> ctypes.CDLL:
    """Load libspecverify.so (building it first when `build` is set)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB
    if build:
        p = build_library()
    if not os.path.exists(p):
        raise RuntimeError(f"libspecverify.so not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    dp = ctypes.c_void_p
    lib.sv_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.sv_workspace_size.restype = sz
    lib.sv_staging_size.argtypes = [i32, i32, i32, i32]
    lib.sv_staging_size.restype = sz
    core = [vp, vp, vp, vp, i32, i32, i32, i32, f32, vp, vp, vp, sz, vp]
    lib.spec_verify.argtypes = core
    lib.spec_verify.restype = i32
    lib.spec_verify_debug.argtypes = core + [dp, dp, dp, dp, dp]
    lib.spec_verify_debug.restype = i32
    lib.spec_verify_profiled.argtypes = core + [vp, vp, vp]
    lib.spec_verify_profiled.restype = i32
    lib.spec_verify_host.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, vp, vp, vp, sz, vp,
                                     sz, vp]
    lib.spec_verify_host.restype = i32
    lib.spec_verify_host_async.argtypes = lib.spec_verify_host.argtypes
    lib.spec_verify_host_async.restype = i32
    lib.sv_read_device_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
    lib.sv_read_device_status.restype = i32
    lib.sv_status_string.argtypes = [i32]
    lib.sv_status_string.restype = ctypes.c_char_p
    lib.spec_verify_static.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, f32, vp, vp, vp]
    lib.spec_verify_static.restype = i32
    lib.sv_sample_workspace_size.argtypes = [i32, i32, i32]
    lib.sv_sample_workspace_size.restype = sz
    lib.spec_draft_sample.argtypes = [vp, vp, i32, i32, i32, f32, vp, dp, vp, sz, vp]
    lib.spec_draft_sample.restype = i32
    lib.sv_greedy_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.sv_greedy_workspace_size.restype = sz
    lib.spec_verify_greedy.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp, sz, vp]
    lib.spec_verify_greedy.restype = i32
    lib.sv_topk_workspace_size.argtypes = [i32, i32, i32, i32, i32]
    lib.sv_topk_workspace_size.restype = sz
    lib.spec_verify_topk.argtypes = core[:9] + [i32] + core[9:]
    lib.spec_verify_topk.restype = i32
    lib.sv_topp_workspace_size.argtypes = [i32, i32, i32, i32]
    lib.sv_topp_workspace_size.restype = sz
    lib.spec_verify_topp.argtypes = core[:9] + [f32] + core[9:11] + [vp] + core[11:]
    lib.spec_verify_topp.restype = i32
    lib.sv_kernels_per_call.argtypes = [i32, i32, i32, i32]
    lib.sv_kernels_per_call.restype = i32
    lib.sv_topp_kernels_per_call.argtypes = [i32, i32, i32, i32]
    lib.sv_topp_kernels_per_call.restype = i32
    lib.sv_force_path.argtypes = [i32]
    lib.sv_force_path.restype = None
    lib.sv_test_withhold_plans.argtypes = [i32]
    lib.sv_test_withhold_plans.restype = None
    lib.sv_lmhead_workspace_size.argtypes = [i32, i32, i32]
    lib.sv_lmhead_workspace_size.restype = sz
    lib.sv_lmhead_stats.argtypes = [vp, vp, vp, i32, i32, i32, f32, dp, dp, vp, vp, sz, vp]
    lib.sv_lmhead_stats.restype = i32
    if path is None:
        _lib = lib
    return lib


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device, stream=None):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


def sv_workspace_size(B: int, K: int, V: int, dtype: int) -> int:
    return int(load_library().sv_workspace_size(B, K, V, dtype))


def sv_staging_size(B: int, K: int, V: int, dtype: int) -> int:
    return int(load_library().sv_staging_size(B, K, V, dtype))


def sv_status_string(code: int) -> str:
    return load_library().sv_status_string(int(code)).decode()


def sv_kernels_per_call(B: int, K: int, V: int, dtype: int) -> int:
    return int(load_library().sv_kernels_per_call(B, K, V, dtype))


def sv_topp_kernels_per_call(B: int, K: int, V: int, dtype: int) -> int:
    return int(load_library().sv_topp_kernels_per_call(B, K, V, dtype))


def sv_test_withhold_plans(on: bool) -> None:
    """Test hook: withhold the plans' release flag so that the fused kernel's
    bounded waits run out (SV_DEV_TIMEOUT), without any GPU fault."""
    load_library().sv_test_withhold_plans(1 if on else 0)


def sv_force_path(path: int) -> None:
    """Test hook: 0 chooses the kernels by size, 1 forces the kernel pair,
    2 the fused kernel."""
    load_library().sv_force_path(int(path))


def _check(target, draft, tokens, uniforms):
    for name, t in (("target", target), ("draft", draft), ("tokens", tokens),
                    ("uniforms", uniforms)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if target.dim() != 3 or draft.dim() != 3:
        raise ValueError("target must be [B, K+1, V] and draft [B, K, V]")
    B, K1, V = target.shape
    K = K1 - 1
    if tuple(draft.shape) != (B, K, V) or draft.dtype != target.dtype:
        raise ValueError("draft must be [B, K, V] with the target's dtype")
    if tuple(tokens.shape) != (B, K) or tokens.dtype != torch.int32:
        raise ValueError("tokens must be [B, K] int32")
    if tuple(uniforms.shape) != (B, K + 2) or uniforms.dtype != torch.float32:
        raise ValueError("uniforms must be [B, K+2] float32")
    return B, K, V, _dtype_code(target)


def new_workspace(B, K, V, dtype, device) -> torch.Tensor:
    n = sv_workspace_size(B, K, V, dtype)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def spec_verify(target, draft, tokens, uniforms, temperature, out_tokens, n_accepted, workspace,
                stream=None) -> int:
    """Direct binding of the C call on torch tensors; returns the host status code."""
    B, K, V, dt = _check(target, draft, tokens, uniforms)
    return int(load_library().spec_verify(
        _ptr(target), _ptr(draft), _ptr(tokens), _ptr(uniforms), B, K, V, dt,
        ctypes.c_float(temperature), _ptr(out_tokens), _ptr(n_accepted), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(target.device, stream)))


def spec_verify_debug(target, draft, tokens, uniforms, temperature, out_tokens, n_accepted,
                      workspace, row_lse=None, thresholds=None, sample_prob=None,
                      row_max=None, ratios=None, stream=None) -> int:
    B, K, V, dt = _check(target, draft, tokens, uniforms)
    return int(load_library().spec_verify_debug(
        _ptr(target), _ptr(draft), _ptr(tokens), _ptr(uniforms), B, K, V, dt,
        ctypes.c_float(temperature), _ptr(out_tokens), _ptr(n_accepted), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(target.device, stream),
        _ptr(row_lse), _ptr(thresholds), _ptr(sample_prob), _ptr(row_max), _ptr(ratios)))


def spec_verify_profiled(target, draft, tokens, uniforms, temperature, out_tokens, n_accepted,
                         workspace, ev_start=None, ev_stats_done=None, ev_end=None,
                         stream=None) -> int:
    """spec_verify recording torch.cuda.Event objects around the streaming kernel."""
    B, K, V, dt = _check(target, draft, tokens, uniforms)

    def evp(e):
        return ctypes.c_void_p(e.cuda_event) if e is not None else None

    return int(load_library().spec_verify_profiled(
        _ptr(target), _ptr(draft), _ptr(tokens), _ptr(uniforms), B, K, V, dt,
        ctypes.c_float(temperature), _ptr(out_tokens), _ptr(n_accepted), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(target.device, stream),
        evp(ev_start), evp(ev_stats_done), evp(ev_end)))


def _host_args(h_target, h_draft, h_tokens, h_uniforms, temperature, h_out_tokens, h_n_accepted,
               staging, workspace, stream):
    for t in (h_target, h_draft, h_tokens, h_uniforms, h_out_tokens, h_n_accepted):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("host tensors must be contiguous CPU tensors")
    B, K1, V = h_target.shape
    K = K1 - 1
    dt = _dtype_code(h_target)
    return (_ptr(h_target), _ptr(h_draft), _ptr(h_tokens), _ptr(h_uniforms), B, K, V, dt,
            ctypes.c_float(temperature), _ptr(h_out_tokens), _ptr(h_n_accepted), _ptr(staging),
            staging.numel() * staging.element_size(), _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream(staging.device, stream))


def spec_verify_host(h_target, h_draft, h_tokens, h_uniforms, temperature, h_out_tokens,
                     h_n_accepted, staging, workspace, stream=None) -> int:
    """Host-buffer call: copies in, verifies, copies out, synchronises. Returns
    a host error code or the device status bits (0 = ok)."""
    return int(load_library().spec_verify_host(*_host_args(
        h_target, h_draft, h_tokens, h_uniforms, temperature, h_out_tokens, h_n_accepted, staging,
        workspace, stream)))


def spec_verify_host_async(h_target, h_draft, h_tokens, h_uniforms, temperature, h_out_tokens,
                           h_n_accepted, staging, workspace, stream=None) -> int:
    """spec_verify_host without the wait: returns the host error code once the
    copies and the step are enqueued; the host outputs are valid once `stream`
    has reached this point."""
    return int(load_library().spec_verify_host_async(*_host_args(
        h_target, h_draft, h_tokens, h_uniforms, temperature, h_out_tokens, h_n_accepted, staging,
        workspace, stream)))


def spec_verify_static(target, draft, tokens, uniforms, temperature, out_tokens, n_accepted,
                       stream=None) -> int:
    """The step with the library's fixed scratch array instead of a workspace,
    for callers that cannot allocate device memory; returns the host status."""
    B, K, V, dt = _check(target, draft, tokens, uniforms)
    return int(load_library().spec_verify_static(
        _ptr(target), _ptr(draft), _ptr(tokens), _ptr(uniforms), B, K, V, dt,
        ctypes.c_float(temperature), _ptr(out_tokens), _ptr(n_accepted),
        _stream(target.device, stream)))


def sv_read_device_status(workspace, stream=None) -> int:
    v = ctypes.c_int(0)
    rc = load_library().sv_read_device_status(_ptr(workspace), _stream(workspace.device, stream),
                                              ctypes.byref(v))
    if rc != SV_OK:
        raise StatusError(rc, "sv_read_device_status")
    return int(v.value)


def verify(target, draft, tokens, uniforms, temperature, *, workspace=None, debug=False,
           stream=None):
    """Allocate outputs (and a workspace if none is given) with torch, run one
    verification step, and return (out_tokens [B,K+1] int32, n_accepted [B]
    int32), plus a dict of intermediate values when `debug` is set."""
    if tokens.dtype == torch.int64:
        tokens = tokens.to(torch.int32)
    B, K, V, dt = _check(target, draft, tokens, uniforms)
    dev = target.device
    out = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
    nacc = torch.empty(B, dtype=torch.int32, device=dev)
    ws = workspace if workspace is not None else new_workspace(B, K, V, dt, dev)
    if debug:
        lse = torch.empty(B, 2 * K + 1, dtype=torch.float64, device=dev)
        thr = torch.empty(B, K, dtype=torch.float64, device=dev)
        prob = torch.empty(B, dtype=torch.float64, device=dev)
        rmax = torch.empty(B, 2 * K + 1, dtype=torch.float64, device=dev)
        ratio = torch.empty(B, K, dtype=torch.float64, device=dev)
        rc = spec_verify_debug(target, draft, tokens, uniforms, temperature, out, nacc, ws,
                               lse, thr, prob, rmax, ratio, stream=stream)
    else:
        rc = spec_verify(target, draft, tokens, uniforms, temperature, out, nacc, ws,
                         stream=stream)
    if rc != SV_OK:
        raise StatusError(rc, "spec_verify")
    if debug:
        return out, nacc, {"row_lse": lse, "thresholds": thr, "sample_prob": prob,
                           "row_max": rmax, "ratios": ratio, "workspace": ws}
    return out, nacc


def sv_topk_workspace_size(B: int, K: int, V: int, dtype: int, top_k: int) -> int:
    return int(load_library().sv_topk_workspace_size(B, K, V, dtype, top_k))


def spec_verify_topk(target, draft, tokens, uniforms, temperature, top_k, out_tokens, n_accepted,
                     workspace, stream=None) -> int:
    """Direct binding of top-k filtered verification; returns the host status code."""
    B, K, V, dt = _check(target, draft, tokens, uniforms)
    return int(load_library().spec_verify_topk(
        _ptr(target), _ptr(draft), _ptr(tokens), _ptr(uniforms), B, K, V, dt,
        ctypes.c_float(temperature), int(top_k), _ptr(out_tokens), _ptr(n_accepted),
        _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(target.device, stream)))


def verify_topk(target, draft, tokens, uniforms, temperature, top_k, *, workspace=None,
                stream=None):
    """Allocate outputs (and a workspace if none is given) and run top-k
    filtered verification; returns (out_tokens [B, K+1] int32, n_accepted [B] int32)."""
    if tokens.dtype == torch.int64:
        tokens = tokens.to(torch.int32)
    B, K, V, dt = _check(target, draft, tokens, uniforms)
    dev = target.device
    out = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
    nacc = torch.empty(B, dtype=torch.int32, device=dev)
    ws = workspace
    if ws is None:
        n = sv_topk_workspace_size(B, K, V, dt, int(top_k))
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    rc = spec_verify_topk(target, draft, tokens, uniforms, temperature, top_k, out, nacc, ws,
                          stream=stream)
    if rc != SV_OK:
        raise StatusError(rc, "spec_verify_topk")
    return out, nacc


def sv_topp_workspace_size(B: int, K: int, V: int, dtype: int) -> int:
    return int(load_library().sv_topp_workspace_size(B, K, V, dtype))


def spec_verify_topp(target, draft, tokens, uniforms, temperature, top_p, out_tokens, n_accepted,
                     workspace, kept_counts=None, stream=None) -> int:
    """Direct binding of nucleus filtered verification; returns the host status code."""
    B, K, V, dt = _check(target, draft, tokens, uniforms)
    return int(load_library().spec_verify_topp(
        _ptr(target), _ptr(draft), _ptr(tokens), _ptr(uniforms), B, K, V, dt,
        ctypes.c_float(temperature), ctypes.c_float(top_p), _ptr(out_tokens), _ptr(n_accepted),
        _ptr(kept_counts), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(target.device, stream)))


def verify_topp(target, draft, tokens, uniforms, temperature, top_p, *, workspace=None,
                stream=None):
    """Allocate outputs (and a workspace if none is given) and run nucleus
    filtered verification; returns (out_tokens [B, K+1] int32, n_accepted [B]
    int32, kept_counts [B, 2K+1] int32)."""
    if tokens.dtype == torch.int64:
        tokens = tokens.to(torch.int32)
    B, K, V, dt = _check(target, draft, tokens, uniforms)
    dev = target.device
    out = torch.empty(B, K + 1, dtype=torch.int32, device=dev)
    nacc = torch.empty(B, dtype=torch.int32, device=dev)
    kept = torch.empty(B, 2 * K + 1, dtype=torch.int32, device=dev)
    ws = workspace
    if ws is None:
        n = sv_topp_workspace_size(B, K, V, dt)
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    rc = spec_verify_topp(target, draft, tokens, uniforms, temperature, top_p, out, nacc, ws,
                          kept, stream=stream)
    if rc != SV_OK:
        raise StatusError(rc, "spec_verify_topp")
    return out, nacc, kept


def sv_sample_workspace_size(N: int, V: int, dtype: int) -> int:
    return int(load_library().sv_sample_workspace_size(N, V, dtype))


def spec_draft_sample(logits, uniforms, temperature, out_tokens, workspace, sample_prob=None,
                      stream=None) -> int:
    """Direct binding of the sampler on torch tensors: logits [N, V] bf16/f32,
    uniforms [N] f32, out_tokens [N] int32; returns the host status code."""
    for name, t in (("logits", logits), ("uniforms", uniforms), ("out_tokens", out_tokens)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if logits.dim() != 2:
        raise ValueError("logits must be [N, V]")
    N, V = logits.shape
    if tuple(uniforms.shape) != (N,) or uniforms.dtype != torch.float32:
        raise ValueError("uniforms must be [N] float32")
    if tuple(out_tokens.shape) != (N,) or out_tokens.dtype != torch.int32:
        raise ValueError("out_tokens must be [N] int32")
    return int(load_library().spec_draft_sample(
        _ptr(logits), _ptr(uniforms), N, V, _dtype_code(logits), ctypes.c_float(temperature),
        _ptr(out_tokens), _ptr(sample_prob), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(logits.device, stream)))


def draft_sample(logits, uniforms, temperature, *, workspace=None, with_prob=False, stream=None):
    """Allocate the outputs (and a workspace if none is given) with torch and
    draw one token per row of `logits`; returns tokens [N] int32 (and the
    drawn tokens' probabilities [N] fp64 when `with_prob`)."""
    N, V = logits.shape
    dev = logits.device
    out = torch.empty(N, dtype=torch.int32, device=dev)
    prob = torch.empty(N, dtype=torch.float64, device=dev) if with_prob else None
    ws = workspace
    if ws is None:
        n = sv_sample_workspace_size(N, V, _dtype_code(logits))
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    rc = spec_draft_sample(logits, uniforms, temperature, out, ws, prob, stream=stream)
    if rc != SV_OK:
        raise StatusError(rc, "spec_draft_sample")
    return (out, prob) if with_prob else out


def sv_greedy_workspace_size(B: int, K: int, V: int, dtype: int) -> int:
    return int(load_library().sv_greedy_workspace_size(B, K, V, dtype))


def spec_verify_greedy(target, tokens, out_tokens, n_accepted, workspace, stream=None) -> int:
    """Direct binding of greedy verification on torch tensors: target [B, K+1, V]
    bf16/f32, tokens [B, K] int32; returns the host status code."""
    for name, t in (("target", target), ("tokens", tokens), ("out_tokens", out_tokens),
                    ("n_accepted", n_accepted)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if target.dim() != 3:
        raise ValueError("target must be [B, K+1, V]")
    B, K1, V = target.shape
    K = K1 - 1
    if tuple(tokens.shape) != (B, K) or tokens.dtype != torch.int32:
        raise ValueError("tokens must be [B, K] int32")
    return int(load_library().spec_verify_greedy(
        _ptr(target), _ptr(tokens), B, K, V, _dtype_code(target), _ptr(out_tokens),
        _ptr(n_accepted), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(target.device, stream)))


def verify_greedy(target, tokens, *, workspace=None, stream=None):
    """Allocate outputs (and a workspace if none is given) and run greedy
    verification; returns (out_tokens [B, K+1] int32, n_accepted [B] int32)."""
    if tokens.dtype == torch.int64:
        tokens = tokens.to(torch.int32)
    B, K1, V = target.shape
    dev = target.device
    out = torch.empty(B, K1, dtype=torch.int32, device=dev)
    nacc = torch.empty(B, dtype=torch.int32, device=dev)
    ws = workspace
    if ws is None:
        n = sv_greedy_workspace_size(B, K1 - 1, V, _dtype_code(target))
        ws = torch.empty(max(n, 256), dtype=torch.uint8, device=dev)
    rc = spec_verify_greedy(target, tokens, out, nacc, ws, stream=stream)
    if rc != SV_OK:
        raise StatusError(rc, "spec_verify_greedy")
    return out, nacc


# ---------------------------------------------------------------- the scoring step's projection

def sv_lmhead_workspace_size(N: int, D: int, V: int) -> int:
    return int(load_library().sv_lmhead_workspace_size(N, D, V))


def sv_lmhead_stats(hidden, weight, tokens, temperature, row_max, lse, at, workspace,
                    stream=None) -> int:
    """Direct binding of the fused projection + row statistics: hidden [N, D]
    and weight [V, D] bf16 CUDA tensors, tokens [N] int32; row_max and lse
    [N] fp64 and at [N] fp32 are written. Returns the host status code."""
    if hidden.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
        raise TypeError("hidden and weight must be bfloat16")
    if hidden.dim() != 2 or weight.dim() != 2 or hidden.shape[1] != weight.shape[1]:
        raise ValueError("hidden [N, D] and weight [V, D] must share D")
    if not (hidden.is_contiguous() and weight.is_contiguous() and tokens.is_contiguous()):
        raise ValueError("inputs must be contiguous")
    if tokens.dtype != torch.int32 or tokens.shape != (hidden.shape[0],):
        raise TypeError("tokens must be int32 [N]")
    N, D = hidden.shape
    V = weight.shape[0]
    return int(load_library().sv_lmhead_stats(
        _ptr(hidden), _ptr(weight), _ptr(tokens), N, D, V, ctypes.c_float(temperature),
        _ptr(row_max), _ptr(lse), _ptr(at), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _stream(hidden.device, stream)))


def lmhead_stats(hidden, weight, tokens, temperature, *, workspace=None, stream=None):
    """Allocate the outputs (and a workspace if none is given) with torch and
    run the fused projection + statistics; returns (row_max, lse, at)."""
    if tokens.dtype == torch.int64:
        tokens = tokens.to(torch.int32)
    N, D = hidden.shape
    V = weight.shape[0]
    dev = hidden.device
    n = sv_lmhead_workspace_size(N, D, V)
    if n == 0:
        raise StatusError(2, "sv_lmhead_workspace_size")
    ws = workspace if workspace is not None else torch.empty(n, dtype=torch.uint8, device=dev)
    row_max = torch.empty(N, dtype=torch.float64, device=dev)
    lse = torch.empty(N, dtype=torch.float64, device=dev)
    at = torch.empty(N, dtype=torch.float32, device=dev)
    rc = sv_lmhead_stats(hidden, weight, tokens, temperature, row_max, lse, at, ws, stream=stream)
    if rc != SV_OK:
        raise StatusError(rc, "sv_lmhead_stats")
    return row_max, lse, at
