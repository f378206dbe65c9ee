"""The C-ABI library: it builds, loads, exports every declared symbol, and its
pure host logic (sizes, argument checks, status strings) behaves; nothing
here launches GPU work."""

import ctypes
import os
import re

import pytest

import speculative_sampling_verification_gb300 as sv
from speculative_sampling_verification_gb300._build import build_library

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    return sv.load_library(build_library())


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)
    keywords = {"if", "sizeof", "defined"}
    return sorted({n for n in names if n not in keywords})


def test_header_declares_the_binding_names():
    assert set(declared_functions()) == set(sv.EXPORTED_SYMBOLS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_workspace_size_is_pure_and_monotone(lib):
    s1 = lib.sv_workspace_size(8, 4, 32000, sv.SV_BF16)
    s2 = lib.sv_workspace_size(64, 8, 128256, sv.SV_BF16)
    s3 = lib.sv_workspace_size(256, 4, 256000, sv.SV_F32)
    assert 0 < s1 < s2 < s3
    assert s1 % 256 == 0 and s2 % 256 == 0
    assert lib.sv_workspace_size(0, 4, 1000, sv.SV_F32) > 0
    for bad in ((-1, 4, 10, 0), (1, 0, 10, 0), (1, 65, 10, 0), (1, 4, 0, 0), (1, 4, 10, 7)):
        assert lib.sv_workspace_size(*bad) == 0
    assert lib.sv_staging_size(8, 4, 32000, sv.SV_BF16) >= 8 * 9 * 32000 * 2


def _call(lib, **kw):
    a = dict(t=1 << 20, d=1 << 20, tok=1 << 20, u=1 << 20, B=2, K=3, V=100, dtype=sv.SV_F32,
             T=1.0, out=1 << 20, nacc=1 << 20, ws=1 << 20, wsb=1 << 30)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.spec_verify(vp(a["t"]), vp(a["d"]), vp(a["tok"]), vp(a["u"]), a["B"], a["K"], a["V"],
                           a["dtype"], ctypes.c_float(a["T"]), vp(a["out"]), vp(a["nacc"]),
                           vp(a["ws"]), a["wsb"], None)


def test_host_validation_codes(lib):
    # Every case fails validation before any CUDA call is made.
    assert _call(lib, dtype=3) == 4
    assert _call(lib, K=0) == 2
    assert _call(lib, K=65) == 2
    assert _call(lib, V=0) == 2
    assert _call(lib, B=-1) == 2
    assert _call(lib, T=0.0) == 3
    assert _call(lib, T=-1.0) == 3
    assert _call(lib, T=float("nan")) == 3
    assert _call(lib, T=float("inf")) == 3
    assert _call(lib, t=0) == 1
    assert _call(lib, ws=0) == 1
    assert _call(lib, nacc=0) == 1
    assert _call(lib, t=(1 << 20) + 2) == 5          # fp32 logits need 4-byte alignment
    assert _call(lib, ws=(1 << 20) + 16) == 5        # workspace needs 256-byte alignment
    assert _call(lib, wsb=16) == 6
    # B == 0 is a no-op that succeeds (nothing is launched).
    assert _call(lib, B=0, t=0, d=0) == 0


def test_status_strings(lib):
    for code in (0, 1, 2, 3, 4, 5, 6, 7, 16, 32, 64, 128, 256):
        s = sv.sv_status_string(code)
        assert s and s != "unknown status"


def test_kernels_per_call(lib):
    # The fused kernel for calls streaming 16 MiB to 1 GiB, else the pair;
    # nothing for invalid sizes or B == 0.
    assert sv.sv_kernels_per_call(8, 4, 32000, sv.SV_BF16) == 2      # 4.6 MB
    assert sv.sv_kernels_per_call(64, 8, 128256, sv.SV_BF16) == 1    # 279 MB
    assert sv.sv_kernels_per_call(256, 4, 256000, sv.SV_F32) == 3    # 2.36 GB
    assert sv.sv_kernels_per_call(0, 4, 1000, sv.SV_F32) == 0
    assert sv.sv_kernels_per_call(1, 0, 1000, sv.SV_F32) == 0


def _call_sample(lib, **kw):
    a = dict(l=1 << 20, u=1 << 20, N=3, V=100, dtype=sv.SV_F32, T=1.0, out=1 << 20, prob=0,
             ws=1 << 20, wsb=1 << 30)
    a.update(kw)
    vp = ctypes.c_void_p
    return lib.spec_draft_sample(vp(a["l"]), vp(a["u"]), a["N"], a["V"], a["dtype"],
                                 ctypes.c_float(a["T"]), vp(a["out"]), vp(a["prob"]) if a["prob"] else None,
                                 vp(a["ws"]), a["wsb"], None)


def test_sampler_workspace_and_validation(lib):
    s1 = lib.sv_sample_workspace_size(32, 32000, sv.SV_BF16)
    s2 = lib.sv_sample_workspace_size(512, 128256, sv.SV_BF16)
    assert 0 < s1 < s2 and s1 % 256 == 0
    for bad in ((-1, 10, 0), (1, 0, 0), (1, 10, 7)):
        assert lib.sv_sample_workspace_size(*bad) == 0
    # Every case fails validation before any CUDA call is made.
    assert _call_sample(lib, dtype=3) == 4
    assert _call_sample(lib, V=0) == 2
    assert _call_sample(lib, N=-1) == 2
    assert _call_sample(lib, T=0.0) == 3
    assert _call_sample(lib, T=float("nan")) == 3
    assert _call_sample(lib, l=0) == 1
    assert _call_sample(lib, u=0) == 1
    assert _call_sample(lib, out=0) == 1
    assert _call_sample(lib, ws=0) == 1
    assert _call_sample(lib, l=(1 << 20) + 2) == 5
    assert _call_sample(lib, u=(1 << 20) + 2) == 5
    assert _call_sample(lib, ws=(1 << 20) + 16) == 5
    assert _call_sample(lib, wsb=16) == 6
    assert _call_sample(lib, N=0, l=0, u=0) == 0


def test_greedy_workspace_and_validation(lib):
    assert 0 < lib.sv_greedy_workspace_size(8, 4, 32000, sv.SV_BF16) < lib.sv_workspace_size(8, 4, 32000, sv.SV_BF16)
    for bad in ((-1, 4, 10, 0), (1, 0, 10, 0), (1, 65, 10, 0), (1, 4, 0, 0), (1, 4, 10, 7)):
        assert lib.sv_greedy_workspace_size(*bad) == 0
    vp = ctypes.c_void_p

    def call(t=1 << 20, tok=1 << 20, B=2, K=3, V=100, dtype=sv.SV_F32, out=1 << 20, nacc=1 << 20,
             ws=1 << 20, wsb=1 << 30):
        return lib.spec_verify_greedy(vp(t), vp(tok), B, K, V, dtype, vp(out), vp(nacc), vp(ws),
                                      wsb, None)

    assert call(dtype=3) == 4
    assert call(K=0) == 2 and call(K=65) == 2 and call(V=0) == 2 and call(B=-1) == 2
    assert call(t=0) == 1 and call(tok=0) == 1 and call(nacc=0) == 1 and call(ws=0) == 1
    assert call(t=(1 << 20) + 2) == 5 and call(ws=(1 << 20) + 16) == 5
    assert call(wsb=16) == 6
    assert call(B=0, t=0, tok=0) == 0


def test_topk_workspace_and_validation(lib):
    full = lib.sv_workspace_size(8, 4, 32000, sv.SV_BF16)
    small = lib.sv_topk_workspace_size(8, 4, 32000, sv.SV_BF16, 50)
    assert 0 < small < full
    # top_k >= V keeps every entry: the unfiltered call and its workspace.
    assert lib.sv_topk_workspace_size(8, 4, 32000, sv.SV_BF16, 32000) == full
    assert lib.sv_topk_workspace_size(8, 4, 100, sv.SV_BF16, 1000) == lib.sv_workspace_size(8, 4, 100, sv.SV_BF16)
    for bad in ((1, 4, 1000, 0, 0), (1, 4, 1000, 0, 257), (1, 4, 1000, 0, -3), (-1, 4, 1000, 0, 8),
                (1, 0, 1000, 0, 8), (1, 65, 1000, 0, 8), (1, 4, 1000, 7, 8)):
        assert lib.sv_topk_workspace_size(*bad) == 0
    vp = ctypes.c_void_p

    def call(t=1 << 20, d=1 << 20, tok=1 << 20, u=1 << 20, B=2, K=3, V=1000, dtype=sv.SV_F32,
             T=1.0, k=20, out=1 << 20, nacc=1 << 20, ws=1 << 20, wsb=1 << 30):
        return lib.spec_verify_topk(vp(t), vp(d), vp(tok), vp(u), B, K, V, dtype,
                                    ctypes.c_float(T), k, vp(out), vp(nacc), vp(ws), wsb, None)

    assert call(dtype=3) == 4
    assert call(k=0) == 2 and call(k=257) == 2 and call(K=0) == 2 and call(B=-1) == 2
    assert call(T=0.0) == 3 and call(T=float("nan")) == 3
    assert call(t=0) == 1 and call(d=0) == 1 and call(u=0) == 1 and call(ws=0) == 1
    assert call(t=(1 << 20) + 2) == 5 and call(tok=(1 << 20) + 2) == 5
    assert call(ws=(1 << 20) + 16) == 5
    assert call(wsb=16) == 6
    # top_k >= V takes the unfiltered entry point, with its own checks.
    assert call(k=5000, wsb=16) == 6 and call(k=5000, T=-1.0) == 3
    assert call(B=0, t=0, d=0, tok=0, u=0) == 0


def test_topp_workspace_and_validation(lib):
    full = lib.sv_workspace_size(8, 4, 32000, sv.SV_BF16)
    assert lib.sv_topp_workspace_size(8, 4, 32000, sv.SV_BF16) >= full + 8 * 9 * 8
    assert sv.sv_topp_kernels_per_call(8, 4, 32000, sv.SV_BF16) == 3
    assert sv.sv_topp_kernels_per_call(256, 4, 256000, sv.SV_F32) == 4
    assert sv.sv_topp_kernels_per_call(0, 4, 1000, sv.SV_F32) == 0
    for bad in ((-1, 4, 10, 0), (1, 0, 10, 0), (1, 65, 10, 0), (1, 4, 0, 0), (1, 4, 10, 7)):
        assert lib.sv_topp_workspace_size(*bad) == 0
    vp = ctypes.c_void_p

    def call(t=1 << 20, d=1 << 20, tok=1 << 20, u=1 << 20, B=2, K=3, V=1000, dtype=sv.SV_F32,
             T=1.0, p=0.9, out=1 << 20, nacc=1 << 20, kept=None, ws=1 << 20, wsb=1 << 30):
        return lib.spec_verify_topp(vp(t), vp(d), vp(tok), vp(u), B, K, V, dtype, ctypes.c_float(T),
                                    ctypes.c_float(p), vp(out), vp(nacc), vp(kept), vp(ws), wsb, None)

    assert call(dtype=3) == 4
    assert call(p=0.0) == 2 and call(p=-1.0) == 2 and call(p=float("nan")) == 2
    assert call(K=0) == 2 and call(B=-1) == 2
    assert call(T=0.0) == 3
    assert call(t=0) == 1 and call(d=0) == 1 and call(ws=0) == 1
    assert call(t=(1 << 20) + 2) == 5 and call(kept=(1 << 20) + 2) == 5
    assert call(wsb=lib.sv_workspace_size(2, 3, 1000, sv.SV_F32)) == 6
    assert call(B=0, t=0, d=0, tok=0, u=0) == 0


@pytest.mark.parametrize("name", ["spec_verify_host", "spec_verify_host_async"])
def test_host_buffer_entry_points_validate_before_any_copy(lib, name):
    vp = ctypes.c_void_p
    fn = getattr(lib, name)

    def call(t=1 << 20, d=1 << 20, tok=1 << 20, u=1 << 20, B=2, K=3, V=100, dtype=sv.SV_F32,
             T=1.0, out=1 << 20, nacc=1 << 20, st=1 << 20, stb=1 << 30, ws=1 << 20, wsb=1 << 30):
        return fn(vp(t), vp(d), vp(tok), vp(u), B, K, V, dtype, ctypes.c_float(T), vp(out),
                  vp(nacc), vp(st), stb, vp(ws), wsb, None)

    assert call(dtype=3) == 4 and call(K=0) == 2 and call(T=0.0) == 3
    assert call(t=0) == 1 and call(st=0) == 1 and call(ws=0) == 1
    assert call(st=(1 << 20) + 16) == 5 and call(ws=(1 << 20) + 16) == 5
    assert call(stb=16) == 6 and call(wsb=16) == 6
    assert call(B=0, t=0, d=0) == 0
