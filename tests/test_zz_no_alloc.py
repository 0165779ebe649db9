"""The allocation-free decode entry point (path_decode_step_noalloc) against the
workspace one (path_decode_step), through the C ABI.

Some callers cannot allocate device memory for this library on their call path (an
engine that owns all device memory behind an allocator its plugins cannot reach, or a
latency-bound loop that may not call cudaMalloc because it can synchronise the device).
For them the decode step keeps its split partials in a fixed array inside the library.
This file sorts last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import pytest
import torch

import path_inputs as pi

pytestmark = pytest.mark.gpu

TOL = 2e-2  # the bf16 absolute tolerance of the parity tests


def _noalloc(lib, s, kc, vc, n, out):
    B, H, cap, d = kc.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return lib._load().path_decode_step_noalloc(
        p(s["q"]), p(s["k"]), p(s["v"]), p(s["w"]), p(s["beta"]), p(kc), p(vc), B, H, n, cap, d,
        lib.BF16, ctypes.c_float(d ** -0.5),
        p(out), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_matches_workspace_decode_on_two_calls(lib):
    wl = pi.DecodeWorkload("noalloc", 2, 3, 2100, 2, 64, torch.bfloat16, 5, 1000)
    cap = wl.n_prefix + wl.steps
    kc_ref, vc_ref = pi.make_decode_prefix(wl, cap, device="cuda")
    kc, vc = kc_ref.clone(), vc_ref.clone()
    for t in range(2):
        s = pi.make_decode_step(wl, t, device="cuda")
        ref = lib.path_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], kc_ref, vc_ref,
                                   wl.n_prefix + t)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(lib, s, kc, vc, wl.n_prefix + t, out) == lib.OK
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert (out.float() - ref.float()).abs().max().item() <= TOL
        assert (kc.float() - kc_ref.float()).abs().max().item() <= TOL
        assert torch.equal(vc, vc_ref)
