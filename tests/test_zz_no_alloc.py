"""The allocation-free decode entry point (path_decode_step_noalloc), through the C ABI,
against the workspace entry point (path_decode_step) and the fp64 oracle.

Some callers cannot allocate device memory for this library on their call path: an
engine that owns all device memory behind an allocator its plugins cannot reach, or a
latency-bound loop that may not call cudaMalloc because it can synchronise the device.
For them the decode step keeps its split partials in a fixed array inside the library.
This file sorts last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import path_inputs as pi

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2   # the bf16 absolute tolerance of the parity tests
F32_REL = 1e-4    # the fp32 normwise relative tolerance of the parity tests
SCRATCH = 16 << 20


def _noalloc(lib, s, kc, vc, n, out):
    B, H, cap, d = kc.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    dt = lib.BF16 if kc.dtype == torch.bfloat16 else lib.F32
    return lib._load().path_decode_step_noalloc(
        p(s["q"]), p(s["k"]), p(s["v"]), p(s["w"]), p(s["beta"]), p(kc), p(vc), B, H, n, cap, d,
        dt, ctypes.c_float(d ** -0.5), p(out),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _close(got, ref, dtype):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    err = np.abs(got - ref).max()
    if dtype == torch.bfloat16:
        return err <= BF16_TOL
    return err / max(np.abs(ref).max(), 1e-30) <= F32_REL


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("n0", [2100, 1023])
def test_noalloc_decode_matches_workspace_decode_and_oracle_on_two_calls(lib, dtype, d, n0):
    # n0 = 1023: the second call has 1024 cached keys (one split), the first 1023; 2100
    # spans three splits
    B, H = 2, 3
    wl = pi.DecodeWorkload("noalloc", B, H, n0, 2, d, dtype, 5, 1000)
    cap = n0 + wl.steps
    kc_ref, vc_ref = pi.make_decode_prefix(wl, cap, device="cuda")
    kc, vc = kc_ref.clone(), vc_ref.clone()
    ocache = oracle.DecodeCache(kc.reshape(B * H, cap, d)[:, :n0].cpu(),
                                vc.reshape(B * H, cap, d)[:, :n0].cpu(), cap)
    for t in range(2):
        s = pi.make_decode_step(wl, t, device="cuda")
        ref = lib.path_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], kc_ref, vc_ref,
                                   n0 + t)
        out = torch.full_like(ref, float("nan"))
        assert _noalloc(lib, s, kc, vc, n0 + t, out) == lib.OK
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert _close(out.double().cpu(), ref.double().cpu(), dtype)
        assert _close(kc.double().cpu(), kc_ref.double().cpu(), dtype)
        assert torch.equal(vc, vc_ref)
        sel = {k: v.reshape(B * H, -1).cpu() for k, v in s.items()}
        want = ocache.step(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"])
        assert _close(out.reshape(B * H, d).double().cpu().numpy(), want, dtype)


def test_noalloc_decode_at_the_scratch_limit(lib):
    # 1025 heads x 62 splits x (64 + 2) fp32 = 16,777,200 bytes: the last head's partials
    # end 16 bytes before the end of the fixed array. Two calls in a row with 62 * 1024 - 1
    # and 62 * 1024 cached keys use all 62 splits; one more key needs a 63rd split per
    # head, which no longer fits and is refused before any launch.
    B, H, d = 1, 1025, 64
    n0 = 62 * 1024 - 1
    assert B * H * 62 * (d + 2) * 4 <= SCRATCH < B * H * 63 * (d + 2) * 4
    torch.cuda.empty_cache()
    wl = pi.DecodeWorkload("noalloc_limit", B, H, n0, 3, d, torch.bfloat16, 7, 2000)
    cap = n0 + 3
    kc, vc = pi.make_decode_prefix(wl, cap, device="cuda")
    heads = [0, 511, 1024]
    ocache = oracle.DecodeCache(kc.reshape(B * H, cap, d)[heads, :n0].cpu(),
                                vc.reshape(B * H, cap, d)[heads, :n0].cpu(), cap)
    for t in range(2):
        s = pi.make_decode_step(wl, t, device="cuda")
        out = torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(lib, s, kc, vc, n0 + t, out) == lib.OK
        torch.cuda.synchronize()
        assert torch.isfinite(out.float()).all()
        sel = {k: v.reshape(B * H, -1)[heads].cpu() for k, v in s.items()}
        want = ocache.step(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"])
        got = out.reshape(B * H, d)[heads].double().cpu().numpy()
        assert np.abs(got - want).max() <= BF16_TOL
    s = pi.make_decode_step(wl, 2, device="cuda")
    out = torch.full((B, H, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(lib, s, kc, vc, n0 + 2, out) == lib.ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()
    del kc, vc
    torch.cuda.empty_cache()
