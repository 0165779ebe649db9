"""C ABI argument checks with fake device pointers: every call here must be rejected (or
be an empty problem) before the library makes any CUDA call, so the pointers are never
dereferenced. As a second guard these tests run only in a process that cannot reach a
GPU: on a machine with one they are skipped here and run by
test_abi.py::test_argument_rejection_runs_where_no_gpu_is_reachable in a child process
with CUDA_VISIBLE_DEVICES empty."""
import ctypes

import pytest


def _gpu_reachable():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


pytestmark = pytest.mark.skipif(_gpu_reachable(),
                                reason="fake device pointers: run only where no GPU is reachable")

FAKE = 0x7F0000000000  # 256-byte aligned, never dereferenced


def _fwd(so, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, w=FAKE, beta=FAKE, out=FAKE, lse=None, B=1, H=1, L=128,
             d=64, dtype=1, scale=0.125, ws=FAKE, ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return so.path_attn_fwd(a["q"], a["k"], a["v"], a["w"], a["beta"], a["out"], a["lse"],
                            a["B"], a["H"], a["L"], a["d"], a["dtype"],
                            ctypes.c_float(a["scale"]), a["ws"], ctypes.c_size_t(a["ws_bytes"]),
                            a["stream"])


@pytest.fixture(scope="module")
def so(lib):
    return lib._load()


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(v=None), 1), (dict(ws=None), 1), (dict(beta=None), 1),
    (dict(d=32), 2), (dict(L=-1), 2), (dict(B=70000), 2), (dict(dtype=3), 3),
    (dict(q=FAKE + 8), 4), (dict(out=FAKE + 4), 4), (dict(ws=FAKE + 16), 4),
    (dict(ws_bytes=1000), 5), (dict(scale=float("inf")), 9), (dict(scale=float("nan")), 9),
])
def test_fwd_rejects_bad_arguments_before_launch(so, kw, code):
    assert _fwd(so, **kw) == code


def test_empty_problems_launch_nothing(so):
    assert _fwd(so, L=0, q=None, k=None, v=None, w=None, beta=None, out=None, ws=None) == 0
    assert _fwd(so, B=0) == 0


def test_head_128_empty_problems_launch_nothing(so):
    assert _fwd(so, d=128, L=0, q=None, k=None, v=None, w=None, beta=None, out=None,
                ws=None) == 0
    assert so.path_fox_fwd(None, None, None, None, None, None, None, None, 1, 1, 0, 128, 1,
                           ctypes.c_float(0.125), None, ctypes.c_size_t(0), None) == 0
    assert so.path_fox_fwd(None, None, None, None, None, None, None, None, 0, 4, 64, 128, 1,
                           ctypes.c_float(0.125), None, ctypes.c_size_t(0), None) == 0


def test_fox_needs_log_f(so):
    r = so.path_fox_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None, 1, 1, 128, 64, 1,
                        ctypes.c_float(0.125), FAKE, ctypes.c_size_t(1 << 30), None)
    assert r == 1


def test_decode_argument_checks(so):
    def call(**kw):
        a = dict(B=1, H=1, cache_len=10, cap=16, d=64, dtype=1, ws_bytes=1 << 20, kc=FAKE)
        a.update(kw)
        return so.path_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, a["kc"], FAKE, a["B"], a["H"],
                                   a["cache_len"], a["cap"], a["d"], a["dtype"],
                                   ctypes.c_float(0.125), FAKE, FAKE,
                                   ctypes.c_size_t(a["ws_bytes"]), None)
    assert call(cache_len=16) == 6
    assert call(cache_len=-1) == 2
    assert call(d=96) == 2
    assert call(d=128, ws_bytes=8) == 5  # head size 128 is accepted by decode
    assert call(kc=None) == 1
    assert call(kc=FAKE + 2) == 4
    assert call(ws_bytes=8) == 5
    assert call(B=0) == 0


def test_fox_decode_argument_checks(so, lib):
    # every case below is rejected before any launch (fake pointers are never used)
    def call(**kw):
        a = dict(B=1, H=1, cache_len=10, cap=16, d=64, dtype=1, ws_bytes=1 << 20, kc=FAKE,
                 lf=FAKE, gc=FAKE)
        a.update(kw)
        return so.path_fox_decode_step(FAKE, FAKE, FAKE, FAKE, FAKE, a["lf"], a["kc"], FAKE,
                                       a["gc"], a["B"], a["H"], a["cache_len"], a["cap"], a["d"],
                                       a["dtype"], ctypes.c_float(0.125), FAKE, FAKE,
                                       ctypes.c_size_t(a["ws_bytes"]), None)
    assert call(cache_len=16) == 6
    assert call(cache_len=-1) == 2
    assert call(d=96) == 2
    assert call(d=128, ws_bytes=8) == 5  # head size 128 accepted, workspace too small
    assert call(dtype=5) == 3
    assert call(lf=None) == 1
    assert call(gc=None) == 1
    assert call(gc=FAKE + 4) == 4
    assert call(lf=FAKE + 2) == 4
    assert call(ws_bytes=8) == 5
    assert call(B=0) == 0
    assert lib.path_workspace_bytes(lib.OP_FOX_DECODE, 2, 2, 2048, 64, lib.BF16) == \
        lib.path_workspace_bytes(lib.OP_DECODE, 2, 2, 2048, 64, lib.BF16)


def test_producer_argument_checks(so, lib):
    # every case below is rejected before any launch (fake pointers are never used)
    def call(**kw):
        a = dict(B=1, L=128, D=128, R=64, H=2, d=64, dtype=1, ws_bytes=1 << 30, x=FAKE,
                 out=FAKE, bmax=1.99)
        a.update(kw)
        return so.path_wbeta_produce(a["x"], FAKE, FAKE, FAKE, FAKE, FAKE,
                                     ctypes.c_float(a["bmax"]), a["out"], FAKE, a["B"], a["L"],
                                     a["D"], a["R"], a["H"], a["d"], a["dtype"], FAKE,
                                     ctypes.c_size_t(a["ws_bytes"]), None)
    assert call(dtype=0) == 3          # bf16 only
    assert call(d=32) == 2
    assert call(D=100) == 2            # D a multiple of 64
    assert call(R=48) == 2             # R a multiple of 64
    assert call(R=192, H=65) == 2      # R + round16(H) > 256
    assert call(H=0) == 2
    assert call(x=None) == 1
    assert call(out=FAKE + 8) == 4
    assert call(ws_bytes=64) == 5
    assert call(bmax=float("nan")) == 9
    assert call(bmax=0.0) == 9
    assert call(L=0) == 0 and call(B=0) == 0
    # workspace: header, z (B*L, R) bf16, three tap-scaled (H*d, R) bf16 matrices
    assert lib.path_wbeta_workspace_bytes(2, 100, 128, 64, 3) == \
        256 + (2 * 100 * 64 * 2 + 255) // 256 * 256 + (3 * 3 * 64 * 64 * 2 + 255) // 256 * 256
    assert lib.path_wbeta_workspace_bytes(2, 100, 128, 64, 3, 64, lib.F32) == 0


def test_noalloc_decode_rejects_problems_beyond_the_fixed_scratch(so):
    # 4096 heads x 17 splits of 1024 keys x 264 B = 18.4 MB > 16 MiB: refused before any
    # launch. The size is checked here first so that these never-dereferenced pointers
    # cannot reach a kernel even if the numbers above were wrong.
    B, H, n = 64, 64, 16 * 1024 + 1
    need = B * H * (-(-n // 1024)) * 66 * 4
    assert need > 16 << 20
    rc = so.path_decode_step_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, B, H, n, n + 1,
                                     64, 1, ctypes.c_float(0.125), FAKE, None)
    assert rc == 5


def test_fox_first_blocks_argument_checks(so):
    def call(**kw):
        a = dict(ws=FAKE, ws_bytes=1 << 30, B=1, H=1, L=128, d=64, dtype=1, first=FAKE)
        a.update(kw)
        return so.path_fox_first_blocks(a["ws"], ctypes.c_size_t(a["ws_bytes"]), a["B"], a["H"],
                                        a["L"], a["d"], a["dtype"], a["first"], None)
    assert call(first=None) == 1
    assert call(ws=None) == 1
    assert call(d=32) == 2
    assert call(first=FAKE + 2) == 4
    assert call(ws=FAKE + 8) == 4
    assert call(ws_bytes=1024) == 5
    assert call(L=0) == 0


def _bwd(so, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, w=FAKE, beta=FAKE, out=FAKE, lse=FAKE, d_out=FAKE, B=1,
             H=1, L=128, d=64, dtype=1, scale=0.125, dq=FAKE, dk=FAKE, dv=FAKE, dw=FAKE,
             dbeta=FAKE, ws=FAKE, ws_bytes=8, stream=None)
    a.update(kw)
    return so.path_attn_bwd(a["q"], a["k"], a["v"], a["w"], a["beta"], a["out"], a["lse"],
                            a["d_out"], a["B"], a["H"], a["L"], a["d"], a["dtype"],
                            ctypes.c_float(a["scale"]), a["dq"], a["dk"], a["dv"], a["dw"],
                            a["dbeta"], a["ws"], ctypes.c_size_t(a["ws_bytes"]), a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), 1), (dict(lse=None), 1), (dict(d_out=None), 1), (dict(dbeta=None), 1),
    (dict(ws=None), 1), (dict(d=96), 2), (dict(L=-1), 2), (dict(dtype=2), 3),
    (dict(d=128), 5),  # head size 128 accepted, workspace too small
    (dict(dw=FAKE + 4), 4), (dict(out=FAKE + 8), 4), (dict(ws=FAKE + 16), 4),
    (dict(scale=float("nan")), 9), (dict(), 5),
])
def test_bwd_rejects_bad_arguments_before_launch(so, kw, code):
    # ws_bytes stays 8 throughout, so nothing can reach a launch
    assert _bwd(so, **kw) == code


def test_bwd_empty_problem_launches_nothing(so):
    assert _bwd(so, L=0, q=None, ws=None) == 0


def _fox_bwd(so, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, w=FAKE, beta=FAKE, log_f=FAKE, out=FAKE, lse=FAKE,
             d_out=FAKE, B=1, H=1, L=128, d=64, dtype=1, scale=0.125, dq=FAKE, dk=FAKE, dv=FAKE,
             dw=FAKE, dbeta=FAKE, dlog_f=FAKE, ws=FAKE, ws_bytes=8, stream=None)
    a.update(kw)
    return so.path_fox_bwd(a["q"], a["k"], a["v"], a["w"], a["beta"], a["log_f"], a["out"],
                           a["lse"], a["d_out"], a["B"], a["H"], a["L"], a["d"], a["dtype"],
                           ctypes.c_float(a["scale"]), a["dq"], a["dk"], a["dv"], a["dw"],
                           a["dbeta"], a["dlog_f"], a["ws"], ctypes.c_size_t(a["ws_bytes"]),
                           a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(log_f=None), 1), (dict(dlog_f=None), 1), (dict(q=None), 1), (dict(d=32), 2),
    (dict(dtype=5), 3), (dict(log_f=FAKE + 4), 4), (dict(dlog_f=FAKE + 8), 4),
    (dict(scale=float("inf")), 9), (dict(), 5),
])
def test_fox_bwd_rejects_bad_arguments_before_launch(so, kw, code):
    assert _fox_bwd(so, **kw) == code


def test_bwd_head_size_128_checks(so):
    # d = 128 passes the size checks of both backwards (the workspace check then stops them)
    assert _bwd(so, d=128, ws_bytes=1000) == 5
    assert _fox_bwd(so, d=128, ws_bytes=1000) == 5
    assert _fox_bwd(so, d=96) == 2


def test_fwd_head_size_128_checks(so):
    # d = 128 passes the size checks of both forwards (the workspace check then stops
    # them); 96 does not; the early-exit extents exist at d = 64 only
    assert _fwd(so, d=128, ws_bytes=1000) == 5
    assert _fwd(so, d=96) == 2
    assert so.path_fox_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 1, 128, 128, 1,
                           ctypes.c_float(0.125), FAKE, ctypes.c_size_t(1000), None) == 5
    assert so.path_fox_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 1, 1, 128, 96, 1,
                           ctypes.c_float(0.125), FAKE, ctypes.c_size_t(1 << 30), None) == 2
    assert so.path_fox_first_blocks(FAKE, ctypes.c_size_t(1 << 30), 1, 1, 128, 128, 1, FAKE,
                                    None) == 2
