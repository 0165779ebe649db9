"""Every entry point is stream-ordered and allocates nothing, so a sequence of calls can be
captured once in a CUDA graph and replayed on new inputs written into the same buffers.
Each test captures on a side stream (after one eager warm-up call), replays on fresh inputs
and compares with eager calls on those inputs bit for bit: the graph runs the same
kernels with the same launch shapes.
"""
import pytest
import torch

import path_inputs as pi

pytestmark = pytest.mark.gpu


def _capture(fn):
    """fn() launched once eagerly on a side stream, then captured; returns the graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _refill(dst, src):
    for k, t in src.items():
        dst[k].copy_(t)


@pytest.mark.parametrize("d,fox", [(64, False), (64, True), (128, False), (128, True)])
def test_forward_graph_replay(lib, d, fox):
    B, H, L = 2, 3, 700
    x = pi.make_fwd_inputs(B, H, L, d=d, seed=61, fox=fox, device="cuda")
    op = lib.OP_FOX_FWD if fox else lib.OP_FWD
    ws = lib.new_workspace(op, B, H, L, lib.BF16, "cuda", d=d)
    out = torch.empty_like(x["q"])
    lse = torch.empty((B, H, L), dtype=torch.float32, device="cuda")

    def fwd():
        if fox:
            lib.path_fox_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], out=out,
                             lse=lse, workspace=ws)
        else:
            lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out=out, lse=lse,
                              workspace=ws)

    g = _capture(fwd)
    x2 = pi.make_fwd_inputs(B, H, L, d=d, seed=62, fox=fox, device="cuda")
    _refill(x, x2)
    g.replay()
    torch.cuda.synchronize()
    got, got_lse = out.clone(), lse.clone()
    fwd()
    torch.cuda.synchronize()
    assert torch.equal(got, out) and torch.equal(got_lse, lse)
    assert lib.path_check_workspace(ws) == lib.OK


def test_backward_graph_replay(lib):
    B, H, L = 1, 2, 300
    x = pi.make_fwd_inputs(B, H, L, seed=63, device="cuda")
    out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    gen = torch.Generator(device="cuda").manual_seed(64)
    d_out = torch.randn(out.shape, generator=gen, device="cuda").to(out.dtype)
    ws = lib.new_workspace(lib.OP_BWD, B, H, L, lib.BF16, "cuda")
    grads = {n: torch.empty((B, H, L, 64), dtype=torch.float32, device="cuda")
             for n in ("dq", "dk", "dv", "dw")}
    grads["dbeta"] = torch.empty((B, H, L), dtype=torch.float32, device="cuda")

    def bwd():
        lib.path_attn_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out, lse, d_out,
                          grads=grads, workspace=ws)

    g = _capture(bwd)
    x2 = pi.make_fwd_inputs(B, H, L, seed=65, device="cuda")
    o2, l2 = lib.path_attn_fwd(x2["q"], x2["k"], x2["v"], x2["w"], x2["beta"])
    _refill(x, x2)
    out.copy_(o2)
    lse.copy_(l2)
    g.replay()
    torch.cuda.synchronize()
    got = {n: t.clone() for n, t in grads.items()}
    bwd()
    torch.cuda.synchronize()
    # the backward accumulates some gradients with atomics: replay and eager may add the
    # same terms in another order, and the bf16 block pass reads those sums as tf32 operands
    # (a 10-bit significand), so an order-dependent last bit can move a result by about
    # 2^-10 of its size; a replay of stale inputs would differ by the whole gradient
    for n, t in grads.items():
        tol = 2e-3 * t.abs().max().item() + 1e-30
        assert (got[n] - t).abs().max().item() <= tol, n


def test_decode_steps_graph_replay(lib):
    # four decode steps (cache lengths fixed at capture) in one graph; replay from the same
    # starting cache equals four eager steps
    wl = pi.DecodeWorkload("graph", 2, 2, 300, 4, 64, torch.bfloat16, 5, 1000)
    cap = 304
    kc, vc = pi.make_decode_prefix(wl, cap, device="cuda")
    k0, v0 = kc.clone(), vc.clone()
    steps = [pi.make_decode_step(wl, t, device="cuda") for t in range(4)]
    ws = lib.new_workspace(lib.OP_DECODE, 2, 2, cap, lib.BF16, "cuda")
    outs = [torch.empty((2, 2, 64), dtype=torch.bfloat16, device="cuda") for _ in range(4)]

    def run():
        for t, s in enumerate(steps):
            lib.path_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], kc, vc, 300 + t,
                                 out=outs[t], workspace=ws)

    g = _capture(run)
    kc.copy_(k0)
    vc.copy_(v0)
    g.replay()
    torch.cuda.synchronize()
    got = [o.clone() for o in outs]
    gk, gv = kc.clone(), vc.clone()
    kc.copy_(k0)
    vc.copy_(v0)
    run()
    torch.cuda.synchronize()
    assert all(torch.equal(a, b) for a, b in zip(got, outs))
    assert torch.equal(gk, kc) and torch.equal(gv, vc)


def test_producer_graph_replay(lib):
    p = pi.make_producer_inputs(2, 300, 256, 64, 4, seed=66, device="cuda")
    w = torch.empty((2, 4, 300, 64), dtype=torch.bfloat16, device="cuda")
    beta = torch.empty((2, 4, 300), dtype=torch.float32, device="cuda")
    ws = torch.empty(lib.path_wbeta_workspace_bytes(2, 300, 256, 64, 4, 64, lib.BF16),
                     dtype=torch.uint8, device="cuda")

    def prod():
        lib.path_wbeta_produce(p["x"], p["w_down"], p["w_up"], p["conv"], p["u"], p["bias"],
                               beta_max=pi.BETA_CLIP, w_out=w, beta_out=beta, workspace=ws)

    g = _capture(prod)
    p2 = pi.make_producer_inputs(2, 300, 256, 64, 4, seed=67, device="cuda")
    _refill(p, p2)
    g.replay()
    torch.cuda.synchronize()
    gw, gb = w.clone(), beta.clone()
    prod()
    torch.cuda.synchronize()
    assert torch.equal(gw, w) and torch.equal(gb, beta)
