"""Parity of the backward pass (path_attn_bwd, through the C ABI) against the fp64 oracle.

The GPU forward supplies out and lse, as a caller's would. Every gradient is compared
normwise: max |g - g*| / max |g*| over the tensor (the denominator at least 1% of the
largest reference gradient of the case).
- fp32 inputs: 1e-4, the fp32 forward's bar (every backward product is fp32 too).
- bf16 inputs: 2e-2, the bf16 forward's bar. The bf16 inputs themselves are exact for both
  sides. What differs is the forward's out, rounded to bf16 (a relative error of 2^-9),
  which enters every dS_ij through dout_i . out_i.
"""
import numpy as np
import pytest
import torch

import oracle
import path_inputs as pi

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
NAMES = ("dq", "dk", "dv", "dw", "dbeta")


def _case(lib, B, H, L, dtype, seed, beta_zero=False, wl=None):
    if wl is None:
        x = pi.make_fwd_inputs(B, H, L, seed=seed, dtype=dtype, device="cuda")
    else:
        x = pi.workload_inputs(wl, device="cuda")
    if beta_zero:
        x["beta"] = torch.zeros_like(x["beta"])
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    d_out = torch.randn((B, H, L, 64), generator=g).to(dtype).cuda()
    out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    grads = lib.path_attn_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out, lse, d_out)
    torch.cuda.synchronize()
    return x, d_out, grads


def _compare(grads, ref, tol, heads=None):
    # a gradient that is exactly zero (one token: the softmax weight is 1, so dS = 0) is
    # measured against 1% of the largest reference gradient instead of against itself
    names = NAMES + (("dlog_f",) if "dlog_f" in ref else ())
    floor = 1e-2 * max(np.abs(ref[n]).max() for n in names)
    for n in names:
        got = grads[n].double().cpu().numpy()
        if heads is not None:
            got = got.reshape(-1, *got.shape[2:])[heads]
        r = ref[n]
        assert np.isfinite(got).all(), n
        err = np.abs(got - r).max() / max(np.abs(r).max(), floor)
        assert err <= tol, "%s: normwise relative error %g (tolerance %g)" % (n, err, tol)


@pytest.mark.parametrize("B,H,L,dtype", [
    (1, 2, 128, torch.float32),    # two blocks
    (1, 2, 200, torch.float32),    # ragged last block
    (2, 2, 130, torch.bfloat16),   # bf16, ragged, three blocks
    (1, 1, 64, torch.float32),     # one block: no inter-block term
    (1, 1, 1, torch.float32),      # one token
    (1, 3, 65, torch.bfloat16),    # one token in the last block
    (1, 1, 384, torch.float32),    # six blocks: interior P_b gradients
])
def test_bwd_matches_oracle(lib, B, H, L, dtype):
    x, d_out, grads = _case(lib, B, H, L, dtype, seed=B * 100 + L)
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out)
    _compare(grads, ref, TOL[dtype])


def test_bwd_beta_zero_is_softmax_attention_gradient(lib):
    # beta = 0: every H_s is the identity, so dw must vanish exactly and dq, dk, dv are the
    # gradients of ordinary causal softmax attention
    x, d_out, grads = _case(lib, 1, 2, 192, torch.float32, seed=3, beta_zero=True)
    assert torch.count_nonzero(grads["dw"]) == 0
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out)
    _compare(grads, ref, 1e-4)


def test_bwd_workload_sampled_heads(lib):
    # the bf16 check workload (B4 H16 L2048, as bench.py times it): the oracle on two heads
    wl = pi.BF16_L2048
    x, d_out, grads = _case(lib, wl.B, wl.H, wl.L, wl.dtype, seed=wl.seed, wl=wl)
    heads = [5, wl.B * wl.H - 1]
    sel = {k: x[k].reshape(-1, *x[k].shape[2:])[heads] for k in ("q", "k", "v", "w", "beta")}
    ref = oracle.path_bwd(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"],
                          d_out.reshape(-1, wl.L, 64)[heads])
    _compare(grads, ref, TOL[torch.bfloat16], heads=heads)


def _fox_case(lib, B, H, L, dtype, seed, gate_scale=1.0, wl=None):
    if wl is None:
        x = pi.make_fwd_inputs(B, H, L, seed=seed, dtype=dtype, fox=True, device="cuda")
    else:
        x = pi.make_fwd_inputs(wl.B, wl.H, wl.L, seed=seed, dtype=wl.dtype, clip=wl.clip,
                               fox=True, device="cuda")
    x["log_f"] = (x["log_f"] * gate_scale).contiguous()
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    d_out = torch.randn((B, H, L, 64), generator=g).to(dtype).cuda()
    out, lse = lib.path_fox_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    grads = lib.path_fox_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], out, lse,
                             d_out)
    torch.cuda.synchronize()
    return x, d_out, grads


@pytest.mark.parametrize("B,H,L,dtype,gate_scale", [
    (1, 2, 200, torch.float32, 1.0),   # workload gate, ragged
    (2, 2, 130, torch.bfloat16, 1.0),  # bf16
    (1, 1, 64, torch.float32, 1.0),    # one block: the diagonal table carries the gate
    (1, 1, 384, torch.float32, 20.0),  # strong gate: the forward's early exit skips blocks
    (1, 2, 320, torch.bfloat16, 5.0),  # bf16, moderate gate
])
def test_fox_bwd_matches_oracle(lib, B, H, L, dtype, gate_scale):
    x, d_out, grads = _fox_case(lib, B, H, L, dtype, seed=7 * L + B, gate_scale=gate_scale)
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out, log_f=x["log_f"])
    _compare(grads, ref, TOL[dtype])


def test_fox_bwd_zero_gate_equals_plain_backward(lib):
    # log f = 0: the forward is plain PaTH, so dq .. dbeta equal the plain backward's within
    # fp32 rounding, while d log f still carries the gradient of the gate
    x, d_out, grads = _fox_case(lib, 1, 2, 256, torch.float32, seed=11, gate_scale=0.0)
    out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    plain = lib.path_attn_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out, lse, d_out)
    for n in NAMES:
        a, b = grads[n].double(), plain[n].double()
        assert (a - b).abs().max().item() <= 1e-5 * max(b.abs().max().item(), 1.0), n
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out, log_f=x["log_f"])
    _compare(grads, ref, 1e-4)


def test_fox_bwd_workload_sampled_heads(lib):
    # the B4 H16 L2048 bf16 workload with the PaTH-FoX gate: the oracle on two heads
    wl = pi.BF16_L2048
    x, d_out, grads = _fox_case(lib, wl.B, wl.H, wl.L, wl.dtype, seed=wl.seed, wl=wl)
    heads = [3, wl.B * wl.H - 2]
    sel = {k: x[k].reshape(-1, *x[k].shape[2:])[heads]
           for k in ("q", "k", "v", "w", "beta", "log_f")}
    ref = oracle.path_bwd(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"],
                          d_out.reshape(-1, wl.L, 64)[heads], log_f=sel["log_f"])
    _compare(grads, ref, TOL[torch.bfloat16], heads=heads)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("kind", ["projection", "reflection", "identity"])
def test_bwd_degenerate_transitions(lib, kind, dtype):
    # beta = 1: every H_s is a projection (singular; the fp32 block pass undoes its steps
    # from the recorded w . x and never inverts H_s, the bf16 one inverts only the unit
    # triangular I + D strictly-upper(W W^T)); beta = 2: exact reflections; w = 0: H = I
    x = pi.make_fwd_inputs(1, 2, 200, seed=31, dtype=dtype, clip=0.0, device="cuda")
    if kind == "projection":
        x["beta"] = torch.ones_like(x["beta"])
    elif kind == "reflection":
        x["beta"] = torch.full_like(x["beta"], 2.0)
    else:
        x["w"] = torch.zeros_like(x["w"])
    g = torch.Generator(device="cpu").manual_seed(32)
    d_out = torch.randn((1, 2, 200, 64), generator=g).to(dtype).cuda()
    out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    grads = lib.path_attn_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out, lse, d_out)
    torch.cuda.synchronize()
    if kind == "identity":
        assert torch.count_nonzero(grads["dw"]) == 0 and torch.count_nonzero(grads["dbeta"]) == 0
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out)
    _compare(grads, ref, TOL[dtype])


def test_bwd_long_head_fp32(lib):
    # one fp32 head of 4096 tokens: 64 blocks, 2016 carried pairs, the fp32 bar throughout
    x, d_out, grads = _case(lib, 1, 1, 4096, torch.float32, seed=41)
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out)
    _compare(grads, ref, 1e-4)


def test_bwd_max_heads(lib):
    # B * H at the 65535 limit (the grid's second dimension), two blocks per head
    B, L = 65535, 65
    x, d_out, grads = _case(lib, B, 1, L, torch.bfloat16, seed=43)
    heads = [0, 1, 32767, B - 1]
    sel = {k: x[k].reshape(-1, *x[k].shape[2:])[heads] for k in ("q", "k", "v", "w", "beta")}
    ref = oracle.path_bwd(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"],
                          d_out.reshape(-1, L, 64)[heads])
    _compare(grads, ref, TOL[torch.bfloat16], heads=heads)


def test_bwd_custom_scale(lib):
    # a softmax scale other than 1/sqrt(d): it multiplies the whole logit, so every
    # gradient but dv carries it
    x = pi.make_fwd_inputs(1, 2, 150, seed=51, dtype=torch.float32, clip=0.0, device="cuda")
    d_out = torch.randn((1, 2, 150, 64), generator=torch.Generator().manual_seed(52)).cuda()
    out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], scale=0.3)
    grads = lib.path_attn_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out, lse, d_out,
                              scale=0.3)
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out, scale=0.3)
    _compare(grads, ref, 1e-4)


@pytest.mark.parametrize("L", [1, 65])
def test_fox_bwd_short(lib, L):
    # one token (every gradient but dv and d log f of a single logit is zero) and one token
    # in the last block
    x, d_out, grads = _fox_case(lib, 1, 2, L, torch.float32, seed=60 + L)
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out, log_f=x["log_f"])
    _compare(grads, ref, 1e-4)


# ---------------------------------------------------------------- bf16: tensor-core query pass

@pytest.mark.parametrize("L", [1, 64, 127, 384, 1000])
def test_bwd_bf16_lengths(lib, L):
    # one token, one block, a ragged second block, six blocks (interior P_b) and 16 blocks
    # with a ragged last one: the tile steps, the diagonal pair and the pass-2 walk
    x, d_out, grads = _case(lib, 1, 2, L, torch.bfloat16, seed=700 + L)
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out)
    _compare(grads, ref, TOL[torch.bfloat16])


@pytest.mark.parametrize("kind", ["beta_zero", "projection", "reflection", "identity", "scale"])
def test_bwd_bf16_special_transitions(lib, kind):
    x = pi.make_fwd_inputs(1, 2, 300, seed=77, dtype=torch.bfloat16, device="cuda")
    scale = None
    if kind == "beta_zero":
        x["beta"] = torch.zeros_like(x["beta"])
    elif kind == "projection":
        x["beta"] = torch.ones_like(x["beta"])
    elif kind == "reflection":
        x["beta"] = torch.full_like(x["beta"], 2.0)
    elif kind == "identity":
        x["w"] = torch.zeros_like(x["w"])
    else:
        scale = 0.3
    d_out = torch.randn((1, 2, 300, 64), generator=torch.Generator().manual_seed(78))
    d_out = d_out.to(torch.bfloat16).cuda()
    out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], scale=scale)
    grads = lib.path_attn_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out, lse, d_out,
                              scale=scale)
    torch.cuda.synchronize()
    if kind in ("beta_zero", "identity"):
        assert torch.count_nonzero(grads["dw"]) == 0
    if kind == "identity":
        assert torch.count_nonzero(grads["dbeta"]) == 0
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out, scale=scale)
    _compare(grads, ref, TOL[torch.bfloat16])


@pytest.mark.parametrize("L,gate_scale", [(1, 1.0), (64, 1.0), (700, 1.0), (700, 20.0)])
def test_fox_bwd_bf16(lib, L, gate_scale):
    x, d_out, grads = _fox_case(lib, 1, 2, L, torch.bfloat16, seed=900 + L,
                                gate_scale=gate_scale)
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out, log_f=x["log_f"])
    _compare(grads, ref, TOL[torch.bfloat16])


def test_bwd_bf16_deterministic_up_to_atomics(lib):
    # two runs agree within fp32 reassociation of the gathered gradients
    x, d_out, g1 = _case(lib, 1, 3, 500, torch.bfloat16, seed=5)
    out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    g2 = lib.path_attn_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out, lse, d_out)
    for n in NAMES:
        a, b = g1[n].double(), g2[n].double()
        assert (a - b).abs().max().item() <= 1e-4 * max(b.abs().max().item(), 1e-6), n


# ---------------------------------------------------------------- head size 128 (fp32 kernels)

def _case128(lib, B, H, L, dtype, seed, fox=False, gate_scale=1.0, mutate=None, x=None):
    if x is None:
        x = pi.make_fwd_inputs(B, H, L, d=128, seed=seed, dtype=dtype, fox=fox, device="cuda")
    if fox:
        x["log_f"] = (x["log_f"] * gate_scale).contiguous()
    if mutate is not None:
        mutate(x)
    g = torch.Generator(device="cpu").manual_seed(seed + 1)
    d_out = torch.randn((B, H, L, 128), generator=g).to(dtype).cuda()
    if fox:
        out, lse = lib.path_fox_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
        grads = lib.path_fox_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], out,
                                 lse, d_out)
    else:
        out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
        grads = lib.path_attn_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out, lse, d_out)
    torch.cuda.synchronize()
    assert grads["dq"].shape == (B, H, L, 128)
    return x, d_out, grads


@pytest.mark.parametrize("B,H,L,dtype", [
    (1, 2, 128, torch.float32),    # two blocks
    (1, 2, 200, torch.float32),    # ragged last block
    (1, 1, 1, torch.float32),      # one token
    (1, 1, 64, torch.float32),     # one block: no inter-block term
    (1, 1, 320, torch.float32),    # five blocks: interior 128 x 128 P_b gradients
    (2, 2, 130, torch.bfloat16),   # bf16, ragged, three blocks
    (1, 2, 384, torch.bfloat16),   # bf16, six blocks
])
def test_bwd_d128_matches_oracle(lib, B, H, L, dtype):
    x, d_out, grads = _case128(lib, B, H, L, dtype, seed=3000 + 10 * B + L)
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out)
    _compare(grads, ref, TOL[dtype])


@pytest.mark.parametrize("B,H,L,dtype,gate_scale", [
    (1, 2, 200, torch.float32, 1.0),   # workload gate, ragged
    (1, 1, 1, torch.float32, 1.0),     # one token
    (1, 1, 384, torch.float32, 20.0),  # strong gate: the forward's early exit skips blocks
    (2, 2, 130, torch.bfloat16, 1.0),  # bf16
    (1, 2, 320, torch.bfloat16, 5.0),  # bf16, moderate gate
])
def test_fox_bwd_d128_matches_oracle(lib, B, H, L, dtype, gate_scale):
    x, d_out, grads = _case128(lib, B, H, L, dtype, seed=3100 + 7 * L + B, fox=True,
                               gate_scale=gate_scale)
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out, log_f=x["log_f"])
    _compare(grads, ref, TOL[dtype])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("kind", ["projection", "reflection", "identity"])
def test_bwd_d128_degenerate_transitions(lib, kind, dtype):
    # beta = 1 (singular projections), beta = 2 (reflections), w = 0 (H = I), at d = 128
    def mutate(x):
        if kind == "projection":
            x["beta"] = torch.ones_like(x["beta"])
        elif kind == "reflection":
            x["beta"] = torch.full_like(x["beta"], 2.0)
        else:
            x["w"] = torch.zeros_like(x["w"])
    x0 = pi.make_fwd_inputs(1, 2, 200, d=128, seed=3200, dtype=dtype, clip=0.0, device="cuda")
    x, d_out, grads = _case128(lib, 1, 2, 200, dtype, seed=3200, mutate=mutate, x=x0)
    if kind == "identity":
        assert torch.count_nonzero(grads["dw"]) == 0 and torch.count_nonzero(grads["dbeta"]) == 0
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out)
    _compare(grads, ref, TOL[dtype])


@pytest.mark.parametrize("fox", [False, True])
def test_bwd_d128_workload_sampled_heads(lib, fox):
    # B4 H8 L2048 bf16 at head size 128 (32 blocks per head, 496 carried pairs): the oracle
    # on two heads
    B, H, L = 4, 8, 2048
    x, d_out, grads = _case128(lib, B, H, L, torch.bfloat16, seed=3300, fox=fox)
    heads = [1, B * H - 1]
    names = ("q", "k", "v", "w", "beta") + (("log_f",) if fox else ())
    sel = {k: x[k].reshape(-1, *x[k].shape[2:])[heads] for k in names}
    ref = oracle.path_bwd(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"],
                          d_out.reshape(-1, L, 128)[heads], log_f=sel.get("log_f"))
    _compare(grads, ref, TOL[torch.bfloat16], heads=heads)


def test_bwd_d128_max_heads(lib):
    # B * H at the 65535 limit (the grid's second dimension), two blocks per head, head
    # size 128 (tensor-core query pass)
    B, L = 65535, 65
    x = pi.make_fwd_inputs(B, 1, L, d=128, seed=3400, dtype=torch.bfloat16, device="cuda")
    x, d_out, grads = _case128(lib, B, 1, L, torch.bfloat16, seed=3400, x=x)
    heads = [0, 1, 32767, B - 1]
    sel = {k: x[k].reshape(-1, *x[k].shape[2:])[heads] for k in ("q", "k", "v", "w", "beta")}
    ref = oracle.path_bwd(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"],
                          d_out.reshape(-1, L, 128)[heads])
    _compare(grads, ref, TOL[torch.bfloat16], heads=heads)


@pytest.mark.parametrize("dtype,fox", [(torch.bfloat16, False), (torch.bfloat16, True),
                                       (torch.float32, False)])
def test_bwd_d128_custom_scale(lib, dtype, fox):
    # a softmax scale other than 1/sqrt(d): the query pass carries dS unscaled and scales
    # its products on output
    x = pi.make_fwd_inputs(1, 2, 150, d=128, seed=3500, dtype=dtype, fox=fox, device="cuda")
    d_out = torch.randn((1, 2, 150, 128), generator=torch.Generator().manual_seed(3501))
    d_out = d_out.to(dtype).cuda()
    if fox:
        out, lse = lib.path_fox_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"],
                                    scale=0.3)
        grads = lib.path_fox_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], out,
                                 lse, d_out, scale=0.3)
    else:
        out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], scale=0.3)
        grads = lib.path_attn_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out, lse, d_out,
                                  scale=0.3)
    torch.cuda.synchronize()
    ref = oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out, scale=0.3,
                          log_f=x["log_f"] if fox else None)
    _compare(grads, ref, TOL[dtype])
