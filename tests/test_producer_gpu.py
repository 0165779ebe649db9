"""Parity of the w / beta producer (through the C ABI) against the fp64 oracle.

Tolerances: w (bf16 out; z and the tap-scaled up-projection are bf16 operands of fp32
contractions) within 2e-2 absolute on every element (the bf16 bar of the attention tests)
and 3e-3 on average; beta (fp32 out of an fp32-accumulated logit) within 1e-4 absolute.
"""
import numpy as np
import pytest
import torch

import oracle
import path_inputs as pi

pytestmark = pytest.mark.gpu

W_MAX_ABS, W_MEAN_ABS, BETA_ABS = 2e-2, 3e-3, 1e-4


def _run(lib, p, beta_max=2.0):
    return lib.path_wbeta_produce(p["x"], p["w_down"], p["w_up"], p["conv"], p["u"], p["bias"],
                                  beta_max=beta_max)


def _check(w, beta, ref_w, ref_beta):
    w = w.double().cpu().numpy()
    beta = beta.double().cpu().numpy()
    assert np.isfinite(w).all() and np.isfinite(beta).all()
    e = np.abs(w - ref_w)
    assert e.max() <= W_MAX_ABS, "w max abs err %g" % e.max()
    assert e.mean() <= W_MEAN_ABS, "w mean abs err %g" % e.mean()
    eb = np.abs(beta - ref_beta).max()
    assert eb <= BETA_ABS, "beta err %g" % eb


@pytest.mark.parametrize("B,L,D,R,H", [
    (2, 300, 128, 64, 3),    # ragged L across 128-token tiles, odd H (half-filled accumulator)
    (1, 1, 64, 64, 1),       # one token: no convolution history
    (3, 2, 64, 64, 2),       # two tokens
    (1, 130, 256, 128, 4),   # two K chunks in both contractions
    (1, 129, 128, 192, 64),  # R + H at the 256-column limit
    (5, 77, 192, 64, 5),     # B * L not a multiple of 128 (P1 tail crosses sequences)
    (3, 2000, 128, 64, 31),  # several (tile, head-pair) units per P2 CTA, runs crossing tiles
])
def test_producer_matches_oracle(lib, B, L, D, R, H):
    p = pi.make_producer_inputs(B, L, D, R, H, seed=B * 1000 + L, device="cuda")
    w, beta = _run(lib, p, beta_max=1.99)
    ref_w, ref_beta = oracle.wbeta_produce(p["x"], p["w_down"], p["w_up"], p["conv"], p["u"],
                                           p["bias"], beta_max=1.99)
    _check(w, beta, ref_w, ref_beta)
    assert w.shape == (B, H, L, 64) and beta.shape == (B, H, L)


def test_producer_zero_convolution_gives_zero_w(lib):
    p = pi.make_producer_inputs(1, 40, 64, 64, 2, seed=7, device="cuda")
    p["conv"] = torch.zeros_like(p["conv"])
    w, beta = _run(lib, p)
    assert torch.count_nonzero(w) == 0
    assert torch.isfinite(beta).all()


def test_producer_workload_sampled_tokens(lib):
    wl = pi.PRODUCER_L4096
    p = pi.make_producer_inputs(wl.B, wl.L, wl.D, wl.R, wl.H, seed=wl.seed, device="cuda")
    w, beta = _run(lib, p, beta_max=pi.BETA_CLIP)
    g = torch.Generator().manual_seed(17)
    bs = torch.randint(0, wl.B, (40,), generator=g).tolist() + [0, wl.B - 1, 3, 5]
    ts = torch.randint(0, wl.L, (40,), generator=g).tolist() + [0, wl.L - 1, 127, 128]
    host = {k: v.cpu() for k, v in p.items() if k != "x"}
    for b, t in zip(bs, ts):
        # w_t depends on x_{t-2..t} only: the oracle on that window is exact for token t
        lo = max(0, t - 2)
        xs = p["x"][b:b + 1, lo:t + 1].cpu()
        ref_w, ref_beta = oracle.wbeta_produce(xs, host["w_down"], host["w_up"], host["conv"],
                                               host["u"], host["bias"], beta_max=pi.BETA_CLIP)
        _check(w[b:b + 1, :, t:t + 1], beta[b:b + 1, :, t:t + 1], ref_w[:, :, -1:],
               ref_beta[:, :, -1:])


def test_producer_feeds_the_attention(lib):
    # the produced w and beta drive path_attn_fwd; the oracle chain is the fp64 producer
    # followed by the fp64 attention on the same rounded w
    B, L, H = 1, 200, 2
    p = pi.make_producer_inputs(B, L, 128, 64, H, seed=21, device="cuda")
    w, beta = _run(lib, p, beta_max=pi.BETA_CLIP)
    x = pi.make_fwd_inputs(B, H, L, seed=22, device="cuda")
    out, _ = lib.path_attn_fwd(x["q"], x["k"], x["v"], w, beta)
    ref_w, ref_beta = oracle.wbeta_produce(p["x"], p["w_down"], p["w_up"], p["conv"], p["u"],
                                           p["bias"], beta_max=pi.BETA_CLIP)
    np.testing.assert_allclose(w.double().cpu().numpy(), ref_w, atol=W_MAX_ABS)
    ref, _ = oracle.path_fwd(x["q"], x["k"], x["v"], w, beta)
    err = np.abs(out.double().cpu().numpy() - ref).max()
    assert err <= 2e-2, err
