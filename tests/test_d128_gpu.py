"""Parity of the head-size-128 PaTH forward (through the C ABI) against the fp64 oracle.

The same bars as the d = 64 forward: fp32 inputs, max normwise relative error <= 1e-4 and
LSE within 1e-4; bf16 inputs, max absolute error <= 2e-2 on every element, mean absolute
error <= 2e-3, LSE within 2e-2. The oracle takes any head size.
"""
import numpy as np
import pytest
import torch

import oracle
import path_inputs as pi
from tests.test_parity_gpu import check_bf16

pytestmark = pytest.mark.gpu

D = 128


def _run(lib, x):
    return lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])


@pytest.mark.parametrize("B,H,L", [(1, 2, 200), (1, 1, 1), (2, 1, 64), (1, 2, 65), (1, 1, 384)])
def test_d128_fp32(lib, B, H, L):
    x = pi.make_fwd_inputs(B, H, L, d=D, dtype=torch.float32, seed=L + 5, clip=0.0, device="cuda")
    out, lse = _run(lib, x)
    assert out.shape == (B, H, L, D)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    rel = np.abs(out.double().cpu().numpy() - ref).max() / np.abs(ref).max()
    assert rel <= 1e-4, rel
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-4


@pytest.mark.parametrize("B,H,L", [(2, 2, 130), (1, 3, 257)])
def test_d128_bf16(lib, B, H, L):
    x = pi.make_fwd_inputs(B, H, L, d=D, dtype=torch.bfloat16, seed=L + 6, device="cuda")
    out, lse = _run(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    check_bf16(out, ref, lse, ref_lse)


def test_d128_two_stages_equal_the_fused_call(lib):
    x = pi.make_fwd_inputs(1, 2, 300, d=D, dtype=torch.bfloat16, seed=9, device="cuda")
    out, lse = _run(lib, x)
    ws = lib.new_workspace(lib.OP_FWD, 1, 2, 300, lib.BF16, x["q"].device, d=D)
    lib.path_fwd_prepare(x["q"], x["k"], x["w"], x["beta"], ws)
    out2, lse2 = lib.path_fwd_scan(x["v"], ws)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_d128_workload_sampled_rows(lib):
    # B4 H8 L2048 (the bf16 check workload's model width, 1024, in heads of 128) on 300
    # sampled rows, including the first and last row of every sampled head
    B, H, L = 4, 8, 2048
    x = pi.make_fwd_inputs(B, H, L, d=D, dtype=torch.bfloat16, seed=12, device="cuda")
    out, lse = _run(lib, x)
    g = np.random.default_rng(3)
    heads = g.integers(0, B * H, 100)
    rows = np.concatenate([np.stack([heads, g.integers(0, L, 100)], 1),
                           np.stack([heads[:100], np.zeros(100, np.int64)], 1),
                           np.stack([heads[:100], np.full(100, L - 1)], 1)]).astype(np.int64)
    ref, ref_lse = oracle.path_rows(x["q"], x["k"], x["v"], x["w"], x["beta"], rows)
    got = out.reshape(B * H, L, D)[rows[:, 0], rows[:, 1]]
    got_lse = lse.reshape(B * H, L)[rows[:, 0], rows[:, 1]]
    check_bf16(got, ref, got_lse, ref_lse)


def test_d128_fox_is_rejected(lib):
    x = pi.make_fwd_inputs(1, 1, 64, d=D, dtype=torch.bfloat16, seed=1, fox=True, device="cuda")
    with pytest.raises(Exception):
        lib.path_fox_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])


def test_d128_custom_scale(lib):
    x = pi.make_fwd_inputs(1, 2, 140, d=D, dtype=torch.float32, seed=21, clip=0.0, device="cuda")
    out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], scale=0.05)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], scale=0.05)
    rel = np.abs(out.double().cpu().numpy() - ref).max() / np.abs(ref).max()
    assert rel <= 1e-4, rel
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-4
