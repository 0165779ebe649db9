"""Parity of the head-size-128 PaTH and PaTH-FoX forward (through the C ABI) against the
fp64 oracle.

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


def test_d128_speed_width_sampled_rows(lib):
    # B32 H16 L4096 d128 (the speed workload's tokens and model width in heads of 128, the
    # bench's head-size-128 leg) on 300 sampled rows, with first and last rows
    B, H, L = 32, 16, 4096
    x = pi.make_fwd_inputs(B, H, L, d=D, dtype=torch.bfloat16, seed=12, device="cuda")
    out, lse = _run(lib, x)
    g = np.random.default_rng(5)
    heads = g.integers(0, B * H, 100)
    rows = np.concatenate([np.stack([heads, g.integers(0, L, 100)], 1),
                           np.stack([heads, np.zeros(100, np.int64)], 1),
                           np.stack([heads, np.full(100, L - 1)], 1)]).astype(np.int64)
    hs = np.unique(heads)
    h = {k: v.reshape(B * H, L, *v.shape[3:])[torch.as_tensor(hs, device=v.device)].cpu()
         for k, v in x.items()}
    loc = np.searchsorted(hs, rows[:, 0])
    ref, ref_lse = oracle.path_rows(h["q"], h["k"], h["v"], h["w"], h["beta"],
                                    np.stack([loc, rows[:, 1]], 1))
    got = out.reshape(B * H, L, D)[rows[:, 0], rows[:, 1]]
    got_lse = lse.reshape(B * H, L)[rows[:, 0], rows[:, 1]]
    check_bf16(got, ref, got_lse, ref_lse)


def _fox(lib, x, scale=None):
    return lib.path_fox_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], scale=scale)


def _check_fp32(out, lse, ref, ref_lse):
    rel = np.abs(out.double().cpu().numpy() - ref).max() / np.abs(ref).max()
    assert rel <= 1e-4, rel
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-4


@pytest.mark.parametrize("B,H,L", [(1, 2, 200), (1, 1, 1), (2, 1, 64), (1, 2, 65), (1, 1, 384)])
def test_d128_fox_fp32(lib, B, H, L):
    x = pi.make_fwd_inputs(B, H, L, d=D, dtype=torch.float32, seed=L + 7, clip=0.0, fox=True,
                           device="cuda")
    out, lse = _fox(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    _check_fp32(out, lse, ref, ref_lse)


@pytest.mark.parametrize("B,H,L", [(2, 2, 130), (1, 3, 257)])
def test_d128_fox_bf16(lib, B, H, L):
    x = pi.make_fwd_inputs(B, H, L, d=D, dtype=torch.bfloat16, seed=L + 8, fox=True,
                           device="cuda")
    out, lse = _fox(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    check_bf16(out, ref, lse, ref_lse)


def test_d128_fox_two_stages_equal_the_fused_call(lib):
    x = pi.make_fwd_inputs(1, 2, 300, d=D, dtype=torch.bfloat16, seed=19, fox=True, device="cuda")
    out, lse = _fox(lib, x)
    ws = lib.new_workspace(lib.OP_FOX_FWD, 1, 2, 300, lib.BF16, x["q"].device, d=D)
    lib.path_fwd_prepare(x["q"], x["k"], x["w"], x["beta"], ws, log_f=x["log_f"])
    out2, lse2 = lib.path_fwd_scan(x["v"], ws, fox=True)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_d128_fox_zero_gate_is_path(lib):
    # log f = 0: every bias is an exact zero, so PaTH-FoX gives PaTH's bits
    x = pi.make_fwd_inputs(1, 2, 333, d=D, dtype=torch.bfloat16, seed=23, fox=True, device="cuda")
    x["log_f"] = torch.zeros_like(x["log_f"])
    out, lse = _fox(lib, x)
    out2, lse2 = _run(lib, x)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_d128_fox_long_gate_sums_fp32(lib):
    # 8192 tokens at log f ~ -1.3: the gate prefix sums reach about -10^4 while the bias
    # against recent keys stays small; it must be accurate to its own size for the fp32
    # bars to hold on rows all along the sequence
    x = pi.make_fwd_inputs(1, 1, 8192, d=D, dtype=torch.float32, seed=47, clip=0.0, fox=True,
                           device="cuda")
    g = torch.Generator(device="cpu").manual_seed(147)
    x["log_f"] = torch.nn.functional.logsigmoid(
        torch.randn(x["log_f"].shape, generator=g) - 1.0).to("cuda").contiguous()
    out, lse = _fox(lib, x)
    rows = np.arange(0, 8192, 61)
    pairs = np.stack([np.zeros_like(rows), rows], axis=1)
    h = {k: v[0].cpu() for k, v in x.items()}
    ref, ref_lse = oracle.path_rows(h["q"], h["k"], h["v"], h["w"], h["beta"], pairs, h["log_f"])
    got = out[0, 0].double().cpu().numpy()[rows]
    assert np.abs(got - ref).max() / np.abs(ref).max() <= 1e-4
    assert np.abs(lse[0, 0].double().cpu().numpy()[rows] - ref_lse).max() <= 1e-4


def test_d128_fox_early_exit_skips_blocks(lib):
    # log f = -5 per token: keys a block or more behind a query weigh about e^-300. The
    # values of blocks 0 and 1 are NaN: a query block that visited them would turn NaN
    # (0 x NaN), so finite rows from block 3 on show the scan stopped above them, and they
    # match the oracle on the clean values (the skipped weights are below e^-40)
    L = 640
    x = pi.make_fwd_inputs(1, 2, L, d=D, dtype=torch.float32, seed=51, clip=0.0, fox=True,
                           device="cuda")
    x["log_f"] = torch.full_like(x["log_f"], -5.0)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    x["v"][:, :, :128] = float("nan")
    out, lse = _fox(lib, x)
    got = out[:, :, 192:].double().cpu().numpy()
    assert np.isfinite(got).all()
    r = ref[:, :, 192:]
    assert np.abs(got - r).max() / np.abs(r).max() <= 1e-4
    assert np.abs(lse[:, :, 192:].double().cpu().numpy() - ref_lse[:, :, 192:]).max() <= 1e-4


def test_d128_fox_early_exit_skips_blocks_bf16(lib):
    # the tensor-core scan (bf16) stops at the extents computed before it: with log f = -5
    # per token and the values of blocks 0 and 1 NaN, rows from block 4 on (128-row tiles of
    # two query blocks) stay finite and match the oracle on the clean values
    L = 640
    x = pi.make_fwd_inputs(1, 2, L, d=D, dtype=torch.bfloat16, seed=52, fox=True, device="cuda")
    x["log_f"] = torch.full_like(x["log_f"], -5.0)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    x["v"][:, :, :128] = float("nan")
    out, lse = _fox(lib, x)
    got = out[:, :, 256:]
    assert torch.isfinite(got).all()
    check_bf16(got, ref[:, :, 256:], lse[:, :, 256:], ref_lse[:, :, 256:])


@pytest.mark.parametrize("L", [384, 1000])
def test_d128_fox_own_block_only_gate(lib, L):
    # log f = -200 per token: every query block needs only its own block (the bf16 scan
    # walks two blocks per tile), with an odd tile count at L = 384
    x = pi.make_fwd_inputs(2, 2, L, d=D, dtype=torch.bfloat16, seed=54, fox=True, device="cuda")
    x["log_f"] = torch.full_like(x["log_f"], -200.0)
    out, lse = _fox(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    check_bf16(out, ref, lse, ref_lse)


def test_d128_fox_mixed_sign_gate(lib):
    # log f of both signs (the bias against older keys can be positive), custom scale
    x = pi.make_fwd_inputs(2, 2, 640, d=D, dtype=torch.bfloat16, seed=49, fox=True, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(149)
    x["log_f"] = (0.5 * torch.randn(x["log_f"].shape, generator=g) - 0.3).to("cuda").contiguous()
    out, lse = _fox(lib, x, scale=0.2)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"],
                                   scale=0.2)
    check_bf16(out, ref, lse, ref_lse)


def test_d128_fox_workload_sampled_rows(lib):
    # PaTH-FoX on B4 H8 L2048 d128 bf16, 300 sampled rows with the first and last rows
    B, H, L = 4, 8, 2048
    x = pi.make_fwd_inputs(B, H, L, d=D, dtype=torch.bfloat16, seed=13, fox=True, device="cuda")
    out, lse = _fox(lib, x)
    g = np.random.default_rng(4)
    heads = g.integers(0, B * H, 100)
    rows = np.concatenate([np.stack([heads, g.integers(0, L, 100)], 1),
                           np.stack([heads, np.zeros(100, np.int64)], 1),
                           np.stack([heads, np.full(100, L - 1)], 1)]).astype(np.int64)
    ref, ref_lse = oracle.path_rows(x["q"], x["k"], x["v"], x["w"], x["beta"], rows, x["log_f"])
    got = out.reshape(B * H, L, D)[rows[:, 0], rows[:, 1]]
    got_lse = lse.reshape(B * H, L)[rows[:, 0], rows[:, 1]]
    check_bf16(got, ref, got_lse, ref_lse)


def test_d128_custom_scale(lib):
    x = pi.make_fwd_inputs(1, 2, 140, d=D, dtype=torch.float32, seed=21, clip=0.0, device="cuda")
    out, lse = lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], scale=0.05)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], scale=0.05)
    rel = np.abs(out.double().cpu().numpy() - ref).max() / np.abs(ref).max()
    assert rel <= 1e-4, rel
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-4


@pytest.mark.parametrize("fox", [False, True])
def test_d128_empty_sequence(lib, fox):
    x = pi.make_fwd_inputs(2, 3, 0, d=D, dtype=torch.bfloat16, seed=1, fox=fox, device="cuda")
    out, lse = _fox(lib, x) if fox else _run(lib, x)
    assert out.shape == (2, 3, 0, D) and lse.shape == (2, 3, 0)


def test_d128_has_no_precomputed_extents(lib):
    x = pi.make_fwd_inputs(1, 1, 128, d=D, dtype=torch.bfloat16, seed=2, fox=True, device="cuda")
    ws = lib.new_workspace(lib.OP_FOX_FWD, 1, 1, 128, lib.BF16, "cuda", d=D)
    lib.path_fwd_prepare(x["q"], x["k"], x["w"], x["beta"], ws, log_f=x["log_f"])
    with pytest.raises(lib.PathError):
        lib.path_fox_first_blocks(ws, 1, 1, 128, torch.bfloat16, d=D)


@pytest.mark.parametrize("fox", [False, True])
def test_d128_max_heads(lib, fox):
    # 65535 heads (the grid's y limit) of 70 tokens (two blocks, the second ragged); sampled
    # rows of sampled heads against the oracle
    B, H, L = 65535, 1, 70
    x = pi.make_fwd_inputs(B, H, L, d=D, dtype=torch.bfloat16, seed=31, fox=fox, device="cuda")
    out, lse = _fox(lib, x) if fox else _run(lib, x)
    g = np.random.default_rng(5)
    heads = np.concatenate([[0, B * H - 1], g.integers(0, B * H, 60)])
    rows = np.stack([heads, g.integers(0, L, heads.size)], 1).astype(np.int64)
    rows = np.concatenate([rows, np.stack([heads, np.full(heads.size, L - 1)], 1)])
    sel = torch.as_tensor(np.unique(rows[:, 0]), device="cuda")
    sub = {k: v.reshape(B * H, *v.shape[2:])[sel] for k, v in x.items()}
    remap = {int(h): i for i, h in enumerate(sel.tolist())}
    local = np.stack([[remap[int(h)] for h in rows[:, 0]], rows[:, 1]], 1).astype(np.int64)
    ref, ref_lse = oracle.path_rows(sub["q"], sub["k"], sub["v"], sub["w"], sub["beta"], local,
                                    sub.get("log_f"))
    got = out.reshape(B * H, L, D)[rows[:, 0], rows[:, 1]]
    got_lse = lse.reshape(B * H, L)[rows[:, 0], rows[:, 1]]
    check_bf16(got, ref, got_lse, ref_lse)


# ---------------------------------------------------------------- bf16: tensor-core kernels

@pytest.mark.parametrize("L", [1, 63, 64, 65, 127, 128, 129, 384, 1000])
def test_d128_bf16_lengths(lib, L):
    # the tile's diagonal pair, a padded odd last block, and walks of up to 16 key blocks
    x = pi.make_fwd_inputs(1, 2, L, d=D, dtype=torch.bfloat16, seed=1100 + L, device="cuda")
    out, lse = _run(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    check_bf16(out, ref, lse, ref_lse)


@pytest.mark.parametrize("gate_scale", [1.0, 8.0])
def test_d128_fox_bf16_lengths_and_gates(lib, gate_scale):
    # PaTH-FoX through the tensor-core scan (no early exit there: vanishing keys weigh 0)
    x = pi.make_fwd_inputs(1, 2, 700, d=D, dtype=torch.bfloat16, seed=1200, fox=True,
                           device="cuda")
    x["log_f"] = (x["log_f"] * gate_scale).contiguous()
    out, lse = _fox(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    check_bf16(out, ref, lse, ref_lse)


@pytest.mark.parametrize("kind", ["beta_zero", "reflection", "identity"])
def test_d128_bf16_special_transitions(lib, kind):
    x = pi.make_fwd_inputs(1, 2, 260, d=D, dtype=torch.bfloat16, seed=1300, device="cuda")
    if kind == "beta_zero":
        x["beta"] = torch.zeros_like(x["beta"])
    elif kind == "reflection":
        x["beta"] = torch.full_like(x["beta"], 1.99)
    else:
        x["w"] = torch.zeros_like(x["w"])
    out, lse = _run(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    check_bf16(out, ref, lse, ref_lse)
