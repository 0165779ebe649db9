"""Parity of the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances: fp32 inputs, max normwise relative error <= 1e-4 (max|o - o*| / max|o*|);
bf16 inputs, max absolute error <= 2e-2 on every output element, plus a mean absolute
error bound (2e-3) that catches systematic drift which the max bound would miss, and
LSE within 2e-2 absolute. The oracle sees exactly the rounded tensors the GPU sees.
"""
import numpy as np
import pytest
import torch

import oracle
import path_inputs as pi

pytestmark = pytest.mark.gpu

BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
F32_MAX_REL = 1e-4


def run_fwd(pa, x, fox=False, scale=None):
    if fox:
        return pa.path_fox_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], scale=scale)
    return pa.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], scale=scale)


def check_bf16(got, ref, lse=None, ref_lse=None):
    got = got.double().cpu().numpy() if hasattr(got, "cpu") else got
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert err.max() <= BF16_MAX_ABS, "max abs err %g" % err.max()
    assert err.mean() <= BF16_MEAN_ABS, "mean abs err %g" % err.mean()
    if lse is not None:
        le = np.abs(lse.double().cpu().numpy() - ref_lse)
        assert le.max() <= BF16_MAX_ABS, "lse err %g" % le.max()


# ---------------------------------------------------------------- fp32

def test_tiny_fp32_workload(lib, record_property):
    x = pi.workload_inputs(pi.TINY_FP32, device="cuda")
    out, lse = run_fwd(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    err = np.abs(out.double().cpu().numpy() - ref)
    rel = err.max() / np.abs(ref).max()
    assert rel <= F32_MAX_REL, rel
    # the element-wise figure |o - o*| / max(|o*|, 1e-3), reported beside the normwise one;
    # the normwise bar implies it is at most 1e-4 * max|o*| / 1e-3 everywhere
    elem = (err / np.maximum(np.abs(ref), 1e-3)).max()
    record_property("normwise_rel", float(rel))
    record_property("elementwise_rel", float(elem))
    print("tiny fp32: normwise %.3g, element-wise %.3g" % (rel, elem))
    assert elem <= F32_MAX_REL * np.abs(ref).max() / 1e-3
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-4


@pytest.mark.parametrize("L", [1, 50, 64, 65, 130, 257])
@pytest.mark.parametrize("fox", [False, True])
def test_fp32_ragged(lib, L, fox):
    x = pi.make_fwd_inputs(2, 2, L, dtype=torch.float32, seed=L, clip=0.0, fox=fox, device="cuda")
    out, lse = run_fwd(lib, x, fox)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x.get("log_f"))
    rel = np.abs(out.double().cpu().numpy() - ref).max() / np.abs(ref).max()
    assert rel <= F32_MAX_REL, rel
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-4


# ---------------------------------------------------------------- bf16, full oracle

@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 127, 128, 129, 200, 384, 515])
def test_bf16_ragged_lengths(lib, L):
    x = pi.make_fwd_inputs(2, 3, L, seed=100 + L, device="cuda")
    out, lse = run_fwd(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    check_bf16(out, ref, lse, ref_lse)


def test_bf16_workload_L2048(lib):
    x = pi.workload_inputs(pi.BF16_L2048, device="cuda")
    out, lse = run_fwd(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    check_bf16(out, ref, lse, ref_lse)


@pytest.mark.parametrize("L", [64, 200, 640])
def test_fox_bf16_full(lib, L):
    x = pi.make_fwd_inputs(2, 2, L, seed=300 + L, fox=True, device="cuda")
    out, lse = run_fwd(lib, x, fox=True)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    check_bf16(out, ref, lse, ref_lse)


def test_beta_extremes_bf16(lib):
    # beta = 0 everywhere is plain causal attention; beta near 2 is the reflection regime
    for lo, hi in ((0.0, 0.0), (1.98, 1.99)):
        x = pi.make_fwd_inputs(1, 2, 333, seed=7, device="cuda")
        x["beta"] = torch.empty_like(x["beta"]).uniform_(lo, hi) if hi > 0 else \
            torch.zeros_like(x["beta"])
        out, lse = run_fwd(lib, x)
        ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
        check_bf16(out, ref, lse, ref_lse)


def test_zero_directions_are_plain_attention(lib):
    # w = 0 makes every transition the identity whatever beta is: plain causal softmax
    # attention, which the oracle computes with beta = 0
    for dtype in (torch.float32, torch.bfloat16):
        x = pi.make_fwd_inputs(2, 2, 300, dtype=dtype, seed=71, device="cuda")
        x["w"] = torch.zeros_like(x["w"])
        out, lse = run_fwd(lib, x)
        ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"],
                                       torch.zeros_like(x["beta"]))
        if dtype == torch.float32:
            rel = np.abs(out.double().cpu().numpy() - ref).max() / np.abs(ref).max()
            assert rel <= F32_MAX_REL, rel
        else:
            check_bf16(out, ref, lse, ref_lse)


def test_exact_reflections_fp32(lib):
    # beta = 2: every transition is a Householder reflection (orthogonal)
    x = pi.make_fwd_inputs(1, 2, 257, dtype=torch.float32, seed=72, clip=0.0, device="cuda")
    x["beta"] = torch.full_like(x["beta"], 2.0)
    out, lse = run_fwd(lib, x)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    rel = np.abs(out.double().cpu().numpy() - ref).max() / np.abs(ref).max()
    assert rel <= F32_MAX_REL, rel
    assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-4


def test_maximum_head_count(lib):
    # B * H at the accepted maximum (65535 heads, the grid's y limit): spot-check heads
    B, H, L = 65535, 1, 64
    x = pi.make_fwd_inputs(B, H, L, seed=73, device="cuda")
    out, lse = run_fwd(lib, x)
    torch.cuda.synchronize()
    heads = [0, 1, 32767, 65533, 65534]
    sel = {k: v[heads].cpu() for k, v in x.items()}
    ref, ref_lse = oracle.path_fwd(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"])
    check_bf16(out[heads], ref, lse[heads], ref_lse)
    assert torch.isfinite(out).all()


def test_very_long_sequence_sampled(lib):
    # one head of 2^18 tokens (4096 key blocks), sampled rows including both ends
    x = pi.make_fwd_inputs(1, 1, 1 << 18, seed=74, device="cuda")
    out, lse = run_fwd(lib, x)
    torch.cuda.synchronize()
    rows = np.array([[0, 0], [0, 1], [0, 63], [0, 64], [0, 131071], [0, 131072],
                     [0, (1 << 18) - 2], [0, (1 << 18) - 1], [0, 200000], [0, 77777]])
    h = {k: v.reshape(1, *v.shape[2:]).cpu() for k, v in x.items()}
    ref, ref_lse = oracle.path_rows(h["q"], h["k"], h["v"], h["w"], h["beta"], rows)
    got = out.reshape(1 << 18, 64)[torch.as_tensor(rows[:, 1], device="cuda")]
    got_lse = lse.reshape(1 << 18)[torch.as_tensor(rows[:, 1], device="cuda")]
    check_bf16(got, ref)
    assert np.abs(got_lse.double().cpu().numpy() - ref_lse).max() <= BF16_MAX_ABS


def test_custom_scale(lib):
    x = pi.make_fwd_inputs(1, 2, 150, seed=9, device="cuda")
    out, lse = run_fwd(lib, x, scale=0.3)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], scale=0.3)
    check_bf16(out, ref, lse, ref_lse)


def test_prepare_then_scan_equals_fused(lib):
    x = pi.make_fwd_inputs(2, 2, 300, seed=11, device="cuda")
    out, lse = run_fwd(lib, x)
    ws = lib.new_workspace(lib.OP_FWD, 2, 2, 300, lib.BF16, "cuda")
    lib.path_fwd_prepare(x["q"], x["k"], x["w"], x["beta"], ws)
    out2, lse2 = lib.path_fwd_scan(x["v"], ws)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)


def test_deterministic(lib):
    x = pi.make_fwd_inputs(2, 4, 700, seed=12, device="cuda")
    a, _ = run_fwd(lib, x)
    b, _ = run_fwd(lib, x)
    assert torch.equal(a, b)


def test_empty_problem_is_a_no_op(lib):
    z = torch.empty((1, 2, 0, 64), dtype=torch.bfloat16, device="cuda")
    beta = torch.empty((1, 2, 0), dtype=torch.float32, device="cuda")
    out, lse = lib.path_attn_fwd(z, z, z, z, beta)
    assert out.shape == (1, 2, 0, 64)


# ---------------------------------------------------------------- preprocessing factors

def _align256(x):
    return (x + 255) // 256 * 256


def _block_reference(q, k, w, beta, log_f, t0, L, scale):
    """fp64 boundary-adjusted rows, dense block transition and diagonal logits (log2
    units) of the 64-token block starting at t0, by explicit Householder products."""
    d = q.shape[1]
    H = [np.eye(d) - beta[t] * np.outer(w[t], w[t]) if t < L else np.eye(d)
         for t in range(t0, t0 + 64)]
    qt = np.zeros((64, d)); kt = np.zeros((64, d)); D = np.full((64, 64), -np.inf)
    P = np.eye(d)
    for m in H:
        P = P @ m
    for i in range(64):
        if t0 + i >= L:
            continue
        x = q[t0 + i].copy()
        for s in range(i, -1, -1):      # (H_0 ... H_i) q_i: H_i first
            x = H[s] @ x
        qt[i] = x
        y = k[t0 + i].copy()
        for s in range(i + 1, 64):      # H_63 ... H_{i+1} k_i: H_{i+1} first
            y = H[s] @ y
        kt[i] = y
    for i in range(64):
        if t0 + i >= L:
            continue
        x = q[t0 + i].copy()
        bias = 0.0
        for j in range(i, -1, -1):
            D[i, j] = scale * (k[t0 + j] @ x) * 1.4426950408889634
            if log_f is not None:
                D[i, j] += bias * 1.4426950408889634
                bias += log_f[t0 + j]
            x = H[j] @ x
    return qt, kt, P, D


@pytest.mark.parametrize("L,fox", [(64, False), (200, False), (130, True)])
def test_prepare_factors_match_explicit_products(lib, L, fox):
    B, H = 1, 2
    x = pi.make_fwd_inputs(B, H, L, seed=50 + L, fox=fox, device="cuda")
    ws = lib.new_workspace(lib.OP_FOX_FWD if fox else lib.OP_FWD, B, H, L, lib.BF16, "cuda")
    ws.zero_()
    lib.path_fwd_prepare(x["q"], x["k"], x["w"], x["beta"], ws, log_f=x.get("log_f"))
    torch.cuda.synchronize()
    nb = (L + 63) // 64
    nblk = nb + (nb & 1)
    Lp = nblk * 64
    BH = B * H
    off_qt = 256
    off_kp = _align256(off_qt + BH * Lp * 64 * 2)
    off_dg = _align256(off_kp + BH * nblk * 128 * 64 * 2)
    qt = ws[off_qt:off_qt + BH * Lp * 64 * 2].view(torch.bfloat16).reshape(BH, Lp, 64)
    kp = ws[off_kp:off_kp + BH * nblk * 128 * 64 * 2].view(torch.bfloat16).reshape(
        BH, nblk, 128, 64)
    dg = ws[off_dg:off_dg + BH * nblk * 64 * 64 * 2].view(torch.float16).reshape(
        BH, nblk, 64, 64)
    off_pr = _align256(off_dg + BH * nblk * 64 * 64 * 2)
    if not fox:
        pr = ws[off_pr:off_pr + BH * (nblk // 2) * 128 * 64 * 2].view(torch.bfloat16).reshape(
            BH, nblk // 2, 128, 64)
    h = {k_: v.reshape(BH, L, *v.shape[3:]).double().cpu().numpy() for k_, v in x.items()}
    for bh in range(BH):
        refs = [_block_reference(h["q"][bh], h["k"][bh], h["w"][bh], h["beta"][bh],
                                 h["log_f"][bh] if fox else None, 64 * b, L, 0.125)
                for b in range(nb)]
        # block-pair products for the two-block scan steps (plain PaTH only): K^ = K~_{2u}
        # P_{2u+1}, Pi = P_{2u} P_{2u+1} (a block past the end is the identity transition)
        for u in range(nblk // 2 if not fox else 0):
            k_lo, p_lo = refs[2 * u][1], refs[2 * u][2]
            p_hi = refs[2 * u + 1][2] if 2 * u + 1 < nb else np.eye(64)
            n = min(64, L - 128 * u)
            g_kh = pr[bh, u, :64].double().cpu().numpy()
            g_pi = pr[bh, u, 64:].double().cpu().numpy()
            assert np.abs(g_kh[:n] - (k_lo @ p_hi)[:n]).max() <= 3e-2
            assert np.abs(g_pi - p_lo @ p_hi).max() <= 1.5e-2
        for b in range(nb):
            rq, rk, rP, rD = refs[b]
            n = min(64, L - 64 * b)
            gq = qt[bh, 64 * b:64 * b + n].double().cpu().numpy()
            gk = kp[bh, b, :n].double().cpu().numpy()
            gP = kp[bh, b, 64:].double().cpu().numpy()
            gD = dg[bh, b, :n].double().cpu().numpy()
            assert np.abs(gq - rq[:n]).max() <= 2e-2
            assert np.abs(gk - rk[:n]).max() <= 2e-2
            assert np.abs(gP - rP).max() <= 1e-2
            fin = np.isfinite(rD[:n])
            assert np.array_equal(fin, np.isfinite(gD))
            assert np.abs(gD[fin] - rD[:n][fin]).max() <= 2e-2


# ---------------------------------------------------------------- full-size workloads, sampled rows

def _sampled_parity(lib, wl, n_heads=12, n_rows=600, seed=0):
    x = pi.workload_inputs(wl, device="cuda")
    out, lse = run_fwd(lib, x, fox=wl.fox)
    torch.cuda.synchronize()
    B, H, L = wl.B, wl.H, wl.L
    g = torch.Generator().manual_seed(seed)
    heads = torch.randperm(B * H, generator=g)[:n_heads]
    sel = {k: v.reshape(B * H, *v.shape[2:])[heads.to(v.device)].cpu() for k, v in x.items()}
    rows = pi.sample_rows(n_heads, L, n_rows, seed=seed)
    ref, ref_lse = oracle.path_rows(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"], rows,
                                    log_f=sel.get("log_f"))
    flat = out.reshape(B * H, L, 64)
    flat_lse = lse.reshape(B * H, L)
    hsel = heads[rows[:, 0]].to(out.device)
    ridx = torch.as_tensor(rows[:, 1], device=out.device)
    got = flat[hsel, ridx].double().cpu().numpy()
    got_lse = flat_lse[hsel, ridx].double().cpu().numpy()
    check_bf16(got, ref)
    assert np.abs(got_lse - ref_lse).max() <= BF16_MAX_ABS
    assert torch.isfinite(out).all()


def test_speed_workload_sampled(lib):
    _sampled_parity(lib, pi.BF16_L4096)


@pytest.mark.parametrize("L", [L for L in pi.SPEED_SWEEP_L if L != 4096])
def test_speed_shape_sweep_sampled(lib, L):
    # the B32 H32 speed shape at the other sequence lengths of the throughput curve, in the
    # launch configuration the sweep times; 300 sampled rows on 8 heads (heads are
    # independent, so the sample is exact for them)
    _sampled_parity(lib, pi.speed_shape(L), n_heads=8, n_rows=300, seed=L)


def test_fox_long_workload_sampled(lib):
    _sampled_parity(lib, pi.FOX_L16384, n_heads=8, n_rows=300)


# ---------------------------------------------------------------- FoX early exit

def _fox_with_extents(lib, x, scale=None):
    """Prepare + scan through the two-stage ABI; returns (extents, out, lse)."""
    B, H, L, _ = x["q"].shape
    code = lib.BF16 if x["q"].dtype == torch.bfloat16 else lib.F32
    ws = lib.new_workspace(lib.OP_FOX_FWD, B, H, L, code, "cuda")
    lib.path_fwd_prepare(x["q"], x["k"], x["w"], x["beta"], ws, log_f=x["log_f"], scale=scale)
    first = lib.path_fox_first_blocks(ws, B, H, L, x["q"].dtype)
    out, lse = lib.path_fwd_scan(x["v"], ws, fox=True, scale=scale)
    return first.cpu().numpy(), out, lse


def _check_extents_safe(x, first, scale=None):
    """Every key a query block skips weighs below e^-40 relative to its row's largest
    logit, by the oracle's fp64 logits; returns the fraction of key blocks skipped."""
    B, H, L, _ = x["q"].shape
    skipped = total = 0
    for b in range(B):
        for h in range(H):
            lg = oracle.path_logits(x["q"][b, h].cpu(), x["k"][b, h].cpu(), x["w"][b, h].cpu(),
                                    x["beta"][b, h].cpu(), x["log_f"][b, h].cpu(), scale)
            m = lg.max(axis=1)
            for qb in range(first.shape[2]):
                f = int(first[b, h, qb])
                assert 0 <= f <= qb
                skipped += f
                total += qb
                if f:
                    rows = slice(64 * qb, min(64 * qb + 64, L))
                    assert (lg[rows, :64 * f] < m[rows, None] - 40.0).all()
    return skipped / max(total, 1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_fox_early_exit_strong_gate(lib, dtype):
    # log f ~ logsigmoid(N(-1, 1)): about -80 nats per 64-token block, so every tile
    # stops within a block or two of its own; the output must still match the oracle's
    # full sum
    x = pi.make_fwd_inputs(1, 2, 1000, dtype=dtype, seed=41, clip=0.0 if dtype == torch.float32
                           else pi.BETA_CLIP, fox=True, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(141)
    x["log_f"] = torch.nn.functional.logsigmoid(
        torch.randn(x["log_f"].shape, generator=g) - 1.0).to("cuda").contiguous()
    first, out, lse = _fox_with_extents(lib, x)
    frac = _check_extents_safe(x, first)
    assert frac > 0.8, frac
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    if dtype == torch.float32:
        rel = np.abs(out.double().cpu().numpy() - ref).max() / np.abs(ref).max()
        assert rel <= F32_MAX_REL, rel
        assert np.abs(lse.double().cpu().numpy() - ref_lse).max() <= 1e-4
    else:
        check_bf16(out, ref, lse, ref_lse)


@pytest.mark.parametrize("L", [384, 1000])
def test_fox_own_block_only_gate(lib, L):
    # log f = -200 per token: a key one token back weighs e^-200 of the query's own key, far
    # below the bound's slack, so every query block's extent is its own block; the PaTH-FoX
    # scan then has tile pairs
    # whose second tile stops at its own lower block (the operand position no MMA reads is
    # skipped) and, at L = 384 (three tiles), a last item with one tile only
    x = pi.make_fwd_inputs(2, 2, L, seed=44, fox=True, device="cuda")
    x["log_f"] = torch.full_like(x["log_f"], -200.0)
    first, out, lse = _fox_with_extents(lib, x)
    nq = (L + 63) // 64
    assert np.array_equal(first, np.broadcast_to(np.arange(nq), (2, 2, nq)))
    _check_extents_safe(x, first)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    check_bf16(out, ref, lse, ref_lse)


def test_fox_early_exit_workload_gate(lib):
    # the FoX workload's gate, logsigmoid(N(2, 1)): the exit is active from a few blocks on
    x = pi.make_fwd_inputs(1, 2, 2048, seed=42, fox=True, device="cuda")
    first, out, lse = _fox_with_extents(lib, x)
    frac = _check_extents_safe(x, first)
    assert frac > 0.3, frac
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    check_bf16(out, ref, lse, ref_lse)


def test_fox_early_exit_mixed_sign_gate(lib):
    # log f of both signs: the prefix sums are not monotone; the bound uses prefix minima
    x = pi.make_fwd_inputs(2, 2, 640, seed=43, fox=True, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(143)
    x["log_f"] = (0.5 * torch.randn(x["log_f"].shape, generator=g) - 0.3).to("cuda").contiguous()
    first, out, lse = _fox_with_extents(lib, x, scale=0.2)
    _check_extents_safe(x, first, scale=0.2)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"],
                                   scale=0.2)
    check_bf16(out, ref, lse, ref_lse)


def test_fox_long_gate_sums_fp32(lib):
    # 8192 tokens at log f ~ -1.3: the gate prefix sums reach about -10^4; the bias
    # c_i - c_j must still be accurate to its own size (fp32 pairs), so that fp32 outputs
    # and LSE stay within 1e-4 of the oracle
    x = pi.make_fwd_inputs(1, 1, 8192, dtype=torch.float32, seed=45, clip=0.0, fox=True,
                           device="cuda")
    g = torch.Generator(device="cpu").manual_seed(145)
    x["log_f"] = torch.nn.functional.logsigmoid(
        torch.randn(x["log_f"].shape, generator=g) - 1.0).to("cuda").contiguous()
    out, lse = run_fwd(lib, x, fox=True)
    rows = np.arange(0, 8192, 61)
    pairs = np.stack([np.zeros_like(rows), rows], axis=1)   # (head, query) pairs
    h = {k: v[0].cpu() for k, v in x.items()}                # (H = 1, L, ...)
    ref, ref_lse = oracle.path_rows(h["q"], h["k"], h["v"], h["w"], h["beta"], pairs, h["log_f"])
    got = out[0, 0].double().cpu().numpy()[rows]
    assert np.abs(got - ref).max() / np.abs(ref).max() <= F32_MAX_REL
    assert np.abs(lse[0, 0].double().cpu().numpy()[rows] - ref_lse).max() <= 1e-4


@pytest.mark.parametrize("dtype,first", [(torch.bfloat16, 256), (torch.float32, 192)])
def test_fox_early_exit_never_reads_skipped_values(lib, dtype, first):
    # log f = -5 per token and the values of blocks 0 and 1 set to NaN: a query block whose
    # scan visited them would turn NaN (0 x NaN). Rows from block 3 on (fp32 scan, one query
    # block per CTA) or block 4 on (tensor-core scan: 128-row tiles of two query blocks)
    # stay finite, so the scan stopped above those blocks, and they match the oracle on the
    # clean values (the skipped weights are below e^-40)
    L = 640
    x = pi.make_fwd_inputs(1, 2, L, dtype=dtype, seed=53, clip=0.0 if dtype == torch.float32
                           else pi.BETA_CLIP, fox=True, device="cuda")
    x["log_f"] = torch.full_like(x["log_f"], -5.0)
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    x["v"][:, :, :128] = float("nan")
    out, lse = run_fwd(lib, x, fox=True)
    got = out[:, :, first:]
    assert torch.isfinite(got).all()
    if dtype == torch.bfloat16:
        check_bf16(got, ref[:, :, first:], lse[:, :, first:], ref_lse[:, :, first:])
    else:
        r = ref[:, :, first:]
        assert np.abs(got.double().cpu().numpy() - r).max() / np.abs(r).max() <= F32_MAX_REL
        assert np.abs(lse[:, :, first:].double().cpu().numpy() - ref_lse[:, :, first:]).max() <= 1e-4


def test_fox_zero_gate_has_no_exit(lib):
    # log f = 0: no bias, nothing can be skipped, and FoX equals PaTH (up to rounding:
    # the FoX scan applies the scale in another order than the PaTH scan)
    x = pi.make_fwd_inputs(1, 2, 700, seed=44, fox=True, device="cuda")
    x["log_f"] = torch.zeros_like(x["log_f"])
    first, out, lse = _fox_with_extents(lib, x)
    assert (first == 0).all()
    ref, ref_lse = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    check_bf16(out, ref, lse, ref_lse)


# ---------------------------------------------------------------- decode

def _decode_run(lib, B, H, n0, steps, dtype, seed, check_heads=None, d=64):
    wl = pi.DecodeWorkload("t", B, H, n0, steps, d, dtype, seed, 1000 + seed)
    cap = n0 + steps
    kc, vc = pi.make_decode_prefix(wl, cap, device="cuda")
    heads = list(range(B * H)) if check_heads is None else check_heads
    hk = kc.reshape(B * H, cap, d)[heads, :n0].cpu()
    hv = vc.reshape(B * H, cap, d)[heads, :n0].cpu()
    ocache = oracle.DecodeCache(hk, hv, cap)
    ws = lib.new_workspace(lib.OP_DECODE, B, H, cap, lib.BF16 if dtype == torch.bfloat16 else lib.F32,
                           "cuda", d)
    worst = 0.0
    for t in range(steps):
        s = pi.make_decode_step(wl, t, device="cuda")
        pre = kc.reshape(B * H, cap, d)[heads[:2], :n0 + t].double().cpu().numpy()
        o = lib.path_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], kc, vc, n0 + t,
                                 workspace=ws)
        sel = {k: v.reshape(B * H, -1)[heads].cpu() for k, v in s.items()}
        ref = ocache.step(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"])
        got = o.reshape(B * H, d)[heads].double().cpu().numpy()
        worst = max(worst, np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))
        if dtype == torch.bfloat16:
            assert np.abs(got - ref).max() <= BF16_MAX_ABS
        # the updated keys equal H_t applied to the pre-step keys, rounded once
        post = kc.reshape(B * H, cap, d)[heads[:2], :n0 + t + 1].double().cpu().numpy()
        w = sel["w"][:2].double().numpy()
        b = sel["beta"][:2].double().numpy().reshape(2, 1)
        expect = pre - b[:, :, None] * np.einsum("hjc,hc->hj", pre, w)[:, :, None] * w[:, None, :]
        expect = torch.from_numpy(expect).to(dtype).double().numpy()
        # fp32 arithmetic then one rounding: within 2 ulps of the fp64 result rounded once
        ulp = np.abs(expect) * (2.0 ** -6 if dtype == torch.bfloat16 else 2.0 ** -21)
        assert np.all(np.abs(post[:, :n0 + t] - expect) <= ulp + 1e-5)
        assert np.array_equal(post[:, n0 + t], sel["k"][:2].double().numpy())
    return worst


def test_decode_small_fp32(lib):
    worst = _decode_run(lib, 2, 3, 200, 12, torch.float32, seed=1)
    assert worst <= F32_MAX_REL


def test_decode_small_bf16_from_empty_and_ragged(lib):
    # empty prefix, then lengths crossing the split boundary (1024 keys per split)
    _decode_run(lib, 1, 2, 0, 5, torch.bfloat16, seed=2)
    worst = _decode_run(lib, 2, 2, 1020, 8, torch.bfloat16, seed=3)
    assert worst <= 5e-2


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_head_dim_128(lib, dtype):
    # head size 128: 16 lanes per bf16 key row (32 per fp32 row); empty prefix, then lengths
    # crossing a split boundary
    _decode_run(lib, 1, 2, 0, 3, dtype, seed=31, d=128)
    worst = _decode_run(lib, 2, 2, 1021, 5, dtype, seed=32, d=128)
    assert worst <= (F32_MAX_REL if dtype == torch.float32 else 5e-2)


def test_decode_workload_sampled_heads(lib):
    # 16 heads spread over the batch, compared with the oracle at every one of the 64 steps
    wl = pi.DECODE_32K
    cap = wl.n_prefix + wl.steps
    kc, vc = pi.make_decode_prefix(wl, cap, device="cuda")
    nh = wl.B * wl.H
    heads = sorted({0, nh - 1} | {int(h) for h in np.linspace(37, nh - 2, 14)})
    assert len(heads) == 16
    ocache = oracle.DecodeCache(kc.reshape(nh, cap, 64)[heads, :wl.n_prefix].cpu(),
                                vc.reshape(nh, cap, 64)[heads, :wl.n_prefix].cpu(), cap)
    ws = lib.new_workspace(lib.OP_DECODE, wl.B, wl.H, cap, lib.BF16, "cuda")
    rel = []
    for t in range(wl.steps):
        s = pi.make_decode_step(wl, t, device="cuda")
        o = lib.path_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], kc, vc,
                                 wl.n_prefix + t, workspace=ws)
        sel = {k: v.reshape(nh, -1)[heads].cpu() for k, v in s.items()}
        ref = ocache.step(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"])
        got = o.reshape(nh, 64)[heads].double().cpu().numpy()
        assert np.abs(got - ref).max() <= BF16_MAX_ABS, t
        rel.append(np.abs(got - ref).max() / np.abs(ref).max())
    assert max(rel) <= 5e-2, rel


# ---------------------------------------------------------------- PaTH-FoX decode

def _fox_decode_run(lib, B, H, n0, steps, dtype, seed, check_heads=None, d=64):
    wl = pi.DecodeWorkload("t", B, H, n0, steps, d, dtype, seed, 1000 + seed)
    cap = n0 + steps
    kc, vc, gc = pi.make_fox_decode_prefix(wl, cap, device="cuda")
    heads = list(range(B * H)) if check_heads is None else check_heads
    ocache = oracle.DecodeCache(kc.reshape(B * H, cap, d)[heads, :n0].cpu(),
                                vc.reshape(B * H, cap, d)[heads, :n0].cpu(), cap, fox=True,
                                g_prefix=gc.reshape(B * H, cap)[heads, :n0].cpu())
    ws = lib.new_workspace(lib.OP_FOX_DECODE, B, H, cap,
                           lib.BF16 if dtype == torch.bfloat16 else lib.F32, "cuda", d)
    worst = 0.0
    for t in range(steps):
        s = pi.make_decode_step(wl, t, device="cuda", fox=True)
        pre_g = gc.reshape(B * H, cap)[heads, :n0 + t].double().cpu().numpy()
        o = lib.path_fox_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], s["log_f"],
                                     kc, vc, gc, n0 + t, workspace=ws)
        sel = {k: v.reshape(B * H, -1)[heads].cpu() for k, v in s.items()}
        ref = ocache.step(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"],
                          log_f=sel["log_f"])
        got = o.reshape(B * H, d)[heads].double().cpu().numpy()
        worst = max(worst, np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-30))
        if dtype == torch.bfloat16:
            assert np.abs(got - ref).max() <= BF16_MAX_ABS
        # gate sums: one fp32 addition of log f_t to the stored value, and 0 appended
        post_g = gc.reshape(B * H, cap)[heads, :n0 + t + 1].double().cpu().numpy()
        lf = sel["log_f"].double().numpy().reshape(-1, 1)
        expect = (pre_g + lf).astype(np.float32).astype(np.float64)
        assert np.all(np.abs(post_g[:, :n0 + t] - expect) <= np.abs(expect) * 2.0 ** -23 + 1e-30)
        assert np.all(post_g[:, n0 + t] == 0)
        # and they stay within fp32 rounding of the oracle's fp64 sums
        assert np.allclose(post_g, ocache.cbias[:, :n0 + t + 1], rtol=1e-5, atol=1e-5)
    return worst


def test_fox_decode_small_fp32(lib):
    worst = _fox_decode_run(lib, 2, 3, 200, 12, torch.float32, seed=11)
    assert worst <= F32_MAX_REL


def test_fox_decode_bf16_from_empty_and_across_splits(lib):
    _fox_decode_run(lib, 1, 2, 0, 5, torch.bfloat16, seed=12)
    worst = _fox_decode_run(lib, 2, 2, 1021, 6, torch.bfloat16, seed=13)
    assert worst <= 5e-2


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_fox_decode_head_dim_128(lib, dtype):
    worst = _fox_decode_run(lib, 2, 2, 1500, 4, dtype, seed=33, d=128)
    assert worst <= (F32_MAX_REL if dtype == torch.float32 else 5e-2)


def test_fox_decode_zero_gate_equals_path_decode(lib):
    # log f = 0 leaves every gate sum at 0 and adds nothing to a logit: the PaTH step, with
    # the same keys bit for bit (the softmax partial sums run in another order, so the
    # outputs agree to rounding)
    wl = pi.DecodeWorkload("t", 2, 2, 1500, 3, 64, torch.bfloat16, 14, 1014)
    cap = wl.n_prefix + wl.steps
    kc, vc = pi.make_decode_prefix(wl, cap, device="cuda")
    kf, vf = kc.clone(), vc.clone()
    gc = torch.zeros((2, 2, cap), dtype=torch.float32, device="cuda")
    for t in range(wl.steps):
        s = pi.make_decode_step(wl, t, device="cuda")
        zero = torch.zeros_like(s["beta"])
        a = lib.path_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], kc, vc,
                                 wl.n_prefix + t)
        b = lib.path_fox_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], zero, kf, vf,
                                     gc, wl.n_prefix + t)
        assert (a.float() - b.float()).abs().max().item() <= 2.0 ** -7 * a.float().abs().max().item()
    assert torch.equal(kc, kf) and torch.equal(vc, vf)
    assert torch.count_nonzero(gc) == 0


@pytest.mark.parametrize("kind", ["strong", "mixed_sign"])
def test_fox_decode_vanishing_keys(lib, kind):
    # strong gates: all but the last few dozen keys weigh below 2^-64 and skip their value
    # rows; mixed-sign gates (log f ~ N(0, 2), so older keys can gain weight): the skip rule
    # still holds because the new key's own logit bounds the row maximum from below
    B, H, n0, steps = 1, 3, 3000, 4
    wl = pi.DecodeWorkload("t", B, H, n0, steps, 64, torch.bfloat16, 15, 1015)
    cap = n0 + steps
    kc, vc, gc = pi.make_fox_decode_prefix(wl, cap, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(99)
    if kind == "strong":
        gc[:, :, :n0] *= 20.0
        lf_scale, lf_shift = 1.0, -3.0
    else:
        gc[:, :, :n0] = torch.cumsum(2.0 * torch.randn((B, H, n0), generator=g, device="cuda"), -1)
        gc[:, :, :n0] -= gc[:, :, n0 - 1:n0].clone()
        lf_scale, lf_shift = 2.0, 0.0
    ocache = oracle.DecodeCache(kc[:, :, :n0].cpu(), vc[:, :, :n0].cpu(), cap, fox=True,
                                g_prefix=gc[:, :, :n0].cpu())
    for t in range(steps):
        s = pi.make_decode_step(wl, t, device="cuda", fox=True)
        s["log_f"] = (lf_scale * torch.randn((B, H, 1), generator=g, device="cuda") + lf_shift)
        o = lib.path_fox_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"],
                                     s["log_f"].contiguous(), kc, vc, gc, n0 + t)
        ref = ocache.step(s["q"].cpu(), s["k"].cpu(), s["v"].cpu(), s["w"].cpu(),
                          s["beta"].cpu(), log_f=s["log_f"].cpu())
        check_bf16(o.reshape(B * H, 64), ref)


def test_fox_decode_workload_sampled_heads(lib):
    wl = pi.FOX_DECODE_32K
    cap = wl.n_prefix + wl.steps
    kc, vc, gc = pi.make_fox_decode_prefix(wl, cap, device="cuda")
    heads = [0, 301, 1023]
    nh = wl.B * wl.H
    ocache = oracle.DecodeCache(kc.reshape(nh, cap, 64)[heads, :wl.n_prefix].cpu(),
                                vc.reshape(nh, cap, 64)[heads, :wl.n_prefix].cpu(), cap,
                                fox=True, g_prefix=gc.reshape(nh, cap)[heads, :wl.n_prefix].cpu())
    ws = lib.new_workspace(lib.OP_FOX_DECODE, wl.B, wl.H, cap, lib.BF16, "cuda")
    for t in range(wl.steps):
        s = pi.make_decode_step(wl, t, device="cuda", fox=True)
        o = lib.path_fox_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], s["log_f"],
                                     kc, vc, gc, wl.n_prefix + t, workspace=ws)
        sel = {k: v.reshape(nh, -1)[heads].cpu() for k, v in s.items()}
        ref = ocache.step(sel["q"], sel["k"], sel["v"], sel["w"], sel["beta"],
                          log_f=sel["log_f"])
        if t % 8 == 7 or t == 0:
            got = o.reshape(nh, 64)[heads].double().cpu().numpy()
            assert np.abs(got - ref).max() <= BF16_MAX_ABS


def test_decode_capacity_error(lib):
    kc = torch.zeros((1, 1, 4, 64), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    s = pi.make_fwd_inputs(1, 1, 1, seed=0, device="cuda")
    with pytest.raises(lib.PathError) as e:
        lib.path_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], kc, vc, 4)
    assert e.value.code == lib.ERR_CAPACITY
    assert torch.count_nonzero(kc) == 0


# ---------------------------------------------------------------- bounded waits

@pytest.mark.parametrize("fox", [False, True])
def test_forced_timeout_reports_status_and_context_survives(lib, monkeypatch, fox):
    # PaTH-FoX: 40 heads x 4 tile pairs = 160 items, more than one per CTA of the persistent
    # scan, so the abort has to stop CTAs in the middle of their item loops
    B, H, L = (1, 40, 1024) if fox else (1, 1, 256)
    x = pi.make_fwd_inputs(B, H, L, seed=5, fox=fox, device="cuda")
    ws = lib.new_workspace(lib.OP_FOX_FWD if fox else lib.OP_FWD, B, H, L, lib.BF16, "cuda")

    def fwd():
        if fox:
            return lib.path_fox_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"],
                                    workspace=ws)
        return lib.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], workspace=ws)

    monkeypatch.setenv("PATH_ATTN_DEBUG_FORCE_TIMEOUT", "1")
    fwd()
    assert lib.path_check_workspace(ws) == lib.ERR_TIMEOUT
    monkeypatch.delenv("PATH_ATTN_DEBUG_FORCE_TIMEOUT")
    out, _ = fwd()
    assert lib.path_check_workspace(ws) == lib.OK
    ref, _ = oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x.get("log_f"))
    check_bf16(out, ref)
