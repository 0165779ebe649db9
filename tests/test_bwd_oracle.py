"""Pins of the oracle's backward pass (CPU only).

The pages give no backward, so the oracle's gradients are the chain rule applied to the
definition (path_oracle.c, oracle_path_bwd). They are pinned here to facts that do not
come from that derivation:
- central finite differences of the forward oracle's loss sum(dout * out), for every input
  entry, plain and PaTH-FoX;
- beta = 0, where PaTH is ordinary causal softmax attention: dq, dk, dv in closed matrix
  form, dw = 0, and dbeta_s = -scale * sum_{j < s <= i} dS_ij (w_s . k_j)(w_s . q_i), the
  first-order change of the logits when H_s leaves the identity;
- w -> -w leaves every H_s unchanged, so every gradient but dw is unchanged and dw flips;
- dv = P^T dout with P the softmax of the forward oracle's own logit matrix.
"""
import math

import numpy as np
import pytest

import oracle


def rand_case(rng, L, d, nh=1):
    q, k, v, dout = (rng.standard_normal((nh, L, d)) for _ in range(4))
    w = rng.standard_normal((nh, L, d))
    w /= np.linalg.norm(w, axis=-1, keepdims=True)
    beta = 2.0 / (1.0 + np.exp(-rng.standard_normal((nh, L))))
    log_f = -np.log1p(np.exp(-(2.0 + rng.standard_normal((nh, L)))))
    return q, k, v, w, beta, log_f, dout


def loss(q, k, v, w, beta, log_f, dout):
    out, _ = oracle.path_fwd(q, k, v, w, beta, log_f=log_f)
    return float((out * dout).sum())


@pytest.mark.parametrize("fox", [False, True])
def test_bwd_matches_finite_differences(fox):
    rng = np.random.default_rng(11 + fox)
    q, k, v, w, beta, log_f, dout = rand_case(rng, 7, 5)
    if not fox:
        log_f = None
    g = oracle.path_bwd(q, k, v, w, beta, dout, log_f=log_f)
    args = {"q": q, "k": k, "v": v, "w": w, "beta": beta, "log_f": log_f}
    names = [("dq", "q"), ("dk", "k"), ("dv", "v"), ("dw", "w"), ("dbeta", "beta")]
    if fox:
        names.append(("dlog_f", "log_f"))
    h = 1e-6
    for gname, aname in names:
        base = args[aname]
        fd = np.zeros_like(base)
        for idx in np.ndindex(base.shape):
            hi, lo = base.copy(), base.copy()
            hi[idx] += h
            lo[idx] -= h
            fd[idx] = (loss(**{**args, aname: hi}, dout=dout) -
                       loss(**{**args, aname: lo}, dout=dout)) / (2 * h)
        err = np.abs(fd - g[gname]).max() / np.abs(fd).max()
        assert err < 1e-6, "%s: relative error %g against finite differences" % (gname, err)


@pytest.mark.parametrize("fox", [False, True])
def test_bwd_head_size_128_matches_finite_differences_sampled(fox):
    # the head size of the second model width: nothing in the derivation or the oracle's
    # loops depends on d, so a few sampled entries per gradient suffice
    rng = np.random.default_rng(21 + fox)
    q, k, v, w, beta, log_f, dout = rand_case(rng, 5, 128)
    if not fox:
        log_f = None
    g = oracle.path_bwd(q, k, v, w, beta, dout, log_f=log_f)
    args = {"q": q, "k": k, "v": v, "w": w, "beta": beta, "log_f": log_f}
    names = [("dq", "q"), ("dk", "k"), ("dv", "v"), ("dw", "w"), ("dbeta", "beta")]
    if fox:
        names.append(("dlog_f", "log_f"))
    h = 1e-6
    for gname, aname in names:
        base = args[aname]
        flat = rng.choice(base.size, size=min(24, base.size), replace=False)
        for f in flat:
            idx = np.unravel_index(f, base.shape)
            hi, lo = base.copy(), base.copy()
            hi[idx] += h
            lo[idx] -= h
            fd = (loss(**{**args, aname: hi}, dout=dout) -
                  loss(**{**args, aname: lo}, dout=dout)) / (2 * h)
            scale = max(np.abs(g[gname]).max(), 1e-3)
            assert abs(fd - g[gname][idx]) <= 1e-6 * scale, (gname, idx, fd, g[gname][idx])


def test_bwd_beta_zero_closed_form():
    rng = np.random.default_rng(5)
    L, d = 23, 8
    q, k, v, w, _, _, dout = rand_case(rng, L, d)
    beta = np.zeros((1, L))
    g = oracle.path_bwd(q, k, v, w, beta, dout)
    Q, K, V, Wm, dO = q[0], k[0], v[0], w[0], dout[0]
    sc = 1.0 / math.sqrt(d)
    S = sc * Q @ K.T
    S[np.triu_indices(L, 1)] = -np.inf
    P = np.exp(S - S.max(1, keepdims=True))
    P /= P.sum(1, keepdims=True)
    dP = dO @ V.T
    dS = P * (dP - (P * dP).sum(1, keepdims=True))
    np.testing.assert_allclose(g["dv"][0], P.T @ dO, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["dq"][0], sc * dS @ K, rtol=0, atol=1e-12)
    np.testing.assert_allclose(g["dk"][0], sc * dS.T @ Q, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(g["dw"], 0.0)
    wq = Wm @ Q.T  # wq[s, i] = w_s . q_i
    wk = Wm @ K.T  # wk[s, j] = w_s . k_j
    ref = np.zeros(L)
    for s in range(L):
        for i in range(s, L):
            for j in range(s):
                ref[s] -= sc * dS[i, j] * wk[s, j] * wq[s, i]
    np.testing.assert_allclose(g["dbeta"][0], ref, rtol=0, atol=1e-12)


def test_bwd_sign_of_w():
    rng = np.random.default_rng(8)
    q, k, v, w, beta, log_f, dout = rand_case(rng, 19, 6, nh=2)
    a = oracle.path_bwd(q, k, v, w, beta, dout, log_f=log_f)
    b = oracle.path_bwd(q, k, v, -w, beta, dout, log_f=log_f)
    for n in ("dq", "dk", "dv", "dbeta", "dlog_f"):
        np.testing.assert_allclose(b[n], a[n], rtol=0, atol=1e-12)
    np.testing.assert_allclose(b["dw"], -a["dw"], rtol=0, atol=1e-12)


def test_bwd_dv_is_p_transpose_dout():
    rng = np.random.default_rng(9)
    L, d = 31, 8
    q, k, v, w, beta, log_f, dout = rand_case(rng, L, d)
    for lf in (None, log_f):
        g = oracle.path_bwd(q, k, v, w, beta, dout, log_f=lf)
        S = oracle.path_logits(q[0], k[0], w[0], beta[0], log_f=None if lf is None else lf[0])
        P = np.exp(S - S.max(1, keepdims=True))
        P /= P.sum(1, keepdims=True)
        np.testing.assert_allclose(g["dv"][0], P.T @ dout[0], rtol=0, atol=1e-12)
