"""Pins of the fp64 oracle against facts the pages and the mathematics fix.

Definition pinned (review "거리에서 경로로, PaTH Attention" §3-§4, §9; technical summary
"技術要約: PaTH Attention" §2-§3): logit(i, j) = sigma * k_j^T (H_{j+1} ... H_i) q_i
[+ sum_{s=j+1..i} log f_s], H_s = I - beta_s w_s w_s^T, causal softmax, weighted sum of V;
decode applies the new H_t to every cached key in place.

Each pin is independent of the oracle's code: a hand-worked example, textbook attention
at beta = 0, explicit d x d matrix products, closed forms and invariants. Every pin has
to fail for at least one plausible mistake; test_oracle_mutants.py plants such mistakes
in copies of the oracle and checks that these pins catch each of them.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- helpers (test side)

def rand_head(rng, L, d, beta_range=(0.0, 2.0)):
    q, k, v, g = (rng.standard_normal((L, d)) for _ in range(4))
    w = g / np.linalg.norm(g, axis=1, keepdims=True)
    beta = rng.uniform(*beta_range, size=L)
    return q, k, v, w, beta


def naive_attention(q, k, v, scale, bias=None):
    """Textbook causal softmax attention; bias[i, j] is added to the scaled logit."""
    L = q.shape[0]
    s = scale * (q @ k.T)
    if bias is not None:
        s = s + bias
    s = np.where(np.tril(np.ones((L, L), bool)), s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


def householder(w, beta):
    return np.eye(w.shape[0]) - beta * np.outer(w, w)


def brute_logits(q, k, w, beta, scale, log_f=None):
    """Explicit d x d products: P = H_{j+1} @ ... @ H_i, logit = scale k_j^T P q_i."""
    L, d = q.shape
    Hs = [householder(w[s], beta[s]) for s in range(L)]
    out = np.full((L, L), -np.inf)
    for i in range(L):
        for j in range(i + 1):
            P = np.eye(d)
            for s in range(j + 1, i + 1):
                P = P @ Hs[s]
            out[i, j] = scale * k[j] @ P @ q[i]
            if log_f is not None:
                out[i, j] += sum(log_f[j + 1:i + 1])
    return out


def softmax_rows(logits, v):
    m = logits.max(axis=1, keepdims=True)
    p = np.exp(logits - m)
    p /= p.sum(axis=1, keepdims=True)
    return p @ v


def cumsum_bias(log_f):
    c = np.cumsum(log_f)
    return c[:, None] - c[None, :]


# ----------------------------------------------------------------- golden hand example

def load_hand():
    L_, O_, F_ = {}, {}, {}
    with open(os.path.join(GOLDEN, "hand_2d.txt")) as f:
        for line in f:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] == "L":
                L_[(int(t[1]), int(t[2]))] = float(t[3])
            elif t[0] == "O":
                O_[int(t[1])] = (float(t[2]), float(t[3]))
            elif t[0] == "F":
                F_[(int(t[1]), int(t[2]))] = float(t[3])
    r2 = 1.0 / math.sqrt(2.0)
    w = np.array([[1, 0], [1, 0], [r2, r2]], float)
    beta = np.ones(3)
    q = np.array([[1, 1], [0, 1], [1, 0]], float)
    k = np.array([[0, 1], [1, 1], [2, 0]], float)
    v = np.array([[1, 0], [0, 1], [0, 0]], float)
    return (q, k, v, w, beta), L_, O_, F_


def test_hand_example_logits_outputs_and_fox():
    (q, k, v, w, beta), L_, O_, F_ = load_hand()
    lg = oracle.path_logits(q, k, w, beta, scale=1.0)
    for (i, j), val in L_.items():
        assert lg[i, j] == pytest.approx(val, abs=1e-14)
    out, _ = oracle.path_fwd(q, k, v, w, beta, scale=1.0)
    for i, val in O_.items():
        np.testing.assert_allclose(out[i], val, atol=1e-14)
    log_f = np.array([0.0, -1.0, -2.0])
    lf = oracle.path_logits(q, k, w, beta, log_f=log_f, scale=1.0)
    for (i, j), val in F_.items():
        assert lf[i, j] == pytest.approx(val, abs=1e-14)


# ----------------------------------------------------------------- special cases

@pytest.mark.parametrize("L,d", [(1, 4), (37, 8), (130, 64), (70, 128)])
def test_beta_zero_is_causal_softmax_attention(L, d):
    rng = np.random.default_rng(L)
    q, k, v, w, _ = rand_head(rng, L, d)
    beta = np.zeros(L)
    out, lse = oracle.path_fwd(q, k, v, w, beta)
    ref = naive_attention(q, k, v, 1 / math.sqrt(d))
    np.testing.assert_allclose(out, ref, atol=1e-12, rtol=0)
    # log-sum-exp of the scaled logits, written out
    s = (q @ k.T) / math.sqrt(d)
    for i in (0, L // 2, L - 1):
        m = s[i, :i + 1].max()
        assert lse[i] == pytest.approx(m + math.log(np.exp(s[i, :i + 1] - m).sum()), abs=1e-12)


def test_diagonal_logit_is_plain_dot_product():
    rng = np.random.default_rng(3)
    q, k, v, w, beta = rand_head(rng, 40, 16)
    lg = oracle.path_logits(q, k, w, beta)
    np.testing.assert_allclose(np.diag(lg), (q * k).sum(1) / 4.0, atol=1e-13, rtol=0)
    assert np.all(np.isneginf(lg[np.triu_indices(40, 1)]))


@pytest.mark.parametrize("L,d", [(2, 3), (9, 8), (16, 64), (10, 128)])
def test_brute_force_explicit_matrices(L, d):
    rng = np.random.default_rng(100 + L)
    q, k, v, w, beta = rand_head(rng, L, d)
    log_f = np.log(rng.uniform(0.2, 1.0, size=L))
    scale = 1 / math.sqrt(d)
    for lf in (None, log_f):
        ref = brute_logits(q, k, w, beta, scale, lf)
        got = oracle.path_logits(q, k, w, beta, log_f=lf)
        np.testing.assert_allclose(got, ref, atol=1e-12, rtol=0)
        out, _ = oracle.path_fwd(q, k, v, w, beta, log_f=lf)
        np.testing.assert_allclose(out, softmax_rows(ref, v), atol=1e-12, rtol=0)


def test_repeated_transition_closed_form():
    # (I - beta w w^T)^n = I - (1 - (1 - beta)^n) w w^T for unit w
    rng = np.random.default_rng(5)
    L, d, b = 50, 16, 1.7
    q, k, v, _, _ = rand_head(rng, L, d)
    g = rng.standard_normal(d)
    w1 = g / np.linalg.norm(g)
    w = np.tile(w1, (L, 1))
    beta = np.full(L, b)
    lg = oracle.path_logits(q, k, w, beta, scale=1.0)
    for i in (0, 7, 49):
        for j in (0, i // 2, i):
            n = i - j
            P = np.eye(d) - (1 - (1 - b) ** n) * np.outer(w1, w1)
            assert lg[i, j] == pytest.approx(k[j] @ P @ q[i], abs=1e-12)


def test_reflections_preserve_norm_and_general_beta_contracts():
    rng = np.random.default_rng(7)
    L, d = 200, 64
    q, _, _, w, _ = rand_head(rng, L, d)
    two = np.full(L, 2.0)
    for (i, j) in [(199, 0), (150, 40), (10, 9)]:
        x = oracle.path_transport(q[i], w, two, i, j)
        assert np.linalg.norm(x) == pytest.approx(np.linalg.norm(q[i]), rel=1e-12)
    beta = rng.uniform(0, 2, size=L)
    for (i, j) in [(199, 0), (120, 100)]:
        x = oracle.path_transport(q[i], w, beta, i, j)
        assert np.linalg.norm(x) <= np.linalg.norm(q[i]) * (1 + 1e-12)
    # the transport equals the explicit product H_{j+1} ... H_i q
    P = np.eye(d)
    for s in range(101, 121):
        P = P @ householder(w[s], beta[s])
    np.testing.assert_allclose(oracle.path_transport(q[120], w, beta, 120, 100), P @ q[120],
                               atol=1e-12, rtol=0)


def test_order_of_transitions_matters():
    rng = np.random.default_rng(11)
    L, d = 12, 8
    q, k, v, w, beta = rand_head(rng, L, d, (0.3, 1.9))
    base = oracle.path_logits(q, k, w, beta)
    w2, b2 = w.copy(), beta.copy()
    w2[[3, 5]] = w2[[5, 3]]
    b2[[3, 5]] = b2[[5, 3]]
    swapped = oracle.path_logits(q, k, w2, b2)
    # pairs whose path crosses both tokens 3 and 5 see a different product
    diff = np.abs(base[5:, :3] - swapped[5:, :3])
    assert diff.min() > 1e-6
    # pairs whose path avoids both tokens are unchanged
    np.testing.assert_allclose(base[2, :3], swapped[2, :3], atol=1e-14)
    np.testing.assert_allclose(base[11, 6:12], swapped[11, 6:12], atol=1e-14)


# ----------------------------------------------------------------- UT form used by the kernels

def ut_factor(W, beta):
    """A = (I + D N)^{-1} D with N = strictly-upper(W W^T) (compact WY / UT form)."""
    C = W.shape[0]
    N = np.triu(W @ W.T, 1)
    return np.linalg.solve(np.eye(C) + np.diag(beta) @ N, np.diag(beta))


def test_ut_identity_and_bounds():
    # H_first ... H_last = I - W^T A W (technical summary §3, UT transform)
    rng = np.random.default_rng(13)
    for C, d in [(2, 5), (16, 64), (64, 64)]:
        _, _, _, W, beta = rand_head(rng, C, d)
        P = np.eye(d)
        for s in range(C):
            P = P @ householder(W[s], beta[s])
        A = ut_factor(W, beta)
        np.testing.assert_allclose(np.eye(d) - W.T @ A @ W, P, atol=1e-12, rtol=0)
        # A_ss = beta_s, |A_su| <= beta_s beta_u above the diagonal (each entry is
        # -beta_s beta_u w_s^T H_{s+1} ... H_{u-1} w_u), and A is upper triangular
        np.testing.assert_allclose(np.diag(A), beta, atol=1e-14)
        assert np.all(np.abs(np.triu(A, 1)) <= np.outer(beta, beta) + 1e-12)
        assert np.all(np.tril(A, -1) == 0)
        # the leading block inverts the leading product
        t = C // 2
        Pt = np.eye(d)
        for s in range(t):
            Pt = Pt @ householder(W[s], beta[s])
        np.testing.assert_allclose(np.eye(d) - W[:t].T @ A[:t, :t] @ W[:t], Pt, atol=1e-12)


# ----------------------------------------------------------------- PaTH-FoX

def test_fox_reductions():
    rng = np.random.default_rng(17)
    L, d = 90, 16
    q, k, v, w, beta = rand_head(rng, L, d)
    plain, _ = oracle.path_fwd(q, k, v, w, beta)
    zero_gate, _ = oracle.path_fwd(q, k, v, w, beta, log_f=np.zeros(L))
    np.testing.assert_allclose(zero_gate, plain, atol=1e-14, rtol=0)
    log_f = np.log(rng.uniform(0.05, 1.0, size=L))
    fox_only, _ = oracle.path_fwd(q, k, v, w, np.zeros(L), log_f=log_f)
    ref = naive_attention(q, k, v, 1 / math.sqrt(d), bias=cumsum_bias(log_f))
    np.testing.assert_allclose(fox_only, ref, atol=1e-12, rtol=0)


# ----------------------------------------------------------------- decode

@pytest.mark.parametrize("fox", [False, True])
def test_decode_from_empty_cache_matches_prefill(fox):
    _decode_from_empty_matches_prefill(fox, 16)


@pytest.mark.parametrize("fox", [False, True])
def test_decode_from_empty_cache_matches_prefill_head_128(fox):
    _decode_from_empty_matches_prefill(fox, 128)


def _decode_from_empty_matches_prefill(fox, d):
    rng = np.random.default_rng(19)
    nh, T = 3, 40
    q, k, v, g = (rng.standard_normal((nh, T, d)) for _ in range(4))
    w = g / np.linalg.norm(g, axis=-1, keepdims=True)
    beta = rng.uniform(0, 2, size=(nh, T))
    log_f = np.log(rng.uniform(0.1, 1.0, size=(nh, T))) if fox else None
    ref, _ = oracle.path_fwd(q, k, v, w, beta, log_f=log_f)
    cache = oracle.DecodeCache(np.zeros((nh, 0, d)), np.zeros((nh, 0, d)), cap=T, fox=fox)
    for t in range(T):
        o = cache.step(q[:, t], k[:, t], v[:, t], w[:, t], beta[:, t],
                       log_f=None if log_f is None else log_f[:, t])
        np.testing.assert_allclose(o, ref[:, t], atol=1e-12, rtol=0)
    # the cache holds the keys transported to the last position: H_{T-1} ... H_{j+1} k_j
    j = 5
    P = np.eye(d)
    for s in range(j + 1, T):
        P = P @ householder(w[1, s], beta[1, s])
    np.testing.assert_allclose(cache.Kc[1, j], P.T @ k[1, j], atol=1e-12)


def test_fox_decode_from_prefill_state_matches_prefill():
    # A PaTH-FoX cache built from a prefix of n0 tokens holds the keys transported to the
    # prefix's last position and, per key j, the gate sum over positions j+1 .. n0-1.
    # Built here from explicit d x d products and plain sums, then stepped by the oracle,
    # it must give the prefill rows n0 .. T-1.
    rng = np.random.default_rng(29)
    nh, T, n0, d = 2, 30, 17, 8
    q, k, v, g = (rng.standard_normal((nh, T, d)) for _ in range(4))
    w = g / np.linalg.norm(g, axis=-1, keepdims=True)
    beta = rng.uniform(0, 2, size=(nh, T))
    log_f = np.log(rng.uniform(0.2, 1.0, size=(nh, T)))
    ref, _ = oracle.path_fwd(q, k, v, w, beta, log_f=log_f)
    kp = np.empty((nh, n0, d))
    gp = np.empty((nh, n0))
    for h in range(nh):
        for j in range(n0):
            P = np.eye(d)
            for s in range(j + 1, n0):
                P = P @ householder(w[h, s], beta[h, s])
            kp[h, j] = P.T @ k[h, j]
            gp[h, j] = sum(log_f[h, s] for s in range(j + 1, n0))
    cache = oracle.DecodeCache(kp, v[:, :n0], cap=T, fox=True, g_prefix=gp)
    for t in range(n0, T):
        o = cache.step(q[:, t], k[:, t], v[:, t], w[:, t], beta[:, t], log_f=log_f[:, t])
        np.testing.assert_allclose(o, ref[:, t], atol=1e-12, rtol=0)


def test_sampled_rows_match_full_forward():
    rng = np.random.default_rng(23)
    B, H, L, d = 2, 3, 70, 8
    q, k, v, g = (rng.standard_normal((B, H, L, d)) for _ in range(4))
    w = g / np.linalg.norm(g, axis=-1, keepdims=True)
    beta = rng.uniform(0, 2, size=(B, H, L))
    out, lse = oracle.path_fwd(q, k, v, w, beta)
    rows = np.array([[0, 0], [5, 69], [3, 33], [1, 64]])
    ro, rl = oracle.path_rows(q, k, v, w, beta, rows)
    flat, flat_lse = out.reshape(-1, L, d), lse.reshape(-1, L)
    for n, (h, i) in enumerate(rows):
        np.testing.assert_array_equal(ro[n], flat[h, i])
        assert rl[n] == flat_lse[h, i]
