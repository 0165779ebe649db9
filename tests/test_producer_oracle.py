"""Pins of the fp64 w / beta producer oracle against facts the pages and the mathematics fix.

Definition pinned (review "거리에서 경로로, PaTH Attention" §3: a low-dimensional linear
projection and a short convolution of size 3 give w, which is L2-normalised, and beta is
twice a sigmoid; technical summary "技術要約: PaTH Attention" §2: beta_s = 2 sigmoid(u^T x_s
+ b); §6: beta is clipped for bf16). Conventions: weights (out, in); conv taps (channel, 3)
with tap 2 on token t, tap 1 on t - 1, tap 0 on t - 2, zero before the first token;
w = y / max(|y|, eps) per head of d channels.

Each pin is independent of the oracle's code: a hand-worked example, a closed form, the
reach of the convolution in time, a shift property, invariances and limits of beta.
test_oracle_mutants.py plants mistakes in the oracle and checks that these pins catch them.
"""
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_producer(rng, B=2, L=12, D=16, R=4, H=3, d=8):
    x = rng.standard_normal((B, L, D))
    w_down = rng.standard_normal((R, D)) / math.sqrt(D)
    w_up = rng.standard_normal((H * d, R)) / math.sqrt(R)
    conv = rng.standard_normal((H * d, 3))
    u = rng.standard_normal((H, D)) / math.sqrt(D)
    b = rng.standard_normal(H)
    return x, w_down, w_up, conv, u, b


def test_hand_example():
    vals = {}
    with open(os.path.join(GOLDEN, "producer_hand.txt")) as f:
        for line in f:
            if line.startswith("#") or ":" not in line:
                continue
            k, v = line.split(":", 1)
            vals[k.strip()] = np.array([float(t) for t in v.split()])
    x = vals["x"].reshape(1, 3, 2)
    w, beta = oracle.wbeta_produce(x, vals["w_down"].reshape(1, 2), vals["w_up"].reshape(2, 1),
                                   vals["conv"].reshape(2, 3), vals["u"].reshape(1, 2),
                                   vals["bias"], beta_max=float(vals["beta_max"][0]))
    np.testing.assert_allclose(w.reshape(-1), vals["w"], atol=1e-15, rtol=0)
    np.testing.assert_allclose(beta.reshape(-1), vals["beta"], atol=1e-15, rtol=0)


def test_rank_one_equal_taps_closed_form():
    # R = 1 and the same taps (a0, a1, a2) on every channel: y'_t = s_t * w_up[:, 0] with
    # s_t = a2 z_t + a1 z_{t-1} + a0 z_{t-2}, so w_t = sign(s_t) * w_up_h / |w_up_h| per head
    rng = np.random.default_rng(3)
    B, L, D, H, d = 1, 9, 5, 2, 4
    x = rng.standard_normal((B, L, D))
    w_down = rng.standard_normal((1, D))
    w_up = rng.standard_normal((H * d, 1))
    a = np.array([0.3, -1.1, 0.7])
    conv = np.tile(a, (H * d, 1))
    w, _ = oracle.wbeta_produce(x, w_down, w_up, conv, np.zeros((H, D)), np.zeros(H))
    z = x[0] @ w_down[0]
    for t in range(L):
        s = a[2] * z[t] + (a[1] * z[t - 1] if t >= 1 else 0.0) + (a[0] * z[t - 2] if t >= 2 else 0.0)
        for h in range(H):
            col = w_up[h * d:(h + 1) * d, 0]
            np.testing.assert_allclose(w[0, h, t], np.sign(s) * col / np.linalg.norm(col),
                                       atol=1e-13, rtol=0)


def test_convolution_reaches_two_tokens_back_and_no_further():
    rng = np.random.default_rng(5)
    x, w_down, w_up, conv, u, b = rand_producer(rng)
    w0, b0 = oracle.wbeta_produce(x, w_down, w_up, conv, u, b)
    x2 = x.copy()
    x2[1, 5] += rng.standard_normal(x.shape[-1])
    w1, b1 = oracle.wbeta_produce(x2, w_down, w_up, conv, u, b)
    diff = np.abs(w1 - w0).max(axis=(1, 3))  # (B, L)
    assert np.all(diff[0] == 0)                      # other sequence untouched
    assert np.all(diff[1, :5] == 0)                  # causal
    assert np.all(diff[1, 5:8] > 1e-6)               # t, t + 1, t + 2 see x_t
    assert np.all(diff[1, 8:] == 0)                  # width 3: no further
    bd = np.abs(b1 - b0).max(axis=1)
    assert np.all(bd[1, [t for t in range(12) if t != 5]] == 0) and bd[1, 5] > 0


def test_lag_one_tap_shifts_the_output_by_one_token():
    rng = np.random.default_rng(7)
    x, w_down, w_up, _, u, b = rand_producer(rng)
    C = w_up.shape[0]
    now = np.tile([0.0, 0.0, 1.0], (C, 1))
    lag1 = np.tile([0.0, 1.0, 0.0], (C, 1))
    w_now, _ = oracle.wbeta_produce(x, w_down, w_up, now, u, b)
    w_lag, _ = oracle.wbeta_produce(x, w_down, w_up, lag1, u, b)
    np.testing.assert_allclose(w_lag[:, :, 1:], w_now[:, :, :-1], atol=1e-14, rtol=0)
    assert np.all(w_lag[:, :, 0] == 0)  # nothing before the first token: zero vector


def test_unit_norm_scale_invariance_and_heads_independent():
    rng = np.random.default_rng(9)
    x, w_down, w_up, conv, u, b = rand_producer(rng)
    w, _ = oracle.wbeta_produce(x, w_down, w_up, conv, u, b)
    np.testing.assert_allclose(np.linalg.norm(w, axis=-1), 1.0, atol=1e-14)
    w3, _ = oracle.wbeta_produce(x, w_down, 3.0 * w_up, conv, u, b)
    np.testing.assert_allclose(w3, w, atol=1e-14)
    wn, _ = oracle.wbeta_produce(x, w_down, -w_up, conv, u, b)
    np.testing.assert_allclose(wn, -w, atol=1e-14)
    d = w.shape[-1]
    w_up2 = w_up.copy()
    w_up2[d:2 * d] = rng.standard_normal(w_up2[d:2 * d].shape)  # only head 1's rows
    w2, _ = oracle.wbeta_produce(x, w_down, w_up2, conv, u, b)
    np.testing.assert_array_equal(w2[:, 0], w[:, 0])
    np.testing.assert_array_equal(w2[:, 2], w[:, 2])
    assert np.abs(w2[:, 1] - w[:, 1]).max() > 1e-3


def test_beta_limits():
    rng = np.random.default_rng(11)
    x, w_down, w_up, conv, u, b = rand_producer(rng)
    H, D = u.shape
    _, beta = oracle.wbeta_produce(x, w_down, w_up, conv, np.zeros((H, D)), np.zeros(H))
    np.testing.assert_array_equal(beta, 1.0)  # 2 sigmoid(0)
    _, beta = oracle.wbeta_produce(x, w_down, w_up, conv, u, b)
    assert np.all((beta > 0) & (beta < 2))
    big = np.full(H, 50.0)
    _, beta = oracle.wbeta_produce(x, w_down, w_up, conv, np.zeros((H, D)), big, beta_max=1.99)
    np.testing.assert_array_equal(beta, 1.99)
    # the logit is u_h . x_t + b_h: one head's u on one coordinate
    u1 = np.zeros((H, D))
    u1[1, 3] = 1.0
    _, beta = oracle.wbeta_produce(x, w_down, w_up, conv, u1, np.zeros(H))
    np.testing.assert_allclose(beta[:, 1], 2.0 / (1.0 + np.exp(-x[:, :, 3])), atol=1e-15)
