"""fp64 CPU oracle for PaTH attention.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. It shares no code with
the CUDA path in ``dependent_position_encoded_gb300``.

Each function computes the method's definition directly (see path_oracle.c):
the logit of query i and key j is
``scale * k_j^T (H_{j+1} ... H_i) q_i [+ sum_{s=j+1..i} log f_s]`` with
``H_s = I - beta_s w_s w_s^T``, followed by a causal softmax and the weighted
sum of V (review "거리에서 경로로, PaTH Attention" §3-§4; technical summary
"技術要約: PaTH Attention" §2). Inputs are upcast to float64 exactly as given:
callers pass the rounded tensors that the GPU sees, and w is not renormalised.

Parity pins: every function here is pinned by tests/test_oracle_pins.py
against closed forms, textbook special cases, brute force with explicit
d x d matrices and a hand-worked example (tests/golden/).
"""
import ctypes
import math

import numpy as np

from . import build as _build

_lib = None


def _configure(lib):
    """Declares the C signatures on a loaded oracle library."""
    dp = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_path_fwd.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_double, dp, dp, ctypes.c_int]
    lib.oracle_path_fwd.restype = ctypes.c_int
    lib.oracle_path_rows.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_double, i64p, ctypes.c_int64,
                                     dp, dp, ctypes.c_int]
    lib.oracle_path_rows.restype = ctypes.c_int
    lib.oracle_path_logits.argtypes = [dp, dp, dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_double, dp]
    lib.oracle_path_logits.restype = None
    lib.oracle_path_transport.argtypes = [dp, dp, dp, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, dp]
    lib.oracle_path_transport.restype = None
    lib.oracle_path_decode_step.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, dp,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_double, dp]
    lib.oracle_path_decode_step.restype = None
    lib.oracle_wbeta_produce.argtypes = [dp, dp, dp, dp, dp, dp, ctypes.c_double] + \
        [ctypes.c_int] * 6 + [ctypes.c_double, dp, dp]
    lib.oracle_wbeta_produce.restype = None
    lib.oracle_path_bwd.argtypes = [dp] * 7 + [ctypes.c_int] * 3 + [ctypes.c_double] + \
        [dp] * 6 + [ctypes.c_int]
    lib.oracle_path_bwd.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(_build.build()))
    return _lib


def swap_library(path):
    """Makes this module call the oracle library at ``path``; returns the previous
    library object (or None). Used by the mutation tests, which load copies of
    the oracle with planted mistakes."""
    global _lib
    prev = _lib
    _lib = None if path is None else _configure(ctypes.CDLL(path))
    return prev


def restore_library(prev):
    global _lib
    _lib = prev


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor -> numpy, exact upcast
        x = x.detach().to("cpu")
        x = x.double().numpy() if x.is_floating_point() else x.numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _heads(x, L, d):
    """Flattens (..., L, d) to (nh, L, d)."""
    return x.reshape(-1, L, d)


def path_fwd(q, k, v, w, beta, log_f=None, scale=None, nthreads=0):
    """Full PaTH (log_f None) or PaTH-FoX forward.

    q, k, v, w: (..., L, d); beta, log_f: (..., L). Returns (out, lse) as
    float64 arrays of shapes (..., L, d) and (..., L).
    """
    q, k, v, w, beta, log_f = map(_f64, (q, k, v, w, beta, log_f))
    lead, L, d = q.shape[:-2], q.shape[-2], q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qh, kh, vh, wh = (np.ascontiguousarray(_heads(t, L, d)) for t in (q, k, v, w))
    nh = qh.shape[0]
    bh = np.ascontiguousarray(beta.reshape(nh, L))
    fh = None if log_f is None else np.ascontiguousarray(log_f.reshape(nh, L))
    out = np.empty((nh, L, d))
    lse = np.empty((nh, L))
    _load().oracle_path_fwd(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(wh), _ptr(bh), _ptr(fh),
                            nh, L, d, float(scale), _ptr(out), _ptr(lse), int(nthreads))
    return out.reshape(*lead, L, d), lse.reshape(*lead, L)


def path_rows(q, k, v, w, beta, rows, log_f=None, scale=None, nthreads=0):
    """Forward for sampled rows only.

    rows: int array of shape (n, 2) holding (flattened head index, query index).
    Returns (out (n, d), lse (n,)).
    """
    q, k, v, w, beta, log_f = map(_f64, (q, k, v, w, beta, log_f))
    L, d = q.shape[-2], q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qh, kh, vh, wh = (np.ascontiguousarray(_heads(t, L, d)) for t in (q, k, v, w))
    nh = qh.shape[0]
    bh = np.ascontiguousarray(beta.reshape(nh, L))
    fh = None if log_f is None else np.ascontiguousarray(log_f.reshape(nh, L))
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    if rows.size and (rows[:, 0].min() < 0 or rows[:, 0].max() >= nh
                      or rows[:, 1].min() < 0 or rows[:, 1].max() >= L):
        raise ValueError("row index out of range")
    n = rows.shape[0]
    out = np.empty((n, d))
    lse = np.empty((n,))
    _load().oracle_path_rows(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(wh), _ptr(bh), _ptr(fh),
                             nh, L, d, float(scale),
                             rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
                             _ptr(out), _ptr(lse), int(nthreads))
    return out, lse


def path_logits(q, k, w, beta, log_f=None, scale=None):
    """(L, L) logit matrix of one head; -inf above the diagonal."""
    q, k, w, beta, log_f = map(_f64, (q, k, w, beta, log_f))
    L, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = np.empty((L, L))
    _load().oracle_path_logits(_ptr(q), _ptr(k), _ptr(w), _ptr(beta), _ptr(log_f),
                               L, d, float(scale), _ptr(out))
    return out


def path_transport(q, w, beta, i, j):
    """x = H_{j+1} ... H_i q for one head (w: (L, d), beta: (L,))."""
    q, w, beta = map(_f64, (q, w, beta))
    d = q.shape[-1]
    x = np.empty(d)
    _load().oracle_path_transport(_ptr(q), _ptr(w), _ptr(beta), int(i), int(j), d, _ptr(x))
    return x


class DecodeCache:
    """fp64 key/value cache for the decode oracle (heads are independent).

    Kc, Vc: (nh, cap, d) float64; length: number of valid entries.
    """

    def __init__(self, k_prefix, v_prefix, cap, fox=False, g_prefix=None):
        """g_prefix (nh or (..., n0)): for a PaTH-FoX cache, the per-key gate sums of the
        prefix keys (sum of log f over positions j+1 .. n0-1); zeros when omitted."""
        k_prefix, v_prefix = _f64(k_prefix), _f64(v_prefix)
        nh = int(np.prod(k_prefix.shape[:-2]))
        n0, d = k_prefix.shape[-2], k_prefix.shape[-1]
        self.nh, self.cap, self.d, self.length = nh, int(cap), d, n0
        self.Kc = np.zeros((nh, cap, d))
        self.Vc = np.zeros((nh, cap, d))
        self.Kc[:, :n0] = k_prefix.reshape(nh, n0, d)
        self.Vc[:, :n0] = v_prefix.reshape(nh, n0, d)
        self.cbias = np.zeros((nh, cap)) if fox else None
        if g_prefix is not None:
            if not fox:
                raise ValueError("g_prefix needs fox=True")
            self.cbias[:, :n0] = _f64(g_prefix).reshape(nh, n0)

    def step(self, q, k, v, w, beta, log_f=None, scale=None):
        """Applies one decode step in place; returns o_t of shape (nh, d)."""
        if self.length + 1 > self.cap:
            raise ValueError("cache full")
        q, k, v, w, beta, log_f = map(_f64, (q, k, v, w, beta, log_f))
        nh, d = self.nh, self.d
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        if (log_f is None) != (self.cbias is None):
            raise ValueError("log_f must be given exactly when the cache was built with fox=True")
        args = [np.ascontiguousarray(t.reshape(nh, d)) for t in (q, k, v, w)]
        b = np.ascontiguousarray(beta.reshape(nh))
        f = None if log_f is None else np.ascontiguousarray(log_f.reshape(nh))
        out = np.empty((nh, d))
        _load().oracle_path_decode_step(*(_ptr(a) for a in args), _ptr(b), _ptr(f),
                                        _ptr(self.Kc), _ptr(self.Vc), _ptr(self.cbias),
                                        nh, self.length, self.cap, d, float(scale), _ptr(out))
        self.length += 1
        return out


def wbeta_produce(x, w_down, w_up, conv, u, bias, beta_max=2.0, eps=1e-12):
    """The w/beta producer (see path_oracle.c): x (B, L, D), w_down (R, D), w_up (H*d, R),
    conv (H*d, 3), u (H, D), bias (H,). Returns (w (B, H, L, d), beta (B, H, L)) float64;
    d is w_up's rows divided by u's rows."""
    x, w_down, w_up, conv, u, bias = map(_f64, (x, w_down, w_up, conv, u, bias))
    B, L, D = x.shape
    R = w_down.shape[0]
    H = u.shape[0]
    d = w_up.shape[0] // H
    if w_down.shape != (R, D) or w_up.shape != (H * d, R) or conv.shape != (H * d, 3) \
            or u.shape != (H, D) or bias.shape != (H,):
        raise ValueError("inconsistent producer shapes")
    w = np.empty((B, H, L, d))
    beta = np.empty((B, H, L))
    _load().oracle_wbeta_produce(_ptr(x), _ptr(w_down), _ptr(w_up), _ptr(conv), _ptr(u),
                                 _ptr(bias), float(beta_max), B, L, D, R, H, d, float(eps),
                                 _ptr(w), _ptr(beta))
    return w, beta


def path_bwd(q, k, v, w, beta, dout, log_f=None, scale=None, nthreads=0):
    """Gradients of the PaTH (log_f None) or PaTH-FoX forward for the loss
    sum(dout * out), by reverse mode through the definition's per-row sweep
    (path_oracle.c, oracle_path_bwd).

    Returns a dict of float64 arrays: dq, dk, dv, dw (..., L, d), dbeta (..., L) and,
    with log_f, dlog_f (..., L).
    """
    q, k, v, w, beta, log_f, dout = map(_f64, (q, k, v, w, beta, log_f, dout))
    lead, L, d = q.shape[:-2], q.shape[-2], q.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    qh, kh, vh, wh, dh = (np.ascontiguousarray(_heads(t, L, d)) for t in (q, k, v, w, dout))
    nh = qh.shape[0]
    bh = np.ascontiguousarray(beta.reshape(nh, L))
    fh = None if log_f is None else np.ascontiguousarray(log_f.reshape(nh, L))
    g = {n: np.empty((nh, L, d)) for n in ("dq", "dk", "dv", "dw")}
    g["dbeta"] = np.empty((nh, L))
    if fh is not None:
        g["dlog_f"] = np.empty((nh, L))
    _load().oracle_path_bwd(_ptr(qh), _ptr(kh), _ptr(vh), _ptr(wh), _ptr(bh), _ptr(fh),
                            _ptr(dh), nh, L, d, float(scale), _ptr(g["dq"]), _ptr(g["dk"]),
                            _ptr(g["dv"]), _ptr(g["dw"]), _ptr(g["dbeta"]),
                            _ptr(g.get("dlog_f")), int(nthreads))
    out = {}
    for n, a in g.items():
        out[n] = a.reshape(*lead, L, d) if a.ndim == 3 else a.reshape(*lead, L)
    return out
