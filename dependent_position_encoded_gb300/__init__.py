"""GB300 (sm_103a) PaTH attention.

A thin Python binding over ``libpath_attn.so``, whose C ABI is declared in
``include/path_attn.h``. Every step of the computation runs in the library's
CUDA kernels; this module only checks tensor arguments, allocates outputs and
workspaces with PyTorch (device memory and streams are PyTorch's job here) and
passes raw pointers. There is no CPU fallback: without the built library or a
CUDA device every call raises.

Entry points keep the C names: ``path_attn_fwd``, ``path_fox_fwd``,
``path_fwd_prepare``, ``path_fwd_scan``, ``path_decode_step``, ``path_fox_decode_step``,
``path_wbeta_produce``,
``path_workspace_bytes``, ``path_check_workspace``, ``path_status_string``.
"""
import ctypes
import math
import os

from . import build as _build

# status codes and enums, mirroring include/path_attn.h
OK, ERR_NULL, ERR_SHAPE, ERR_DTYPE, ERR_ALIGN, ERR_WORKSPACE, ERR_CAPACITY, ERR_TIMEOUT, \
    ERR_CUDA, ERR_ARG = range(10)
F32, BF16 = 0, 1
OP_FWD, OP_FOX_FWD, OP_DECODE, OP_FOX_DECODE, OP_BWD, OP_FOX_BWD = 0, 1, 2, 3, 4, 5
HEAD_DIM = 64

EXPORTED = ("path_workspace_bytes", "path_attn_fwd", "path_fox_fwd", "path_fwd_prepare",
            "path_fwd_scan", "path_decode_step", "path_check_workspace", "path_status_string",
            "path_decode_step_noalloc", "path_fox_first_blocks", "path_fox_decode_step",
            "path_wbeta_workspace_bytes", "path_wbeta_produce", "path_attn_bwd",
            "path_fox_bwd")

_lib = None


class PathError(RuntimeError):
    def __init__(self, code, where):
        self.code = code
        super().__init__("%s: %s" % (where, path_status_string(code)))


def library_path():
    return _build.LIB


def ensure_built():
    """Builds libpath_attn.so if it is missing or older than its sources."""
    if not _build.up_to_date():
        _build.build()
    return _build.LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise RuntimeError("libpath_attn.so is not built; run dependent_position_encoded_gb300."
                           "build.build() (or __graft_entry__.build())")
    lib = ctypes.CDLL(_build.LIB)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.path_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.path_workspace_bytes.restype = S
    lib.path_attn_fwd.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F, P, S, P]
    lib.path_attn_fwd.restype = I
    lib.path_fox_fwd.argtypes = [P, P, P, P, P, P, P, P, I, I, I, I, I, F, P, S, P]
    lib.path_fox_fwd.restype = I
    lib.path_fwd_prepare.argtypes = [P, P, P, P, P, I, I, I, I, I, F, P, S, P]
    lib.path_fwd_prepare.restype = I
    lib.path_fwd_scan.argtypes = [P, P, P, I, I, I, I, I, I, F, P, S, P]
    lib.path_fwd_scan.restype = I
    lib.path_decode_step.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, S, P]
    lib.path_decode_step.restype = I
    lib.path_fox_decode_step.argtypes = [P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, P, S,
                                         P]
    lib.path_fox_decode_step.restype = I
    lib.path_wbeta_workspace_bytes.argtypes = [I, I, I, I, I, I, I]
    lib.path_wbeta_workspace_bytes.restype = S
    lib.path_wbeta_produce.argtypes = [P, P, P, P, P, P, F, P, P, I, I, I, I, I, I, I, P, S, P]
    lib.path_wbeta_produce.restype = I
    lib.path_attn_bwd.argtypes = [P] * 8 + [I] * 5 + [F] + [P] * 6 + [S, P]
    lib.path_attn_bwd.restype = I
    lib.path_fox_bwd.argtypes = [P] * 9 + [I] * 5 + [F] + [P] * 7 + [S, P]
    lib.path_fox_bwd.restype = I
    lib.path_decode_step_noalloc.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, F, P, P]
    lib.path_decode_step_noalloc.restype = I
    lib.path_fox_first_blocks.argtypes = [P, S, I, I, I, I, I, P, P]
    lib.path_fox_first_blocks.restype = I
    lib.path_check_workspace.argtypes = [P, P]
    lib.path_check_workspace.restype = I
    lib.path_status_string.argtypes = [I]
    lib.path_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def path_status_string(code):
    return _load().path_status_string(int(code)).decode()


def _check(code, where):
    if code != OK:
        raise PathError(code, where)


# ---------------------------------------------------------------- marshalling helpers

def _torch():
    import torch
    return torch


def _dtype_code_of(dtype):
    torch = _torch()
    if dtype == torch.bfloat16:
        return BF16
    if dtype == torch.float32:
        return F32
    raise TypeError("unsupported dtype %s (bfloat16 or float32)" % dtype)


def _dtype_code(t):
    return _dtype_code_of(t.dtype)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _cuda_tensor(t, name, dtype=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t


def _stream(stream, device):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _scale(scale, d):
    return 1.0 / math.sqrt(d) if scale is None else float(scale)


def path_workspace_bytes(op, B, H, L, d=HEAD_DIM, dtype=BF16):
    return int(_load().path_workspace_bytes(int(op), int(B), int(H), int(L), int(d), int(dtype)))


def new_workspace(op, B, H, L, dtype, device, d=HEAD_DIM):
    """A device workspace sized by path_workspace_bytes (256-byte aligned by PyTorch)."""
    torch = _torch()
    n = path_workspace_bytes(op, B, H, L, d, dtype)
    if n == 0:
        raise PathError(ERR_SHAPE, "path_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _fwd_args(q, k, v, w, beta):
    torch = _torch()
    _cuda_tensor(q, "q")
    dt = q.dtype
    for t, n in ((k, "k"), (v, "v"), (w, "w")):
        _cuda_tensor(t, n, dt)
        if t.shape != q.shape:
            raise ValueError("%s has shape %s, expected %s" % (n, tuple(t.shape), tuple(q.shape)))
    if q.dim() != 4:
        raise ValueError("q must be (B, H, L, d)")
    B, H, L, d = q.shape
    _cuda_tensor(beta, "beta", torch.float32)
    if beta.shape != (B, H, L):
        raise ValueError("beta must be (B, H, L) float32")
    return B, H, L, d, _dtype_code(q)


def _outputs(q, out, lse, B, H, L):
    torch = _torch()
    if out is None:
        out = torch.empty_like(q)
    else:
        _cuda_tensor(out, "out", q.dtype)
    if lse is True:
        lse = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
    elif lse is not None and lse is not False:
        _cuda_tensor(lse, "lse", torch.float32)
    else:
        lse = None
    return out, lse


def path_attn_fwd(q, k, v, w, beta, out=None, lse=True, scale=None, workspace=None, stream=None):
    """PaTH forward; returns (out, lse or None). lse=True allocates it, None skips it."""
    B, H, L, d, dt = _fwd_args(q, k, v, w, beta)
    out, lse = _outputs(q, out, lse, B, H, L)
    if workspace is None:
        workspace = new_workspace(OP_FWD, B, H, L, dt, q.device, d=d)
    _check(_load().path_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(out),
                                 _ptr(lse), B, H, L, d, dt, _scale(scale, d), _ptr(workspace),
                                 workspace.numel(), _stream(stream, q.device)), "path_attn_fwd")
    return out, lse


def _bwd_grads(q, grads, B, H, L, d, fox):
    torch = _torch()
    g = dict(grads or {})
    for n in ("dq", "dk", "dv", "dw"):
        if n not in g:
            g[n] = torch.empty((B, H, L, d), dtype=torch.float32, device=q.device)
        _cuda_tensor(g[n], n, torch.float32)
    names = ("dbeta", "dlog_f") if fox else ("dbeta",)
    for n in names:
        if n not in g:
            g[n] = torch.empty((B, H, L), dtype=torch.float32, device=q.device)
        _cuda_tensor(g[n], n, torch.float32)
    return g


def _bwd_checks(q, out, lse, d_out, B, H, L):
    torch = _torch()
    _cuda_tensor(out, "out", q.dtype)
    _cuda_tensor(d_out, "d_out", q.dtype)
    _cuda_tensor(lse, "lse", torch.float32)
    if out.shape != q.shape or d_out.shape != q.shape or lse.shape != (B, H, L):
        raise ValueError("out, d_out must be (B, H, L, d) and lse (B, H, L)")


def path_attn_bwd(q, k, v, w, beta, out, lse, d_out, scale=None, grads=None, workspace=None,
                  stream=None):
    """PaTH backward; returns a dict of fp32 gradients dq, dk, dv, dw (B, H, L, d) and
    dbeta (B, H, L). `out` and `lse` are the forward's outputs for the same inputs and scale;
    `grads` may hold preallocated fp32 buffers under those names."""
    B, H, L, d, dt = _fwd_args(q, k, v, w, beta)
    _bwd_checks(q, out, lse, d_out, B, H, L)
    g = _bwd_grads(q, grads, B, H, L, d, False)
    if workspace is None:
        workspace = new_workspace(OP_BWD, B, H, L, dt, q.device, d=d)
    _check(_load().path_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(out),
                                 _ptr(lse), _ptr(d_out), B, H, L, d, dt, _scale(scale, d),
                                 _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["dw"]),
                                 _ptr(g["dbeta"]), _ptr(workspace), workspace.numel(),
                                 _stream(stream, q.device)), "path_attn_bwd")
    return g


def path_fox_bwd(q, k, v, w, beta, log_f, out, lse, d_out, scale=None, grads=None,
                 workspace=None, stream=None):
    """PaTH-FoX backward; as path_attn_bwd plus dlog_f (B, H, L) fp32. `out` and `lse` are
    path_fox_fwd's outputs."""
    torch = _torch()
    B, H, L, d, dt = _fwd_args(q, k, v, w, beta)
    _cuda_tensor(log_f, "log_f", torch.float32)
    if log_f.shape != (B, H, L):
        raise ValueError("log_f must be (B, H, L) float32")
    _bwd_checks(q, out, lse, d_out, B, H, L)
    g = _bwd_grads(q, grads, B, H, L, d, True)
    if workspace is None:
        workspace = new_workspace(OP_FOX_BWD, B, H, L, dt, q.device, d=d)
    _check(_load().path_fox_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(log_f),
                                _ptr(out), _ptr(lse), _ptr(d_out), B, H, L, d, dt,
                                _scale(scale, d), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
                                _ptr(g["dw"]), _ptr(g["dbeta"]), _ptr(g["dlog_f"]),
                                _ptr(workspace), workspace.numel(), _stream(stream, q.device)),
           "path_fox_bwd")
    return g


def path_fox_fwd(q, k, v, w, beta, log_f, out=None, lse=True, scale=None, workspace=None,
                 stream=None):
    """PaTH-FoX forward; returns (out, lse or None)."""
    torch = _torch()
    B, H, L, d, dt = _fwd_args(q, k, v, w, beta)
    _cuda_tensor(log_f, "log_f", torch.float32)
    if log_f.shape != (B, H, L):
        raise ValueError("log_f must be (B, H, L) float32")
    out, lse = _outputs(q, out, lse, B, H, L)
    if workspace is None:
        workspace = new_workspace(OP_FOX_FWD, B, H, L, dt, q.device, d=d)
    _check(_load().path_fox_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(w), _ptr(beta), _ptr(log_f),
                                _ptr(out), _ptr(lse), B, H, L, d, dt, _scale(scale, d),
                                _ptr(workspace), workspace.numel(), _stream(stream, q.device)),
           "path_fox_fwd")
    return out, lse


def path_fwd_prepare(q, k, w, beta, workspace, log_f=None, scale=None, stream=None):
    """First stage (UT preprocessing) into `workspace`."""
    torch = _torch()
    B, H, L, d, dt = _fwd_args(q, k, q, w, beta)
    if log_f is not None:
        _cuda_tensor(log_f, "log_f", torch.float32)
    _check(_load().path_fwd_prepare(_ptr(q), _ptr(k), _ptr(w), _ptr(beta), _ptr(log_f), B, H, L,
                                    d, dt, _scale(scale, d), _ptr(workspace), workspace.numel(),
                                    _stream(stream, q.device)), "path_fwd_prepare")


def path_fwd_scan(v, workspace, out=None, lse=True, fox=False, scale=None, stream=None):
    """Second stage (block scan) from `workspace`; returns (out, lse or None)."""
    _cuda_tensor(v, "v")
    B, H, L, d = v.shape
    dt = _dtype_code(v)
    out, lse = _outputs(v, out, lse, B, H, L)
    _check(_load().path_fwd_scan(_ptr(v), _ptr(out), _ptr(lse), int(bool(fox)), B, H, L, d, dt,
                                 _scale(scale, d), _ptr(workspace), workspace.numel(),
                                 _stream(stream, v.device)), "path_fwd_scan")
    return out, lse


def path_fox_first_blocks(workspace, B, H, L, dtype, stream=None, d=HEAD_DIM):
    """PaTH-FoX early-exit extents left in `workspace` by path_fwd_prepare(..., log_f):
    an int32 tensor (B, H, ceil(L / 64)) of the lowest key block each query block needs.
    Head size 64 only: the head-size-128 scan decides its exit as it runs (d = 128 raises
    PathError with ERR_SHAPE)."""
    torch = _torch()
    nq = (L + 63) // 64
    first = torch.empty((B, H, nq), dtype=torch.int32, device=workspace.device)
    _check(_load().path_fox_first_blocks(_ptr(workspace), workspace.numel(), B, H, L, int(d),
                                         _dtype_code_of(dtype), _ptr(first),
                                         _stream(stream, workspace.device)),
           "path_fox_first_blocks")
    return first


def _decode_args(q, k, v, w, beta, k_cache, v_cache, out):
    """Checks the decode arguments and returns (inputs, out, (B, H, cap, d)). Shapes and
    dtypes are checked before devices, so every size error is raised before any call."""
    torch = _torch()
    named = [(k_cache, "k_cache"), (v_cache, "v_cache"), (q, "q"), (k, "k"), (v, "v"),
             (w, "w"), (beta, "beta")] + ([(out, "out")] if out is not None else [])
    for t, n in named:
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a tensor" % n)
    if k_cache.dim() != 4:
        raise ValueError("k_cache must have shape (B, H, cap, d)")
    dt_t = k_cache.dtype
    B, H, cap, d = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("v_cache must match k_cache")
    for t, n, dt, count in ((v_cache, "v_cache", dt_t, None), (q, "q", dt_t, B * H * d),
                            (k, "k", dt_t, B * H * d), (v, "v", dt_t, B * H * d),
                            (w, "w", dt_t, B * H * d), (beta, "beta", torch.float32, B * H),
                            (out, "out", dt_t, B * H * d)):
        if t is None:
            continue
        if t.dtype != dt:
            raise TypeError("%s must be %s, got %s" % (n, dt, t.dtype))
        if count is not None and t.numel() != count:
            raise ValueError("%s must hold %d values, got %d" % (n, count, t.numel()))
    for t, n in named:
        _cuda_tensor(t, n)
        if t.device != k_cache.device:
            raise ValueError("%s must be on %s" % (n, k_cache.device))
    if out is None:
        out = torch.empty((B, H, d), dtype=dt_t, device=k_cache.device)
    return [q, k, v, w], out, (B, H, cap, d)


def path_decode_step(q, k, v, w, beta, k_cache, v_cache, cache_len, scale=None, out=None,
                     workspace=None, stream=None):
    """One decode step: updates k_cache in place, appends (k, v) at cache_len and returns
    the attention output (B, H, d). q, k, v, w: (B, H, d) (a trailing length-1 axis is
    accepted); beta: (B, H); caches: (B, H, cap, d)."""
    ins, out, (B, H, cap, d) = _decode_args(q, k, v, w, beta, k_cache, v_cache, out)
    if workspace is None:
        workspace = new_workspace(OP_DECODE, B, H, cap, _dtype_code(k_cache), k_cache.device, d)
    _check(_load().path_decode_step(_ptr(ins[0]), _ptr(ins[1]), _ptr(ins[2]), _ptr(ins[3]),
                                    _ptr(beta), _ptr(k_cache), _ptr(v_cache), B, H,
                                    int(cache_len), cap, d, _dtype_code(k_cache),
                                    _scale(scale, d), _ptr(out), _ptr(workspace),
                                    workspace.numel(), _stream(stream, k_cache.device)),
           "path_decode_step")
    return out


def path_fox_decode_step(q, k, v, w, beta, log_f, k_cache, v_cache, g_cache, cache_len,
                         scale=None, out=None, workspace=None, stream=None):
    """One PaTH-FoX decode step: as path_decode_step, plus the per-key gate sums g_cache
    (B, H, cap) fp32, updated in place (g_j += log_f for j < cache_len, g = 0 appended), and
    the bias g_j on every logit. log_f: (B, H) fp32, the new token's log forget gate."""
    torch = _torch()
    ins, out, (B, H, cap, d) = _decode_args(q, k, v, w, beta, k_cache, v_cache, out)
    _cuda_tensor(log_f, "log_f", torch.float32)
    if log_f.numel() != B * H:
        raise ValueError("log_f must hold (B, H) values")
    _cuda_tensor(g_cache, "g_cache", torch.float32)
    if tuple(g_cache.shape) != (B, H, cap):
        raise ValueError("g_cache must have shape (B, H, cap)")
    if workspace is None:
        workspace = new_workspace(OP_FOX_DECODE, B, H, cap, _dtype_code(k_cache), k_cache.device,
                                  d)
    _check(_load().path_fox_decode_step(_ptr(ins[0]), _ptr(ins[1]), _ptr(ins[2]), _ptr(ins[3]),
                                        _ptr(beta), _ptr(log_f), _ptr(k_cache), _ptr(v_cache),
                                        _ptr(g_cache), B, H, int(cache_len), cap, d,
                                        _dtype_code(k_cache), _scale(scale, d), _ptr(out),
                                        _ptr(workspace), workspace.numel(),
                                        _stream(stream, k_cache.device)),
           "path_fox_decode_step")
    return out


def path_check_workspace(workspace, stream=None):
    """Synchronises the stream and returns the status code left by kernels in `workspace`."""
    return int(_load().path_check_workspace(_ptr(workspace), _stream(stream, workspace.device)))


def path_decode_step_noalloc(q, k, v, w, beta, k_cache, v_cache, cache_len, scale=None, out=None,
                             stream=None):
    """path_decode_step without a workspace, for callers that may not allocate device memory
    for the library on the call path. The split partials live in a fixed 16 MiB array inside
    the library; calls that overlap on one GPU share it and must be serialised. Raises
    PathError(ERR_WORKSPACE) when B * H * ceil(cache_len / 1024) partials do not fit."""
    ins, out, (B, H, cap, d) = _decode_args(q, k, v, w, beta, k_cache, v_cache, out)
    _check(_load().path_decode_step_noalloc(_ptr(ins[0]), _ptr(ins[1]), _ptr(ins[2]),
                                            _ptr(ins[3]), _ptr(beta), _ptr(k_cache),
                                            _ptr(v_cache), B, H, int(cache_len), cap, d,
                                            _dtype_code(k_cache), _scale(scale, d), _ptr(out),
                                            _stream(stream, k_cache.device)),
           "path_decode_step_noalloc")
    return out


def path_wbeta_workspace_bytes(B, L, D, R, H, d=HEAD_DIM, dtype=BF16):
    return int(_load().path_wbeta_workspace_bytes(int(B), int(L), int(D), int(R), int(H), int(d),
                                                  int(dtype)))


def path_wbeta_produce(x, w_down, w_up, conv, u, bias, beta_max=2.0, w_out=None, beta_out=None,
                       workspace=None, stream=None):
    """The w / beta producer: x (B, L, D) bf16; w_down (R, D), w_up (H*d, R), u (H, D) bf16;
    conv (H*d, 3) and bias (H,) fp32. Returns (w (B, H, L, d) bf16, beta (B, H, L) fp32),
    the layouts path_attn_fwd takes."""
    torch = _torch()
    _cuda_tensor(x, "x", torch.bfloat16)
    B, L, D = x.shape
    _cuda_tensor(w_down, "w_down", torch.bfloat16)
    _cuda_tensor(w_up, "w_up", torch.bfloat16)
    _cuda_tensor(u, "u", torch.bfloat16)
    _cuda_tensor(conv, "conv", torch.float32)
    _cuda_tensor(bias, "bias", torch.float32)
    R, H = w_down.shape[0], u.shape[0]
    d = w_up.shape[0] // H
    if (tuple(w_down.shape) != (R, D) or tuple(w_up.shape) != (H * d, R)
            or tuple(u.shape) != (H, D) or tuple(conv.shape) != (H * d, 3)
            or tuple(bias.shape) != (H,)):
        raise ValueError("inconsistent producer shapes")
    if w_out is None:
        w_out = torch.empty((B, H, L, d), dtype=torch.bfloat16, device=x.device)
    if beta_out is None:
        beta_out = torch.empty((B, H, L), dtype=torch.float32, device=x.device)
    if workspace is None:
        n = path_wbeta_workspace_bytes(B, L, D, R, H, d, BF16)
        if n == 0:
            raise PathError(ERR_SHAPE, "path_wbeta_workspace_bytes")
        workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    _check(_load().path_wbeta_produce(_ptr(x), _ptr(w_down), _ptr(w_up), _ptr(conv), _ptr(u),
                                      _ptr(bias), float(beta_max), _ptr(w_out), _ptr(beta_out), B,
                                      L, D, R, H, d, BF16, _ptr(workspace), workspace.numel(),
                                      _stream(stream, x.device)),
           "path_wbeta_produce")
    return w_out, beta_out
