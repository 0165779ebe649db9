"""Seeded synthetic inputs for PaTH attention workloads.

This module only draws random tensors in the distributions the workloads name.
It holds none of the method's arithmetic, and both the CUDA path's tests and
the oracle read their inputs from it.

Recipe (draw order q, k, v, g, z[, u] from one generator per seed):
  q, k, v ~ N(0, 1)                       shape (B, H, L, d)
  w = g / ||g||,  g ~ N(0, I_d)           unit directions, normalised in fp32
  beta = 2 * sigmoid(z),  z ~ N(0, 1)     fp32, optionally clipped from above
  log f = logsigmoid(u),  u ~ N(2, 1)     fp32 (PaTH-FoX only)
q, k, v, w are rounded once to the workload dtype; beta and log f stay fp32
(bf16 would round a 1.99 clip up to 1.9921875). Consumers use the rounded
tensors as given; w is not renormalised after rounding.

Decode caches are synthetic cache contents: prefix keys and values ~ N(0, 1)
(the keys stand for already-transformed cache entries). A PaTH-FoX cache also
holds per-key gate sums; the synthetic ones are those a gate log f =
logsigmoid(u), u ~ N(2, 1), at every prefix position leaves behind: the entry of
key j is the sum of the draws at positions j+1 .. n-1 (fp64, stored fp32), so
the last key holds 0.
"""
from dataclasses import dataclass

import torch

D = 64
BETA_CLIP = 1.99


@dataclass(frozen=True)
class FwdWorkload:
    name: str
    B: int
    H: int
    L: int
    d: int
    dtype: torch.dtype
    seed: int
    clip: float  # 0 disables the clip
    fox: bool


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    n_prefix: int
    steps: int
    d: int
    dtype: torch.dtype
    seed: int
    step_seed: int


# The five workloads: tiny fp32 check, bf16 check, the bf16 speed shape,
# PaTH-FoX at long context, and 64 decode steps over a 32K-token cache.
TINY_FP32 = FwdWorkload("path_fwd_tiny_fp32_B1H2L128", 1, 2, 128, D, torch.float32, 0, 0.0, False)
BF16_L2048 = FwdWorkload("path_fwd_bf16_B4H16L2048", 4, 16, 2048, D, torch.bfloat16, 2, BETA_CLIP, False)
# the same model width (1024) in eight heads of 128
BF16_L2048_D128 = FwdWorkload("path_fwd_bf16_B4H8L2048_d128", 4, 8, 2048, 128, torch.bfloat16, 2, BETA_CLIP, False)
BF16_L4096 = FwdWorkload("path_fwd_bf16_B32H32L4096", 32, 32, 4096, D, torch.bfloat16, 3, BETA_CLIP, False)
FOX_L16384 = FwdWorkload("path_fox_fwd_bf16_B8H16L16384", 8, 16, 16384, D, torch.bfloat16, 4, BETA_CLIP, True)
DECODE_32K = DecodeWorkload("path_decode_bf16_B32H32N32768x64", 32, 32, 32768, 64, D, torch.bfloat16, 5, 1000)
# Head size 128 at the same model width (H*d = 2048): 16 heads of 128.
DECODE_32K_D128 = DecodeWorkload("path_decode_bf16_B32H16d128N32768x64", 32, 16, 32768, 64, 128, torch.bfloat16, 5, 1000)
# PaTH-FoX decode: the same cache and steps plus forget gates (prefix gate sums, log f per step).
FOX_DECODE_32K = DecodeWorkload("path_fox_decode_bf16_B32H32N32768x64", 32, 32, 32768, 64, D, torch.bfloat16, 5, 1000)

SPEED_SWEEP_L = (1024, 2048, 4096, 8192, 16384)


def speed_shape(L):
    """The B=32, H=32 bf16 speed shape at sequence length L (seed 3)."""
    return FwdWorkload("path_fwd_bf16_B32H32L%d" % L, 32, 32, L, D, torch.bfloat16, 3, BETA_CLIP, False)


def _gen(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_fwd_inputs(B, H, L, d=D, dtype=torch.bfloat16, seed=0, clip=BETA_CLIP, fox=False,
                    device="cpu"):
    """Returns dict(q, k, v, w, beta[, log_f]) drawn per the module recipe."""
    g = _gen(seed, device)
    shape = (B, H, L, d)
    f32 = torch.float32
    q = torch.randn(shape, generator=g, device=device, dtype=f32)
    k = torch.randn(shape, generator=g, device=device, dtype=f32)
    v = torch.randn(shape, generator=g, device=device, dtype=f32)
    gw = torch.randn(shape, generator=g, device=device, dtype=f32)
    w = gw / gw.norm(dim=-1, keepdim=True)
    del gw
    z = torch.randn((B, H, L), generator=g, device=device, dtype=f32)
    beta = 2.0 * torch.sigmoid(z)
    if clip:
        beta = beta.clamp(max=clip)
    out = {"q": q.to(dtype), "k": k.to(dtype), "v": v.to(dtype), "w": w.to(dtype),
           "beta": beta.contiguous()}
    if fox:
        u = torch.randn((B, H, L), generator=g, device=device, dtype=f32) + 2.0
        out["log_f"] = torch.nn.functional.logsigmoid(u).contiguous()
    return out


def workload_inputs(wl, device="cpu", L=None):
    """Inputs of a forward workload (optionally at another sequence length)."""
    return make_fwd_inputs(wl.B, wl.H, wl.L if L is None else L, wl.d, wl.dtype, wl.seed,
                           wl.clip, wl.fox, device)


def make_decode_prefix(wl, cap, device="cpu"):
    """Cache tensors (B, H, cap, d) holding n_prefix N(0,1) keys and values."""
    g = _gen(wl.seed, device)
    shape = (wl.B, wl.H, wl.n_prefix, wl.d)
    kc = torch.zeros((wl.B, wl.H, cap, wl.d), device=device, dtype=wl.dtype)
    vc = torch.zeros_like(kc)
    kc[:, :, :wl.n_prefix] = torch.randn(shape, generator=g, device=device).to(wl.dtype)
    vc[:, :, :wl.n_prefix] = torch.randn(shape, generator=g, device=device).to(wl.dtype)
    return kc, vc


def make_fox_decode_prefix(wl, cap, device="cpu"):
    """(k_cache, v_cache, g_cache): make_decode_prefix's caches (same draws) plus the gate
    sums (B, H, cap) fp32 of the n_prefix cached keys (see the module recipe)."""
    g = _gen(wl.seed, device)
    shape = (wl.B, wl.H, wl.n_prefix, wl.d)
    kc = torch.zeros((wl.B, wl.H, cap, wl.d), device=device, dtype=wl.dtype)
    vc = torch.zeros_like(kc)
    kc[:, :, :wl.n_prefix] = torch.randn(shape, generator=g, device=device).to(wl.dtype)
    vc[:, :, :wl.n_prefix] = torch.randn(shape, generator=g, device=device).to(wl.dtype)
    u = torch.randn((wl.B, wl.H, wl.n_prefix), generator=g, device=device) + 2.0
    draws = torch.nn.functional.logsigmoid(u).double()
    gc = torch.zeros((wl.B, wl.H, cap), device=device, dtype=torch.float32)
    if wl.n_prefix > 0:
        # entry j: draws at positions j+1 .. n-1 (a suffix sum shifted by one)
        tail = torch.flip(torch.cumsum(torch.flip(draws, [-1]), -1), [-1])
        gc[:, :, :wl.n_prefix - 1] = tail[:, :, 1:].float()
    return kc, vc, gc


@dataclass(frozen=True)
class ProducerWorkload:
    name: str
    B: int
    L: int
    D: int
    R: int
    H: int
    seed: int


# The w / beta producer at the speed shape: B=32 sequences of L=4096 tokens, model width
# D = H*d = 2048, a rank-64 projection, 32 heads.
PRODUCER_L4096 = ProducerWorkload("path_wbeta_bf16_B32L4096D2048R64H32", 32, 4096, 2048, 64, 32, 6)


def make_producer_inputs(B, L, D, R, H, d=D, seed=0, device="cpu"):
    """Seeded producer inputs (draw order x, w_down, w_up, conv, u, bias): activations
    x ~ N(0, 1); projection weights ~ N(0, 1 / fan_in) (rows = output features), so that
    every intermediate is of unit scale; conv taps ~ N(0, 1/3); u ~ N(0, 1 / D);
    bias ~ N(0, 1). x and the weight matrices bf16, conv and bias fp32."""
    g = _gen(seed, device)
    f32 = torch.float32
    x = torch.randn((B, L, D), generator=g, device=device, dtype=f32)
    w_down = torch.randn((R, D), generator=g, device=device, dtype=f32) * D ** -0.5
    w_up = torch.randn((H * d, R), generator=g, device=device, dtype=f32) * R ** -0.5
    conv = torch.randn((H * d, 3), generator=g, device=device, dtype=f32) * 3 ** -0.5
    u = torch.randn((H, D), generator=g, device=device, dtype=f32) * D ** -0.5
    bias = torch.randn((H,), generator=g, device=device, dtype=f32)
    bf = torch.bfloat16
    return {"x": x.to(bf), "w_down": w_down.to(bf).contiguous(), "w_up": w_up.to(bf).contiguous(),
            "conv": conv.contiguous(), "u": u.to(bf).contiguous(), "bias": bias}


def make_decode_step(wl, t, device="cpu", fox=False, B=None, H=None):
    """Inputs of decode step t: q, k, v, w (B, H, d) and beta (B, H), seed step_seed + t."""
    B = wl.B if B is None else B
    H = wl.H if H is None else H
    return make_fwd_inputs(B, H, 1, wl.d, wl.dtype, wl.step_seed + t, BETA_CLIP, fox,
                           device)


def sample_rows(nh, L, n, seed=0, block=64):
    """Seeded (head, query) pairs for sampled parity: n random rows plus the
    edge rows of every sampled head (first and last row, block boundaries)."""
    g = torch.Generator().manual_seed(int(seed) + 7919)
    heads = torch.randint(0, nh, (n,), generator=g)
    rows = torch.randint(0, L, (n,), generator=g)
    edges = [0, L - 1] + [b for x in range(block, L, block) for b in (x - 1, x)][:8]
    eh = torch.randint(0, nh, (len(edges),), generator=g)
    pairs = torch.cat([torch.stack([heads, rows], 1),
                       torch.stack([eh, torch.tensor(edges, dtype=torch.int64)], 1)])
    return pairs.numpy()
