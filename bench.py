"""Benchmark of the PaTH attention hot path on GB300.

One step = one PaTH forward (UT preprocessing + block scan) over the bf16 speed
workload B=32, H=32, L=4096, d=64, inputs resident in HBM (2.1 GB of inputs per
step, larger than the 129 MB L2, so no flush is needed between steps). Timed
with CUDA events on the launching stream. The line also carries the PaTH-FoX
forward (B=8, H=16, L=16384) and the decode step (B=32, H=32, 32K-token cache,
64 steps) as sub-objects, an end-to-end figure through the C ABI from pinned
host buffers, the roofline of the dominant kernel and the fp64 oracle timed on
the host cores.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch one process per GPU with torch.distributed.run; every rank runs
its own batch of the workload (weak scaling, no collective on the data path).
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import path_inputs as pi  # noqa: E402

C = 64
METRIC = "PaTH attn fwd tokens/s & TFLOP/s (B32 H32 d64 L4096 bf16), % roofline; decode GB/s"


def fwd_flops(B, H, L, d=64):
    """Algorithmic FLOPs of one forward: causal QK^T + PV, the rank-C state updates of
    the block scan, and the per-block UT preprocessing."""
    f_attn = 2.0 * B * H * L * L * d
    f_corr = 2.0 * B * H * d * L * (L - C)
    f_pre = B * H * L * (12.0 * C * d + 2.0 / 3.0 * C * C)
    return f_attn, f_corr, f_pre


def scan_executed_flops(B, H, L, first=None):
    """Tensor-core FLOPs the block-scan kernels actually issue, on 128-row tiles t (query
    blocks 2t, 2t+1) in units of mm = one 128 x 64 x 64 product.
    first None (PaTH, two key blocks per step): per visited key block S = X K~^T, except at
    the last block X P_b^T (as pair products), P V every block.
    first given (PaTH-FoX, one key block per step): the early-exit extents (B*H rows of
    per-query-block lowest key blocks, as path_fox_first_blocks returns them); a tile walks
    key blocks 2t+1 down to the lower extent of its two query blocks, with [S | X'] =
    X [K~_b; P_b]^T (N = 128) at every block but its first and P V_b at every block."""
    nblk = (L + C - 1) // C
    nq = nblk
    nblk += nblk & 1
    mm = 2.0 * 128 * 64 * 64

    if first is None:
        def tile_flops(steps):
            return (steps - 1) * mm + (steps - 2) * mm + steps * mm
        return B * H * sum(tile_flops(2 * t + 2) for t in range(nblk // 2))
    total = 0.0
    for row in first:
        for t in range(nblk // 2):
            lo = row[2 * t] if 2 * t + 1 >= nq else min(row[2 * t], row[2 * t + 1])
            n = 2 * t + 2 - min(lo, 2 * t)
            total += 2 * (n - 1) * mm + n * mm
    return total


def decode_bytes(B, H, n, d=64):
    """HBM bytes of one decode step over n cached keys: key read + key write + value
    read (2 bytes each) plus the new token's q, k, v, w, o."""
    return B * H * (6.0 * n * d + 12.0 * d)


def fox_decode_bytes(B, H, n, d=64):
    """HBM bytes every PaTH-FoX decode step must move over n cached keys: key read + key
    write (2 bytes each) and the per-key gate sum (4 bytes read, 4 written), plus the new
    token's q, k, v, w, o, log f and appended gate sum. Value rows of keys whose weight
    vanishes under the gate are not read, so they are not counted: a lower bound of the
    traffic, and GB/s on this basis never overstates the achieved bandwidth."""
    return B * H * (4.0 * n * d + 8.0 * n + 12.0 * d + 8.0)


def producer_bytes(wl, d=64):
    """HBM bytes of one w / beta production: x read, w and beta written, the bf16
    intermediate z written and read back, and the weights read (w_up once to form the three
    tap-scaled copies, written once and read once each)."""
    B, L, D, R, H = wl.B, wl.L, wl.D, wl.R, wl.H
    per_token = 2.0 * D + 2.0 * H * d + 4.0 * H + 2.0 * 2 * R
    weights = 2.0 * (R * D + H * D) + 2.0 * H * d * R * (1 + 3 + 3) + 4.0 * H * d * 3
    return B * L * per_token + weights


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def compact(obj, sig=5):
    """Rounds every float in a nested dict/list to `sig` significant digits (keeps the JSON
    line short; integers and strings pass through)."""
    if isinstance(obj, float):
        if obj == 0.0 or not math.isfinite(obj):
            return obj
        return float("%.*g" % (sig, obj))
    if isinstance(obj, dict):
        return {k: compact(v, sig) for k, v in obj.items()}
    if isinstance(obj, (list, tuple)):
        return [compact(v, sig) for v in obj]
    return obj


# Legs that end the JSON line, in this order: a reader that keeps only the line's end (the
# last 3 KB) still finds them.
LINE_END = ("fwd_d128", "bwd", "bwd_d128", "decode", "fox", "sweep_L")


def order_line(line):
    """The line's keys in print order: everything else first (insertion order), then the
    LINE_END legs that are present."""
    ordered = {k: v for k, v in line.items() if k not in LINE_END}
    ordered.update({k: line[k] for k in LINE_END if k in line})
    return ordered


def kernel_source_hash(name):
    src = os.path.join(ROOT, "dependent_position_encoded_gb300", "csrc", name)
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def ncu_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current source of that kernel (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        j = json.load(f)
    e = j.get(kernel_key)
    if not e or e.get("source_sha") != kernel_source_hash(e["source"]):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    t = [x.strip() for x in line.split(",")]
                    if len(t) >= 9:
                        rows.append(t)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        loaded = sorted(sm)[len(sm) // 2:] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def time_forward(pa, x, steps, warmup, fox=False):
    """Times `steps` forwards (prepare + scan); returns (total_ms, scan_ms_list, prep_ms_list)."""
    B, H, L, d = x["q"].shape
    op = pa.OP_FOX_FWD if fox else pa.OP_FWD
    dt = pa.F32 if x["q"].dtype == torch.float32 else pa.BF16
    ws = pa.new_workspace(op, B, H, L, dt, x["q"].device, d=d)
    out = torch.empty_like(x["q"])
    lse = torch.empty((B, H, L), dtype=torch.float32, device=x["q"].device)
    log_f = x.get("log_f") if fox else None
    stream = torch.cuda.current_stream()

    def one(evs=None):
        if evs:
            evs[0].record(stream)
        pa.path_fwd_prepare(x["q"], x["k"], x["w"], x["beta"], ws, log_f=log_f)
        if evs:
            evs[1].record(stream)
        pa.path_fwd_scan(x["v"], ws, out=out, lse=lse, fox=fox)
        if evs:
            evs[2].record(stream)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        one(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    status = pa.path_check_workspace(ws)
    if status != pa.OK:
        raise RuntimeError("kernel status " + pa.path_status_string(status))
    total = start.elapsed_time(end)
    prep = [e[0].elapsed_time(e[1]) for e in evs]
    scan = [e[1].elapsed_time(e[2]) for e in evs]
    return total, scan, prep


def time_e2e(pa, x, steps, warmup):
    """The same forward through the C ABI, end to end: every step copies its own inputs
    from pinned host memory and reads its output back. Copies run on their own streams
    with double-buffered device tensors, so step k's host-to-device copy and step k-1's
    read-back overlap step k-1's and step k's forward (the pipelining a serving loop does);
    the timed region spans the first copy-in to the last read-back."""
    keys = ("q", "k", "v", "w", "beta")
    host = [{k: x[k].cpu().pin_memory() for k in keys} for _ in range(2)]
    dev = [{k: torch.empty_like(x[k]) for k in keys} for _ in range(2)]
    B, H, L, _ = x["q"].shape
    ws = [pa.new_workspace(pa.OP_FWD, B, H, L, pa.BF16, x["q"].device) for _ in range(2)]
    out = [torch.empty_like(x["q"]) for _ in range(2)]
    out_h = [torch.empty(out[0].shape, dtype=out[0].dtype).pin_memory() for _ in range(2)]
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=False)  # noqa: E731

    def run(n):
        in_ready, comp_done, out_done = [None] * n, [None] * n, [None] * n
        for k in range(n):
            i = k % 2
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(comp_done[k - 2])  # buffer i no longer read
                for key in keys:
                    dev[i][key].copy_(host[i][key], non_blocking=True)
                in_ready[k] = ev()
                in_ready[k].record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(in_ready[k])
                if k >= 2:
                    s_cmp.wait_event(out_done[k - 2])  # out[i] has been read back
                pa.path_attn_fwd(dev[i]["q"], dev[i]["k"], dev[i]["v"], dev[i]["w"],
                                 dev[i]["beta"], out=out[i], lse=None, workspace=ws[i],
                                 stream=s_cmp)
                comp_done[k] = ev()
                comp_done[k].record(s_cmp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[k])
                out_h[i].copy_(out[i], non_blocking=True)
                out_done[k] = ev()
                out_done[k].record(s_out)
        return out_done[n - 1]

    run(warmup)
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    last = run(steps)
    s_out.wait_event(last)
    end.record(s_out)
    torch.cuda.synchronize()
    h2d = sum(host[0][k].numel() * host[0][k].element_size() for k in keys)
    d2h = out_h[0].numel() * out_h[0].element_size()
    return start.elapsed_time(end), h2d, d2h


def time_decode(pa, wl, reps=2, fox=False):
    """Times the 64-step decode sequence (cache reset to the prefix length each repetition;
    the cache content drifts across repetitions, which does not change the work). With
    fox, the PaTH-FoX step over the same cache plus its gate sums."""
    dev = torch.device("cuda")
    cap = wl.n_prefix + wl.steps
    if fox:
        kc, vc, gc = pi.make_fox_decode_prefix(wl, cap, device=dev)
    else:
        kc, vc = pi.make_decode_prefix(wl, cap, device=dev)
    steps = [pi.make_decode_step(wl, t, device=dev, fox=fox) for t in range(wl.steps)]
    ws = pa.new_workspace(pa.OP_FOX_DECODE if fox else pa.OP_DECODE, wl.B, wl.H, cap, pa.BF16,
                          dev, wl.d)
    out = torch.empty((wl.B, wl.H, wl.d), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()
    per_step = []
    for r in range(reps + 1):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(wl.steps + 1)]
        evs[0].record(stream)
        for t, s in enumerate(steps):
            if fox:
                pa.path_fox_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], s["log_f"],
                                        kc, vc, gc, wl.n_prefix + t, out=out, workspace=ws)
            else:
                pa.path_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], kc, vc,
                                    wl.n_prefix + t, out=out, workspace=ws)
            evs[t + 1].record(stream)
        torch.cuda.synchronize()
        if r > 0:  # the first pass is the warm-up
            per_step.append([evs[t].elapsed_time(evs[t + 1]) for t in range(wl.steps)])
    ms = [statistics.mean(col) for col in zip(*per_step)]
    bytes_fn = fox_decode_bytes if fox else decode_bytes
    nbytes = [bytes_fn(wl.B, wl.H, wl.n_prefix + t, wl.d) for t in range(wl.steps)]
    gbs = sum(nbytes) / (sum(ms) * 1e-3) / 1e9
    return {"ms_per_step": sum(ms) / len(ms), "gbs": gbs,
            "tokens_per_s": wl.B / (sum(ms) / len(ms) * 1e-3),
            "bytes_per_step": sum(nbytes) / len(nbytes), "launches_per_step": 2}


def time_producer(pa, wl, steps=5, warmup=3):
    """Times the w / beta producer (its three launches) on the workload, inputs resident."""
    dev = torch.device("cuda")
    p = pi.make_producer_inputs(wl.B, wl.L, wl.D, wl.R, wl.H, seed=wl.seed, device=dev)
    n = pa.path_wbeta_workspace_bytes(wl.B, wl.L, wl.D, wl.R, wl.H)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    w = torch.empty((wl.B, wl.H, wl.L, 64), dtype=torch.bfloat16, device=dev)
    beta = torch.empty((wl.B, wl.H, wl.L), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def one():
        pa.path_wbeta_produce(p["x"], p["w_down"], p["w_up"], p["conv"], p["u"], p["bias"],
                              beta_max=pi.BETA_CLIP, w_out=w, beta_out=beta, workspace=ws)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    if pa.path_check_workspace(ws) != pa.OK:
        raise RuntimeError("producer kernel status")
    ms = e0.elapsed_time(e1) / steps
    nbytes = producer_bytes(wl)
    return {"workload": wl.name, "ms_per_step": ms, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "tokens_per_s": wl.B * wl.L / (ms * 1e-3), "bytes_per_step": nbytes,
            "launches_per_step": 3}


# FP32 FMA peak of the CUDA cores, from the unit counts and the maximum SM clock:
# 152 SMs x 128 FP32 lanes x 2 FLOP per FMA x 2.07 GHz (nominal; no measured FP32 figure)
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12


def bwd_flops(B, H, L, d=64):
    """Algorithmic FLOPs of the backward's query pass: per pair of query block a and key block
    b < a, the logits, dout V_b^T, the dk~ and dv terms and dT K~_b (5 products of
    2 * 64^2 * d each), plus X P_b^T, G P_b and the dP_b term when b > 0 (3 products of
    2 * 64 * d^2); per diagonal block dout V^T and p^T dout (2 * 64^2 * d each)."""
    nb = (L + 63) // 64
    pairs = nb * (nb - 1) // 2
    t, u = 2 * 64 * 64 * d, 2 * 64 * d * d
    return B * H * (5 * t * pairs + 3 * u * (pairs - (nb - 1)) + 2 * t * nb)


def time_bwd(pa, wl, steps=5, warmup=3, fox=False):
    """Times path_attn_bwd (path_fox_bwd with fox) on the workload (forward outputs and
    d_out resident)."""
    dev = torch.device("cuda")
    x = pi.make_fwd_inputs(wl.B, wl.H, wl.L, wl.d, wl.dtype, wl.seed, wl.clip, fox, dev)
    g = torch.Generator(device=dev).manual_seed(wl.seed + 1)
    d_out = torch.randn((wl.B, wl.H, wl.L, wl.d), generator=g, device=dev).to(wl.dtype)
    if fox:
        out, lse = pa.path_fox_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"])
    else:
        out, lse = pa.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    ws = pa.new_workspace(pa.OP_FOX_BWD if fox else pa.OP_BWD, wl.B, wl.H, wl.L,
                          pa.BF16 if wl.dtype == torch.bfloat16 else pa.F32, dev, d=wl.d)
    grads = {n: torch.empty((wl.B, wl.H, wl.L, wl.d), dtype=torch.float32, device=dev)
             for n in ("dq", "dk", "dv", "dw")}
    grads["dbeta"] = torch.empty((wl.B, wl.H, wl.L), dtype=torch.float32, device=dev)
    grads["dlog_f"] = torch.empty((wl.B, wl.H, wl.L), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def one():
        if fox:
            pa.path_fox_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["log_f"], out, lse,
                            d_out, grads=grads, workspace=ws)
        else:
            pa.path_attn_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], out, lse, d_out,
                             grads=grads, workspace=ws)

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        one()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    fl = bwd_flops(wl.B, wl.H, wl.L, wl.d)
    name = wl.name.replace("path_fwd", "path_fox_bwd" if fox else "path_bwd")
    return {"workload": name, "ms_per_step": ms,
            "tokens_per_s": wl.B * wl.L / (ms * 1e-3), "query_pass_flops": fl,
            "workspace_bytes": ws.numel(),
            # UT preparation, query pass, block pass; FoX adds the gate sums and d log f (and,
            # at d = 128, the preparation's exit-bound pass)
            "launches_per_step": (6 if wl.d == 128 else 5) if fox else 3}


def cpu_baseline(x_cpu, wl, target_s=12.0):
    """The fp64 oracle on whole heads of the workload, timed on the host cores."""
    import oracle
    B, H, L = wl.B, wl.H, wl.L
    nh_total = B * H
    # x_cpu holds a subset of heads drawn in the workload's distribution
    sel = {k: v.reshape(-1, *v.shape[2:]) for k, v in x_cpu.items()}
    nh_avail = sel["q"].shape[0]

    def run(n):
        t0 = time.perf_counter()
        oracle.path_fwd(sel["q"][:n], sel["k"][:n], sel["v"][:n], sel["w"][:n],
                        sel["beta"][:n], log_f=sel.get("log_f", None) if wl.fox else None)
        return time.perf_counter() - t0

    t1 = run(1)
    n = max(1, min(nh_avail, int(target_s / max(t1, 1e-3))))
    t = run(n) if n > 1 else t1
    cores = os.cpu_count()
    t_full = t * nh_total / n
    return {"value": B * L / t_full, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "%d of %d heads of the workload, every query row (%.1f s); full-workload "
                      "time extrapolated by head count" % (n, nh_total, t)}


def leg_cpu_baselines(wl_bwd, wl_dec, wl_prod, wl_fox=None):
    """The fp64 oracle beside the backward, decode and producer legs, each on a bounded
    sample of its workload's shapes and distributions (fresh draws of a few heads or
    tokens), extrapolated to the workload in the leg's own unit."""
    import numpy as np
    import oracle
    out = {}
    # backward: two whole heads of L tokens
    x = pi.make_fwd_inputs(1, 2, wl_bwd.L, seed=wl_bwd.seed, device="cpu")
    d_out = torch.randn((1, 2, wl_bwd.L, 64), generator=torch.Generator().manual_seed(1))
    t0 = time.perf_counter()
    oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out.to(torch.bfloat16))
    t = (time.perf_counter() - t0) * (wl_bwd.B * wl_bwd.H) / 2
    out["bwd"] = {"value": wl_bwd.B * wl_bwd.L / t, "unit": "tokens/s", "cores": 2,
                  "kind": "oracle", "sample": "2 of %d heads, L %d, one thread per head; "
                  "time extrapolated by head count" % (wl_bwd.B * wl_bwd.H, wl_bwd.L)}
    # backward at head size 128 (B4 H8 L2048): two whole heads
    wl_b2 = pi.BF16_L2048_D128
    x = pi.make_fwd_inputs(1, 2, wl_b2.L, d=128, seed=wl_b2.seed, device="cpu")
    d_out = torch.randn((1, 2, wl_b2.L, 128), generator=torch.Generator().manual_seed(1))
    t0 = time.perf_counter()
    oracle.path_bwd(x["q"], x["k"], x["v"], x["w"], x["beta"], d_out.to(torch.bfloat16))
    t = (time.perf_counter() - t0) * (wl_b2.B * wl_b2.H) / 2
    out["bwd_d128"] = {"value": wl_b2.B * wl_b2.L / t, "unit": "tokens/s", "cores": 2,
                       "kind": "oracle", "sample": "2 of %d heads, L %d, d 128, one thread per "
                       "head; time extrapolated by head count" % (wl_b2.B * wl_b2.H, wl_b2.L)}
    # decode: one step over 4 heads of the prefix cache
    nh, n0 = 4, wl_dec.n_prefix
    g = torch.Generator().manual_seed(wl_dec.seed)
    cache = oracle.DecodeCache(torch.randn((nh, n0, 64), generator=g).to(torch.bfloat16),
                               torch.randn((nh, n0, 64), generator=g).to(torch.bfloat16), n0 + 1)
    q, k, v = (torch.randn((nh, 64), generator=g) for _ in range(3))
    w = torch.nn.functional.normalize(torch.randn((nh, 64), generator=g), dim=-1)
    beta = 2 * torch.sigmoid(torch.randn((nh,), generator=g))
    t0 = time.perf_counter()
    cache.step(q, k, v, w, beta)
    t = (time.perf_counter() - t0) * (wl_dec.B * wl_dec.H) / nh
    out["decode"] = {"value": decode_bytes(wl_dec.B, wl_dec.H, n0) / t / 1e9, "unit": "GB/s",
                     "cores": 1, "kind": "oracle",
                     "sample": "one step over %d of %d heads of a %d-key cache; time "
                               "extrapolated by head count" % (nh, wl_dec.B * wl_dec.H, n0)}
    # producer: one sequence of 256 tokens
    Lp = 256
    pr = pi.make_producer_inputs(1, Lp, wl_prod.D, wl_prod.R, wl_prod.H, seed=wl_prod.seed)
    t0 = time.perf_counter()
    oracle.wbeta_produce(pr["x"], pr["w_down"], pr["w_up"], pr["conv"], pr["u"], pr["bias"],
                         beta_max=pi.BETA_CLIP)
    t = (time.perf_counter() - t0) * (wl_prod.B * wl_prod.L) / Lp
    out["producer"] = {"value": producer_bytes(wl_prod) / t / 1e9, "unit": "GB/s", "cores": 1,
                       "kind": "oracle", "sample": "%d of %d tokens; time extrapolated by "
                       "token count" % (Lp, wl_prod.B * wl_prod.L)}
    # the bf16 check workload (B4 H16 L2048): two whole heads, every query row
    x = pi.make_fwd_inputs(1, 2, wl_bwd.L, seed=wl_bwd.seed, device="cpu")
    t0 = time.perf_counter()
    oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    t = (time.perf_counter() - t0) * (wl_bwd.B * wl_bwd.H) / 2
    out["fwd_L2048"] = {"value": wl_bwd.B * wl_bwd.L / t, "unit": "tokens/s",
                        "cores": os.cpu_count(), "kind": "oracle",
                        "sample": "2 of %d heads, every query row; time extrapolated by head "
                                  "count" % (wl_bwd.B * wl_bwd.H)}
    if wl_fox is not None:
        # PaTH-FoX (B8 H16 L16384): two whole fresh heads, every query row
        x = pi.make_fwd_inputs(1, 2, wl_fox.L, seed=wl_fox.seed, fox=True, device="cpu")
        t0 = time.perf_counter()
        oracle.path_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], log_f=x["log_f"])
        t = time.perf_counter() - t0
        t_full = t * (wl_fox.B * wl_fox.H) / 2
        out["fox"] = {"value": wl_fox.B * wl_fox.L / t_full, "unit": "tokens/s",
                      "cores": os.cpu_count(), "kind": "oracle",
                      "sample": "2 of %d heads, every query row (%.1f s); time extrapolated "
                                "by head count" % (wl_fox.B * wl_fox.H, t)}
    return out


# kernels of one bf16 forward at head size 64: UT preprocessing, block-pair products, scan
LAUNCHES_PER_FWD = 3


def bench_parity(pa, x, n_rows=300):
    """Parity figures carried in the bench line: the tiny fp32 workload against the oracle
    in full (normwise max|o - o*| / max|o*| and element-wise max |o - o*| / max(|o*|, 1e-3)),
    and `n_rows` seeded sampled rows of the timed workload (max absolute error, bf16)."""
    import numpy as np
    import oracle
    t = pi.workload_inputs(pi.TINY_FP32, device="cuda")
    out, _ = pa.path_attn_fwd(t["q"], t["k"], t["v"], t["w"], t["beta"])
    ref, _ = oracle.path_fwd(t["q"], t["k"], t["v"], t["w"], t["beta"])
    got = out.double().cpu().numpy()
    err = np.abs(got - ref)
    res = {"tiny_fp32": {"normwise_rel": float(err.max() / np.abs(ref).max()),
                         "elementwise_rel": float((err / np.maximum(np.abs(ref), 1e-3)).max()),
                         "bar": "normwise <= 1e-4"}}
    B, H, L, d = x["q"].shape
    rows = pi.sample_rows(B * H, L, n_rows, seed=3)
    out, _ = pa.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"])
    got = out.reshape(B * H, L, d)[torch.as_tensor(rows[:, 0]), torch.as_tensor(rows[:, 1])]
    cpu = {k: v.reshape(B * H, L, -1)[torch.as_tensor(np.unique(rows[:, 0]))].cpu()
           for k, v in x.items()}
    remap = {h: i for i, h in enumerate(np.unique(rows[:, 0]))}
    r2 = np.array([[remap[h], i] for h, i in rows])
    ref, _ = oracle.path_rows(cpu["q"], cpu["k"], cpu["v"], cpu["w"], cpu["beta"][..., 0], r2)
    res["speed_workload_rows"] = {"rows": int(len(rows)),
                                  "max_abs": float(np.abs(got.double().cpu().numpy() - ref).max()),
                                  "bar": "max_abs <= 2e-2"}
    return res


def run_legs(pa, peaks, dev, rank):
    """The secondary legs: the bf16 check workload, the producer, the backward (plain and
    PaTH-FoX), head size 128 (forward and decode), fp32 inputs and the PaTH-FoX decode."""
    legs = {}
    wl2 = shard_workload(pi.BF16_L2048, rank)
    x2 = pi.workload_inputs(wl2, device=dev)
    t2, sc2, pr2 = time_forward(pa, x2, 5, 3)
    a, c, p = fwd_flops(wl2.B, wl2.H, wl2.L)
    legs["fwd_L2048"] = {"workload": wl2.name, "ms_per_step": t2 / 5,
                         "tokens_per_s": wl2.B * wl2.L / (t2 / 5 * 1e-3),
                         "tflops": (a + c + p) / (t2 / 5 * 1e-3) / 1e12}
    del x2
    prod = time_producer(pa, pi.PRODUCER_L4096)
    t_down, t_up = ncu_traffic("producer_down_kernel"), ncu_traffic("producer_up_kernel")
    prod["roofline"] = {"bound": "hbm", "achieved": prod["gbs"], "peak": peaks["hbm_gbs"],
                        "unit": "GB/s", "frac": prod["gbs"] / peaks["hbm_gbs"],
                        "traffic": (t_down + t_up) if (t_down and t_up) else None}
    legs["producer"] = prod
    torch.cuda.empty_cache()
    for fox in (False, True):
        wlb = pi.BF16_L2048
        bwd = time_bwd(pa, wlb, fox=fox)
        sec = bwd["ms_per_step"] * 1e-3
        ach = bwd["query_pass_flops"] / sec / 1e12
        ex = bwd_tc_executed_flops(wlb.B, wlb.H, wlb.L) / sec / 1e12
        bwd["roofline"] = BWD_ROOFLINE(ach, peaks, fox, ex)
        legs["fox_bwd" if fox else "bwd"] = bwd
        torch.cuda.empty_cache()
    # the backward at head size 128 on the same model width (bf16: warp-level tensor-core query
    # pass, block pass in matrix form)
    bwd = time_bwd(pa, pi.BF16_L2048_D128)
    ach = bwd["query_pass_flops"] / (bwd["ms_per_step"] * 1e-3) / 1e12
    bwd["roofline"] = {"kernels": "query-pass FLOPs over the whole call (mma.sync bf16)",
                       "bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
                       "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
                       "traffic": ncu_traffic("bwd_query128_mma_kernel"),
                       "peak_source": "%s bf16 dense (burst)" % peaks["source"]}
    legs["bwd_d128"] = bwd
    torch.cuda.empty_cache()
    # head size 128 at the speed workload's tokens and model width (B32, 16 heads of 128 =
    # 32 heads of 64), and on the bf16 check workload's width in 8 heads (B4 H8 L2048)
    # (the small case first, so that the main figures end the leg's entry in the line)
    for key, (B_, H_, L_) in (("small_", (4, 8, 2048)), ("", (32, 16, 4096))):
        xd = pi.make_fwd_inputs(B_, H_, L_, d=128, dtype=torch.bfloat16, seed=12, device=dev)
        d_tot, d_scan, d_prep = time_forward(pa, xd, 3, 3)
        d_ms = d_tot / 3
        fa, fc, fp = fwd_flops(B_, H_, L_, d=128)
        d_ach = (fa + fc + fp) / (d_ms * 1e-3) / 1e12
        del xd
        xd = pi.make_fwd_inputs(B_, H_, L_, d=128, dtype=torch.bfloat16, seed=12, fox=True,
                                device=dev)
        f_tot, _, _ = time_forward(pa, xd, 3, 3, fox=True)
        del xd
        torch.cuda.empty_cache()
        name = "path_fwd_bf16_B%dH%dL%d_d128" % (B_, H_, L_)
        if key:
            legs["fwd_d128"] = {"small_workload": name, "small_ms_per_step": d_ms,
                                "small_tflops": d_ach,
                                "small_frac": d_ach / peaks["bf16_tflops"],
                                "small_fox_ms_per_step": f_tot / 3}
        else:
            legs["fwd_d128"].update({"workload": name, "roofline": D128_ROOFLINE(d_ach, peaks),
                                     "scan_ms": statistics.mean(d_scan),
                                     "prepare_ms": statistics.mean(d_prep),
                                     "fox_ms_per_step": f_tot / 3,
                                     "tokens_per_s": B_ * L_ / (d_ms * 1e-3),
                                     "ms_per_step": d_ms})
    # fp32 inputs (fp32 CUDA-core preparation and scan) on the bf16 check workload's shape
    x32 = pi.make_fwd_inputs(4, 16, 2048, dtype=torch.float32, seed=2, clip=0.0, device=dev)
    s_tot, s_scan, s_prep = time_forward(pa, x32, 3, 3)
    s_ms = s_tot / 3
    fa, fc, fp = fwd_flops(4, 16, 2048)
    s_ach = (fa + fc + fp) / (s_ms * 1e-3) / 1e12
    legs["fwd_f32"] = {"workload": "path_fwd_f32_B4H16L2048", "ms_per_step": s_ms,
                       "tokens_per_s": 4 * 2048 / (s_ms * 1e-3),
                       "roofline": {"bound": "alu", "achieved": s_ach, "peak": FP32_ALU_TFLOPS,
                                    "unit": "TFLOP/s", "frac": s_ach / FP32_ALU_TFLOPS,
                                    "traffic": None}}
    del x32
    torch.cuda.empty_cache()
    for key, wl, fox, kern in (("decode_d128", pi.DECODE_32K_D128, False, "decode_split_kernel_d128"),
                               ("fox_decode", pi.FOX_DECODE_32K, True, "decode_split_kernel_fox")):
        r = time_decode(pa, wl, fox=fox)
        r["workload"] = wl.name
        r["roofline"] = {"bound": "hbm", "achieved": r["gbs"], "peak": peaks["hbm_gbs"],
                         "unit": "GB/s", "frac": r["gbs"] / peaks["hbm_gbs"],
                         "traffic": ncu_traffic(kern)}
        legs[key] = r
        torch.cuda.empty_cache()
    return legs


def run_headline_legs(pa, peaks, dev, rank):
    """The decode step on the 32K cache and the PaTH-FoX forward: printed last in the line."""
    out = {}
    dec = time_decode(pa, pi.DECODE_32K)
    dec["workload"] = pi.DECODE_32K.name
    dec["roofline"] = {"kernel": "decode_split_kernel", "bound": "hbm", "achieved": dec["gbs"],
                       "peak": peaks["hbm_gbs"], "unit": "GB/s",
                       "frac": dec["gbs"] / peaks["hbm_gbs"],
                       "traffic": ncu_traffic("decode_split_kernel"),
                       "peak_source": "%s HBM copy" % peaks["source"]}
    out["decode"] = dec
    torch.cuda.empty_cache()
    fw = shard_workload(pi.FOX_L16384, rank)
    xf = pi.workload_inputs(fw, device=dev)
    fox_total, fox_scan, fox_prep = time_forward(pa, xf, 3, 3, fox=True)
    fox_ms = fox_total / 3
    # the early exit skips the key blocks whose weights vanish, so the fixed algorithmic-FLOP
    # formula does not describe the work done: the scan's rate is taken on the tensor-core
    # FLOPs of the key blocks it visits (from the recorded extents)
    wsf = pa.new_workspace(pa.OP_FOX_FWD, fw.B, fw.H, fw.L, pa.BF16, dev)
    pa.path_fwd_prepare(xf["q"], xf["k"], xf["w"], xf["beta"], wsf, log_f=xf["log_f"])
    first = pa.path_fox_first_blocks(wsf, fw.B, fw.H, fw.L, xf["q"].dtype).cpu()
    f_ex = scan_executed_flops(fw.B, fw.H, fw.L, first.reshape(fw.B * fw.H, -1).tolist())
    del wsf, xf
    torch.cuda.empty_cache()
    f_scan = statistics.mean(fox_scan)
    f_ach = f_ex / (f_scan * 1e-3) / 1e12
    out["fox"] = {"workload": fw.name, "ms_per_step": fox_ms,
                  "tokens_per_s": fw.B * fw.L / (fox_ms * 1e-3), "early_exit": True,
                  "scan_ms": f_scan, "prepare_ms": statistics.mean(fox_prep),
                  "roofline": {"kernel": "path_scan_tc_fox_kernel", "bound": "tensor",
                               "achieved": f_ach, "peak": peaks["bf16_tflops"],
                               "unit": "TFLOP/s", "frac": f_ach / peaks["bf16_tflops"],
                               "traffic": ncu_traffic("path_scan_tc_fox_kernel"),
                               "basis": "executed tensor FLOPs of the visited key blocks",
                               "executed_flops_per_launch": f_ex}}
    return out


def bwd_tc_executed_flops(B, H, L):
    """Tensor-core FLOPs the bf16 backward's query pass issues (128-row tiles t of query
    blocks 2t, 2t+1): pass 1, per key block, [S|X'] = X [K~; P]^T (N = 128, not at the tile's
    first, diagonal-only step), dout V^T (N = 64) and [p^T; dT^T][X | dout] (N = 128,
    K = 128); pass 2, per key block, dT K~ and, past the first, G_hi P + G_lo P and
    [G_hi^T; G_lo^T] X (K = 128)."""
    nbe = -(-L // 64)
    nbe += nbe & 1
    u = 2.0 * 128 * 64 * 64  # one M = 128, N = 64, K = 64 product
    total = 0.0
    for t in range(nbe // 2):
        s1 = 2 * t + 2
        total += (s1 - 1) * 2 * u + s1 * u + s1 * 4 * u
        s2 = 2 * t + 1
        total += s2 * u + (s2 - 1) * (2 * u + 2 * u)
    return B * H * total


def BWD_ROOFLINE(ach, peaks, fox, executed=None):
    return {"kernels": "query-pass FLOPs (64^3 gradient products) over the whole call",
            "bound": "tensor",
            "achieved": ach, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
            "frac": ach / peaks["bf16_tflops"],
            "traffic": ncu_traffic("bwd_query_tc_kernel_fox" if fox else "bwd_query_tc_kernel"),
            "executed_tensor_tflops": executed,
            "peak_source": "%s bf16 dense (burst)" % peaks["source"]}


def D128_ROOFLINE(ach, peaks):
    return {"kernels": "ut_prepare_tc128_kernel + scan_tc128_kernel (tcgen05)",
            "bound": "tensor", "achieved": ach, "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": ach / peaks["bf16_tflops"],
            "traffic": ncu_traffic("scan_tc128_kernel"),
            "peak_source": "%s bf16 dense (burst)" % peaks["source"]}


PROFILE_CASES = {
    # a quarter of the speed workload: 1.3 GB on the device, inputs larger than L2
    "fwd": pi.FwdWorkload("path_fwd_bf16_B8H32L4096", 8, 32, 4096, 64, torch.bfloat16, 3,
                          pi.BETA_CLIP, False),
    "fox": pi.FwdWorkload("path_fox_fwd_bf16_B2H16L16384", 2, 16, 16384, 64, torch.bfloat16, 4,
                          pi.BETA_CLIP, True),
    "decode": pi.DecodeWorkload("path_decode_bf16_B8H32N32768x4", 8, 32, 32768, 4, 64,
                                torch.bfloat16, 5, 1000),
    "fox_decode": pi.DecodeWorkload("path_fox_decode_bf16_B8H32N32768x4", 8, 32, 32768, 4, 64,
                                    torch.bfloat16, 5, 1000),
    # a quarter of the producer workload: x 134 MB, w 134 MB (both larger than L2)
    "producer": pi.ProducerWorkload("path_wbeta_bf16_B8L4096D2048R64H32", 8, 4096, 2048, 64, 32, 6),
    # the backward legs' own workload (1.3 GB of workspace, stash larger than L2)
    "bwd": pi.BF16_L2048,
    "fox_bwd": pi.BF16_L2048,
    "bwd_d128": pi.BF16_L2048_D128,
    # a quarter of the head-size-128 forward leg's workload (B8 of B32, H16 L4096 d128)
    "fwd_d128": pi.FwdWorkload("path_fwd_bf16_B8H16L4096_d128", 8, 16, 4096, 128, torch.bfloat16, 12,
                               pi.BETA_CLIP, False),
    # the fp32-input forward leg's own workload (fp32 CUDA-core kernels)
    "fwd_f32": pi.FwdWorkload("path_fwd_f32_B4H16L2048", 4, 16, 2048, 64, torch.float32, 2, 0.0,
                              False),
    # a quarter of the head-size-128 decode workload (B8 H16 d128, 32K cache)
    "decode_d128": pi.DecodeWorkload("path_decode_bf16_B8H16d128N32768x4", 8, 16, 32768, 4, 128,
                                     torch.bfloat16, 5, 1000),
}


def run_profile_case(args):
    """Runs one operation on its reduced case: warm-up launches, then `steps` launches."""
    import dependent_position_encoded_gb300 as pa
    pa.ensure_built()
    dev = torch.device("cuda")
    wl = PROFILE_CASES[args.profile]
    if args.profile in ("decode", "decode_d128"):
        cap = wl.n_prefix + args.warmup + args.steps
        kc, vc = pi.make_decode_prefix(wl, cap, device=dev)
        ws = pa.new_workspace(pa.OP_DECODE, wl.B, wl.H, cap, pa.BF16, dev, wl.d)
        s = pi.make_decode_step(wl, 0, device=dev)
        for t in range(args.warmup + args.steps):
            pa.path_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], kc, vc,
                                wl.n_prefix + t, workspace=ws)
    elif args.profile == "producer":
        r = time_producer(pa, wl, steps=args.steps, warmup=args.warmup)
        print(json.dumps(r))
    elif args.profile in ("bwd", "fox_bwd", "bwd_d128"):
        r = time_bwd(pa, wl, steps=args.steps, warmup=args.warmup, fox=args.profile == "fox_bwd")
        print(json.dumps(r))
    elif args.profile == "fox_decode":
        cap = wl.n_prefix + args.warmup + args.steps
        kc, vc, gc = pi.make_fox_decode_prefix(wl, cap, device=dev)
        ws = pa.new_workspace(pa.OP_FOX_DECODE, wl.B, wl.H, cap, pa.BF16, dev)
        s = pi.make_decode_step(wl, 0, device=dev, fox=True)
        for t in range(args.warmup + args.steps):
            pa.path_fox_decode_step(s["q"], s["k"], s["v"], s["w"], s["beta"], s["log_f"], kc,
                                    vc, gc, wl.n_prefix + t, workspace=ws)
    else:
        x = pi.workload_inputs(wl, device=dev)
        total, scan, prep = time_forward(pa, x, args.steps, args.warmup, fox=wl.fox)
        print(json.dumps({"profile": wl.name, "scan_ms": scan, "prepare_ms": prep}))
    torch.cuda.synchronize()


def dist_setup(n_gpus, backend=None):
    if n_gpus <= 1 and "WORLD_SIZE" not in os.environ:
        return 0, 1, 0
    import torch.distributed as dist
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    backend = backend or ("nccl" if torch.cuda.is_available() else "gloo")
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend=backend)
    return rank, world, local


def shard_workload(wl, rank):
    """The rank's shard of the global batch: its own B rows, drawn from their own seed.

    Batch rows are independent problems, so ranks share nothing on the data path; rank 0's
    shard is the single-GPU workload itself.
    """
    import dataclasses
    return wl if rank == 0 else dataclasses.replace(wl, seed=wl.seed + 7919 * rank)


def aggregate(local_ms, world, rows_per_rank, L, steps):
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    t_max = max_over_ranks(local_ms, world)
    return t_max, t_max / steps, world * rows_per_rank * L * steps / (t_max * 1e-3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world <= 1:
        return x
    import torch.distributed as dist
    on_gpu = dist.get_backend() == "nccl"
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    """The fp64 oracle as the reference arm, on rank 0 only."""
    if rank != 0:
        return
    wl = pi.BF16_L4096
    # one head per step: the oracle on the full workload would take hours
    import oracle
    g = pi.make_fwd_inputs(1, 2, wl.L, seed=wl.seed, device="cpu")
    sel = {k: v.reshape(2, *v.shape[2:]) for k, v in g.items()}

    def step():
        t0 = time.perf_counter()
        oracle.path_fwd(sel["q"][:1], sel["k"][:1], sel["v"][:1], sel["w"][:1], sel["beta"][:1])
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        step()
    times = [step() for _ in range(args.steps)]
    t_head = statistics.mean(times)
    t_full = t_head * wl.B * wl.H
    value = wl.B * wl.L / t_full
    cores = os.cpu_count()
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_full * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "L": wl.L, "d": 64},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "one head (all %d query rows) per step; full-workload "
                                       "time = per-head time x %d heads" % (wl.L, wl.B * wl.H)},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip FoX, decode and e2e legs")
    ap.add_argument("--no-sweep", action="store_true", help="skip the L sweep")
    ap.add_argument("--profile", choices=["fwd", "fox", "decode", "fox_decode", "producer", "bwd", "fwd_d128",
                                          "decode_d128", "fox_bwd", "bwd_d128", "fwd_f32"],
                    help="run only that operation on a reduced case (for ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.profile:
        run_profile_case(args)
        return
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import dependent_position_encoded_gb300 as pa
    pa.ensure_built() if rank == 0 else None
    barrier(world)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    wl = shard_workload(pi.BF16_L4096, rank)
    x = pi.workload_inputs(wl, device=dev)
    B, H, L = wl.B, wl.H, wl.L
    f_attn, f_corr, f_pre = fwd_flops(B, H, L)
    F = f_attn + f_corr + f_pre

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        total_ms, scan_ms, prep_ms = time_forward(pa, x, args.steps, args.warmup)
    barrier(world)
    torch.cuda.synchronize()
    clocks = clk.summary()
    t_max, ms_step, value = aggregate(total_ms, world, B, L, args.steps)

    scan_avg = statistics.mean(scan_ms)
    prep_avg = statistics.mean(prep_ms)
    achieved = (f_attn + f_corr) / (scan_avg * 1e-3) / 1e12
    roofline = {"kernel": "path_scan_tc_kernel", "bound": "tensor", "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"],
                "traffic": ncu_traffic("path_scan_tc_kernel"),
                "peak_source": "%s bf16 dense (burst)" % peaks["source"],
                "algorithmic_flops_per_launch": f_attn + f_corr,
                "executed_tensor_tflops": scan_executed_flops(B, H, L) / (scan_avg * 1e-3) / 1e12,
                "ms_per_launch": scan_avg}
    head = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": wl.name, "B": B, "H": H, "L": L, "d": 64,
                       "per_rank_batch": B, "global_batch": world * B,
                       "l2": "inputs 2.1 GB per step (> L2), no flush",
                       "parallelism": "dp%d (batch shards)" % world if world > 1 else "single"},
            "tflops": F / (ms_step * 1e-3) / 1e12 * world,
            "fa_equiv_tflops": f_attn / (ms_step * 1e-3) / 1e12 * world,
            "fwd_roofline_frac": F / (ms_step * 1e-3) / 1e12 / peaks["bf16_tflops"],
            "prepare_ms": prep_avg, "scan_ms": scan_avg,
            "roofline": roofline, "clocks": clocks,
            "gpu_launches": LAUNCHES_PER_FWD * args.steps}
    legs = {}    # secondary legs, printed before the headline legs
    tail = {}    # decode, PaTH-FoX and the L sweep: printed last

    if not args.no_extras:
        n_e2e = max(4, args.steps)
        e2e_ms, h2d, d2h = time_e2e(pa, x, n_e2e, 3)
        head["e2e"] = {"value": aggregate(e2e_ms, world, B, L, n_e2e)[2], "unit": "tokens/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                       "overlap": "copy-in, forward and read-back on three streams, "
                                  "double-buffered; every step moves its own bytes"}
        if rank == 0:
            head["parity"] = bench_parity(pa, x)
        del x
        torch.cuda.empty_cache()
        legs.update(run_legs(pa, peaks, dev, rank))
        tail.update(run_headline_legs(pa, peaks, dev, rank))

    if not args.no_sweep and rank == 0:
        sweep = {}
        for Ls in pi.SPEED_SWEEP_L:
            xs = pi.workload_inputs(pi.speed_shape(Ls), device=dev)
            tot, sc, pr = time_forward(pa, xs, 3, 3)
            a, c, p = fwd_flops(32, 32, Ls)
            sweep[str(Ls)] = {"ms": tot / 3, "tflops": (a + c + p) / (tot / 3 * 1e-3) / 1e12,
                              "frac": (a + c + p) / (tot / 3 * 1e-3) / 1e12 / peaks["bf16_tflops"],
                              "Mtok_s": 32 * Ls / (tot / 3 * 1e-3) / 1e6}
            del xs
            torch.cuda.empty_cache()
        tail["sweep_L"] = sweep

    if rank == 0 and not args.no_cpu_baseline:
        if not args.no_extras:
            for name, cb in leg_cpu_baselines(pi.BF16_L2048, pi.DECODE_32K, pi.PRODUCER_L4096,
                                              pi.FOX_L16384).items():
                target = tail if name in tail else legs
                if name in target:
                    target[name]["cpu_baseline"] = cb
        xc = pi.make_fwd_inputs(1, 64, wl.L, seed=wl.seed, device="cpu")
        head["cpu_baseline"] = cpu_baseline(xc, pi.FwdWorkload(wl.name, wl.B, wl.H, wl.L, 64,
                                                               wl.dtype, wl.seed, wl.clip, False))
    if rank == 0:
        line = dict(head)
        line.update(legs)
        line.update(tail)
        print(json.dumps(compact(order_line(line))))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
