"""The seeded input generator: determinism, shapes and the stated distributions."""
import torch

import path_inputs as pi


def test_seeded_and_deterministic():
    a = pi.make_fwd_inputs(2, 3, 70, seed=5, fox=True)
    b = pi.make_fwd_inputs(2, 3, 70, seed=5, fox=True)
    for key in a:
        assert torch.equal(a[key], b[key])
    c = pi.make_fwd_inputs(2, 3, 70, seed=6, fox=True)
    assert not torch.equal(a["q"], c["q"])


def test_distributions_and_dtypes():
    x = pi.make_fwd_inputs(4, 4, 512, seed=1, fox=True)
    assert x["q"].dtype == torch.bfloat16 and x["beta"].dtype == torch.float32
    assert x["q"].shape == (4, 4, 512, 64) and x["beta"].shape == (4, 4, 512)
    norms = x["w"].float().norm(dim=-1)
    assert torch.all((norms - 1).abs() < 1e-2)  # unit in fp32, then rounded to bf16
    assert float(x["beta"].min()) > 0 and float(x["beta"].max()) <= pi.BETA_CLIP
    assert float(x["log_f"].max()) < 0
    q = x["q"].float()
    assert abs(float(q.mean())) < 0.02 and abs(float(q.std()) - 1) < 0.02
    # log f = logsigmoid(N(2, 1)): mean about -0.17
    assert -0.25 < float(x["log_f"].mean()) < -0.1


def test_unclipped_tiny_workload():
    x = pi.workload_inputs(pi.TINY_FP32)
    assert x["q"].dtype == torch.float32 and x["q"].shape == (1, 2, 128, 64)
    assert "log_f" not in x


def test_decode_inputs():
    wl = pi.DECODE_32K
    small = pi.DecodeWorkload("t", 2, 2, 100, 3, 64, torch.bfloat16, 5, 1000)
    kc, vc = pi.make_decode_prefix(small, cap=110)
    assert kc.shape == (2, 2, 110, 64) and torch.all(kc[:, :, 100:] == 0)
    s0 = pi.make_decode_step(small, 0)
    assert s0["q"].shape == (2, 2, 1, 64) and s0["beta"].shape == (2, 2, 1)
    assert wl.n_prefix == 32768 and wl.steps == 64


def test_sample_rows_in_range():
    r = pi.sample_rows(10, 300, 50, seed=3)
    assert r.shape[1] == 2 and r[:, 0].max() < 10 and r[:, 1].max() < 300
    assert 0 in r[:, 1] and 299 in r[:, 1]


def test_fox_decode_prefix_gate_sums():
    wl = pi.DecodeWorkload("t", 2, 3, 50, 1, 64, torch.bfloat16, 7, 100)
    kc, vc = pi.make_decode_prefix(wl, 60)
    kf, vf, gc = pi.make_fox_decode_prefix(wl, 60)
    # same key/value draws as the plain decode cache
    assert torch.equal(kc, kf) and torch.equal(vc, vf)
    assert gc.dtype == torch.float32 and gc.shape == (2, 3, 60)
    # the last cached key carries no gate, earlier keys ever more negative sums, and the
    # slots past the prefix are zero
    assert torch.all(gc[:, :, 49:] == 0)
    step = gc[:, :, :48] - gc[:, :, 1:49]
    assert torch.all(step < 0) and torch.all(step > -10)
