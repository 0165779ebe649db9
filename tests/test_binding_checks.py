"""The Python binding's decode argument checks, on CPU tensors: every size or dtype
mismatch is raised before the library is called (the C entry points cannot see tensor
sizes, so a short buffer would otherwise be read or written out of bounds)."""
import pytest
import torch

import dependent_position_encoded_gb300 as pa

B, H, CAP, D = 2, 3, 40, 64


def _args(**kw):
    a = dict(q=torch.zeros(B, H, D, dtype=torch.bfloat16),
             k=torch.zeros(B, H, D, dtype=torch.bfloat16),
             v=torch.zeros(B, H, D, dtype=torch.bfloat16),
             w=torch.zeros(B, H, D, dtype=torch.bfloat16),
             beta=torch.zeros(B, H, dtype=torch.float32),
             k_cache=torch.zeros(B, H, CAP, D, dtype=torch.bfloat16),
             v_cache=torch.zeros(B, H, CAP, D, dtype=torch.bfloat16))
    a.update(kw)
    return a


ENTRY = [pa.path_decode_step, pa.path_decode_step_noalloc]


@pytest.mark.parametrize("fn", ENTRY)
@pytest.mark.parametrize("kw,exc", [
    (dict(v_cache=torch.zeros(B, H, CAP - 1, D, dtype=torch.bfloat16)), ValueError),
    (dict(q=torch.zeros(B, H, D - 1, dtype=torch.bfloat16)), ValueError),
    (dict(w=torch.zeros(B, H - 1, D, dtype=torch.bfloat16)), ValueError),
    (dict(beta=torch.zeros(B * H - 1, dtype=torch.float32)), ValueError),
    (dict(beta=torch.zeros(B, H, dtype=torch.bfloat16)), TypeError),
    (dict(k=torch.zeros(B, H, D, dtype=torch.float32)), TypeError),
    (dict(v_cache=torch.zeros(B, H, CAP, D, dtype=torch.float32)), TypeError),
    (dict(k_cache=torch.zeros(B, H, CAP * D, dtype=torch.bfloat16)), ValueError),
])
def test_decode_size_and_dtype_errors_raise_before_any_call(fn, kw, exc):
    a = _args(**kw)
    with pytest.raises(exc):
        fn(a["q"], a["k"], a["v"], a["w"], a["beta"], a["k_cache"], a["v_cache"], 5)


@pytest.mark.parametrize("fn", ENTRY)
def test_decode_out_is_checked(fn):
    a = _args()
    with pytest.raises(TypeError):
        fn(a["q"], a["k"], a["v"], a["w"], a["beta"], a["k_cache"], a["v_cache"], 5,
           out=torch.zeros(B, H, D, dtype=torch.float32))
    with pytest.raises(ValueError):
        fn(a["q"], a["k"], a["v"], a["w"], a["beta"], a["k_cache"], a["v_cache"], 5,
           out=torch.zeros(B, H, D - 8, dtype=torch.bfloat16))


def test_well_formed_cpu_tensors_still_need_a_gpu():
    # once every size matches, host tensors are refused as not being on a CUDA device
    a = _args()
    with pytest.raises(TypeError, match="CUDA"):
        pa.path_decode_step_noalloc(a["q"], a["k"], a["v"], a["w"], a["beta"], a["k_cache"],
                                    a["v_cache"], 5)
