"""kda_check_range on the device: the log-decay precondition g in [-5, 0] is
reported through the caller's status word (KDA_ERR_RANGE), in agreement with
numpy's element test, for bf16 and fp32, ragged counts and NaN."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
from kimi_delta_attention_chunk_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_workload_gates_pass(dtype):
    d = synth.direct_inputs(333, 3, 128, 128, dtype, seed=81)
    kda.check_range(d["g"].cuda())  # raises on a violation


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("where,value", [(0, 0.5), (-1, -5.5), (12345, float("nan")), (777, -5.0), (778, 0.0)])
def test_single_element_decides(dtype, where, value):
    g = torch.full((1, 131, 3, 128), -1.0, dtype=dtype)
    g.view(-1)[where] = value
    expect_bad = not (-5.0 <= float(g.view(-1)[where]) <= 0.0)
    st = kda.check_range(g.cuda(), sync=False)
    torch.cuda.synchronize()
    assert int(st.item()) == (5 if expect_bad else 0)
    assert bool(np.any(~((g.float().numpy() >= -5.0) & (g.float().numpy() <= 0.0)))) == expect_bad
    if expect_bad:
        with pytest.raises(kda.KDAError) as err:
            kda.check_range(g.cuda())
        assert err.value.status == 5


def test_empty_and_custom_bounds():
    st = kda.check_range(torch.empty(0, device="cuda"), sync=False)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    x = torch.linspace(-1.0, 1.0, 1001, device="cuda")
    kda.check_range(x, lo=-1.0, hi=1.0)
    with pytest.raises(kda.KDAError):
        kda.check_range(x, lo=-0.5, hi=1.0)
