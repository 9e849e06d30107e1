"""kda_output_gate against the oracle: out = o / sqrt(mean(o^2) + eps) * w *
sigmoid(gate) per (token, head) row, element by element, through the C ABI."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
import oracle
from kimi_delta_attention_chunk_gb300 import synth
from tests.kda_testutil import TOL_F32, rel_err

pytestmark = pytest.mark.gpu


def run(shape, gdt, odt, with_weight, seed, eps=1e-6, in_place=False):
    d = synth.output_gate_inputs(shape, gdt, seed)
    w = d["weight"] if with_weight else None
    ref = oracle.output_gate(d["o"], d["gate"], w, eps=eps)
    o = d["o"].cuda()
    out = o if in_place else None
    got = kda.output_gate(o, d["gate"].cuda(), None if w is None else w.cuda(), eps=eps, out_dtype=odt, out=out)
    torch.cuda.synchronize()
    return got, ref


def check(got, ref, odt):
    if odt == torch.float32:
        e = rel_err(got, ref)
        assert e <= TOL_F32, f"err {e:.3e}"
    else:
        # one rounding to bf16 of a value within fp32 error of the exact one
        x = got.cpu().double().numpy()
        rms = float(np.sqrt(np.mean(ref * ref)))
        bad = np.abs(x - ref) > 2.0 ** -8 * np.abs(ref) + 1e-6 * rms
        assert not bad.any(), f"{int(bad.sum())} values off by more than a bf16 rounding"


@pytest.mark.parametrize("V", [64, 128])
@pytest.mark.parametrize("gdt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("odt", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("with_weight", [True, False])
def test_small_shapes(V, gdt, odt, with_weight):
    got, ref = run((2, 37, 3, V), gdt, odt, with_weight, seed=501)
    check(got, ref, odt)


def test_in_place_and_decode_layout():
    got, ref = run((256, 96, 128), torch.bfloat16, torch.float32, True, seed=502, in_place=True)
    check(got, ref, torch.float32)


def test_eps_dominates_tiny_rows():
    # rows of magnitude ~1e-4 with eps = 1e-2: the output scales with o / sqrt(eps)
    d = synth.output_gate_inputs((1, 16, 2, 128), torch.float32, 503)
    o = d["o"] * 1e-4
    ref = oracle.output_gate(o, d["gate"], d["weight"], eps=1e-2)
    got = kda.output_gate(o.cuda(), d["gate"].cuda(), d["weight"].cuda(), eps=1e-2)
    torch.cuda.synchronize()
    assert rel_err(got, ref) <= TOL_F32


def test_empty_is_a_no_op():
    o = torch.empty((1, 0, 96, 128), device="cuda")
    out = kda.output_gate(o, torch.empty_like(o, dtype=torch.bfloat16))
    assert out.shape == o.shape


def test_prefill_size():
    # the 4096-token, 96-head workload: every element
    got, ref = run((1, 4096, 96, 128), torch.bfloat16, torch.float32, True, seed=504)
    check(got, ref, torch.float32)
