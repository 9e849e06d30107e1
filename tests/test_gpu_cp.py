"""Context parallelism on one GPU against the oracle: the state composition
kernel, the segment transition (kda_chunk_fwd with v = 0 from the identity),
and a sequence cut into segments, each run independently, composed and rerun,
against the oracle's recurrence over the whole sequence."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
import oracle
from kimi_delta_attention_chunk_gb300 import cp, synth
from tests.kda_testutil import TOL_BF16, TOL_F32, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (128, 64)])
@pytest.mark.parametrize("mode", ["plain", "no_addend", "in_place"])
def test_state_compose(K, V, mode):
    g = torch.Generator().manual_seed(71)
    H = 5
    M = torch.randn(H, K, K, generator=g) / K ** 0.5
    S = torch.randn(H, K, V, generator=g)
    A = torch.randn(H, K, V, generator=g)
    ref = oracle.state_compose(M, S, None if mode == "no_addend" else A)
    Md, Sd, Ad = M.cuda(), S.cuda(), A.cuda()
    if mode == "plain":
        got = kda.state_compose(Md, Sd, Ad)
    elif mode == "no_addend":
        got = kda.state_compose(Md, Sd)
    else:
        got = kda.state_compose(Md, Sd, Ad, out=Ad)
    torch.cuda.synchronize()
    assert rel_err(got, ref) <= TOL_F32


@pytest.mark.parametrize("T,gscale", [(150, 0.01), (20, 1.0)])
def test_segment_transition_matches_the_product_of_factors(T, gscale):
    # (with the workloads' gates a long segment forgets its start entirely, M
    # underflows to zero; weak gates or a short segment keep M of order one)
    d = synth.direct_inputs(T, 2, 128, 128, torch.bfloat16, seed=72)
    g = (d["g"].float() * gscale).to(torch.bfloat16)
    M = cp.segment_transition(d["k"].cuda(), g.cuda(), d["beta"].cuda())
    torch.cuda.synchronize()
    ref = oracle.segment_transition(d["k"][0], g[0], d["beta"][0])
    assert rel_err(M[0], ref) <= TOL_BF16


@pytest.mark.parametrize("bounds", [[64], [200, 450], [1, 333, 334, 640]])
@pytest.mark.parametrize("gscale", [1.0, 0.01])
def test_segmented_prefill_equals_the_whole_sequence(bounds, gscale):
    d = synth.direct_inputs(700, 3, 128, 128, torch.bfloat16, seed=73, init_state=True)
    d["g"] = (d["g"].float() * gscale).to(torch.bfloat16)  # weak gates: long memories across segments
    dd = to_dev(d)
    o, sT = cp.chunk_fwd_segmented(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], bounds, scale=d["scale"],
                                   initial_state=dd["initial_state"])
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.kda_forward(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                                      initial_state=d["initial_state"])
    eo, es = rel_err(o, o_ref), rel_err(sT, s_ref)
    assert eo <= TOL_BF16 and es <= TOL_BF16, f"o err {eo:.3e}, state err {es:.3e}"
