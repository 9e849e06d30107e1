"""GPU parity of the projections ahead of the gate (kda_gate_proj) against the
fp64 oracle: gate_x = f_b (f_a x) and beta = sigmoid(b_proj x) per token.

Tolerance, per element: |got - ref| <= 2^-8 |ref| + 1e-3 rms(ref).  The outputs
are bf16, whose rounding alone moves a value by up to 2^-9 of itself; the fp32
accumulations (over D for f_a x and b_proj x, over R for f_b y with y kept as a
bf16 hi/lo pair, 2^-17 of itself) add errors near 1e-5 rms, which the floor
covers where the reference is close to zero.  A transposed operand, a wrong
tile offset or a dropped lo term of y (2^-9 of y in every term) fails it.
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
import oracle
from kimi_delta_attention_chunk_gb300 import synth
from tests.kda_testutil import rel_err

pytestmark = pytest.mark.gpu

CHAIN_TOL = 2e-2  # gate projections then the fused prefill, vs the oracle chain (see below)


def check(got, ref, what):
    g = got.detach().float().cpu().double().numpy()
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, (g.shape, ref.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3 * rms
    bad = np.abs(g - ref) > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements off, worst "
                           f"{float(np.max(np.abs(g - ref) - bound)):.3e} beyond the bound")


def run(inp, **kw):
    d = {k: v.cuda() for k, v in inp.items()}
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    gx, beta = kda.gate_proj(d["x"], d["f_a"], d["f_b"], d["b_proj"], status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return gx, beta


@pytest.mark.parametrize("B,T,D,R,HK,NH", [
    (1, 300, 512, 128, 512, 96),    # three 128-token tiles, the last one ragged (44 tokens)
    (2, 130, 256, 64, 256, 16),     # two sequences, rank 64, one 256-channel tile
    (1, 128, 64, 128, 768, 128),    # a single K stage; R + NH = 256, the widest tile
    (1, 1, 640, 128, 256, 32),      # one token
])
def test_gate_proj_matches_the_oracle(B, T, D, R, HK, NH):
    inp = synth.gate_proj_inputs(B, T, D, R, HK, NH, seed=1200 + T)
    gx, beta = run(inp)
    ref_gx, ref_beta = oracle.gate_proj(inp["x"], inp["f_a"], inp["f_b"], inp["b_proj"])
    check(gx, ref_gx, "gate_x")
    check(beta, ref_beta, "beta")


def test_gate_proj_full_size_on_sampled_tokens():
    # the model's shapes: D = 7168, rank 128, H*K = 96*128, 96 heads; 4096 tokens
    B, T, D, R, HK, NH = 1, 4096, 7168, 128, 12288, 96
    inp = synth.gate_proj_inputs(B, T, D, R, HK, NH, seed=1299)
    gx, beta = run(inp)
    rng = np.random.default_rng(7)
    rows = sorted(set([0, 1, 127, 128, 2047, 2048, 4095] + rng.choice(T, 25, replace=False).tolist()))
    ref_gx, ref_beta = oracle.gate_proj(inp["x"][0, rows], inp["f_a"], inp["f_b"], inp["b_proj"])
    check(gx[0, rows], ref_gx, "gate_x")
    check(beta[0, rows], ref_beta, "beta")


def test_gate_proj_feeds_the_fused_prefill():
    # gate_x [B,T,H*K] and beta [B,T,H] go straight into the fused prefill as its
    # gate input [B,T,H,K] and beta; the oracle chain is the same with both stored
    # in bf16 between the two steps, as the prefill's inputs are.  The two sides
    # round the intermediates to bf16 independently, and where an fp32 sum lies
    # next to a rounding boundary they pick neighbouring values: one ulp of a gate
    # input near 2 (2^-6) moves its decay e^g by up to 4% (dg/dx reaches e), which
    # moves state entries by a few 1e-3 of the rms.  Each step's own parity is
    # checked at its own tolerance (above; the prefill's in test_gpu_parity); this
    # test checks that the two compose (layouts, shapes), where a mistake is O(1).
    B, T, H, K, D, R = 1, 192, 16, 128, 256, 128
    pin = synth.prologue_inputs(T, H, K, K, torch.bfloat16, seed=1301)
    gin = synth.gate_proj_inputs(B, T, D, R, H * K, H, seed=1303)
    gx, beta = run(gin)
    d = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in pin.items()}
    o, sT = kda.chunk_fwd_fused(d["q_raw"], d["k_raw"], d["v_raw"], gx.view(B, T, H, K), beta, d["conv_w"],
                                d["A_log"], d["dt_bias"], scale=d["scale"], initial_state=d["initial_state"])
    torch.cuda.synchronize()
    gx_ref, beta_ref = oracle.gate_proj(gin["x"], gin["f_a"], gin["f_b"], gin["b_proj"])
    gx_ref = torch.from_numpy(gx_ref).to(torch.bfloat16).view(B, T, H, K)
    beta_ref = torch.from_numpy(beta_ref).to(torch.bfloat16)
    cw = pin["conv_w"]
    q, k, v, g = oracle.prologue(pin["q_raw"][0], pin["k_raw"][0], pin["v_raw"][0], gx_ref[0],
                                 (cw[0, :H * K], cw[1, :H * K], cw[2, :H * K]), pin["A_log"], pin["dt_bias"])
    o_ref, s_ref = oracle.kda_forward(q, k, v, g, beta_ref[0], scale=pin["scale"],
                                      initial_state=pin["initial_state"])
    eo, es = rel_err(o[0], o_ref), rel_err(sT, s_ref)
    assert eo <= CHAIN_TOL and es <= CHAIN_TOL, (eo, es)


def test_gate_proj_with_no_tokens():
    inp = synth.gate_proj_inputs(1, 0, 128, 128, 256, 16, seed=1302)
    gx, beta = run(inp)
    assert gx.shape == (1, 0, 256) and beta.shape == (1, 0, 16)
