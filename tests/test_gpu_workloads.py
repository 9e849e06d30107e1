"""Full-size workloads, in the launch configuration bench.py times, checked
against the fp64 oracle on sampled heads (or sampled (sequence, head) pairs for
decode): every KDA chain is independent, so a sampled chain's outputs and final
state are exactly what the oracle computes for that chain alone.

Workloads: 4096-token prefill (96 heads); 16-sequence varlen prefill (lengths
512..8192, packed by cu_seqlens, nonzero initial states); 256-sequence decode
over 64 steps; 65536-token prefill with the fused prologue.  bf16 inputs, fp32
state and output, tolerance 2e-3 of the reference RMS.
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
import oracle
from kimi_delta_attention_chunk_gb300 import synth
from tests.kda_testutil import TOL_BF16, rel_err, to_dev

pytestmark = pytest.mark.gpu


def _sub_heads(inp, heads):
    out = {}
    for key in ("q", "k", "v", "g", "beta"):
        out[key] = inp[key][:, :, heads]
    s0 = inp["initial_state"]
    out["initial_state"] = s0[:, heads] if s0 is not None else None
    return out


def test_prefill_4096_tokens_96_heads():
    w = synth.WORKLOADS["prefill"]
    inp = synth.workload_inputs("prefill")
    d = to_dev(inp)
    o, sT = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"])
    torch.cuda.synchronize()
    assert torch.isfinite(o).all()
    heads = [0, 37, 95]
    s = _sub_heads(inp, heads)
    o_ref, s_ref = oracle.kda_forward(s["q"], s["k"], s["v"], s["g"], s["beta"], scale=inp["scale"])
    assert o.shape == (1, w.T, w.H, w.V)
    eo = rel_err(o[:, :, heads].cpu(), o_ref)
    es = rel_err(sT[:, heads].cpu(), s_ref)
    assert eo <= TOL_BF16 and es <= TOL_BF16, (eo, es)


def test_prefill_512_tokens_every_one_of_96_heads():
    """Every head of a 96-head prefill against the oracle, element by element:
    the persistent chunk-local kernel hands (chunk, head) tasks to CTAs by
    chunk * H + h, so a mapping fault confined to some heads would show here
    (8 chunks x 96 heads = 768 tasks: every CTA runs several)."""
    inp = synth.direct_inputs(512, 96, 128, 128, torch.bfloat16, seed=11, init_state=True)
    d = to_dev(inp)
    st = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    o, sT = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                          initial_state=d["initial_state"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    o_ref, s_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=inp["scale"],
                                      initial_state=inp["initial_state"])
    for h in range(96):
        eo = rel_err(o[:, :, h].cpu(), o_ref[:, :, h])
        es = rel_err(sT[:, h].cpu(), s_ref[:, h])
        assert eo <= TOL_BF16 and es <= TOL_BF16, (h, eo, es)


def test_varlen_16_sequences():
    inp = synth.workload_inputs("varlen")
    d = to_dev(inp)
    o, sT = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                          initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"])
    torch.cuda.synchronize()
    heads = [5, 60]
    s = _sub_heads(inp, heads)
    o_ref, s_ref = oracle.kda_forward(s["q"], s["k"], s["v"], s["g"], s["beta"], scale=inp["scale"],
                                      initial_state=s["initial_state"], cu_seqlens=inp["cu_seqlens"])
    eo = rel_err(o[:, :, heads].cpu(), o_ref)
    es = rel_err(sT[:, heads].cpu(), s_ref)
    assert eo <= TOL_BF16 and es <= TOL_BF16, (eo, es)
    # every token of every sequence was written and is finite
    assert torch.isfinite(o).all()


def test_decode_256_sequences_64_steps():
    w = synth.WORKLOADS["decode"]
    inp = synth.workload_inputs("decode")
    d = to_dev(inp)
    state = d["state"].clone()
    outs = []
    for s in range(w.decode_steps):
        outs.append(kda.recurrent_step(d["q"][s], d["k"][s], d["v"][s], d["g"][s], d["beta"][s], state,
                                       scale=inp["scale"]))
    o = torch.stack(outs, dim=1)  # [N, steps, H, V]
    torch.cuda.synchronize()
    seqs, heads = [0, 131, 255], [0, 50, 95]
    tr = lambda x: x[:, seqs][:, :, heads].transpose(0, 1).contiguous()  # noqa: E731  [N_s, steps, H_s, D]
    s0 = inp["state"][seqs][:, heads]
    o_ref, s_ref = oracle.kda_forward(tr(inp["q"]), tr(inp["k"]), tr(inp["v"]), tr(inp["g"]), tr(inp["beta"]),
                                      scale=inp["scale"], initial_state=s0)
    eo = rel_err(o[seqs][:, :, heads].cpu(), o_ref)
    es = rel_err(state[seqs][:, heads].cpu(), s_ref)
    assert eo <= TOL_BF16 and es <= TOL_BF16, (eo, es)


def test_long_prefill_with_fused_prologue():
    w = synth.WORKLOADS["long"]
    inp = synth.workload_inputs("long")
    d = to_dev(inp)
    o, sT = kda.chunk_fwd_fused(d["q_raw"], d["k_raw"], d["v_raw"], d["gate_x"], d["beta"], d["conv_w"],
                                d["A_log"], d["dt_bias"], scale=d["scale"], initial_state=d["initial_state"])
    torch.cuda.synchronize()
    H, K, V = w.H, w.K, w.V
    heads = [3, 90]
    cw = inp["conv_w"]
    rows = lambda D: np.concatenate([np.arange(h * D, (h + 1) * D) for h in heads])  # noqa: E731
    sl = lambda x: x[0][:, heads].contiguous()  # noqa: E731
    q, k, v, g = oracle.prologue(sl(inp["q_raw"]), sl(inp["k_raw"]), sl(inp["v_raw"]), sl(inp["gate_x"]),
                                 (cw[0][rows(K)], cw[1][rows(K)], cw[2][rows(V)]), inp["A_log"],
                                 inp["dt_bias"][rows(K)])
    o_ref, s_ref = oracle.kda_forward(q, k, v, g, sl(inp["beta"]), scale=inp["scale"],
                                      initial_state=inp["initial_state"][:, heads])
    eo = rel_err(o[0][:, heads].cpu(), o_ref)
    es = rel_err(sT[:, heads].cpu(), s_ref)
    assert eo <= TOL_BF16 and es <= TOL_BF16, (eo, es)
