"""GPU parity: libkda.so (through its C ABI) against the fp64 CPU oracle.

Every input comes from the seeded generators in
kimi_delta_attention_chunk_gb300.synth; the oracle sees the exact values the
GPU sees.  Metric: max|x - x_ref| / rms(x_ref) per output tensor, <= 2e-3 for
bf16 inputs (fp32 state, fp32 output) and <= 1e-5 for fp32 inputs.
"""
import numpy as np
import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
import oracle
from kimi_delta_attention_chunk_gb300 import synth
from tests.kda_testutil import rel_err, to_dev, tol_for

pytestmark = pytest.mark.gpu


def run_chunk(inp, **kw):
    d = to_dev(inp)
    o, sT = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                          initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"], **kw)
    torch.cuda.synchronize()
    return o.cpu(), sT.cpu()


def run_oracle(inp, heads=None):
    q, k, v, g, b, s0 = (inp[n] for n in ("q", "k", "v", "g", "beta", "initial_state"))
    if heads is not None:
        q, k, v, g, b = (x[:, :, heads] for x in (q, k, v, g, b))
        s0 = s0[:, heads] if s0 is not None else None
    return oracle.kda_forward(q, k, v, g, b, scale=inp["scale"], initial_state=s0,
                              cu_seqlens=inp["cu_seqlens"])


def check(o, sT, o_ref, s_ref, dtype, heads=None):
    if heads is not None:
        o, sT = o[:, :, heads], sT[:, heads]
    tol = tol_for(dtype)
    eo, es = rel_err(o, o_ref), rel_err(sT, s_ref)
    assert eo <= tol and es <= tol, f"o err {eo:.3e}, state err {es:.3e}, tol {tol:.0e}"
    return eo, es


# ------------------------------------------------------------------ small cases
def test_tiny_fp32_workload():
    w = synth.WORKLOADS["tiny"]
    inp = synth.direct_inputs(w.T, w.H, w.K, w.V, w.dtype, w.seed)
    o, sT = run_chunk(inp)
    o_ref, s_ref = run_oracle(inp)
    check(o, sT, o_ref, s_ref, torch.float32)


@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (128, 64), (64, 128)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_ragged_tail_and_initial_state(K, V, dtype):
    # 5 full chunks and a 13-token tail; 3 heads; nonzero initial state
    inp = synth.direct_inputs(333, 3, K, V, dtype, seed=100 + K + V, B=2, init_state=True)
    o, sT = run_chunk(inp)
    o_ref, s_ref = run_oracle(inp)
    check(o, sT, o_ref, s_ref, dtype)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_varlen_edge_lengths(dtype):
    lengths = [1, 0, 63, 64, 65, 200, 2, 128]
    inp = synth.direct_inputs(0, 4, 128, 128, dtype, seed=7, lengths=lengths, init_state=True)
    o, sT = run_chunk(inp)
    o_ref, s_ref = run_oracle(inp)
    check(o, sT, o_ref, s_ref, dtype)
    # the empty sequence returns its initial state unchanged
    torch.testing.assert_close(sT[1], inp["initial_state"][1], rtol=0, atol=0)


def test_varlen_equals_separate_sequences():
    lengths = [70, 5, 130]
    inp = synth.direct_inputs(0, 2, 128, 128, torch.bfloat16, seed=8, lengths=lengths, init_state=True)
    o, sT = run_chunk(inp)
    cu = inp["cu_seqlens"].tolist()
    for n in range(len(lengths)):
        sub = {key: inp[key][:, cu[n]:cu[n + 1]] for key in ("q", "k", "v", "g", "beta")}
        sub.update(scale=inp["scale"], cu_seqlens=None, initial_state=inp["initial_state"][n:n + 1])
        on, sn = run_chunk(sub)
        torch.testing.assert_close(on, o[:, cu[n]:cu[n + 1]], rtol=0, atol=0)
        torch.testing.assert_close(sn[0], sT[n], rtol=0, atol=0)


def test_split_prefill_hands_off_state():
    inp = synth.direct_inputs(256, 2, 128, 128, torch.bfloat16, seed=9, init_state=True)
    o, sT = run_chunk(inp)
    cut = 100
    first = {key: inp[key][:, :cut].contiguous() for key in ("q", "k", "v", "g", "beta")}
    first.update(scale=inp["scale"], cu_seqlens=None, initial_state=inp["initial_state"])
    o1, s1 = run_chunk(first)
    second = {key: inp[key][:, cut:].contiguous() for key in ("q", "k", "v", "g", "beta")}
    second.update(scale=inp["scale"], cu_seqlens=None, initial_state=s1)
    o2, s2 = run_chunk(second)
    o_ref, s_ref = run_oracle(inp)
    assert rel_err(torch.cat([o1, o2], dim=1), o_ref) <= 2e-3
    assert rel_err(s2, s_ref) <= 2e-3


def test_in_place_state_update_and_bf16_output():
    inp = synth.direct_inputs(150, 2, 128, 128, torch.bfloat16, seed=10, init_state=True)
    d = to_dev(inp)
    state = d["initial_state"].clone()
    o, sT = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=state,
                          final_state=state, o_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert sT.data_ptr() == state.data_ptr() and o.dtype == torch.bfloat16
    o_ref, s_ref = run_oracle(inp)
    assert rel_err(state.cpu(), s_ref) <= 2e-3
    # o rounded to bf16: each element within half a bf16 ulp (2^-9 relative) plus the fp32-output bar
    ob = o.float().cpu().double().numpy()
    rms = np.sqrt(np.mean(o_ref ** 2))
    assert np.all(np.abs(ob - o_ref) <= np.abs(o_ref) * 2.0 ** -8 + 2e-3 * rms)


def test_empty_inputs():
    d = to_dev(synth.direct_inputs(0, 2, 64, 64, torch.bfloat16, seed=11, init_state=True))
    o, sT = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["initial_state"])
    torch.cuda.synchronize()
    assert o.numel() == 0
    torch.testing.assert_close(sT, d["initial_state"], rtol=0, atol=0)


def test_gate_at_lower_bound():
    """g = -5 everywhere: the in-chunk decay reaches e^-320; nothing overflows."""
    inp = synth.direct_inputs(200, 2, 128, 128, torch.bfloat16, seed=12, init_state=True)
    inp["g"] = torch.full_like(inp["g"], -5.0)
    o, sT = run_chunk(inp)
    assert torch.isfinite(o).all() and torch.isfinite(sT).all()
    o_ref, s_ref = run_oracle(inp)
    check(o, sT, o_ref, s_ref, torch.bfloat16)


# ------------------------------------------------------------------ fused prologue
# bf16 with K = V = 128 runs the prologue inside the tensor-core chunk-local
# kernel; the other combinations run the CUDA-core kernel's prologue.
@pytest.mark.parametrize("dtype,K,V", [(torch.bfloat16, 128, 128), (torch.float32, 128, 128),
                                       (torch.bfloat16, 64, 64)])
@pytest.mark.parametrize("act", [0, 1])
def test_fused_prologue_small(act, dtype, K, V):
    lengths = [5, 64, 131, 1, 70]
    H = 3
    inp = synth.prologue_inputs(0, H, K, V, dtype, seed=13 + K + act, lengths=lengths)
    d = to_dev(inp)
    o, sT = kda.chunk_fwd_fused(d["q_raw"], d["k_raw"], d["v_raw"], d["gate_x"], d["beta"], d["conv_w"],
                                d["A_log"], d["dt_bias"], scale=d["scale"], initial_state=d["initial_state"],
                                cu_seqlens=d["cu_seqlens"], conv_act=act)
    torch.cuda.synchronize()
    cw = inp["conv_w"]
    q, k, v, g = oracle.prologue(inp["q_raw"][0], inp["k_raw"][0], inp["v_raw"][0], inp["gate_x"][0],
                                 (cw[0, :H * K], cw[1, :H * K], cw[2, :H * V]), inp["A_log"], inp["dt_bias"],
                                 cu_seqlens=inp["cu_seqlens"], act=act)
    o_ref, s_ref = oracle.kda_forward(q, k, v, g, inp["beta"][0], scale=inp["scale"],
                                      initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"])
    check(o.cpu()[0], sT.cpu(), o_ref, s_ref, dtype)


# ------------------------------------------------------------------ decode
@pytest.mark.parametrize("K,V", [(128, 128), (64, 64), (128, 64)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_steps_small(K, V, dtype):
    steps, N, H = 5, 7, 3
    inp = synth.decode_inputs(N, H, K, V, steps, dtype, seed=14)
    d = to_dev(inp)
    state = d["state"].clone()
    outs = []
    # unaligned beta rows are fine: beta needs only element alignment
    for s in range(steps):
        outs.append(kda.recurrent_step(d["q"][s], d["k"][s], d["v"][s], d["g"][s], d["beta"][s], state,
                                       scale=inp["scale"]).cpu())
    torch.cuda.synchronize()
    # the oracle sees each sequence as `steps` tokens: [N, steps, H, D]
    tr = lambda x: x.transpose(0, 1).contiguous()  # noqa: E731
    o_ref, s_ref = oracle.kda_forward(tr(inp["q"]), tr(inp["k"]), tr(inp["v"]), tr(inp["g"]), tr(inp["beta"]),
                                      scale=inp["scale"], initial_state=inp["state"])
    o = torch.stack(outs, dim=1)
    tol = tol_for(dtype)
    assert rel_err(o, o_ref) <= tol and rel_err(state.cpu(), s_ref) <= tol


def test_decode_equals_prefill():
    """T decode steps from a state == one prefill over the same T tokens."""
    T, H = 40, 2
    inp = synth.direct_inputs(T, H, 128, 128, torch.bfloat16, seed=15, B=3, init_state=True)
    d = to_dev(inp)
    o_p, s_p = kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], initial_state=d["initial_state"])
    state = d["initial_state"].clone()
    o_d = torch.stack([kda.recurrent_step(d["q"][:, t].contiguous(), d["k"][:, t].contiguous(),
                                          d["v"][:, t].contiguous(), d["g"][:, t].contiguous(),
                                          d["beta"][:, t].contiguous(), state) for t in range(T)], dim=1)
    torch.cuda.synchronize()
    assert rel_err(o_d.cpu(), o_p.cpu().double().numpy()) <= 1e-3
    assert rel_err(state.cpu(), s_p.cpu().double().numpy()) <= 1e-3


# ------------------------------------------------------------------ timing hook
def test_trace_events_bracket_the_two_kernels():
    inp = synth.direct_inputs(300, 4, 128, 128, torch.bfloat16, seed=21)
    d = to_dev(inp)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    kda.trace_events(*ev)
    kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"])
    torch.cuda.synchronize()
    t_local, t_state = ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])
    assert t_local > 0 and t_state > 0
    # the setting is consumed by that call: the next call records nothing new
    before = ev[2].query()
    kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"])
    torch.cuda.synchronize()
    assert before and ev[0].elapsed_time(ev[2]) == pytest.approx(t_local + t_state, rel=1e-3, abs=1e-3)
