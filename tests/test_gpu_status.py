"""Device-side failures reported through the caller's status word, without
any GPU fault: a bounded wait inside the prefill's kernels that gives up (a
testing hook makes it wait on an mbarrier that nothing arrives on, with a short
poll limit), and a backward call whose
malformed offsets make it skip a sequence.  After either, the context stays
usable and a normal call matches the oracle."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
import oracle
from kimi_delta_attention_chunk_gb300 import synth
from tests.kda_testutil import TOL_BF16, TOL_F32, rel_err, to_dev

pytestmark = pytest.mark.gpu

KDA_OK, KDA_ERR_RANGE, KDA_ERR_TIMEOUT = 0, 5, 6


def status_word(fill=-1):
    return torch.full((1,), fill, dtype=torch.int32, device="cuda")


def prefill(d, status, fused=False):
    if fused:
        return kda.chunk_fwd_fused(d["q_raw"], d["k_raw"], d["v_raw"], d["gate_x"], d["beta"], d["conv_w"],
                                   d["A_log"], d["dt_bias"], scale=d["scale"], initial_state=d["initial_state"],
                                   cu_seqlens=d["cu_seqlens"], status=status)
    return kda.chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"],
                         initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"], status=status)


def test_status_word_reads_ok_after_a_normal_call():
    d = to_dev(synth.direct_inputs(200, 3, 128, 128, torch.bfloat16, seed=70, init_state=True))
    st = status_word()
    prefill(d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == KDA_OK
    # the CUDA-core path sets it too
    d = to_dev(synth.direct_inputs(100, 2, 64, 64, torch.float32, seed=72))
    st = status_word()
    prefill(d, st)
    torch.cuda.synchronize()
    assert int(st.item()) == KDA_OK


@pytest.mark.parametrize("kernel", [1, 2])
@pytest.mark.parametrize("fused", [False, True])
def test_a_wait_that_gives_up_reports_timeout_and_the_context_stays_usable(fused, kernel):
    """kernel 1: every CTA of the chunk-local kernel, kernel 2: the state
    kernel's MMA issuer, first waits on an mbarrier that nothing arrives on."""
    if fused:
        inp = synth.prologue_inputs(0, 4, 128, 128, torch.bfloat16, seed=73, lengths=[300, 212])
    else:
        inp = synth.direct_inputs(512, 8, 128, 128, torch.bfloat16, seed=71, init_state=True)
    d = to_dev(inp)
    st = status_word()
    kda.set_wait_limit(2000)   # a short limit, so that the injected wait gives up quickly
    kda.inject_wait_timeout(kernel)
    try:
        prefill(d, st, fused)
        torch.cuda.synchronize()
    finally:
        kda.set_wait_limit(0)
        kda.inject_wait_timeout(0)
    assert int(st.item()) == KDA_ERR_TIMEOUT
    # the kernels exited cleanly: the same call with the default limit succeeds
    st = status_word()
    o, s = prefill(d, st, fused)
    torch.cuda.synchronize()
    assert int(st.item()) == KDA_OK
    if fused:
        cw, H = inp["conv_w"], 4
        q, k, v, g = oracle.prologue(inp["q_raw"][0], inp["k_raw"][0], inp["v_raw"][0], inp["gate_x"][0],
                                     (cw[0, :H * 128], cw[1, :H * 128], cw[2, :H * 128]), inp["A_log"],
                                     inp["dt_bias"], cu_seqlens=inp["cu_seqlens"])
        o_ref, s_ref = oracle.kda_forward(q, k, v, g, inp["beta"][0], scale=inp["scale"],
                                          initial_state=inp["initial_state"], cu_seqlens=inp["cu_seqlens"])
        o = o[0]
    else:
        o_ref, s_ref = oracle.kda_forward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], scale=inp["scale"],
                                          initial_state=inp["initial_state"])
    assert rel_err(o, o_ref) <= TOL_BF16 and rel_err(s, s_ref) <= TOL_BF16


def test_backward_skipping_a_malformed_sequence_reports_range():
    # offsets [0, 640, 0, 640]: the third sequence covers the first one's tokens
    # again, so the chains need more checkpoints than the workspace holds; that
    # sequence is skipped (NaN gradients, status KDA_ERR_RANGE), every access
    # stays in bounds, and the first sequence's dS0 is still exact
    T, H, K, V = 640, 2, 64, 64
    inp = synth.direct_inputs(T, H, K, V, torch.float32, seed=74, init_state=False)
    d = to_dev(inp)
    cu = torch.tensor([0, 640, 0, 640], dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(75)
    dO = torch.from_numpy(rng.standard_normal((1, T, H, V)).astype(np.float32))
    st = status_word()
    g = kda.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], dO.cuda(), scale=d["scale"], cu_seqlens=cu,
                      status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == KDA_ERR_RANGE
    dS0 = g["dS0"].cpu()
    assert torch.isnan(dS0[2]).all()
    ref = oracle.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dO, scale=inp["scale"])
    assert rel_err(dS0[0:1], ref["dS0"]) <= TOL_F32
    # a well-formed call afterwards reads OK
    st = status_word()
    kda.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], dO.cuda(), scale=d["scale"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == KDA_OK


@pytest.mark.parametrize("kernel", [3, 4])
def test_backward_wait_that_gives_up_reports_timeout_and_the_context_stays_usable(kernel):
    """kernel 3: the chunked backward's chain kernel, kernel 4: its chunk kernel,
    first waits (in every CTA) on an mbarrier that nothing arrives on."""
    T, H = 200, 3
    inp = synth.direct_inputs(T, H, 128, 128, torch.bfloat16, seed=76, init_state=True)
    d = to_dev(inp)
    rng = np.random.default_rng(77)
    dO = torch.from_numpy(rng.standard_normal((1, T, H, 128)).astype(np.float32))
    st = status_word()
    kda.set_wait_limit(2000)
    kda.inject_wait_timeout(kernel)
    try:
        kda.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], dO.cuda(), scale=d["scale"],
                      initial_state=d["initial_state"], status=st)
        torch.cuda.synchronize()
    finally:
        kda.set_wait_limit(0)
        kda.inject_wait_timeout(0)
    assert int(st.item()) == KDA_ERR_TIMEOUT
    # the kernels exited cleanly: the same call with the default limit succeeds
    st = status_word()
    got = kda.chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], dO.cuda(), scale=d["scale"],
                        initial_state=d["initial_state"], status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == KDA_OK
    ref = oracle.kda_backward(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], dO, scale=inp["scale"],
                              initial_state=inp["initial_state"])
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dS0"):
        assert rel_err(got[key], ref[key]) <= TOL_BF16, key
