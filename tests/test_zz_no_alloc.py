"""kda_chunk_fwd_noalloc: the prefill for callers that cannot allocate device
memory while they run (a serving process that reserved all free HBM for its own
state pool, a runtime whose memory belongs to its own allocator).

The entry point keeps its workspace in a fixed 64 MiB device array instead of
a workspace the caller provides.  Its results must match the fp64 oracle within
the bf16 tolerance, and match kda_chunk_fwd (the existing entry point) within
the same tolerance, also on a second call that finds the previous call's data
in the array; a call that needs more scratch than the array holds must be
rejected before anything runs.  (This file is collected last so that a run
stopping at the first failure has run every other test already.)
"""
import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
import oracle
from kimi_delta_attention_chunk_gb300 import synth
from tests.kda_testutil import TOL_BF16, rel_err, to_dev

pytestmark = pytest.mark.gpu


def both(d):
    args = (d["q"], d["k"], d["v"], d["g"], d["beta"])
    kw = dict(scale=d["scale"], initial_state=d["initial_state"], cu_seqlens=d["cu_seqlens"])
    o_ref, s_ref = kda.chunk_fwd(*args, **kw)
    o, s = kda.chunk_fwd_noalloc(*args, **kw)
    torch.cuda.synchronize()
    return (o, s), (o_ref, s_ref)


def oracle_of(inp, heads=None):
    q, k, v, g, b, s0 = (inp[n] for n in ("q", "k", "v", "g", "beta", "initial_state"))
    if heads is not None:
        q, k, v, g, b = (x[:, :, heads] for x in (q, k, v, g, b))
        s0 = s0[:, heads] if s0 is not None else None
    return oracle.kda_forward(q, k, v, g, b, scale=inp["scale"], initial_state=s0, cu_seqlens=inp["cu_seqlens"])


def assert_close(got, ref, exact, heads=None):
    (o, s), (o_ref, s_ref) = got, ref
    # against the existing entry point
    eo = rel_err(o, o_ref.cpu().double().numpy())
    es = rel_err(s, s_ref.cpu().double().numpy())
    assert eo <= TOL_BF16 and es <= TOL_BF16, f"vs kda_chunk_fwd: o err {eo:.3e}, state err {es:.3e}"
    # against the oracle
    if heads is not None:
        o, s = o[:, :, heads], s[:, heads]
    eo = rel_err(o, exact[0])
    es = rel_err(s, exact[1])
    assert eo <= TOL_BF16 and es <= TOL_BF16, f"vs the oracle: o err {eo:.3e}, state err {es:.3e}"


def test_noalloc_matches_the_oracle_and_chunk_fwd_on_two_calls_in_a_row():
    # call 1: two dense sequences with a ragged tail and an initial state
    inp1 = synth.direct_inputs(333, 3, 128, 128, torch.bfloat16, seed=901, B=2, init_state=True)
    assert_close(*both(to_dev(inp1)), oracle_of(inp1))
    # call 2: packed sequences (chunk bookkeeping in the array too), after call 1
    # left its data in the array
    lengths = [1, 64, 100, 0, 250]
    inp2 = synth.direct_inputs(sum(lengths), 4, 128, 128, torch.bfloat16, seed=902, init_state=True,
                               lengths=lengths)
    assert_close(*both(to_dev(inp2)), oracle_of(inp2))


def test_noalloc_at_capacity_and_rejects_beyond():
    # H = 96: 4 chunks per head fit in 64 MiB (4 * 96 * 147968 bytes), 5 do not
    inp = synth.direct_inputs(256, 96, 128, 128, torch.bfloat16, seed=903)
    heads = [0, 41, 95]
    assert_close(*both(to_dev(inp)), oracle_of(inp, heads), heads=heads)
    d = to_dev(synth.direct_inputs(320, 96, 128, 128, torch.bfloat16, seed=904))
    o = torch.full((1, 320, 96, 128), 7.0, device="cuda")
    with pytest.raises(kda.KDAError) as err:
        kda.chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], scale=d["scale"], o=o)
    assert err.value.status == 3  # KDA_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((o == 7.0).all()), "a rejected call must not write its output"
