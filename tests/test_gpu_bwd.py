"""The backward against the oracle's reverse-mode backward of the recurrence:
every gradient (dq, dk, dv, dg, dbeta, dS0), element by element, bf16 and fp32
inputs, dense and packed sequences, with and without an initial state and a
final-state gradient.  kda_chunk_bwd (chunk by chunk for bf16 with K = V = 128,
token by token otherwise) and kda_recurrent_bwd (token by token) both."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
import oracle
from kimi_delta_attention_chunk_gb300 import synth
from tests.kda_testutil import TOL_BF16, TOL_F32, rel_err, to_dev

pytestmark = pytest.mark.gpu


def check(d, dO, dST, tol, token_by_token=False):
    dd = to_dev(d)
    got = kda.chunk_bwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dO.cuda(),
                        dS_T=None if dST is None else dST.cuda(), scale=d["scale"],
                        initial_state=dd["initial_state"], cu_seqlens=dd["cu_seqlens"],
                        token_by_token=token_by_token)
    torch.cuda.synchronize()
    lead = d["q"].shape[:2]
    flat = (lambda x: x[0]) if d["cu_seqlens"] is not None else (lambda x: x)
    ref = oracle.kda_backward(flat(d["q"]), flat(d["k"]), flat(d["v"]), flat(d["g"]), flat(d["beta"]),
                              flat(dO), dS_T=dST, scale=d["scale"], initial_state=d["initial_state"],
                              cu_seqlens=d["cu_seqlens"])
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dS0"):
        g = got[key][0] if (d["cu_seqlens"] is not None and key != "dS0") else got[key]
        e = rel_err(g, ref[key])
        assert e <= tol, f"{key}: err {e:.3e}"
    assert got["dq"].shape[:2] == lead


@pytest.mark.parametrize("token_by_token", [False, True])
def test_bf16_dense_with_state_gradient(token_by_token):
    # three chunks, the last one ragged
    d = synth.direct_inputs(150, 2, 128, 128, torch.bfloat16, seed=111, init_state=True)
    gen = torch.Generator().manual_seed(1)
    dO = torch.randn(1, 150, 2, 128, generator=gen)
    dST = torch.randn(1, 2, 128, 128, generator=gen)
    check(d, dO, dST, TOL_BF16, token_by_token)


def test_bf16_chunked_packed_sequences():
    # lengths 1, exactly one chunk, ragged, empty, several chunks
    lengths = [1, 64, 100, 0, 130]
    d = synth.direct_inputs(sum(lengths), 3, 128, 128, torch.bfloat16, seed=114, init_state=True, lengths=lengths)
    gen = torch.Generator().manual_seed(4)
    dO = torch.randn(1, sum(lengths), 3, 128, generator=gen)
    dST = torch.randn(len(lengths), 3, 128, 128, generator=gen)
    check(d, dO, dST, TOL_BF16)


def test_bf16_chunked_two_dense_rows_no_state():
    d = synth.direct_inputs(256, 4, 128, 128, torch.bfloat16, seed=115, B=2)
    dO = torch.randn(2, 256, 4, 128, generator=torch.Generator().manual_seed(5))
    check(d, dO, None, TOL_BF16)


def test_bf16_chunked_full_size_on_sampled_heads():
    # the 4096-token, 96-head workload through the chunked path; the oracle's reverse
    # mode on two of the heads (the heads are independent)
    T, H = 4096, 96
    d = synth.direct_inputs(T, H, 128, 128, torch.bfloat16, seed=116)
    dO = torch.randn(1, T, H, 128, generator=torch.Generator().manual_seed(6))
    dd = to_dev(d)
    got = kda.chunk_bwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dO.cuda(), scale=d["scale"])
    torch.cuda.synchronize()
    for h in (0, 77):
        sl = lambda x: x[0, :, h:h + 1]  # noqa: E731
        ref = oracle.kda_backward(sl(d["q"]), sl(d["k"]), sl(d["v"]), sl(d["g"]), d["beta"][0, :, h:h + 1],
                                  sl(dO), scale=d["scale"])
        for key in ("dq", "dk", "dv", "dg", "dbeta"):
            e = rel_err(got[key][0, :, h:h + 1], ref[key])
            assert e <= TOL_BF16, f"head {h} {key}: err {e:.3e}"
        e = rel_err(got["dS0"][:, h:h + 1], ref["dS0"])
        assert e <= TOL_BF16, f"head {h} dS0: err {e:.3e}"


def test_fp32_packed_sequences():
    lengths = [30, 0, 70, 5]
    d = synth.direct_inputs(sum(lengths), 3, 64, 64, torch.float32, seed=112, init_state=True, lengths=lengths)
    dO = torch.randn(1, sum(lengths), 3, 64, generator=torch.Generator().manual_seed(2))
    check(d, dO, None, TOL_F32)


def test_fp32_two_dense_rows_no_initial_state():
    d = synth.direct_inputs(65, 2, 128, 64, torch.float32, seed=113, B=2)
    dO = torch.randn(2, 65, 2, 64, generator=torch.Generator().manual_seed(3))
    check(d, dO, None, TOL_F32)


def test_bf16_chunked_all_heads():
    # every one of the 96 heads at 512 tokens (768 (chunk, head) tasks over the chunk
    # kernel's persistent CTAs, several per CTA), with an initial state and a
    # final-state gradient: a mistake in the task-to-head mapping would show here
    T, H = 512, 96
    d = synth.direct_inputs(T, H, 128, 128, torch.bfloat16, seed=117, init_state=True)
    gen = torch.Generator().manual_seed(7)
    dO = torch.randn(1, T, H, 128, generator=gen)
    dST = torch.randn(1, H, 128, 128, generator=gen)
    check(d, dO, dST, TOL_BF16)
