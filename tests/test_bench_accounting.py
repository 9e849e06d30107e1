"""bench.py's roofline arithmetic on the host: the algorithmic bytes of the prefill
and decode lines counted a second way, from the shapes and dtypes of the tensors
the call reads and writes, and the slot size charged to the two-kernel prefill
checked against the library's own workspace-size query.  No GPU is used."""
import importlib.util
import os

import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
from kimi_delta_attention_chunk_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_accounting", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def nbytes(shape, dtype):
    return torch.empty(shape, dtype=dtype, device="meta").numel() * torch.empty((), dtype=dtype).element_size()


@pytest.mark.parametrize("T,H,K,V,N,dt,reads_state", [
    (4096, 96, 128, 128, 1, torch.bfloat16, False),   # the headline prefill
    (68645, 96, 128, 128, 16, torch.bfloat16, True),  # packed sequences with initial states
    (333, 3, 64, 64, 2, torch.float32, True),
])
def test_prefill_bytes_are_the_tensors_moved(bench, T, H, K, V, N, dt, reads_state):
    """q, k, g [T,H,K], v [T,H,V], beta [T,H] in the input dtype read once; o [T,H,V]
    fp32 written once; the final state [N,H,K,V] fp32 written (and the initial one
    read) once."""
    moved = (3 * nbytes((T, H, K), dt) + nbytes((T, H, V), dt) + nbytes((T, H), dt)
             + nbytes((T, H, V), torch.float32) + nbytes((N, H, K, V), torch.float32) * (2 if reads_state else 1))
    in_bytes = torch.empty((), dtype=dt).element_size()
    assert bench.prefill_bytes(T, H, K, V, N, in_bytes, reads_state) == moved


def test_headline_prefill_bytes(bench):
    # the figure the bench line divides by its time (4096 tokens, 96 heads, K = V = 128)
    assert bench.prefill_bytes(4096, 96, 128, 128, 1, 2, False) == 611_057_664


def test_decode_bytes_are_the_tensors_moved(bench):
    """One step of 256 sequences: the fp32 state read and written, the step's q, k,
    g, v, beta in bf16 read, o fp32 written."""
    N, H, K, V = 256, 96, 128, 128
    moved = (2 * nbytes((N, H, K, V), torch.float32) + 3 * nbytes((N, H, K), torch.bfloat16)
             + nbytes((N, H, V), torch.bfloat16) + nbytes((N, H), torch.bfloat16) + nbytes((N, H, V), torch.float32))
    assert bench.decode_bytes(N, H, K, V, 2) == moved == 3_259_023_360


@pytest.mark.parametrize("T,N,reads_state", [(4096, 1, False), (65536, 1, True), (1000, 3, True)])
def test_kernel_split_adds_the_slot_round_trip(bench, T, N, reads_state):
    """The two kernels' design bytes are the call's algorithmic bytes plus each
    (chunk, head) slot written once and read back once."""
    H, K, V = 96, 128, 128
    n_chunks = N * -(-T // 64)
    local, state = bench.kernel_bytes(T * N, n_chunks, H, K, V, N, reads_state, prologue=False)
    assert local + state == (bench.prefill_bytes(T * N, H, K, V, N, 2, reads_state)
                             + 2 * n_chunks * H * bench.SLOT_BYTES)


def test_slot_bytes_match_the_library(bench):
    """The slot the bench charges is the one the library's workspace query sizes:
    each further 64-token chunk of one head adds exactly one slot."""
    kbuild.build()
    lib = kda.load_library()
    ws = lib.kda_chunk_fwd_workspace_size
    for H in (1, 96):
        assert ws(1, 1, 128, H, 128, 128, 1, 0) - ws(1, 1, 64, H, 128, 128, 1, 0) == H * bench.SLOT_BYTES
