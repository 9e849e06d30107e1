"""The C ABI on the host: libkda.so builds, loads and exports every symbol that
include/kda.h declares; host-side argument checks reject bad calls before any
GPU work.  No kernel is launched here."""
import ctypes
import os
import re

import pytest
import torch

import kimi_delta_attention_chunk_gb300 as kda
from kimi_delta_attention_chunk_gb300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")

INVALID_ARG, UNSUPPORTED, WORKSPACE = 1, 2, 3
SLOT = 147968  # workspace bytes per (chunk, head) of the tensor-core prefill


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"KDA_API[^;(]*?\b(kda_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kda.load_library()


def test_header_declares_the_boundary():
    syms = declared_symbols()
    for name in ("kda_chunk_fwd", "kda_chunk_fwd_fused", "kda_recurrent_step", "kda_status_string"):
        assert name in syms


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert sorted(kda.SIGNATURES) == declared_symbols()


def test_status_strings_and_version(lib):
    assert lib.kda_abi_version() >= 1
    for s in range(7):
        assert lib.kda_status_string(s)
    assert lib.kda_status_string(99) == b"unknown kda_status"


# Fake, 16-byte aligned, never-dereferenced addresses: every call below must be
# rejected on the host before anything is launched.
P = ctypes.c_void_p(0x10000)
Pm = ctypes.c_void_p(0x10008)  # misaligned


BIG_WS = ctypes.c_void_p(0x40000000)  # fake workspace address


def chunk(lib, *, q=P, k=P, v=P, g=P, beta=P, dt=1, s0=None, cu=None, B=1, T=64, H=2, K=128, V=128,
          N=1, o=P, odt=0, sT=None, ws=BIG_WS, ws_bytes=1 << 30, status=None):
    return lib.kda_chunk_fwd(q, k, v, g, beta, dt, 0.0, s0, cu, B, T, H, K, V, N, o, odt, sT, ws, ws_bytes,
                             status, None)


def test_chunk_rejects_bad_arguments(lib):
    assert chunk(lib, K=96) == UNSUPPORTED
    assert chunk(lib, V=32) == UNSUPPORTED
    assert chunk(lib, dt=7) == UNSUPPORTED
    assert chunk(lib, odt=3) == UNSUPPORTED
    assert chunk(lib, q=None) == INVALID_ARG
    assert chunk(lib, o=None) == INVALID_ARG
    assert chunk(lib, k=Pm) == INVALID_ARG
    assert chunk(lib, T=-1) == INVALID_ARG
    assert chunk(lib, H=0) == INVALID_ARG
    assert chunk(lib, B=2, N=1) == INVALID_ARG          # N must equal B without cu_seqlens
    assert chunk(lib, B=2, N=3, cu=P) == INVALID_ARG    # packed sequences need B == 1
    assert chunk(lib, s0=ctypes.c_void_p(0x100000), sT=ctypes.c_void_p(0x100000 + 4096)) == INVALID_ARG
    assert chunk(lib, status=ctypes.c_void_p(0x10002)) == INVALID_ARG   # status word not 4-byte aligned
    assert chunk(lib, ws=Pm) == INVALID_ARG                             # workspace not 16-byte aligned


def test_workspace_size_formula(lib):
    """The size query gives the documented formula: a 147968-byte slot per
    64-token chunk and head, plus the packed-sequence bookkeeping rounded up to
    1 KiB; the CUDA-core path (fp32 or a head size of 64) needs none."""
    ws = lib.kda_chunk_fwd_workspace_size
    assert ws(1, 1, 4096, 96, 128, 128, 1, 0) == 64 * 96 * SLOT
    assert ws(1, 2, 333, 3, 128, 128, 2, 0) == 2 * 6 * 3 * SLOT
    assert ws(1, 1, 0, 3, 128, 128, 1, 0) == 0
    assert ws(1, 1, 64, 4, 128, 128, 0, 1) == 0        # N * H == 0
    # packed: max_chunks = ceil(T / 64) + N, bookkeeping 4 * (2 N + 1 + max_chunks) bytes
    T, N, H = 68645, 16, 96
    mc = -(-T // 64) + N
    hdr = -(-(4 * (2 * N + 1 + mc)) // 1024) * 1024
    assert ws(1, 1, T, H, 128, 128, N, 1) == hdr + mc * H * SLOT
    assert ws(0, 1, 4096, 96, 128, 128, 1, 0) == 0     # fp32 inputs: CUDA-core path
    assert ws(1, 1, 4096, 96, 64, 128, 1, 0) == 0      # K = 64: CUDA-core path
    assert ws(1, -1, 4096, 96, 128, 128, 1, 0) == 0    # invalid sizes


def test_chunk_rejects_a_small_workspace_before_launching(lib):
    need = lib.kda_chunk_fwd_workspace_size(1, 1, 64, 2, 128, 128, 1, 0)
    assert need == 2 * SLOT
    assert chunk(lib, ws_bytes=need - 1) == WORKSPACE
    assert chunk(lib, ws=None, ws_bytes=0) == WORKSPACE


def test_fused_rejects_bad_arguments(lib):
    def fused(**kw):
        a = dict(conv_act=0, lb=-5.0, eps=1e-6, cq=P, ck=P, cv=P, A=P, db=P, K=128)
        a.update(kw)
        return lib.kda_chunk_fwd_fused(P, P, P, P, P, 1, a["cq"], a["ck"], a["cv"], a["conv_act"], a["A"],
                                       a["db"], a["lb"], a["eps"], 0.0, None, None, 1, 64, 2, a["K"], 128, 1,
                                       P, 0, None, a.get("ws", BIG_WS), a.get("wsb", 1 << 30), None, None)
    assert fused(conv_act=2) == INVALID_ARG
    assert fused(lb=1.0) == INVALID_ARG
    assert fused(eps=-1.0) == INVALID_ARG
    assert fused(A=None) == INVALID_ARG
    assert fused(cv=Pm) == INVALID_ARG
    assert fused(K=80) == UNSUPPORTED
    assert fused(wsb=1000) == WORKSPACE


def test_decode_rejects_bad_arguments(lib):
    def step(**kw):
        a = dict(q=P, st=P, N=4, H=2, K=128, V=128, dt=1)
        a.update(kw)
        return lib.kda_recurrent_step(a["q"], P, P, P, P, a["dt"], 0.0, a["st"], a["N"], a["H"], a["K"],
                                      a["V"], P, 0, None)
    assert step(K=100) == UNSUPPORTED
    assert step(dt=5) == UNSUPPORTED
    assert step(st=None) == INVALID_ARG
    assert step(q=Pm) == INVALID_ARG
    assert step(N=-1) == INVALID_ARG
    assert step(N=0, q=None) == 0   # nothing to do


def test_output_gate_rejects_bad_arguments(lib):
    big = ctypes.c_void_p(0x1000000)

    def og(**kw):
        a = dict(o=P, g=big, gdt=1, w=None, eps=1e-6, B=1, T=64, H=2, V=128, out=ctypes.c_void_p(0x2000000),
                 odt=0)
        a.update(kw)
        return lib.kda_output_gate(a["o"], a["g"], a["gdt"], a["w"], a["eps"], a["B"], a["T"], a["H"],
                                   a["V"], a["out"], a["odt"], None)
    assert og(V=96) == UNSUPPORTED
    assert og(gdt=4) == UNSUPPORTED
    assert og(odt=9) == UNSUPPORTED
    assert og(o=None) == INVALID_ARG
    assert og(w=Pm) == INVALID_ARG
    assert og(eps=-1.0) == INVALID_ARG
    assert og(eps=float("inf")) == INVALID_ARG
    assert og(H=0) == INVALID_ARG
    assert og(out=P, odt=1) == INVALID_ARG                        # bf16 out over the fp32 o
    assert og(out=ctypes.c_void_p(0x10000 + 1024)) == INVALID_ARG   # partial overlap with o
    assert og(out=big) == INVALID_ARG                               # out over the gate
    assert og(T=0, o=None, g=None, out=None) == 0                   # nothing to do


def test_check_range_rejects_bad_arguments(lib):
    def chk(**kw):
        a = dict(x=P, dt=1, n=100, lo=-5.0, hi=0.0, st=P)
        a.update(kw)
        return lib.kda_check_range(a["x"], a["dt"], a["n"], a["lo"], a["hi"], a["st"], None)
    assert chk(dt=3) == UNSUPPORTED
    assert chk(n=-1) == INVALID_ARG
    assert chk(lo=1.0, hi=0.0) == INVALID_ARG
    assert chk(lo=float("nan")) == INVALID_ARG
    assert chk(st=None) == INVALID_ARG
    assert chk(st=ctypes.c_void_p(0x10002)) == INVALID_ARG   # status word not 4-byte aligned
    assert chk(x=None) == INVALID_ARG
    assert chk(x=ctypes.c_void_p(0x10001)) == INVALID_ARG    # bf16 elements need 2-byte alignment


def test_backward_rejects_bad_arguments(lib):
    def bwd(**kw):
        a = dict(dq=P, dO=P, K=128, dt=1, dbeta=P)
        a.update(kw)
        return lib.kda_recurrent_bwd(P, P, P, P, P, a["dt"], 0.0, None, None, 1, 64, 2, a["K"], 128, 1, a["dO"],
                                     None, a["dq"], P, P, P, a["dbeta"], None, a.get("ws", BIG_WS),
                                     a.get("wsb", 1 << 30), a.get("st", None), None)
    assert bwd(K=96) == UNSUPPORTED
    assert bwd(dt=4) == UNSUPPORTED
    assert bwd(dO=None) == INVALID_ARG
    assert bwd(dq=None) == INVALID_ARG
    assert bwd(dq=Pm) == INVALID_ARG
    assert bwd(dbeta=ctypes.c_void_p(0x10002)) == INVALID_ARG
    need = lib.kda_recurrent_bwd_workspace_size(1, 1, 64, 2, 128, 128, 1, 0)
    assert need == 4 * 128 * 128 * (1 * 2 + 64 * 2)
    assert bwd(wsb=need - 1) == WORKSPACE
    assert bwd(st=ctypes.c_void_p(0x10001)) == INVALID_ARG


def test_gate_proj_rejects_bad_arguments(lib):
    # fake, disjoint, 16-byte aligned addresses (x [B*T, D], weights, outputs)
    X, FA, FB, BP = (ctypes.c_void_p(a) for a in (0x10000000, 0x20000000, 0x30000000, 0x40000000))
    GX, BE, WS = (ctypes.c_void_p(a) for a in (0x50000000, 0x60000000, 0x70000000))

    def gp(**kw):
        a = dict(x=X, fa=FA, fb=FB, bp=BP, dt=1, B=1, T=300, D=7168, R=128, HK=12288, NH=96, gx=GX, be=BE,
                 ws=WS, wsb=1 << 30, st=None)
        a.update(kw)
        return lib.kda_gate_proj(a["x"], a["fa"], a["fb"], a["bp"], a["dt"], a["B"], a["T"], a["D"], a["R"],
                                 a["HK"], a["NH"], a["gx"], a["be"], a["ws"], a["wsb"], a["st"], None)
    need = lib.kda_gate_proj_workspace_size(1, 300, 7168, 128, 96)
    # y as bf16 hi and lo, and the fp32 partial sums of 8 ranges of D (3 tiles of 128 tokens)
    assert need == 300 * 128 * 2 * 2 + 8 * 224 * 300 * 4
    # 64 tiles: 2 ranges; D = 64: a single range
    assert lib.kda_gate_proj_workspace_size(1, 8192, 7168, 128, 96) == 8192 * (512 + 2 * 224 * 4)
    assert lib.kda_gate_proj_workspace_size(1, 300, 64, 128, 96) == 300 * (512 + 224 * 4)
    assert lib.kda_gate_proj_workspace_size(1, 300, 7168, 96, 96) == 0
    assert gp(dt=0) == UNSUPPORTED                        # bf16 only
    assert gp(D=7000) == UNSUPPORTED                      # D a multiple of 64
    assert gp(R=96) == UNSUPPORTED
    assert gp(NH=100) == UNSUPPORTED                      # NH a multiple of 16
    assert gp(R=128, NH=144) == UNSUPPORTED               # R + NH > 256
    assert gp(HK=12000) == UNSUPPORTED                    # HK a multiple of 256
    assert gp(B=-1) == INVALID_ARG
    assert gp(D=0) == INVALID_ARG
    assert gp(B=1 << 16, T=1 << 16) == INVALID_ARG        # more than 2^31 - 1 tokens
    assert gp(x=None) == INVALID_ARG
    assert gp(fb=Pm) == INVALID_ARG
    assert gp(be=ctypes.c_void_p(0x60000008)) == INVALID_ARG
    assert gp(st=ctypes.c_void_p(0x10002)) == INVALID_ARG
    assert gp(wsb=need - 1) == WORKSPACE
    assert gp(ws=None) == WORKSPACE
    assert gp(gx=ctypes.c_void_p(0x10000000 + 4096)) == INVALID_ARG   # gate_x over x
    assert gp(be=ctypes.c_void_p(0x50000000 + 1024)) == INVALID_ARG   # beta over gate_x
    assert gp(ws=ctypes.c_void_p(0x20000000)) == INVALID_ARG          # workspace over f_a
    assert gp(T=0, x=None, gx=None, be=None, ws=None, wsb=0) == 0    # nothing to do


def test_binding_refuses_cpu_tensors(lib):
    x = torch.zeros(1, 64, 2, 128, dtype=torch.bfloat16)
    b = torch.zeros(1, 64, 2, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        kda.chunk_fwd(x, x, x, x, b)


def test_segmented_driver_checks_its_cuts_on_the_host():
    from kimi_delta_attention_chunk_gb300 import cp
    x = torch.zeros(1, 100, 2, 128, dtype=torch.bfloat16)
    b = torch.zeros(1, 100, 2, dtype=torch.bfloat16)
    for bounds in ([0], [100], [50, 50], [60, 40]):
        with pytest.raises(ValueError):
            cp.chunk_fwd_segmented(x, x, x, x, b, bounds)
