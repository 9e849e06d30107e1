"""Seeded synthetic inputs for KDA workloads.

This module only draws random numbers and shapes them into the value
distributions of the workloads (it holds none of the KDA arithmetic): both the
CUDA path and the CPU oracle are fed from here, and neither is imported here.

Every draw comes from ``numpy.random.Generator(PCG64(seed))`` in a fixed order
(q, k, v, gate pre-activation, beta pre-activation, initial state, conv weights,
A_log, dt_bias), in float32 (beta in float64), block by block over tokens so
that the 65536-token workload stays within a few GB of host memory; the shaping
transforms run in float32 torch CPU ops.  Each tensor is rounded once
(round-to-nearest-even) to its storage dtype; the oracle reads exactly the
rounded values.

Workloads (token-major layouts, as the K3 gate tensor ``(B, T, 96, 128)``):

* ``tiny``    B=1, T=128, H=2, K=V=64, fp32, zero initial state.
* ``prefill`` B=1, T=4096, H=96, K=V=128, bf16, zero initial state.
* ``varlen``  16 sequences with lengths uniform on [512, 8192] packed by
  cu_seqlens, H=96, K=V=128, bf16, initial states ~ N(0, 0.02^2) fp32.
* ``decode``  256 sequences, one token per step, 64 steps, H=96, K=V=128,
  bf16 inputs, fp32 state ~ N(0, 0.02^2).
* ``long``    B=1, T=65536, H=96, K=V=128, bf16 raw projections for the fused
  prologue (short conv width 4, L2-norm, per-channel gate), nonzero state.

Distributions for the direct (non-prologue) inputs: q, k ~ N(0,1) then divided
by their per-(token, head) Euclidean norm; v ~ N(0,1); beta = sigmoid(N(0,1));
g = max(-5, -softplus(N(0,1))).  These shape the inputs; the method's own
L2-norm and gate (the prologue) are computed by the kernels and the oracle.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

GATE_LOWER_BOUND = -5.0
STATE_STD = 0.02
TOKEN_BLOCK = 2048


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    K: int
    V: int
    dtype: torch.dtype
    seed: int
    n_seqs: int = 0          # >0: varlen with this many sequences
    init_state: bool = False
    decode_steps: int = 0    # >0: decode workload with N = B sequences
    prologue: bool = False


WORKLOADS = {
    "tiny": Workload("tiny", 1, 128, 2, 64, 64, torch.float32, seed=0),
    "prefill": Workload("prefill", 1, 4096, 96, 128, 128, torch.bfloat16, seed=1),
    "varlen": Workload("varlen", 1, 0, 96, 128, 128, torch.bfloat16, seed=2, n_seqs=16,
                       init_state=True),
    "decode": Workload("decode", 256, 1, 96, 128, 128, torch.bfloat16, seed=3,
                       init_state=True, decode_steps=64),
    "long": Workload("long", 1, 65536, 96, 128, 128, torch.bfloat16, seed=4, init_state=True,
                     prologue=True),
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _to(x: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dtype)


def _normal(rng, shape, dtype, std=1.0, unit_rows=False) -> torch.Tensor:
    """N(0, std^2) draws in token blocks; optionally each last-axis row scaled to unit norm."""
    out = torch.empty(shape, dtype=dtype)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1) if len(shape) > 1 else out.view(-1, 1)
    rows = flat.shape[0]
    for b in range(0, rows, TOKEN_BLOCK):
        e = min(rows, b + TOKEN_BLOCK)
        x = torch.from_numpy(rng.standard_normal((e - b,) + tuple(shape[1:]), dtype=np.float32))
        if std != 1.0:
            x *= std
        if unit_rows:
            x = x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)
        flat[b:e] = x.to(dtype).reshape(e - b, -1)
    return out


def _beta(rng, shape, dtype) -> torch.Tensor:
    z = torch.from_numpy(rng.standard_normal(shape))
    return torch.sigmoid(z).to(dtype)


def _log_decay(rng, shape, dtype) -> torch.Tensor:
    out = torch.empty(shape, dtype=dtype)
    for b in range(0, shape[0], TOKEN_BLOCK):
        e = min(shape[0], b + TOKEN_BLOCK)
        z = torch.from_numpy(rng.standard_normal((e - b,) + tuple(shape[1:]), dtype=np.float32))
        out[b:e] = torch.clamp(-torch.nn.functional.softplus(z), min=GATE_LOWER_BOUND).to(dtype)
    return out


def varlen_lengths(seed: int, n: int = 16, lo: int = 512, hi: int = 8192) -> np.ndarray:
    """Sequence lengths uniform on the integers [lo, hi] (both ends included)."""
    return _rng(seed).integers(lo, hi, n, endpoint=True).astype(np.int64)


def cu_from_lengths(lengths) -> torch.Tensor:
    lengths = np.asarray(lengths, dtype=np.int64)
    return torch.from_numpy(np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32))


def direct_inputs(T: int, H: int, K: int, V: int, dtype: torch.dtype, seed: int, B: int = 1,
                  lengths=None, init_state: bool = False, n_state: int | None = None) -> dict:
    """q, k, v, g, beta (+ cu_seqlens, initial_state) on the host.

    With ``lengths`` the tokens form one packed stream (B=1) of sum(lengths)
    tokens with ``cu_seqlens``; otherwise B sequences of T tokens each.
    Shapes: q, k, g [B, T, H, K]; v [B, T, H, V]; beta [B, T, H];
    initial_state [N, H, K, V] fp32 (N = number of sequences).
    """
    rng = _rng(seed)
    cu = None
    if lengths is not None:
        B = 1
        T = int(np.sum(lengths))
        cu = cu_from_lengths(lengths)
    BT = B * T
    q = _normal(rng, (BT, H, K), dtype, unit_rows=True).view(B, T, H, K)
    k = _normal(rng, (BT, H, K), dtype, unit_rows=True).view(B, T, H, K)
    v = _normal(rng, (BT, H, V), dtype).view(B, T, H, V)
    g = _log_decay(rng, (BT, H, K), dtype).view(B, T, H, K)
    beta = _beta(rng, (BT, H), dtype).view(B, T, H)
    N = n_state if n_state is not None else (len(lengths) if lengths is not None else B)
    s0 = _normal(rng, (N, H, K, V), torch.float32, std=STATE_STD) if init_state else None
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta, "cu_seqlens": cu, "initial_state": s0,
            "scale": float(K) ** -0.5}


def prologue_inputs(T: int, H: int, K: int, V: int, dtype: torch.dtype, seed: int, B: int = 1,
                    lengths=None, init_state: bool = True) -> dict:
    """Raw inputs for the fused prologue.

    q_raw, k_raw, gate_x [B, T, H, K] and v_raw [B, T, H, V] ~ N(0,1); beta as in
    :func:`direct_inputs`; initial_state ~ N(0, 0.02^2); conv weights
    [3, H*max(K,V), 4] fp32 ~ N(0, 0.5^2) (q uses rows [0, H*K), k the same,
    v rows [0, H*V)); A_log [K] ~ U(-1, 1); dt_bias [H*K] ~ U(-1, 1).
    """
    rng = _rng(seed)
    cu = None
    if lengths is not None:
        B = 1
        T = int(np.sum(lengths))
        cu = cu_from_lengths(lengths)
    BT = B * T
    q = _normal(rng, (BT, H, K), dtype).view(B, T, H, K)
    k = _normal(rng, (BT, H, K), dtype).view(B, T, H, K)
    v = _normal(rng, (BT, H, V), dtype).view(B, T, H, V)
    gx = _normal(rng, (BT, H, K), dtype).view(B, T, H, K)
    beta = _beta(rng, (BT, H), dtype).view(B, T, H)
    N = len(lengths) if lengths is not None else B
    s0 = _normal(rng, (N, H, K, V), torch.float32, std=STATE_STD) if init_state else None
    D = max(K, V)
    conv_w = torch.from_numpy((rng.standard_normal((3, H * D, 4)) * 0.5).astype(np.float32))
    A_log = torch.from_numpy(rng.uniform(-1.0, 1.0, K).astype(np.float32))
    dt_bias = torch.from_numpy(rng.uniform(-1.0, 1.0, H * K).astype(np.float32))
    return {"q_raw": q, "k_raw": k, "v_raw": v, "gate_x": gx, "beta": beta, "cu_seqlens": cu,
            "initial_state": s0, "conv_w": conv_w, "A_log": A_log, "dt_bias": dt_bias,
            "scale": float(K) ** -0.5, "lower_bound": GATE_LOWER_BOUND, "l2_eps": 1e-6}


def decode_inputs(N: int, H: int, K: int, V: int, steps: int, dtype: torch.dtype, seed: int) -> dict:
    """Per-step decode inputs: q, k, g [steps, N, H, K]; v [steps, N, H, V]; beta
    [steps, N, H]; state [N, H, K, V] fp32 ~ N(0, 0.02^2)."""
    rng = _rng(seed)
    q = _normal(rng, (steps * N, H, K), dtype, unit_rows=True).view(steps, N, H, K)
    k = _normal(rng, (steps * N, H, K), dtype, unit_rows=True).view(steps, N, H, K)
    v = _normal(rng, (steps * N, H, V), dtype).view(steps, N, H, V)
    g = _log_decay(rng, (steps * N, H, K), dtype).view(steps, N, H, K)
    beta = _beta(rng, (steps * N, H), dtype).view(steps, N, H)
    s0 = _normal(rng, (N, H, K, V), torch.float32, std=STATE_STD)
    return {"q": q, "k": k, "v": v, "g": g, "beta": beta, "state": s0, "scale": float(K) ** -0.5}


def device_inputs(name: str, device, seed_offset: int = 0) -> dict:
    """Inputs of a named workload drawn directly on a CUDA device (torch's seeded
    Philox generator), with the same shapes and value distributions as the host
    generators above.  For timing only: the host generators are the ones the
    parity tests share with the oracle."""
    w = WORKLOADS[name]
    gen = torch.Generator(device=device)
    gen.manual_seed(1000003 * (w.seed + 1) + seed_offset)
    lengths = varlen_lengths(w.seed, w.n_seqs) if w.n_seqs else None
    B, T = (1, int(np.sum(lengths))) if lengths is not None else (w.B, w.T)
    H, K, V, dt = w.H, w.K, w.V, w.dtype
    rn = lambda *shape: torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)  # noqa: E731
    unit = lambda x: x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)  # noqa: E731
    out = {"scale": float(K) ** -0.5,
           "cu_seqlens": cu_from_lengths(lengths).to(device) if lengths is not None else None}
    N = len(lengths) if lengths is not None else B
    if w.prologue:
        out.update(q_raw=rn(B, T, H, K).to(dt), k_raw=rn(B, T, H, K).to(dt), v_raw=rn(B, T, H, V).to(dt),
                   gate_x=rn(B, T, H, K).to(dt), beta=torch.sigmoid(rn(B, T, H)).to(dt),
                   conv_w=(0.5 * rn(3, H * max(K, V), 4)),
                   A_log=torch.rand(K, generator=gen, device=device) * 2 - 1,
                   dt_bias=torch.rand(H * K, generator=gen, device=device) * 2 - 1)
    else:
        out.update(q=unit(rn(B, T, H, K)).to(dt), k=unit(rn(B, T, H, K)).to(dt), v=rn(B, T, H, V).to(dt),
                   g=torch.clamp(-torch.nn.functional.softplus(rn(B, T, H, K)), min=GATE_LOWER_BOUND).to(dt),
                   beta=torch.sigmoid(rn(B, T, H)).to(dt))
    out["initial_state"] = STATE_STD * rn(N, H, K, V) if w.init_state else None
    return out


def workload_inputs(name: str) -> dict:
    """Full-size inputs of a named workload."""
    w = WORKLOADS[name]
    if w.decode_steps:
        return decode_inputs(w.B, w.H, w.K, w.V, w.decode_steps, w.dtype, w.seed)
    if w.prologue:
        return prologue_inputs(w.T, w.H, w.K, w.V, w.dtype, w.seed, B=w.B, init_state=w.init_state)
    lengths = varlen_lengths(w.seed, w.n_seqs) if w.n_seqs else None
    return direct_inputs(w.T, w.H, w.K, w.V, w.dtype, w.seed, B=w.B, lengths=lengths,
                         init_state=w.init_state)


def output_gate_inputs(shape, gate_dtype: torch.dtype, seed: int) -> dict:
    """Inputs of the layer's output gate: o fp32 ~ N(0,1) times a per-row scale
    10^U(-2, 1) (rows of very different magnitude, as attention outputs have),
    gate pre-activation ~ N(0,1) in ``gate_dtype``, weight [V] ~ U(0.5, 1.5) fp32."""
    rng = _rng(seed)
    V = shape[-1]
    o = rng.standard_normal(shape, dtype=np.float32)
    o *= (10.0 ** rng.uniform(-2.0, 1.0, tuple(shape[:-1]) + (1,))).astype(np.float32)
    gate = rng.standard_normal(shape, dtype=np.float32)
    w = rng.uniform(0.5, 1.5, V).astype(np.float32)
    return {"o": _to(o, torch.float32), "gate": _to(gate, gate_dtype), "weight": _to(w, torch.float32)}


def gate_proj_inputs(B: int, T: int, D: int, R: int, HK: int, NH: int, seed: int,
                     dtype: torch.dtype = torch.bfloat16) -> dict:
    """Inputs of the projections ahead of the gate: the layer input x [B,T,D] ~ N(0,1)
    (a normalised hidden state) and weights drawn with fan-in scaling, f_a [R,D] and
    b_proj [NH,D] ~ N(0, 1/D), f_b [HK,R] ~ N(0, 1/R), so that f_a x, f_b (f_a x) and
    b_proj x all have unit variance.  Drawn in the order x, f_a, f_b, b_proj."""
    rng = _rng(seed)
    x = _normal(rng, (B * T, D), dtype).view(B, T, D)
    f_a = _normal(rng, (R, D), dtype, std=D ** -0.5)
    f_b = _normal(rng, (HK, R), dtype, std=R ** -0.5)
    b_proj = _normal(rng, (NH, D), dtype, std=D ** -0.5)
    return {"x": x, "f_a": f_a, "f_b": f_b, "b_proj": b_proj}

