"""KDA oracle: the plain, slow, double-precision CPU statement of the method.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this
package.  The CUDA path never imports it, and it never imports the CUDA path:
the two share no code, header, table or helper.  The only thing both sides see
is the seeded input generator module, which holds none of the method's
arithmetic.

The arithmetic lives in ``kda_oracle.c`` (plain C, fp64, no fast-math), built
with gcc into ``oracle/_build/libkda_oracle.so`` on first use.  Functions:

* :func:`kda_forward` -- the KDA recurrence, token by token, per (sequence,
  head): channel-wise decay ``S <- Diag(exp(g_t)) S``, delta update
  ``S <- S - beta_t k_t (k_t^T S) + beta_t k_t v_t^T``, read-out
  ``o_t = scale * S^T q_t`` (sources: "ISEEKYAN/k3" README; "kimi-k3-mlx"
  review, sections "The A_log shape mismatch ..." and "Attention is 93
  layers ...").
* :func:`short_conv` -- causal depthwise convolution of width 4 restarted at
  each sequence start ("kimi-k3-mlx" review, "Attention is 93 layers ...").
* :func:`l2norm` -- per-row ``x / sqrt(sum x^2 + eps)``.
* :func:`gate` -- ``g = max(lower_bound, -exp(A_log[c]) * softplus(x + dt_bias))``
  with ``A_log`` broadcast along the 128-wide channel axis and shared by all
  heads ("kimi-k3-mlx" review, "The A_log shape mismatch ...").
* :func:`prologue` -- short_conv on q, k, v, then l2norm on q and k, then gate.
* :func:`segment_transition`, :func:`state_compose` -- context parallelism
  over consecutive segments of a sequence: the recurrence is affine in the
  state, S_end = M S_start + S_zero with M the product of the per-token
  factors ``(I - beta k k^T) Diag(e^g)`` (later tokens on the left), and the
  prefix ``S_in(r+1) = M_r S_in(r) + S_zero_r`` ("ISEEKYAN/k3" README, on the
  initial path without context parallelism; the affine form follows from the
  recurrence above).
* :func:`kda_backward` -- gradients of <dO, o> + <dS_T, S_T> with respect to
  q, k, v, g, beta and the initial state, by reverse mode through the same
  recurrence, token by token (pinned by central finite differences, the T=1
  closed forms and the adjoint identity of the map (v, S0) -> (o, S_T)).
* :func:`gate_proj` -- the projections ahead of the gate, per token:
  ``gate_x = f_b (f_a x)`` (the low-rank forget gate; its input to
  :func:`gate`) and ``beta = sigmoid(b_proj x)`` ("kimi-k3-mlx" review,
  "Attention is 93 layers ...": low-rank forget gate through f_a and f_b;
  "The A_log shape mismatch ...": b_proj is [96, H]).
* :func:`output_gate` -- the layer's output gate on o: per (token, head)
  ``o / sqrt(mean_v o^2 + eps) * w * sigmoid(gate)`` ("kimi-k3-mlx" review,
  "Attention is 93 layers ...": a full-rank output gate; "NeMo AutoModel
  draft_kimi_k3": RMS norms with fp32 variance, sigmoid output gates).

Pins (tests/test_oracle_pins.py): the T=1 closed form, the delta-rule
overwrite invariant, the beta=0 pure-decay invariant, brute-force products of
``(I - beta k k^T) Diag(e^g)``, the scalar-decay (gated delta rule) special
case, linearity in (v, S0), the Householder norm invariant, padding tokens,
a hand-worked golden fixture, and library routines for the prologue
(``numpy.convolve``, ``numpy.linalg.norm``, ``numpy.logaddexp``); for the output
gate, degree-0 homogeneity in o, the sigmoid reflection, unit RMS of the normed
rows, per-channel equivariance and the constant-row closed form; for the gate
projections, the rank-1 outer-product closed form, brute-force sums on tiny
shapes written as Python loops, beta = 1/2 for b_proj = 0, the sigmoid
reflection, and linearity of gate_x in x.  No function here is "parity
unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile ``kda_oracle.c`` with gcc (-O2, no fast-math); return the .so path."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11", "-fPIC",
               "-shared", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.kda_oracle_forward.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64p,
                                               ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_double, _dp, _dp,
                                               ctypes.c_int]
            lib.kda_oracle_forward.restype = ctypes.c_int
            lib.kda_oracle_short_conv.argtypes = [_dp, _dp, _i64p, ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.c_int64, ctypes.c_int, _dp]
            lib.kda_oracle_short_conv.restype = ctypes.c_int
            lib.kda_oracle_l2norm.argtypes = [_dp, ctypes.c_int64, ctypes.c_int64, ctypes.c_double]
            lib.kda_oracle_l2norm.restype = ctypes.c_int
            lib.kda_oracle_gate.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_double, _dp]
            lib.kda_oracle_gate.restype = ctypes.c_int
            lib.kda_oracle_output_gate.argtypes = [_dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                                   ctypes.c_double, _dp]
            lib.kda_oracle_output_gate.restype = ctypes.c_int
            lib.kda_oracle_gate_proj.argtypes = [_dp, _dp, _dp, _dp, ctypes.c_int64, ctypes.c_int64,
                                                 ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _dp, _dp]
            lib.kda_oracle_gate_proj.restype = ctypes.c_int
            lib.kda_oracle_backward.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64p, ctypes.c_int64,
                                                ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                ctypes.c_double, _dp, _dp, _dp, _dp, _dp, _dp, _dp, _dp,
                                                ctypes.c_int]
            lib.kda_oracle_backward.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor: exact upcast of its stored values
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _seqlens(cu_seqlens, Ttot: int, B: int, T: int) -> np.ndarray:
    if cu_seqlens is None:
        return np.arange(B + 1, dtype=np.int64) * T
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu().numpy() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    if cu.ndim != 1 or cu[0] != 0 or cu[-1] != Ttot or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must be non-decreasing, start at 0 and end at the token count")
    return cu


def kda_forward(q, k, v, g, beta, scale=None, initial_state=None, cu_seqlens=None,
                nthreads: int | None = None):
    """Sequential fp64 KDA forward.

    q, k, g: [B, T, H, K] or [Ttot, H, K]; v: [..., H, V]; beta: [..., H].
    With ``cu_seqlens`` (length N+1) the token axis is one packed stream
    (B must be 1); without it each of the B rows is its own sequence.
    initial_state: [N, H, K, V] or None (zeros).  scale: None means K**-0.5.
    Returns (o [same leading shape, V] float64, final_state [N, H, K, V] float64).
    """
    q, k, v, g, beta = (_f64(a) for a in (q, k, v, g, beta))
    lead = q.shape[:-2]
    H, K = q.shape[-2:]
    V = v.shape[-1]
    if len(lead) == 2:
        B, T = lead
    elif len(lead) == 1:
        B, T = 1, lead[0]
    else:
        raise ValueError("q must be [B,T,H,K] or [T,H,K]")
    if cu_seqlens is not None and B != 1:
        raise ValueError("cu_seqlens requires B == 1")
    Ttot = B * T
    cu = _seqlens(cu_seqlens, Ttot, B, T)
    N = cu.shape[0] - 1
    for name, a, last in (("k", k, K), ("g", g, K), ("v", v, V)):
        if a.shape[:-2] != lead or a.shape[-2:] != (H, last):
            raise ValueError(f"{name} has shape {a.shape}")
    if beta.shape != lead + (H,):
        raise ValueError(f"beta has shape {beta.shape}")
    s0 = None
    if initial_state is not None:
        s0 = _f64(initial_state)
        if s0.shape != (N, H, K, V):
            raise ValueError(f"initial_state has shape {s0.shape}, expected {(N, H, K, V)}")
    if scale is None:
        scale = float(K) ** -0.5
    o = np.zeros(lead + (H, V), dtype=np.float64)
    sT = np.zeros((N, H, K, V), dtype=np.float64)
    nt = nthreads or default_threads()
    rc = _load().kda_oracle_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                    _ptr(s0) if s0 is not None else None,
                                    cu.ctypes.data_as(_i64p), N, H, K, V, float(scale),
                                    _ptr(o), _ptr(sT), int(nt))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_forward failed with status {rc}")
    return o, sT


def short_conv(x, w, cu_seqlens=None, act: int = 0):
    """Causal depthwise conv, width w.shape[-1].  x: [B,T,C] / [T,C]; w: [C, W]."""
    x = _f64(x)
    w = _f64(w)
    lead = x.shape[:-1]
    C = x.shape[-1]
    B, T = (lead if len(lead) == 2 else (1, lead[0]))
    cu = _seqlens(cu_seqlens, B * T, B, T)
    if w.ndim != 2 or w.shape[0] != C:
        raise ValueError("w must be [C, W]")
    y = np.zeros_like(x)
    rc = _load().kda_oracle_short_conv(_ptr(x), _ptr(w), cu.ctypes.data_as(_i64p), cu.shape[0] - 1,
                                       C, w.shape[1], int(act), _ptr(y))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_short_conv failed with status {rc}")
    return y


def l2norm(x, eps: float = 1e-6):
    """Rows of the last axis divided by sqrt(sum of squares + eps)."""
    x = _f64(x).copy()
    D = x.shape[-1]
    rc = _load().kda_oracle_l2norm(_ptr(x), x.size // D, D, float(eps))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_l2norm failed with status {rc}")
    return x


def gate(x, A_log, dt_bias, lower_bound: float = -5.0):
    """g = max(lower_bound, -exp(A_log[c]) * softplus(x + dt_bias[h*K + c])); x: [..., H, K]."""
    x = _f64(x)
    A = _f64(A_log)
    db = _f64(dt_bias)
    H, K = x.shape[-2:]
    if A.shape != (K,) or db.shape != (H * K,):
        raise ValueError("A_log must be [K] and dt_bias [H*K]")
    g = np.zeros_like(x)
    rc = _load().kda_oracle_gate(_ptr(x), _ptr(A), _ptr(db), x.size // (H * K), H, K,
                                 float(lower_bound), _ptr(g))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_gate failed with status {rc}")
    return g


def prologue(q_raw, k_raw, v_raw, gate_x, conv_w, A_log, dt_bias, cu_seqlens=None,
             lower_bound: float = -5.0, l2_eps: float = 1e-6, act: int = 0):
    """Short conv on q, k, v; L2-norm of q, k over the head dim; per-channel gate.

    q_raw, k_raw, gate_x: [B,T,H,K]; v_raw: [B,T,H,V]; conv_w: sequence of three
    [H*D, 4] weight arrays (q, k, v).  Returns fp64 (q, k, v, g) in the input shapes.
    """
    out = []
    for x, w in zip((q_raw, k_raw, v_raw), conv_w):
        x = _f64(x)
        shp = x.shape
        y = short_conv(x.reshape(shp[:-2] + (shp[-2] * shp[-1],)), w, cu_seqlens, act)
        out.append(y.reshape(shp))
    q, k, v = out
    q = l2norm(q, l2_eps)
    k = l2norm(k, l2_eps)
    g = gate(gate_x, A_log, dt_bias, lower_bound)
    return q, k, v, g


def output_gate(o, gate, weight=None, eps: float = 1e-6):
    """Output gate of the layer on o: per row of the last axis (length V),
    ``o / sqrt(mean(o^2) + eps) * weight * sigmoid(gate)``.

    o, gate: [..., V]; weight: [V] or None (ones).  Returns float64 in o's shape.
    """
    o = _f64(o)
    g = _f64(gate)
    if g.shape != o.shape:
        raise ValueError(f"gate has shape {g.shape}, expected {o.shape}")
    V = o.shape[-1]
    w = None
    if weight is not None:
        w = _f64(weight)
        if w.shape != (V,):
            raise ValueError(f"weight must be [{V}]")
    out = np.zeros_like(o)
    rc = _load().kda_oracle_output_gate(_ptr(o), _ptr(g), _ptr(w) if w is not None else None,
                                        o.size // V, V, float(eps), _ptr(out))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_output_gate failed with status {rc}")
    return out


def gate_proj(x, f_a, f_b, b_proj):
    """The forget gate's input and beta from the layer input (plain fp64 loops):
    per token, ``gate_x = f_b (f_a x)`` with the low-rank activation ``f_a x``
    kept unrounded, and ``beta = sigmoid(b_proj x)``.

    x: [..., D]; f_a [R, D]; f_b [HK, R]; b_proj [NH, D].  Returns float64
    (gate_x [..., HK], beta [..., NH]).
    """
    x, fa, fb, bp = (_f64(a) for a in (x, f_a, f_b, b_proj))
    D = x.shape[-1]
    R, HK, NH = fa.shape[0], fb.shape[0], bp.shape[0]
    if fa.shape != (R, D) or fb.shape != (HK, R) or bp.shape != (NH, D):
        raise ValueError("f_a must be [R, D], f_b [HK, R] and b_proj [NH, D]")
    rows = x.size // D
    gx = np.zeros(x.shape[:-1] + (HK,))
    beta = np.zeros(x.shape[:-1] + (NH,))
    rc = _load().kda_oracle_gate_proj(_ptr(x), _ptr(fa), _ptr(fb), _ptr(bp), rows, D, R, HK, NH, _ptr(gx),
                                      _ptr(beta))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_gate_proj failed with status {rc}")
    return gx, beta


def segment_transition(k, g, beta):
    """M = prod_t (I - beta_t k_t k_t^T) Diag(exp(g_t)) over a segment, later tokens
    on the left, per head: k, g [T, H, K] (or [1, T, H, K]), beta [T, H] -> M [H, K, K]
    float64 (explicit K x K products, numpy matmul)."""
    k, g, beta = (_f64(a) for a in (k, g, beta))
    if k.ndim == 4:
        k, g, beta = k[0], g[0], beta[0]
    T, H, K = k.shape
    M = np.broadcast_to(np.eye(K), (H, K, K)).copy()
    for t in range(T):
        for h in range(H):
            kt = k[t, h]
            step = (np.eye(K) - beta[t, h] * np.outer(kt, kt)) * np.exp(g[t, h])[None, :]
            M[h] = step @ M[h]
    return M


def state_compose(M, S, A=None):
    """M @ S + A per head (numpy matmul in float64): M [..., K, K], S and A [..., K, V]."""
    M, S = _f64(M), _f64(S)
    out = np.matmul(M, S)
    if A is not None:
        out = out + _f64(A)
    return out


def kda_backward(q, k, v, g, beta, dO, dS_T=None, scale=None, initial_state=None, cu_seqlens=None,
                 nthreads: int | None = None):
    """Gradients of ``<dO, o> + <dS_T, S_T>`` through :func:`kda_forward` (same
    shapes and conventions; dS_T [N, H, K, V] or None).  Returns a dict with dq,
    dk, dv, dg, dbeta (input shapes) and dS0 ([N, H, K, V]), all float64."""
    q, k, v, g, beta, dO = (_f64(a) for a in (q, k, v, g, beta, dO))
    lead = q.shape[:-2]
    H, K = q.shape[-2:]
    V = v.shape[-1]
    B, T = (lead if len(lead) == 2 else (1, lead[0]))
    if cu_seqlens is not None and B != 1:
        raise ValueError("cu_seqlens requires B == 1")
    cu = _seqlens(cu_seqlens, B * T, B, T)
    N = cu.shape[0] - 1
    if dO.shape != lead + (H, V):
        raise ValueError(f"dO has shape {dO.shape}")
    s0 = None if initial_state is None else _f64(initial_state)
    dst = None if dS_T is None else _f64(dS_T)
    for name, a in (("initial_state", s0), ("dS_T", dst)):
        if a is not None and a.shape != (N, H, K, V):
            raise ValueError(f"{name} has shape {a.shape}, expected {(N, H, K, V)}")
    if scale is None:
        scale = float(K) ** -0.5
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v), "dg": np.zeros_like(g),
           "dbeta": np.zeros_like(beta), "dS0": np.zeros((N, H, K, V))}
    rc = _load().kda_oracle_backward(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(s0) if s0 is not None else None, cu.ctypes.data_as(_i64p),
                                     N, H, K, V, float(scale), _ptr(dO), _ptr(dst) if dst is not None else None,
                                     _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                                     _ptr(out["dbeta"]), _ptr(out["dS0"]), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_backward failed with status {rc}")
    return out
