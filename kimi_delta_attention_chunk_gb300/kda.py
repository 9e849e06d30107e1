"""Thin ctypes binding of libkda.so (C ABI in include/kda.h).

Marshalling only: every function checks that the tensors live on the current
CUDA device, picks the dtype codes, and forwards raw device pointers, sizes and
the current CUDA stream to the library.  All arithmetic runs in the library's
kernels; there is no CPU or PyTorch fallback, and a missing library raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "libkda.so"
_lock = threading.Lock()
_lib = None

KDA_F32, KDA_BF16 = 0, 1
_STATUS = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_WORKSPACE",
           4: "KDA_ERR_CUDA", 5: "KDA_ERR_RANGE", 6: "KDA_ERR_TIMEOUT"}

# (name, restype, argtypes) of every exported symbol of include/kda.h
_vp, _fp, _i32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
_i, _f, _sz, _u32 = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint32
SIGNATURES = {
    "kda_status_string": (ctypes.c_char_p, [_i]),
    "kda_abi_version": (_i, []),
    "kda_chunk_fwd_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "kda_chunk_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _f, _fp, _i32p, _i, _i, _i, _i, _i, _i,
                           _vp, _i, _fp, _vp, _sz, _i32p, _vp]),
    "kda_chunk_fwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _f, _fp, _i32p, _i, _i, _i, _i, _i,
                                   _i, _vp, _i, _fp, _vp]),
    "kda_chunk_fwd_fused": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _fp, _fp, _fp, _i, _fp, _fp, _f, _f,
                                 _f, _fp, _i32p, _i, _i, _i, _i, _i, _i, _vp, _i, _fp, _vp, _sz, _i32p,
                                 _vp]),
    "kda_trace_events": (None, [_vp, _vp, _vp]),
    "kda_set_wait_limit": (None, [_u32]),
    "kda_inject_wait_timeout": (None, [_i]),
    "kda_recurrent_step": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _f, _fp, _i, _i, _i, _i, _vp, _i,
                                _vp]),
    "kda_output_gate": (_i, [_fp, _vp, _i, _fp, _f, _i, _i, _i, _i, _vp, _i, _vp]),
    "kda_gate_proj_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "kda_gate_proj": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _sz, _i32p, _vp]),
    "kda_state_compose": (_i, [_fp, _fp, _fp, _fp, _i, _i, _i, _vp]),
    "kda_check_range": (_i, [_vp, _i, ctypes.c_int64, _f, _f, _vp, _vp]),
    "kda_recurrent_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "kda_chunk_bwd_workspace_size": (_sz, [_i, _i, _i, _i, _i, _i, _i, _i]),
    "kda_chunk_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _f, _fp, _i32p, _i, _i, _i, _i, _i, _i,
                           _fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, _vp, _sz, _i32p, _vp]),
    "kda_recurrent_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _f, _fp, _i32p, _i, _i, _i, _i, _i, _i,
                               _fp, _fp, _fp, _fp, _fp, _fp, _fp, _fp, _vp, _sz, _i32p, _vp]),
}


class KDAError(RuntimeError):
    """A libkda.so call returned a non-OK status."""

    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)}")
        self.status = status


def library_path() -> str:
    return os.environ.get("KDA_LIBRARY", os.path.join(_PKG, _LIB_NAME))


def load_library():
    """Load libkda.so (built by ``build.py``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise ImportError(f"{path} is missing: build it with "
                                  "`python -m kimi_delta_attention_chunk_gb300.build`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensors passed to libkda must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to libkda must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise KDAError(fn, status)


def _dt_of(dtype) -> int:
    if dtype == torch.bfloat16:
        return KDA_BF16
    if dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {dtype}")


def workspace_size(in_dtype, B: int, T: int, H: int, K: int, V: int, N: int, packed: bool) -> int:
    """Device workspace bytes ``kda_chunk_fwd`` / ``kda_chunk_fwd_fused`` need."""
    return int(load_library().kda_chunk_fwd_workspace_size(_dt_of(in_dtype), B, T, H, K, V, N, int(packed)))


def bwd_workspace_size(in_dtype, B: int, T: int, H: int, K: int, V: int, N: int, packed: bool,
                       token_by_token: bool = False) -> int:
    """Device workspace bytes ``kda_chunk_bwd`` (or, with ``token_by_token``,
    ``kda_recurrent_bwd``) needs."""
    lib = load_library()
    fn = lib.kda_recurrent_bwd_workspace_size if token_by_token else lib.kda_chunk_bwd_workspace_size
    return int(fn(_dt_of(in_dtype), B, T, H, K, V, N, int(packed)))


def _workspace(nbytes: int, device, workspace):
    """The caller's workspace tensor (checked), or a fresh uint8 one of nbytes."""
    if workspace is None:
        if nbytes == 0:
            return None, 0
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
    elif workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError(f"workspace holds {workspace.numel() * workspace.element_size()} bytes, "
                         f"the call needs {nbytes}")
    return workspace, workspace.numel() * workspace.element_size()


def set_wait_limit(iterations: int = 0):
    """Testing hook: polls before a bounded device-side wait of the tensor-core
    prefill gives up (0 restores the default)."""
    load_library().kda_set_wait_limit(int(iterations))


def inject_wait_timeout(kernel: int):
    """Testing hook: the next tensor-core prefill or chunked backward call on this
    thread makes the first wait of its chunk-local (1), state (2), backward chain
    (3) or backward chunk (4) kernel one that nothing completes, so that it gives
    up and reports KDA_ERR_TIMEOUT."""
    load_library().kda_inject_wait_timeout(int(kernel))


def chunk_fwd(q, k, v, g, beta, scale: float | None = None, initial_state=None, cu_seqlens=None,
              output_final_state: bool = True, o_dtype=torch.float32, o=None, final_state=None,
              workspace=None, status=None):
    """Chunked KDA prefill.  q, k, g: [B,T,H,K]; v: [B,T,H,V]; beta: [B,T,H].

    Returns (o [B,T,H,V] in ``o_dtype``, final_state [N,H,K,V] fp32 or None).
    ``cu_seqlens`` (int32 [N+1], on the device) packs N sequences into B == 1.
    ``final_state`` may be the ``initial_state`` tensor itself (in-place update).
    ``workspace``: a device tensor of at least :func:`workspace_size` bytes (a
    fresh one from torch's allocator when None).  ``status``: an optional device
    int32 tensor that receives the call's device-side status (0, or 6 =
    KDA_ERR_TIMEOUT when a bounded wait gave up); read it after the stream work.
    """
    lib = load_library()
    B, T, H, K = q.shape
    V = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty((B, T, H, V), dtype=o_dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, K, V), dtype=torch.float32, device=q.device)
    ws, ws_bytes = _workspace(workspace_size(q.dtype, B, T, H, K, V, N, cu_seqlens is not None), q.device,
                              workspace)
    st = lib.kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dt(q),
                           float(scale or 0.0), _ptr(initial_state), _ptr(cu_seqlens),
                           B, T, H, K, V, N, _ptr(o), _dt(o), _ptr(final_state), _ptr(ws), ws_bytes,
                           _ptr(status), _stream(q.device))
    _check("kda_chunk_fwd", st)
    return o, final_state


def chunk_fwd_noalloc(q, k, v, g, beta, scale: float | None = None, initial_state=None, cu_seqlens=None,
                      output_final_state: bool = True, o_dtype=torch.float32, o=None, final_state=None):
    """``chunk_fwd`` through ``kda_chunk_fwd_noalloc``: the library allocates no
    device memory for the call (its workspace is a fixed 64 MiB array, so only
    small calls fit; bf16 inputs with K = V = 128 only).  For callers whose
    device memory is all reserved by their own allocator.  ``o`` and
    ``final_state`` can be passed in so that nothing at all is allocated."""
    lib = load_library()
    B, T, H, K = q.shape
    V = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty((B, T, H, V), dtype=o_dtype, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, K, V), dtype=torch.float32, device=q.device)
    st = lib.kda_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dt(q),
                                   float(scale or 0.0), _ptr(initial_state), _ptr(cu_seqlens),
                                   B, T, H, K, V, N, _ptr(o), _dt(o), _ptr(final_state), _stream(q.device))
    _check("kda_chunk_fwd_noalloc", st)
    return o, final_state


def chunk_fwd_fused(q_raw, k_raw, v_raw, gate_x, beta, conv_w, A_log, dt_bias,
                    scale: float | None = None, initial_state=None, cu_seqlens=None,
                    lower_bound: float = -5.0, l2_eps: float = 1e-6, conv_act: int = 0,
                    output_final_state: bool = True, o_dtype=torch.float32, o=None,
                    final_state=None, workspace=None, status=None):
    """Chunked prefill with the fused prologue (short conv, L2-norm, gate).

    conv_w: a sequence (conv_q [H*K,4], conv_k [H*K,4], conv_v [H*V,4]) of fp32
    tensors, or one [3, H*D, 4] tensor whose leading rows are used.  ``workspace``
    and ``status`` as for :func:`chunk_fwd`.
    """
    lib = load_library()
    B, T, H, K = q_raw.shape
    V = v_raw.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    if isinstance(conv_w, torch.Tensor):
        cq = conv_w[0, : H * K].contiguous()
        ck = conv_w[1, : H * K].contiguous()
        cv = conv_w[2, : H * V].contiguous()
    else:
        cq, ck, cv = (w.contiguous() for w in conv_w)
    if o is None:
        o = torch.empty((B, T, H, V), dtype=o_dtype, device=q_raw.device)
    if final_state is None and output_final_state:
        final_state = torch.empty((N, H, K, V), dtype=torch.float32, device=q_raw.device)
    ws, ws_bytes = _workspace(workspace_size(q_raw.dtype, B, T, H, K, V, N, cu_seqlens is not None),
                              q_raw.device, workspace)
    st = lib.kda_chunk_fwd_fused(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(gate_x), _ptr(beta),
                                 _dt(q_raw), _ptr(cq), _ptr(ck), _ptr(cv), int(conv_act), _ptr(A_log),
                                 _ptr(dt_bias), float(lower_bound), float(l2_eps), float(scale or 0.0),
                                 _ptr(initial_state), _ptr(cu_seqlens), B, T, H, K, V, N, _ptr(o),
                                 _dt(o), _ptr(final_state), _ptr(ws), ws_bytes, _ptr(status),
                                 _stream(q_raw.device))
    _check("kda_chunk_fwd_fused", st)
    return o, final_state


def trace_events(begin=None, split=None, end=None):
    """Have the next prefill call on this thread record these torch.cuda.Event
    objects on its stream: before its first kernel, after the chunk-local
    kernel, after its last kernel (tensor-core path only)."""
    lib = load_library()
    h = []
    for e in (begin, split, end):
        if e is None:
            h.append(None)
        else:
            if not e.cuda_event:  # torch creates the CUDA event on first record
                e.record()
            h.append(e.cuda_event)
    lib.kda_trace_events(*h)


def recurrent_step(q, k, v, g, beta, state, scale: float | None = None, o_dtype=torch.float32, o=None):
    """One decode token per sequence; ``state`` [N,H,K,V] fp32 is updated in place.

    q, k, g: [N,H,K]; v: [N,H,V]; beta: [N,H].  Returns o [N,H,V].
    """
    lib = load_library()
    N, H, K = q.shape
    V = v.shape[-1]
    if o is None:
        o = torch.empty((N, H, V), dtype=o_dtype, device=q.device)
    st = lib.kda_recurrent_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dt(q),
                                float(scale or 0.0), _ptr(state), N, H, K, V, _ptr(o), _dt(o),
                                _stream(q.device))
    _check("kda_recurrent_step", st)
    return o


def output_gate(o, gate, weight=None, eps: float = 1e-6, out_dtype=torch.float32, out=None):
    """The layer's output gate, ``o / sqrt(mean(o^2) + eps) * weight * sigmoid(gate)``
    per (token, head) row of V values.

    o: [B,T,H,V] or [N,H,V] fp32; gate: same shape (bf16 or fp32); weight: [V] fp32
    or None.  ``out`` may be ``o`` itself for an fp32 result.  Returns out.
    """
    lib = load_library()
    if o.dim() == 3:
        (B, T), (H, V) = (1, o.shape[0]), o.shape[1:]
    else:
        B, T, H, V = o.shape
    if tuple(gate.shape) != tuple(o.shape):
        raise ValueError(f"gate has shape {tuple(gate.shape)}, expected {tuple(o.shape)}")
    if out is None:
        out = torch.empty(o.shape, dtype=out_dtype, device=o.device)
    st = lib.kda_output_gate(_ptr(o), _ptr(gate), _dt(gate), _ptr(weight), float(eps), B, T, H, V,
                             _ptr(out), _dt(out), _stream(o.device))
    _check("kda_output_gate", st)
    return out


def gate_proj_workspace_size(B: int, T: int, D: int, R: int, NH: int) -> int:
    """Device workspace bytes ``kda_gate_proj`` needs (the split partial sums and
    y = f_a x between its kernels)."""
    return int(load_library().kda_gate_proj_workspace_size(B, T, D, R, NH))


def gate_proj(x, f_a, f_b, b_proj, gate_x=None, beta=None, workspace=None, status=None):
    """The projections ahead of the gate: ``gate_x = f_b (f_a x)`` and
    ``beta = sigmoid(b_proj x)`` per token, bf16 in and out.

    x: [B,T,D] (or [T,D]); f_a [R,D]; f_b [HK,R]; b_proj [NH,D].  Returns
    (gate_x [B,T,HK], beta [B,T,NH]), the shapes ``chunk_fwd_fused`` takes as
    [B,T,H,K] and [B,T,H].  ``workspace``/``status`` as for :func:`chunk_fwd`.
    """
    lib = load_library()
    xs = x if x.dim() == 3 else x.unsqueeze(0)
    B, T, D = xs.shape
    R, HK, NH = f_a.shape[0], f_b.shape[0], b_proj.shape[0]
    if tuple(f_a.shape) != (R, D) or tuple(f_b.shape) != (HK, R) or tuple(b_proj.shape) != (NH, D):
        raise ValueError("f_a must be [R, D], f_b [HK, R] and b_proj [NH, D]")
    for t in (f_a, f_b, b_proj):
        if t.dtype != x.dtype:
            raise TypeError("x, f_a, f_b and b_proj must share one dtype")
    if gate_x is None:
        gate_x = torch.empty((B, T, HK), dtype=x.dtype, device=x.device)
    if beta is None:
        beta = torch.empty((B, T, NH), dtype=x.dtype, device=x.device)
    ws, ws_bytes = _workspace(gate_proj_workspace_size(B, T, D, R, NH), x.device, workspace)
    st = lib.kda_gate_proj(_ptr(xs), _ptr(f_a), _ptr(f_b), _ptr(b_proj), _dt(x), B, T, D, R, HK, NH,
                           _ptr(gate_x), _ptr(beta), _ptr(ws), ws_bytes, _ptr(status), _stream(x.device))
    _check("kda_gate_proj", st)
    return gate_x, beta


def state_compose(M, S, A=None, out=None):
    """out[h] = M[h] @ S[h] + A[h] for every head: M [..., H, K, K], S and A
    [..., H, K, V] fp32 (leading dims flattened into heads).  ``out`` may be A."""
    lib = load_library()
    K, V = S.shape[-2:]
    H = S.numel() // (K * V)
    if M.shape[-2:] != (K, K) or M.numel() != H * K * K:
        raise ValueError(f"M has shape {tuple(M.shape)}")
    if out is None:
        out = torch.empty_like(S)
    st = lib.kda_state_compose(_ptr(M), _ptr(S), _ptr(A), _ptr(out), H, K, V, _stream(S.device))
    _check("kda_state_compose", st)
    return out


def check_range(x, lo: float = -5.0, hi: float = 0.0, status=None, sync: bool = True):
    """Debug range check on the device (default: the log-decay precondition
    g in [-5, 0]).  With ``sync`` the stream is synchronised and KDAError
    (KDA_ERR_RANGE) is raised for an element outside [lo, hi] or NaN; without it
    the device status word (int32 tensor, 0 or 5) is returned for the caller to
    read later."""
    lib = load_library()
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=x.device)
    st = lib.kda_check_range(_ptr(x), _dt(x), x.numel(), float(lo), float(hi), _ptr(status),
                             _stream(x.device))
    _check("kda_check_range", st)
    if sync:
        code = int(status.item())
        _check("kda_check_range", code)
    return status


def chunk_bwd(q, k, v, g, beta, dO, dS_T=None, scale: float | None = None, initial_state=None,
              cu_seqlens=None, workspace=None, status=None, token_by_token: bool = False):
    """Gradients of <dO, o> + <dS_T, S_T> through :func:`chunk_fwd` (same shapes;
    dO fp32 [B,T,H,V], dS_T fp32 [N,H,K,V] or None).  Returns a dict of fp32
    tensors dq, dk, dv, dg, dbeta and dS0 ([N,H,K,V]).  ``workspace`` (at least
    :func:`bwd_workspace_size` bytes) and ``status`` as for :func:`chunk_fwd`
    (the status word reads 5 = KDA_ERR_RANGE when malformed offsets made the
    token-by-token path skip a sequence).  ``kda_chunk_bwd`` runs by default
    (chunk by chunk for bf16 with K = V = 128); ``token_by_token`` calls
    ``kda_recurrent_bwd``."""
    lib = load_library()
    B, T, H, K = q.shape
    V = v.shape[-1]
    N = B if cu_seqlens is None else cu_seqlens.numel() - 1
    dev = q.device
    f32 = torch.float32
    out = {"dq": torch.empty((B, T, H, K), dtype=f32, device=dev),
           "dk": torch.empty((B, T, H, K), dtype=f32, device=dev),
           "dv": torch.empty((B, T, H, V), dtype=f32, device=dev),
           "dg": torch.empty((B, T, H, K), dtype=f32, device=dev),
           "dbeta": torch.empty((B, T, H), dtype=f32, device=dev),
           "dS0": torch.empty((N, H, K, V), dtype=f32, device=dev)}
    ws, ws_bytes = _workspace(bwd_workspace_size(q.dtype, B, T, H, K, V, N, cu_seqlens is not None,
                                                 token_by_token), dev, workspace)
    name = "kda_recurrent_bwd" if token_by_token else "kda_chunk_bwd"
    st = getattr(lib, name)(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _dt(q), float(scale or 0.0),
                            _ptr(initial_state), _ptr(cu_seqlens), B, T, H, K, V, N, _ptr(dO), _ptr(dS_T),
                            _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]),
                            _ptr(out["dbeta"]), _ptr(out["dS0"]), _ptr(ws), ws_bytes, _ptr(status),
                            _stream(dev))
    _check(name, st)
    return out
