"""Context-parallel KDA prefill: one sequence split into consecutive segments.

The recurrence is affine in the state.  Over a segment of tokens,

    S_end = M S_start + S_zero,   M = prod_t (I - beta_t k_t k_t^T) Diag(e^{g_t})

(later tokens on the left), S_zero the segment's final state from a zero start.
Each segment (one per rank) therefore computes, independently of the others,

1. S_zero: ``kda_chunk_fwd`` over the segment from a zero state;
2. M: ``kda_chunk_fwd`` over the segment with v = 0, K-wide values and the
   identity as initial state (its final state is M itself);

then the segments exchange their (M, S_zero) -- one all-gather -- and every
rank forms its initial state by the prefix S_in(r + 1) = M_r S_in(r) + S_zero_r
(``kda_state_compose``), and reruns its segment from S_in(r) for its o and
final state.  The last rank's final state is the sequence's.

Two drivers share the prefix: :func:`cp_chunk_fwd` (one segment per rank of a
``torch.distributed`` group, the exchange an ``all_gather``) and
:func:`chunk_fwd_segmented` (all segments on one device, in turn).  Every step
runs in libkda.so's kernels; the segments are dense (B = 1, no cu_seqlens) and
need K = V.
"""
from __future__ import annotations

import torch

from .kda import chunk_fwd, state_compose


def segment_transition(k, g, beta):
    """M [1, H, K, K] of the segment (k, g [1, T, H, K], beta [1, T, H])."""
    B, T, H, K = k.shape
    if B != 1:
        raise ValueError("a segment is one sequence (B = 1)")
    zeros = torch.zeros_like(k)
    eye = torch.eye(K, dtype=torch.float32, device=k.device).expand(1, H, K, K).contiguous()
    _, M = chunk_fwd(k, k, zeros, g, beta, initial_state=eye)
    return M


def prefix_state(Ms, Ss, initial_state, upto: int, compose=None):
    """S_in of segment ``upto``: start from ``initial_state`` (None: zeros) and apply
    S <- M_r S + S_zero_r for r < upto.  ``compose(M, S, A)`` defaults to the
    library's state composition."""
    compose = compose or (lambda M, S, A: state_compose(M, S, A))
    S = initial_state if initial_state is not None else torch.zeros_like(Ss[0])
    for r in range(upto):
        S = compose(Ms[r], S, Ss[r])
    return S


def cp_chunk_fwd(q, k, v, g, beta, scale: float | None = None, initial_state=None, group=None):
    """This rank's segment of a sequence split across the ranks of ``group`` in rank
    order.  q, k, g [1, T_r, H, K]; v [1, T_r, H, V]; beta [1, T_r, H];
    initial_state: the sequence's initial state [1, H, K, V] (used by every rank;
    None: zeros).  Returns (o of the segment, the state after the segment)."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    _, s_zero = chunk_fwd(q, k, v, g, beta, scale=scale)
    M = segment_transition(k, g, beta)
    Ms = [torch.empty_like(M) for _ in range(world)]
    Ss = [torch.empty_like(s_zero) for _ in range(world)]
    dist.all_gather(Ms, M, group=group)
    dist.all_gather(Ss, s_zero, group=group)
    s_in = prefix_state(Ms, Ss, initial_state, rank)
    return chunk_fwd(q, k, v, g, beta, scale=scale, initial_state=s_in)


def chunk_fwd_segmented(q, k, v, g, beta, bounds, scale: float | None = None, initial_state=None):
    """The same on one device: the token axis of one sequence is cut at ``bounds``
    (increasing token offsets strictly inside (0, T)).  Returns (o, final state)."""
    T = q.shape[1]
    cuts = [0] + [int(b) for b in bounds] + [T]
    if any(b <= a for a, b in zip(cuts, cuts[1:])):
        raise ValueError("bounds must be increasing and strictly inside (0, T)")
    segs = [slice(a, b) for a, b in zip(cuts, cuts[1:])]
    parts = [tuple(x[:, s].contiguous() for x in (q, k, v, g, beta)) for s in segs]
    Ss, Ms = [], []
    for sq, sk, sv, sg, sb in parts:
        Ss.append(chunk_fwd(sq, sk, sv, sg, sb, scale=scale)[1])
        Ms.append(segment_transition(sk, sg, sb))
    outs, s_end = [], None
    for r, (sq, sk, sv, sg, sb) in enumerate(parts):
        s_in = prefix_state(Ms, Ss, initial_state, r)
        o, s_end = chunk_fwd(sq, sk, sv, sg, sb, scale=scale, initial_state=s_in)
        outs.append(o)
    return torch.cat(outs, dim=1), s_end
