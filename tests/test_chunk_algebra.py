"""The chunked form of the KDA forward, written out in fp64 numpy, equals the
oracle's token-by-token recurrence.

This is the algebra the CUDA prefill kernels implement (chunk size 64, 16-token
sub-blocks for the gated intra-chunk products, UT transform, inter-chunk state
passing).  It is a check of that derivation against the oracle -- it shares no
code with the kernels and is not itself an oracle.  CPU only.
"""
import numpy as np
import pytest

import oracle

C = 64
SUB = 16


def chunk_forward(q, k, v, g, beta, scale, s0, cu):
    """q, k, g: [Ttot, H, K]; v: [Ttot, H, V]; beta: [Ttot, H]; s0: [N, H, K, V]."""
    Ttot, H, K = q.shape
    V = v.shape[-1]
    N = len(cu) - 1
    o = np.zeros((Ttot, H, V))
    sT = np.zeros((N, H, K, V))
    for n in range(N):
        for h in range(H):
            S = s0[n, h].copy()
            for c0 in range(cu[n], cu[n + 1], C):
                L = min(C, cu[n + 1] - c0)
                pad = lambda x: np.concatenate([x, np.zeros((C - L,) + x.shape[1:])])  # noqa: E731
                qc, kc, gc = pad(q[c0:c0 + L, h]), pad(k[c0:c0 + L, h]), pad(g[c0:c0 + L, h])
                vc, bc = pad(v[c0:c0 + L, h]), pad(beta[c0:c0 + L, h])
                G = np.cumsum(gc, axis=0)
                A = np.zeros((C, C))
                P = np.zeros((C, C))
                for R in range(C // SUB):
                    r0 = R * SUB
                    ref = G[r0 - 1] if r0 > 0 else np.zeros(K)
                    rows = slice(r0, r0 + SUB)
                    lk = kc[rows] * np.exp(G[rows] - ref)        # <= 1
                    lq = qc[rows] * np.exp(G[rows] - ref)
                    rk = kc[:r0 + SUB] * np.exp(ref - G[:r0 + SUB])  # <= 1 off-diagonal, <= e^80 on it
                    A[rows, :r0 + SUB] = lk @ rk.T
                    P[rows, :r0 + SUB] = lq @ rk.T
                A = np.tril(A, -1)
                P = np.tril(P)
                Tm = np.linalg.inv(np.eye(C) + bc[:, None] * A)
                Kt = kc * np.exp(G)
                Qt = qc * np.exp(G)
                Kb = kc * np.exp(G[-1] - G)
                W = Tm @ (bc[:, None] * Kt)
                Ut = Tm @ (bc[:, None] * vc)
                U = Ut - W @ S
                O = scale * (Qt @ S + P @ U)
                S = np.exp(G[-1])[:, None] * S + Kb.T @ U
                o[c0:c0 + L, h] = O[:L]
            sT[n, h] = S
    return o, sT


@pytest.mark.parametrize("lens", [[128], [64], [1], [200, 7, 64, 65, 0, 130]])
def test_chunk_form_equals_recurrence(lens):
    rng = np.random.default_rng(sum(lens) + len(lens))
    H, K, V = 2, 16, 8
    Ttot = sum(lens)
    q = rng.standard_normal((Ttot, H, K))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((Ttot, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((Ttot, H, V))
    g = np.maximum(-5.0, -np.logaddexp(0.0, rng.standard_normal((Ttot, H, K))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((Ttot, H))))
    s0 = rng.standard_normal((len(lens), H, K, V)) * 0.1
    cu = np.concatenate([[0], np.cumsum(lens)])
    o_ref, s_ref = oracle.kda_forward(q, k, v, g, beta, scale=K ** -0.5, initial_state=s0, cu_seqlens=cu)
    o, s = chunk_forward(q, k, v, g, beta, K ** -0.5, s0, cu)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12 * np.abs(o_ref).max())
    np.testing.assert_allclose(s, s_ref, rtol=0, atol=1e-12 * np.abs(s_ref).max())


def test_chunk_form_at_the_gate_lower_bound():
    """g = -5 everywhere: the in-chunk decay reaches e^-320; the sub-block
    reference points keep every factor finite and the result exact."""
    rng = np.random.default_rng(5)
    T, H, K, V = 130, 1, 8, 4
    q = rng.standard_normal((T, H, K))
    k = rng.standard_normal((T, H, K))
    v = rng.standard_normal((T, H, V))
    g = np.full((T, H, K), -5.0)
    beta = np.full((T, H), 0.5)
    cu = np.array([0, T])
    s0 = np.zeros((1, H, K, V))
    o_ref, s_ref = oracle.kda_forward(q, k, v, g, beta, scale=0.3, initial_state=s0, cu_seqlens=cu)
    o, s = chunk_forward(q, k, v, g, beta, 0.3, s0, cu)
    assert np.all(np.isfinite(o))
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12 * np.abs(o_ref).max())
    np.testing.assert_allclose(s, s_ref, rtol=0, atol=1e-12 * np.abs(s_ref).max())
