"""The chunked form of the KDA backward, written out in fp64 numpy, equals the
oracle's token-by-token reverse mode.

Per chunk of C = 64 tokens (entering state S, G the in-chunk cumulative
log-decay, E = e^G, E_C = e^{G_C}):

    forward   X = k E,  Y = k / E,  Xq = q E,  A = tril(X Y^T, -1),  P = tril(Xq Y^T)
              T = (I + Diag(beta) A)^{-1},  W = T Diag(beta) X,  U~ = T Diag(beta) v
              U = U~ - W S,  O = scale (Xq S + P U),  S' = Diag(E_C) S + Kb^T U  (Kb = k E_C / E)
    backward  dU = scale P^T dO + Kb dS',   dS = scale Xq^T dO + Diag(E_C) dS' - W^T dU
              dP = scale tril(dO U^T),  dW = -dU S^T,  dKb = U dS'^T
              dT = dW (Diag(beta) X)^T + dU (Diag(beta) v)^T,  dM = -T^T dT T^T
              dA = Diag(beta) tril(dM, -1),  dbeta = rowsum(dM A) + rowsum((T^T dW) X) + rowsum((T^T dU) v)
              then the products X Y^T, Xq Y^T and the factors e^{+-G} back to k, q and G,
              and dg = reverse cumulative sum of dG over the chunk.

The chunks run backwards with dS carried between them (the reverse of the
forward's state passing), from the entry states of a forward sweep.  This is
the derivation a chunked backward kernel implements, checked against the
oracle; it shares no code with the CUDA path and is not itself an oracle.
CPU only.
"""
import numpy as np
import pytest

import oracle

C = 64


def _chunks(lo, hi):
    return [(c0, min(C, hi - c0)) for c0 in range(lo, hi, C)]


def chunk_backward(q, k, v, g, beta, scale, s0, cu, dO, dST):
    """q, k, g [Ttot, H, K]; v, dO [Ttot, H, V]; beta [Ttot, H]; s0, dST [N, H, K, V]."""
    Ttot, H, K = q.shape
    V = v.shape[-1]
    N = len(cu) - 1
    out = {"dq": np.zeros_like(q), "dk": np.zeros_like(k), "dv": np.zeros_like(v), "dg": np.zeros_like(g),
           "dbeta": np.zeros_like(beta), "dS0": np.zeros((N, H, K, V))}
    for n in range(N):
        for h in range(H):
            chunks = _chunks(cu[n], cu[n + 1])

            def pad(x, c0, L):
                return np.concatenate([x[c0:c0 + L, h], np.zeros((C - L,) + x.shape[2:])])

            # forward sweep: the state entering each chunk
            S = s0[n, h].copy()
            S_in, saved = [], []
            for c0, L in chunks:
                qc, kc, vc, gc, bc = (pad(x, c0, L) for x in (q, k, v, g, beta))
                G = np.cumsum(gc, axis=0)
                E, EC = np.exp(G), np.exp(G[-1])
                X, Y, Xq, Kb = kc * E, kc / E, qc * E, kc * EC / E
                A = np.tril(X @ Y.T, -1)
                P = np.tril(Xq @ Y.T)
                Tm = np.linalg.inv(np.eye(C) + bc[:, None] * A)
                W = Tm @ (bc[:, None] * X)
                Ut = Tm @ (bc[:, None] * vc)
                U = Ut - W @ S
                S_in.append(S)
                saved.append((qc, kc, vc, bc, E, EC, X, Y, Xq, Kb, A, P, Tm, W, U))
                S = EC[:, None] * S + Kb.T @ U
            # backward sweep
            dS = dST[n, h].copy()
            for (c0, L), S, sv in zip(reversed(chunks), reversed(S_in), reversed(saved)):
                qc, kc, vc, bc, E, EC, X, Y, Xq, Kb, A, P, Tm, W, U = sv
                dOc = pad(dO, c0, L)
                dU = scale * P.T @ dOc + Kb @ dS
                dS_prev = scale * Xq.T @ dOc + EC[:, None] * dS - W.T @ dU
                dXq = scale * dOc @ S.T                      # through O = scale Xq S
                dP = scale * np.tril(dOc @ U.T)
                dKb = U @ dS.T
                dEC = np.sum(dS * S, axis=1)                 # through Diag(E_C) S
                dW = -dU @ S.T
                dT = dW @ (bc[:, None] * X).T + dU @ (bc[:, None] * vc).T
                dBk, dBv = Tm.T @ dW, Tm.T @ dU
                dM = -Tm.T @ dT @ Tm.T
                dA = bc[:, None] * np.tril(dM, -1)
                db = np.sum(dM * A, axis=1) + np.sum(dBk * X, axis=1) + np.sum(dBv * vc, axis=1)
                dX = bc[:, None] * dBk + dA @ Y              # W = T Diag(beta) X and A = X Y^T
                dY = dA.T @ X + dP.T @ Xq                    # A and P = Xq Y^T
                dXq = dXq + dP @ Y
                dvc = bc[:, None] * dBv
                dkc = dX * E + dY / E + dKb * EC / E
                dqc = dXq * E
                dG = dX * X - dY * Y + dXq * Xq - dKb * Kb
                dG[-1] += dEC * EC + np.sum(dKb * Kb, axis=0)  # G_C = G[-1]
                dgc = np.cumsum(dG[::-1], axis=0)[::-1]        # G = cumsum(g)
                sl = slice(c0, c0 + L)
                out["dq"][sl, h] = dqc[:L]
                out["dk"][sl, h] = dkc[:L]
                out["dv"][sl, h] = dvc[:L]
                out["dg"][sl, h] = dgc[:L]
                out["dbeta"][sl, h] = db[:L]
                dS = dS_prev
            out["dS0"][n, h] = dS
    return out


@pytest.mark.parametrize("lens", [[64], [130], [1], [70, 0, 5, 64]])
def test_chunk_backward_equals_reverse_mode(lens):
    rng = np.random.default_rng(7 * sum(lens) + len(lens))
    H, K, V = 2, 8, 5
    Ttot = sum(lens)
    q = rng.standard_normal((Ttot, H, K))
    k = rng.standard_normal((Ttot, H, K))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((Ttot, H, V))
    g = np.maximum(-5.0, -np.logaddexp(0.0, rng.standard_normal((Ttot, H, K))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((Ttot, H))))
    s0 = rng.standard_normal((len(lens), H, K, V)) * 0.1
    dO = rng.standard_normal((Ttot, H, V))
    dST = rng.standard_normal((len(lens), H, K, V))
    cu = np.concatenate([[0], np.cumsum(lens)])
    ref = oracle.kda_backward(q, k, v, g, beta, dO, dS_T=dST, scale=K ** -0.5, initial_state=s0, cu_seqlens=cu)
    got = chunk_backward(q, k, v, g, beta, K ** -0.5, s0, cu, dO, dST)
    for key in ("dq", "dk", "dv", "dg", "dbeta", "dS0"):
        scale_ = max(np.abs(ref[key]).max(), 1e-30)
        np.testing.assert_allclose(got[key], ref[key], rtol=0, atol=1e-12 * scale_, err_msg=key)
