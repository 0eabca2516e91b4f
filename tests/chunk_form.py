"""Chunkwise form of the KDA recurrence in fp64 numpy (test-only).

This is the re-association the CUDA prefill kernel is built on, written out
plainly so the CPU tests can pin the algebra against the token-by-token
oracle.  It is not used by the product.

Derivation (one head, one chunk of C tokens, incoming state S0).  With
alpha_t = exp(g_t) the recurrence of "Kimi K3 Architecture Explained",
Step 3, multiplies out to

    S_t = Diag(alpha_t) S_{t-1} + k_t u_t^T,
    u_t = beta_t (v_t - S_{t-1}^T (alpha_t * k_t)).

Let G_t = sum_{s<=t} g_s inside the chunk, K+ = exp(G) * K, K- = exp(-G) * K,
Q+ = exp(G) * Q.  Unrolling gives

    (I + L) U = diag(beta) (V - K+ S0),  L = strict_lower(diag(beta) K+ K-^T)
    U  = Ut - W S0,   W = (I+L)^-1 diag(beta) K+,   Ut = (I+L)^-1 diag(beta) V
    O  = Q+ S0 + P U, P = lower_with_diagonal(Q+ K-^T)   (read after update)
    S_C = Diag(exp(G_C)) S0 + Khat^T U,  Khat_t = exp(G_C - G_t) * k_t

which is the "UT transform and pseudo-value term" that "From GPT-2 to Kimi
K3, from first principles", Chapter 6, names without the algebra.
"""
import numpy as np


def chunk_recurrence(q, k, v, g, beta, S0, C):
    """One head, one document.  q,k,g: [T, dk]; v: [T, dv]; beta: [T]."""
    T = q.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    out = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, C):
        sl = slice(c0, min(c0 + C, T))
        n = sl.stop - sl.start
        G = np.cumsum(g[sl], axis=0)
        Kp, Km, Qp = np.exp(G) * k[sl], np.exp(-G) * k[sl], np.exp(G) * q[sl]
        b = beta[sl][:, None]
        L = np.tril(b * (Kp @ Km.T), -1)
        A = np.eye(n) + L
        W = np.linalg.solve(A, b * Kp)
        Ut = np.linalg.solve(A, b * v[sl])
        U = Ut - W @ S
        P = np.tril(Qp @ Km.T)
        out[sl] = Qp @ S + P @ U
        Khat = np.exp(G[-1] - G) * k[sl]
        S = np.exp(G[-1])[:, None] * S + Khat.T @ U
    return out, S
