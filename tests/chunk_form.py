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


def chunk_recurrence(q, k, v, g, beta, S0, C, reassociated=False):
    """One head, one document.  q,k,g: [T, dk]; v: [T, dv]; beta: [T].

    reassociated=True takes U = Tb (V - K+ S0) with Tb = (I+L)^-1 diag(beta)
    (the order the CUDA prefill computes it in: the state products first,
    then one product with Tb) instead of Ut - W S0."""
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
        if reassociated:
            Tb = np.linalg.solve(A, np.diag(beta[sl]))
            U = Tb @ (v[sl] - Kp @ S)
        else:
            W = np.linalg.solve(A, b * Kp)
            Ut = np.linalg.solve(A, b * v[sl])
            U = Ut - W @ S
        P = np.tril(Qp @ Km.T)
        out[sl] = Qp @ S + P @ U
        Khat = np.exp(G[-1] - G) * k[sl]
        S = np.exp(G[-1])[:, None] * S + Khat.T @ U
    return out, S


def gram_tiled(k, q, g, beta, tile=16):
    """L and P of one chunk through per-tile reference points, the way the
    CUDA prefill forms its Gram operands so that every factor stays inside
    fp32 range.  k, q, g: [C, dk] (C a multiple of `tile`); beta: [C].

    Row tile a (tokens of tile a) uses its start s_a = G before the tile:
    left rows k_i e^{G_i - s_a} (and q_i e^{G_i - s_a}).  A column token j of
    tile b <= a uses its tile's end e_b = G after tile b: k_j e^{e_b - G_j},
    times e^{s_a - e_b} per channel.  The product of the three factors is
    e^{G_i - G_j}, so L = strict_lower(diag(beta) K+ K-^T) and
    P = lower_with_diagonal(Q+ K-^T) come out unchanged.  Returns (L, P, the
    largest factor used)."""
    C, dk = k.shape
    G = np.cumsum(g, axis=0)
    start = np.vstack([np.zeros((1, dk)), G[tile - 1:-1:tile]])   # s_a, one row per tile
    end = G[tile - 1::tile]                                         # e_b
    L, P = np.zeros((C, C)), np.zeros((C, C))
    biggest = 0.0
    for a in range(C // tile):
        rows = slice(a * tile, (a + 1) * tile)
        left_k = np.exp(G[rows] - start[a]) * k[rows]
        left_q = np.exp(G[rows] - start[a]) * q[rows]
        biggest = max(biggest, float(np.exp(G[rows] - start[a]).max()))
        for b in range(a + 1):
            cols = slice(b * tile, (b + 1) * tile)
            f_col = np.exp(end[b] - G[cols])
            f_pair = np.exp(start[a] - end[b])
            biggest = max(biggest, float(f_col.max()), float(f_pair.max()))
            right = f_col * f_pair * k[cols]
            L[rows, cols] = left_k @ right.T
            P[rows, cols] = left_q @ right.T
    return np.tril(beta[:, None] * L, -1), np.tril(P), biggest


def verify_pairs(q, k, v, g, beta, S0):
    """Draft tokens two per pass, the algebra of the CUDA verify kernel.
    One head; q, k, g: [K, dk]; v: [K, dv]; beta: [K].  For tokens t, t+1:

        a_t = (alpha_t k_t)^T S,  b_t = (alpha_t q_t)^T S
        u_t = beta_t (v_t - a_t),  o_t = b_t + u_t (k_t . q_t)
        (D_{t+1} S_t)^T x = (alpha_{t+1} alpha_t x)^T S + ((alpha_{t+1} x) . k_t) u_t

    for x = k_{t+1} (its error term) and x = q_{t+1} (its read), with S the
    state before token t; then S <- D_{t+1} (D_t S + k_t u_t^T) + k_{t+1} u_{t+1}^T.
    An odd last token runs alone.  Returns (outputs [K, dv], final state)."""
    S = np.array(S0, dtype=np.float64, copy=True)
    K = q.shape[0]
    out = np.zeros((K, v.shape[1]))
    t = 0
    while t < K:
        a1 = np.exp(g[t])
        u1 = beta[t] * (v[t] - (a1 * k[t]) @ S)
        out[t] = (a1 * q[t]) @ S + u1 * (k[t] @ q[t])
        if t + 1 == K:
            S = a1[:, None] * S + np.outer(k[t], u1)
            break
        a2 = np.exp(g[t + 1])
        e2 = (a2 * a1 * k[t + 1]) @ S + ((a2 * k[t + 1]) @ k[t]) * u1
        r2 = (a2 * a1 * q[t + 1]) @ S + ((a2 * q[t + 1]) @ k[t]) * u1
        u2 = beta[t + 1] * (v[t + 1] - e2)
        out[t + 1] = r2 + u2 * (k[t + 1] @ q[t + 1])
        S = a2[:, None] * (a1[:, None] * S + np.outer(k[t], u1)) + np.outer(k[t + 1], u2)
        t += 2
    return out, S



def block_inverse(L, tile=16):
    """T = (I + L)^-1 for a strictly lower 64 x 64 L, in the stages of the
    CUDA prefill (16 x 16 blocks, a, b = 0..3).  With N = I + L split into
    its diagonal blocks and the rest, D = the inverses of the diagonal blocks
    (forward substitution) and M = N_offdiag D (strictly block lower, M^4 = 0):

        T = D (I + M)^-1 = D (I - M + M^2 - M^3)

    stage 1: the six M_ab = L_ab D_bb;
    stage 2: T_{a,a-1} = -D_aa M_{a,a-1},  V20 = M21 M10 - M20,
             V31 = M32 M21 - M31,  Y30 = M31 M10 - M30;
    stage 3: T20 = D22 V20,  T31 = D33 V31,  T30 = D33 Y30 + T32 V20."""
    n = L.shape[0]
    nb = n // tile
    assert nb == 4
    blk = lambda X, a, b: X[a * tile:(a + 1) * tile, b * tile:(b + 1) * tile]
    D = []
    for a in range(nb):                          # forward substitution per diagonal block
        Na = np.eye(tile) + blk(L, a, a)
        Da = np.zeros((tile, tile))
        for i in range(tile):
            Da[i, i] = 1.0
            for j in range(i):
                Da[i, j] = -sum(Na[i, m] * Da[m, j] for m in range(j, i))
        D.append(Da)
    M = {(a, b): blk(L, a, b) @ D[b] for a in range(nb) for b in range(a)}
    T = np.zeros((n, n))
    put = lambda a, b, X: T.__setitem__((slice(a * tile, (a + 1) * tile),
                                         slice(b * tile, (b + 1) * tile)), X)
    for a in range(nb):
        put(a, a, D[a])
    for a in range(1, nb):
        put(a, a - 1, -D[a] @ M[a, a - 1])
    V20 = M[2, 1] @ M[1, 0] - M[2, 0]
    V31 = M[3, 2] @ M[2, 1] - M[3, 1]
    Y30 = M[3, 1] @ M[1, 0] - M[3, 0]
    put(2, 0, D[2] @ V20)
    put(3, 1, D[3] @ V31)
    T32 = -D[3] @ M[3, 2]
    put(3, 0, D[3] @ Y30 + T32 @ V20)
    return T


def segmented_three_pass(q, k, v, g, beta, S0, nseg, prefill):
    """One document as `nseg` segments of whole 64-token chunks, joined the
    way the segment-scan prefill joins them (test-only; `prefill` is any
    exact single-document prefill, here the oracle's recurrence).  The
    recurrence is linear in (v, S_in), and over a segment S_out = P S_in + R:
      1. v as given, segment 0 from S0, the others from zero: outputs o^0, R_s;
      2. v = 0 from the identity: P_s;
      3. S_1 = R_0, S_{s+1} = P_s S_s + R_s;
      4. v = 0 from S_s: the outputs the incoming state adds, o = o^0 + o^S.
    Shapes as the oracle's: q, k, g [T, H, d]; v [T, H, d]; S0 [1, H, d, d]."""
    T, H, d = q.shape
    chunks = -(-T // 64)
    seg_len = -(-chunks // nseg) * 64
    bounds = [(s0, min(s0 + seg_len, T)) for s0 in range(0, T, seg_len)]
    out = np.zeros_like(v, dtype=np.float64)
    eye = np.broadcast_to(np.eye(d), (1, H, d, d)).copy()
    zero_state = np.zeros((1, H, d, d))
    R, P = [], []
    for i, (a, b) in enumerate(bounds):
        sl = slice(a, b)
        o0, r = prefill(q[sl], k[sl], v[sl], g[sl], beta[sl], S0 if i == 0 else zero_state)
        _, p = prefill(q[sl], k[sl], np.zeros_like(v[sl]), g[sl], beta[sl], eye)
        out[sl] = o0
        R.append(r)
        P.append(p)
    S = R[0]
    for i in range(1, len(bounds)):
        a, b = bounds[i]
        sl = slice(a, b)
        oS, _ = prefill(q[sl], k[sl], np.zeros_like(v[sl]), g[sl], beta[sl], S)
        out[sl] += oS
        S = np.einsum("hij,hjk->hik", P[i][0], S[0])[None] + R[i]
    return out, S
