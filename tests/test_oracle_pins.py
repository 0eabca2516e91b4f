"""Pins for the fp64 oracle: facts the pages and mathematics fix, checked
without reusing the oracle's own formula.

Each test names the passage it follows (page title -- section).  A plausible
slip in the oracle (decay applied after the write, a transposed state, the
read taken before the update, a missing beta, conv taps reversed, the wrong
log base) fails at least one of them; see test_planted_mistakes_are_caught.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from tests.chunk_form import (block_inverse, chunk_recurrence, gram_tiled,
                              segmented_three_pass, verify_pairs)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def rand_inputs(rng, T, H, dk, dv, unit=True, beta_range=(0.0, 1.0), g_scale=1.0):
    q = rng.standard_normal((T, H, dk))
    k = rng.standard_normal((T, H, dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, dv))
    g = -5.0 * g_scale / (1.0 + np.exp(-rng.standard_normal((T, H, dk))))
    beta = rng.uniform(*beta_range, size=(T, H))
    return q, k, v, g, beta


def close(a, b, rtol=1e-12, atol=1e-12):
    np.testing.assert_allclose(a, b, rtol=rtol, atol=atol)


# ---------------------------------------------------------------- decay only

def test_decay_only_closed_form():
    """beta = 0: memory only decays, row i by exp(sum_t g_t[i]).
    From GPT-2 to Kimi K3, Chapter 5 ('Retain: scale each row of old memory
    by its own alpha'); Kimi K3 Architecture Explained, Step 3."""
    rng = np.random.default_rng(1)
    T, H, dk, dv = 37, 3, 8, 5
    q, k, v, g, _ = rand_inputs(rng, T, H, dk, dv)
    beta = np.zeros((T, H))
    S0 = rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.recurrence(q, k, v, g, beta, S0)
    Gam = np.cumsum(g, axis=0)                       # [T, H, dk]
    close(fin[0], np.exp(Gam[-1])[:, :, None] * S0[0])
    for t in (0, 11, T - 1):
        St = np.exp(Gam[t])[:, :, None] * S0[0]      # [H, dk, dv]
        close(out[t], np.einsum("hij,hi->hj", St, q[t]))


@pytest.mark.parametrize("case", golden("half_life.json")["cases"])
def test_half_life_matches_pages(case):
    """Constant alpha, no writes: the stored value halves after about
    ln 2 / -ln(alpha) tokens -- 69 for 0.99 and 693 for 0.999 (From GPT-2 to
    Kimi K3, Chapter 4)."""
    alpha, about = case["alpha"], case["half_life_tokens_about"]
    T = 2 * about
    g = np.full((T, 1, 1), math.log(alpha))
    ones = np.ones((T, 1, 1))
    out, _ = oracle.recurrence(ones, ones, ones, g, np.zeros((T, 1)),
                               np.ones((1, 1, 1, 1)))
    trace = out[:, 0, 0]                              # S_t read with q = 1
    first_below = int(np.argmax(trace <= 0.5)) + 1    # tokens until halved
    assert abs(first_below - about) <= 1
    assert abs(trace[about - 1] - 0.5) < 0.005


def test_decay_bound_pages():
    """g = gmin*sigmoid(z) stays in (-5, 0); exp(-5) ~ 0.0067 is never
    attained; 16 tokens of decay stay above -80 (From GPT-2 to Kimi K3,
    Chapter 5, K3's lower-bounded decay)."""
    gb = golden("decay_bound.json")
    z = np.concatenate([np.linspace(-30, 30, 2001), [0.0]])   # fp64 resolves the bound here
    g = oracle.decay_gate(z, gb["gmin"])
    assert np.all(g > gb["gmin"]) and np.all(g < 0)
    assert g[-1] == gb["gmin"] / 2                   # sigmoid(0) = 1/2
    assert round(math.exp(gb["gmin"]), gb["alpha_infimum_digits"]) == gb["alpha_infimum"]
    tile = g[np.argsort(g)][: gb["tile_tokens"]].sum()   # 16 strongest decays
    assert tile > gb["tile_cumulative_log_decay_floor"]
    assert gb["tile_tokens"] * gb["gmin"] == gb["tile_cumulative_log_decay_floor"]


def test_state_size_pages():
    """96 x 128 x 128 numbers per layer and request, ~3 MiB in BF16, ~207 MiB
    over 69 KDA layers (From GPT-2 to Kimi K3, Chapter 5)."""
    s = golden("state_size.json")
    n = s["heads"] * s["d_k"] * s["d_v"]
    assert n == s["numbers_per_layer_per_request"]
    assert round(n * 2 / 2**20) == s["bf16_mib_per_layer_about"]
    assert round(n * 2 * s["kda_layers"] / 2**20) == s["bf16_mib_all_layers_about"]


# ---------------------------------------------------------------- special cases

def test_deltanet_is_a_gradient_step():
    """alpha = 1 reduces KDA to DeltaNet, which is one gradient step of
    0.5*||S^T k - v||^2 with learning rate beta (From GPT-2 to Kimi K3,
    Chapter 3 'Why this is an online learning step').  The reference below
    takes the gradient with torch autograd, not with the oracle's formula."""
    rng = np.random.default_rng(2)
    T, H, dk, dv = 12, 2, 6, 4
    q, k, v, _, beta = rand_inputs(rng, T, H, dk, dv)
    g = np.zeros((T, H, dk))
    S0 = rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.recurrence(q, k, v, g, beta, S0)
    for h in range(H):
        S = torch.tensor(S0[0, h], dtype=torch.float64)
        for t in range(T):
            Sv = S.clone().requires_grad_(True)
            kt = torch.tensor(k[t, h])
            vt = torch.tensor(v[t, h])
            loss = 0.5 * ((Sv.T @ kt - vt) ** 2).sum()
            (grad,) = torch.autograd.grad(loss, Sv)
            S = S - float(beta[t, h]) * grad
            close(out[t, h], (S.T @ torch.tensor(q[t, h])).numpy())
        close(fin[0, h], S.numpy())


def test_gated_deltanet_scalar_alpha():
    """alpha equal across channels reduces KDA to Gated DeltaNet,
    S_t = alpha_t (I - beta k k^T) S_{t-1} + beta k v^T (Kimi K3 Architecture
    Explained, Step 3 'The first fix: a forget gate'), evaluated here with
    explicit d x d matrices and the scalar applied after the projection."""
    rng = np.random.default_rng(3)
    T, H, dk, dv = 10, 2, 5, 3
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    gs = g[:, :, :1]
    g = np.repeat(gs, dk, axis=2)
    S0 = rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.recurrence(q, k, v, g, beta, S0)
    for h in range(H):
        S = S0[0, h].copy()
        for t in range(T):
            a = math.exp(gs[t, h, 0])
            S = a * (np.eye(dk) - beta[t, h] * np.outer(k[t, h], k[t, h])) @ S \
                + beta[t, h] * np.outer(k[t, h], v[t, h])
            close(out[t, h], S.T @ q[t, h])
        close(fin[0, h], S)


def test_exact_overwrite_unit_key():
    """With ||k|| = 1, beta = 1 and alpha = 1 a write makes S_t^T k_t = v_t
    exactly, whatever the prior state (From GPT-2 to Kimi K3, Chapter 3 'A
    complete overwrite')."""
    rng = np.random.default_rng(4)
    T, H, dk, dv = 9, 3, 16, 7
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    _, S_prev = oracle.recurrence(q, k, v, g, beta, rng.standard_normal((1, H, dk, dv)))
    kt = rng.standard_normal((1, H, dk))
    kt /= np.linalg.norm(kt, axis=-1, keepdims=True)
    vt = rng.standard_normal((1, H, dv))
    _, S = oracle.recurrence(kt, kt, vt, np.zeros((1, H, dk)), np.ones((1, H)), S_prev)
    close(np.einsum("hij,hi->hj", S[0], kt[0]), vt[0], rtol=1e-13, atol=1e-13)


def test_overwrite_worked_example():
    """The 2-d worked example of Chapter 3 (golden/overwrite_2d.json)."""
    ex = golden("overwrite_2d.json")
    k = np.array(ex["key"])[None, None]
    v = np.array(ex["value"])[None, None]
    S0 = np.array(ex["state_before"])[None, None]
    assert np.allclose(S0[0, 0].T @ k[0, 0], ex["prediction_before"])
    out, S = oracle.recurrence(k, k, v, np.zeros_like(k), np.array([[ex["beta"]]]), S0)
    assert np.array_equal(S[0, 0], np.array(ex["state_after"]))
    assert np.array_equal(out[0, 0], np.array(ex["read_after"]))


def product_reference(q, k, v, g, beta, S0):
    """Outputs and final state from explicit transition matrices:
    S_t = M_t...M_1 S_0 + sum_s M_t...M_{s+1} beta_s k_s v_s^T,
    M_t = (I - beta_t k_t k_t^T) Diag(alpha_t), o_t = S_t^T q_t."""
    T, H, dk = q.shape
    dv = v.shape[2]
    out = np.zeros((T, H, dv))
    fin = np.zeros((1, H, dk, dv))
    for h in range(H):
        M = [(np.eye(dk) - beta[t, h] * np.outer(k[t, h], k[t, h])) @ np.diag(np.exp(g[t, h]))
             for t in range(T)]
        for tt in range(T):
            prod = np.eye(dk)
            St = np.zeros((dk, dv))
            for t in range(tt, -1, -1):     # prod = M_tt ... M_{t+1}
                St += prod @ (beta[t, h] * np.outer(k[t, h], v[t, h]))
                prod = prod @ M[t]
            St += prod @ S0[0, h]
            out[tt, h] = St.T @ q[tt, h]
            fin[0, h] = St
    return out, fin


def test_unrolled_product_of_transitions():
    """T <= 8: the oracle equals the explicit product of transition matrices
    M_t = (I - beta_t k_t k_t^T) Diag(alpha_t) for every output and the final
    state (Kimi K3 Architecture Explained, Step 3; infra diagram, KDA card)."""
    rng = np.random.default_rng(5)
    T, H, dk, dv = 8, 2, 4, 3
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv, unit=False)
    S0 = rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.recurrence(q, k, v, g, beta, S0)
    ref_out, ref_fin = product_reference(q, k, v, g, beta, S0)
    close(out, ref_out, rtol=1e-11, atol=1e-12)
    close(fin, ref_fin, rtol=1e-11, atol=1e-12)


def test_exact_rational_arithmetic():
    """Brute force in exact rationals (sympy) on a 3-token, 2x2 example of
    the published matrix equation; alpha is chosen rational and fed to the
    oracle as g = ln(alpha)."""
    sympy = pytest.importorskip("sympy")
    R = sympy.Rational
    ks = [[R(3, 5), R(4, 5)], [R(1), R(0)], [R(-5, 13), R(12, 13)]]
    vs = [[R(1), R(-2)], [R(1, 2), R(3)], [R(-1), R(1, 4)]]
    qs = [[R(1), R(1, 3)], [R(-2, 7), R(1)], [R(0), R(-1)]]
    al = [[R(1, 2), R(9, 10)], [R(3, 4), R(1, 5)], [R(99, 100), R(2, 3)]]
    bs = [R(1, 3), R(1), R(3, 4)]
    S = sympy.Matrix([[R(1, 7), R(0)], [R(-1), R(2, 9)]])
    S0 = np.array(S.tolist(), dtype=np.float64)
    exp_out = []
    for t in range(3):
        kk = sympy.Matrix(ks[t])
        S = (sympy.eye(2) - bs[t] * kk * kk.T) * sympy.diag(*al[t]) * S \
            + bs[t] * kk * sympy.Matrix(vs[t]).T
        exp_out.append([float(x) for x in (S.T * sympy.Matrix(qs[t]))])
    f = lambda x: np.array(x, dtype=np.float64)[:, None, :]
    g = np.log(np.array(al, dtype=np.float64))[:, None, :]
    out, fin = oracle.recurrence(f(qs), f(ks), f(vs), g,
                                 np.array(bs, dtype=np.float64)[:, None], S0[None, None])
    close(out[:, 0], np.array(exp_out), rtol=1e-14, atol=1e-14)
    close(fin[0, 0], np.array(S.tolist(), dtype=np.float64), rtol=1e-14, atol=1e-14)


# ---------------------------------------------------------------- structure

def _segment_map(q, k, g, beta, dk):
    """(P, R) of a segment: S_out = P S_in + R (From GPT-2 to Kimi K3,
    Chapter 6 'Context parallelism is not simple summation')."""
    T, H = beta.shape
    I = np.broadcast_to(np.eye(dk), (1, H, dk, dk)).copy()
    _, P = oracle.recurrence(q, k, np.zeros((T, H, dk)), g, beta, I)
    return P


def test_affine_segment_composition():
    """A segment acts on its incoming state as an affine map, and maps compose
    associatively: (P2, R2) o (P1, R1) = (P2 P1, P2 R1 + R2)."""
    rng = np.random.default_rng(6)
    T1, T2, H, dk, dv = 7, 9, 2, 5, 4
    q, k, v, g, beta = rand_inputs(rng, T1 + T2, H, dk, dv)
    S_in = rng.standard_normal((1, H, dk, dv))
    _, whole = oracle.recurrence(q, k, v, g, beta, S_in)
    a, b = slice(0, T1), slice(T1, T1 + T2)
    _, mid = oracle.recurrence(q[a], k[a], v[a], g[a], beta[a], S_in)
    _, two = oracle.recurrence(q[b], k[b], v[b], g[b], beta[b], mid)
    close(whole, two, rtol=1e-11, atol=1e-12)
    P1, P2 = _segment_map(q[a], k[a], g[a], beta[a], dk), _segment_map(q[b], k[b], g[b], beta[b], dk)
    _, R1 = oracle.recurrence(q[a], k[a], v[a], g[a], beta[a], None)
    _, R2 = oracle.recurrence(q[b], k[b], v[b], g[b], beta[b], None)
    close(P1[0] @ S_in[0] + R1[0], mid[0], rtol=1e-11, atol=1e-12)
    P12 = P2[0] @ P1[0]
    R12 = P2[0] @ R1[0] + R2[0]
    close(P12 @ S_in[0] + R12, whole[0], rtol=1e-11, atol=1e-12)


def test_non_expansion_unit_keys():
    """Unit keys, beta in [0,1], alpha in (0,1], no writes: the spectral norm
    of the state never grows (Kimi K3 Architecture Explained, 'Inside a KDA
    Layer': a key of length 1 means (I - beta k k^T) can only keep or shrink)."""
    rng = np.random.default_rng(7)
    T, H, dk, dv = 40, 2, 6, 6
    q, k, _, g, beta = rand_inputs(rng, T, H, dk, dv, g_scale=0.05)
    S = rng.standard_normal((1, H, dk, dv))
    prev = [np.linalg.norm(S[0, h], 2) for h in range(H)]
    for t in range(T):
        sl = slice(t, t + 1)
        _, S = oracle.recurrence(q[sl], k[sl], np.zeros((1, H, dv)), g[sl], beta[sl], S)
        for h in range(H):
            n = np.linalg.norm(S[0, h], 2)
            assert n <= prev[h] * (1 + 1e-12)
            prev[h] = n


def test_linear_in_values_and_state():
    """For fixed q, k, g, beta the outputs and final state are linear in
    (V, S0) jointly -- the recurrence is affine in both."""
    rng = np.random.default_rng(8)
    T, H, dk, dv = 15, 2, 5, 4
    q, k, v1, g, beta = rand_inputs(rng, T, H, dk, dv)
    v2 = rng.standard_normal(v1.shape)
    s1, s2 = rng.standard_normal((2, 1, H, dk, dv))
    o1, f1 = oracle.recurrence(q, k, v1, g, beta, s1)
    o2, f2 = oracle.recurrence(q, k, v2, g, beta, s2)
    o3, f3 = oracle.recurrence(q, k, 2.0 * v1 - 3.0 * v2, g, beta, 2.0 * s1 - 3.0 * s2)
    close(o3, 2.0 * o1 - 3.0 * o2, rtol=1e-10, atol=1e-11)
    close(f3, 2.0 * f1 - 3.0 * f2, rtol=1e-10, atol=1e-11)


def test_packed_documents_are_independent():
    """Packed documents delimited by cumulative offsets never see each other
    (infra diagram: 'cumulative sequence offsets preserve their boundaries');
    a zero-length document returns its initial state."""
    rng = np.random.default_rng(9)
    lengths = [5, 0, 7, 1, 3]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, H, dk, dv = cu[-1], 2, 4, 3
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    S0 = rng.standard_normal((len(lengths), H, dk, dv))
    out, fin = oracle.recurrence(q, k, v, g, beta, S0, cu)
    for n, L in enumerate(lengths):
        sl = slice(cu[n], cu[n + 1])
        o, f = oracle.recurrence(q[sl], k[sl], v[sl], g[sl], beta[sl], S0[n:n + 1])
        close(out[sl], o)
        close(fin[n], f[0])
    close(fin[1], S0[1], rtol=0, atol=0)


@pytest.mark.parametrize("C", [1, 4, 16, 64])
def test_chunkwise_form_matches_recurrence(C):
    """The chunked re-association (UT transform + pseudo-values, From GPT-2 to
    Kimi K3, Chapter 6) equals the token recurrence to fp64 rounding; this pins
    the algebra the CUDA prefill uses."""
    rng = np.random.default_rng(10 + C)
    T, H, dk, dv = 150, 2, 16, 8
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    S0 = 0.1 * rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.recurrence(q, k, v, g, beta, S0)
    for h in range(H):
        o, f = chunk_recurrence(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], S0[0, h], C)
        close(o, out[:, h], rtol=1e-9, atol=1e-10)
        close(f, fin[0, h], rtol=1e-9, atol=1e-10)


@pytest.mark.parametrize("C", [16, 64])
def test_reassociated_chunk_form_matches_recurrence(C):
    """U = Tb (V - K+ S0), the order the CUDA prefill computes it in (state
    products first, then one product with Tb = (I+L)^-1 diag(beta)), equals
    the pages' Ut - W S0 and the token recurrence to fp64 rounding."""
    rng = np.random.default_rng(30 + C)
    T, H, dk, dv = 150, 2, 16, 8
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv)
    S0 = 0.1 * rng.standard_normal((1, H, dk, dv))
    out, fin = oracle.recurrence(q, k, v, g, beta, S0)
    for h in range(H):
        o, f = chunk_recurrence(q[:, h], k[:, h], v[:, h], g[:, h], beta[:, h], S0[0, h], C,
                                reassociated=True)
        close(o, out[:, h], rtol=1e-9, atol=1e-10)
        close(f, fin[0, h], rtol=1e-9, atol=1e-10)


def test_tiled_gram_matches_direct_and_stays_in_fp32_range():
    """The per-tile reference points of the CUDA prefill's Gram (16-token
    tiles of a 64-token chunk) give L and P unchanged, and with the bounded
    gate (g > -5 per token and channel, Kimi K3's lower-bounded decay) no
    factor exceeds e^(5 x 16) = e^80, inside fp32 range (about e^88.7) --
    while the direct factors e^{-G} of a whole chunk reach e^320."""
    rng = np.random.default_rng(41)
    C, dk = 64, 32
    k = rng.standard_normal((C, dk)); k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((C, dk)); q /= np.linalg.norm(q, axis=1, keepdims=True)
    beta = 1 / (1 + np.exp(-rng.standard_normal(C)))
    for g in (-5 / (1 + np.exp(-rng.standard_normal((C, dk)))),      # the workloads' gate
              -0.01 / (1 + np.exp(-rng.standard_normal((C, dk)))),   # weak: far tiles count
              np.full((C, dk), -5 + 1e-9)):                           # at the bound
        G = np.cumsum(g, axis=0)
        Kp, Km, Qp = np.exp(G) * k, np.exp(-G) * k, np.exp(G) * q
        L_ref = np.tril(beta[:, None] * (Kp @ Km.T), -1)
        P_ref = np.tril(Qp @ Km.T)
        L, P, biggest = gram_tiled(k, q, g, beta)
        close(L, L_ref, rtol=1e-10, atol=1e-12)
        close(P, P_ref, rtol=1e-10, atol=1e-12)
        assert biggest <= np.exp(80.0) < np.finfo(np.float32).max
    assert np.exp(-G).max() > np.exp(300)                               # why the tiles exist


def test_block_inverse_stages_match_the_inverse():
    """The prefill's block inverse of I + L (diagonal blocks by forward
    substitution, then the three stages of products) equals the matrix
    inverse, for the L of a chunk with the workloads' distributions and with
    a decay 500 times weaker.  Under the workloads' decay the blocks two
    tiles apart weigh about e^-40, so only the weak decay (close to DeltaNet)
    makes every stage's formula count: a flipped sign or swapped factor in
    V20, Y30, T30 or T31 then moves T by 0.08 to 0.6."""
    rng = np.random.default_rng(61)
    C, dk = 64, 32
    for scale in (1.0, 500.0):
        k = rng.standard_normal((C, dk)); k /= np.linalg.norm(k, axis=1, keepdims=True)
        g = -5 / (1 + np.exp(-rng.standard_normal((C, dk)))) / scale
        beta = 1 / (1 + np.exp(-rng.standard_normal(C)))
        G = np.cumsum(g, axis=0)
        L = np.tril(beta[:, None] * ((np.exp(G) * k) @ (np.exp(-G) * k).T), -1)
        T = block_inverse(L)
        close(T, np.linalg.inv(np.eye(C) + L), rtol=1e-9, atol=1e-11)
        close(T @ (np.eye(C) + L), np.eye(C), rtol=0, atol=1e-10)


@pytest.mark.parametrize("nseg", [1, 2, 3, 5])
def test_segment_scan_three_prefills_match_recurrence(nseg):
    """The segment-scan prefill's decomposition (three prefills of the
    segments as independent documents, then the scan of their affine maps,
    From GPT-2 to Kimi K3, Chapter 6, context parallelism) gives the
    one-document recurrence's outputs and final state, with an initial state
    and a ragged last segment."""
    rng = np.random.default_rng(70 + nseg)
    T, H, d = 300, 2, 8
    q, k, v, g, beta = rand_inputs(rng, T, H, d, d, g_scale=0.05)   # a slow decay: segments interact
    S0 = 0.1 * rng.standard_normal((1, H, d, d))
    out, fin = oracle.recurrence(q, k, v, g, beta, S0)
    prefill = lambda *a: oracle.recurrence(*a)
    o, f = segmented_three_pass(q, k, v, g, beta, S0, nseg, prefill)
    close(o, out, rtol=1e-9, atol=1e-11)
    close(f, fin, rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("K", [1, 2, 5, 6])
def test_two_drafts_per_pass_match_recurrence(K):
    """The verify kernel's pass over the state for two draft tokens at once
    (the second token's sums expanded over the state before the first) gives
    the token recurrence's outputs and state; an odd last token alone."""
    rng = np.random.default_rng(50 + K)
    dk, dv = 16, 8
    q, k, v, g, beta = rand_inputs(rng, K, 1, dk, dv)
    S0 = 0.1 * rng.standard_normal((1, 1, dk, dv))
    out, fin = oracle.recurrence(q, k, v, g, beta, S0)
    o, f = verify_pairs(q[:, 0], k[:, 0], v[:, 0], g[:, 0], beta[:, 0], S0[0, 0])
    close(o, out[:, 0], rtol=1e-11, atol=1e-13)
    close(f, fin[0, 0], rtol=1e-11, atol=1e-13)


# ---------------------------------------------------------------- prologue

def test_short_conv_matches_lfilter():
    """Width-4 depthwise causal conv with zero history at each document start
    (infra diagram, KDA card) equals scipy's FIR filter per channel and per
    document, taps reversed into filter order."""
    signal = pytest.importorskip("scipy.signal")
    rng = np.random.default_rng(11)
    lengths = [6, 1, 0, 9]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, C = cu[-1], 5
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, 4))
    y = oracle.short_conv(x, w, cu)
    for n in range(len(lengths)):
        sl = slice(cu[n], cu[n + 1])
        if lengths[n] == 0:
            continue
        for c in range(C):
            close(y[sl, c], signal.lfilter(w[c, ::-1], [1.0], x[sl, c]))


def test_short_conv_one_hot_taps():
    """Tap 3 alone is the identity; tap 2 alone delays by one token and
    feeds zero at every document start."""
    rng = np.random.default_rng(12)
    cu = np.array([0, 4, 9])
    x = rng.standard_normal((9, 3))
    w = np.zeros((3, 4))
    w[:, 3] = 1.0
    close(oracle.short_conv(x, w, cu), x, rtol=0, atol=0)
    w[:] = 0.0
    w[:, 2] = 1.0
    y = oracle.short_conv(x, w, cu)
    assert np.all(y[[0, 4]] == 0.0)
    close(y[1:4], x[0:3], rtol=0, atol=0)
    close(y[5:9], x[4:8], rtol=0, atol=0)


def test_swish_sigmoid_gate_match_expit():
    special = pytest.importorskip("scipy.special")
    z = np.random.default_rng(13).standard_normal(1000) * 6
    close(oracle.sigmoid(z), special.expit(z), rtol=1e-15, atol=1e-16)
    close(oracle.swish(z), z * special.expit(z), rtol=1e-14, atol=1e-16)
    close(oracle.decay_gate(z), -5.0 * special.expit(z), rtol=1e-14, atol=1e-16)


def test_l2norm_unit_length_same_direction():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((50, 3, 16)) * 4
    y = oracle.l2norm(x, eps=0.0)
    close(np.linalg.norm(y, axis=-1), np.ones((50, 3)), rtol=1e-14, atol=0)
    cos = (x * y).sum(-1) / np.linalg.norm(x, axis=-1)
    close(cos, np.ones((50, 3)), rtol=1e-14, atol=0)
    small = oracle.l2norm(np.full((1, 4), 1e-4), eps=1e-6)   # eps matters
    assert np.linalg.norm(small) < 0.25


def test_prologue_composes_conv_swish_norm():
    """ShortConv -> Swish; q and k then L2Norm; v not normalised (infra
    diagram: 'q, k, v ... ShortConv, Swish; q and k then L2Norm')."""
    rng = np.random.default_rng(15)
    T, H, d = 10, 2, 8
    raw = [rng.standard_normal((T, H, d)) for _ in range(3)]
    w = np.zeros((3, H * d, 4))
    w[:, :, 3] = 1.0                                   # identity conv
    zg, zb = rng.standard_normal((T, H, d)), rng.standard_normal((T, H))
    q, k, v, g, b = oracle.prologue(*raw, w, zg, zb, eps=0.0)
    sw = lambda x: x / (1 + np.exp(-x))
    for got, r in ((q, raw[0]), (k, raw[1])):
        s = sw(r)
        close(got, s / np.linalg.norm(s, axis=-1, keepdims=True), rtol=1e-13, atol=1e-15)
    close(v, sw(raw[2]), rtol=1e-14, atol=1e-16)
    assert np.all((g > -5) & (g < 0)) and np.all((b > 0) & (b < 1))


# ---------------------------------------------------------------- the pins bite

def _planted(q, k, v, g, beta, S0, mistake):
    """The recurrence with one plausible mistake planted (numpy, CPU)."""
    T, H, dk = q.shape
    dv = v.shape[2]
    out = np.zeros((T, H, dv))
    S = S0[0].copy()
    for t in range(T):
        for h in range(H):
            a = np.exp(g[t, h]) if mistake != "log2" else 2.0 ** g[t, h]
            kt, vt, qt, bt = k[t, h], v[t, h], q[t, h], beta[t, h]
            if mistake == "decay_after_write":
                S[h] = S[h] + bt * np.outer(kt, vt - S[h].T @ kt)
                S[h] = a[:, None] * S[h]
            elif mistake == "decay_columns":
                R = S[h] * a[None, :dv] if dv == dk else S[h]
                S[h] = R + bt * np.outer(kt, vt - R.T @ kt)
            else:
                R = a[:, None] * S[h]
                bb = 1.0 if mistake == "no_beta" else bt
                S[h] = R + bb * np.outer(kt, vt - R.T @ kt)
            out[t, h] = (S[h].T @ qt) if mistake != "read_before" else (
                (S[h] - bt * np.outer(kt, vt - S[h].T @ kt)).T @ qt)
    return out, S[None]


@pytest.mark.parametrize("mistake", ["decay_after_write", "decay_columns", "no_beta",
                                     "log2", "read_before"])
def test_planted_mistakes_are_caught(mistake):
    """A copy of the oracle's loop with one plausible slip planted fails the
    explicit transition-matrix pin, while the unplanted copy passes it."""
    rng = np.random.default_rng(16)
    T, H, dk, dv = 6, 1, 4, 4
    q, k, v, g, beta = rand_inputs(rng, T, H, dk, dv, unit=False)
    S0 = rng.standard_normal((1, H, dk, dv))
    ref_out, ref_fin = product_reference(q, k, v, g, beta, S0)
    bad_out, bad_fin = _planted(q, k, v, g, beta, S0, mistake)
    ok_out, ok_fin = _planted(q, k, v, g, beta, S0, "none")
    close(ok_out, ref_out, rtol=1e-12, atol=1e-12)
    assert not (np.allclose(bad_out, ref_out, rtol=1e-6) and np.allclose(bad_fin, ref_fin, rtol=1e-6))


# ---------------------------------------------------------------- output gate

def test_output_gate_matches_torch_rms_norm_and_sigmoid():
    """Head RMSNorm x sigmoid(gate) (From GPT-2 to Kimi K3, Chapter 5 'A third
    gate'; infra diagram 'Head RMSNorm + gate') equals torch's rms_norm and
    sigmoid in fp64."""
    rng = np.random.default_rng(17)
    o = rng.standard_normal((30, 4, 16)) * 3
    z = rng.standard_normal((30, 4, 16)) * 2
    w = rng.uniform(0.5, 1.5, 16)
    y = oracle.output_gate(o, z, w, eps=1e-6)
    ref = torch.nn.functional.rms_norm(torch.tensor(o), (16,), torch.tensor(w), eps=1e-6) \
        * torch.sigmoid(torch.tensor(z))
    close(y, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_output_gate_invariants():
    """Scale invariance of the norm, odd symmetry, unit RMS when the gate is
    open and w = 1, and sigmoid(0) = 1/2."""
    rng = np.random.default_rng(18)
    o = rng.standard_normal((20, 8))
    z = rng.standard_normal((20, 8))
    y = oracle.output_gate(o, z, eps=0.0)
    close(oracle.output_gate(7.5 * o, z, eps=0.0), y, rtol=1e-13, atol=1e-15)
    close(oracle.output_gate(-o, z, eps=0.0), -y, rtol=0, atol=0)
    open_ = oracle.output_gate(o, np.full_like(z, 60.0), eps=0.0)
    close(np.sqrt(np.mean(open_ ** 2, axis=-1)), np.ones(20), rtol=1e-13, atol=0)
    half = oracle.output_gate(o, np.zeros_like(z), eps=0.0)
    close(2 * half, open_, rtol=1e-14, atol=1e-16)
