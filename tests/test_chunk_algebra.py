"""The chunked WY/UT form that the device build kernel evaluates, written out
in float64 and checked against the oracle's token recurrence.

This is a CPU check of the kernel's mathematics, not part of the oracle.  Per
chunk of n <= 64 tokens with keys K [n, dk], values V [n, dv], write weights
beta and within-chunk cumulative log-decay c_i = g_1 + ... + g_i:

  G   = K K^T
  L_Q = strictly-lower(diag(beta) G)
  L_S = strictly-lower(diag(beta) G * exp(c_i - c_j))
  W   = (I + L_Q)^-1 diag(beta) K,   U = (I + L_S)^-1 diag(beta) V
  Q  <- Q - K^T (W Q)
  S  <- e^{c_n} S + K^T (diag(e^{c_n - c_i}) U - e^{c_n} W S)

with the decay of T carried as a log: T = e^{sum g} Q.

The seam window's chunk form that the tensor-core compose evaluates (chunks
of up to 8 tokens, only the products with the running state done on the
chain) is checked the same way against the oracle's token-by-token seam
advance (``seam_chunked`` below).
"""
import numpy as np
import pytest

from oracle import linear_state as ls


def chunked(k, v, beta, g, C=64, pad_to_chunk=False, rescale=False):
    L, dk = k.shape
    dv = v.shape[1]
    Q = np.eye(dk)
    S = np.zeros((dk, dv))
    logG = 0.0
    e = 0
    for c0 in range(0, L, C):
        K, V = k[c0:c0 + C], v[c0:c0 + C]
        b, gg = beta[c0:c0 + C], g[c0:c0 + C]
        if pad_to_chunk and len(K) < C:
            pad = C - len(K)
            K = np.concatenate([K, np.zeros((pad, dk))])
            V = np.concatenate([V, np.zeros((pad, dv))])
            b = np.concatenate([b, np.zeros(pad)])
            gg = np.concatenate([gg, np.zeros(pad)])
        n = len(K)
        c = np.cumsum(gg)
        G = K @ K.T
        LQ = np.tril(b[:, None] * G, -1)
        LS = np.tril(b[:, None] * G * np.exp(c[:, None] - c[None, :]), -1)
        W = np.linalg.solve(np.eye(n) + LQ, b[:, None] * K)
        U = np.linalg.solve(np.eye(n) + LS, b[:, None] * V)
        Gn = np.exp(c[-1])
        Q = Q + K.T @ (-(W @ Q))
        S = Gn * S + K.T @ (np.exp(c[-1] - c)[:, None] * U - Gn * (W @ S))
        logG += c[-1]
        if rescale:
            m = np.abs(Q).max()
            if m > 0:
                s = -int(np.floor(np.log2(m)))
                Q = np.ldexp(Q, s)
                e -= s
    return Q, e, logG, S


def tokens(rng, L, dk, dv, x_mean=-4.0):
    k = rng.standard_normal((L, dk))
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    return (k, rng.standard_normal((L, dv)), rng.random(L),
            -np.logaddexp(0.0, rng.normal(x_mean, 1.0, L)))


@pytest.mark.parametrize("L", [1, 5, 63, 64, 65, 130, 200])
def test_chunked_equals_token_recurrence(L):
    rng = np.random.default_rng(100 + L)
    k, v, beta, g = tokens(rng, L, 32, 24)
    ref = ls.segment_pair("gdn", k, v, beta, g, want_T=False)
    for pad in (False, True):
        Q, e, logG, S = chunked(k, v, beta, g, C=64, pad_to_chunk=pad)
        assert ls.rel_fro(Q, ref["Q"]) < 1e-12
        assert ls.rel_fro(S, ref["S"]) < 1e-12
        assert abs(logG - ref["logG"]) < 1e-12


def test_chunked_with_power_of_two_rescale():
    rng = np.random.default_rng(7)
    k, v, beta, g = tokens(rng, 700, 16, 16)
    ref = ls.segment_pair("gdn", k, v, beta, g, want_T=False)
    Q, e, logG, S = chunked(k, v, beta, g, C=64, rescale=True)
    assert 1.0 <= np.abs(Q).max() < 2.0
    assert ls.rel_fro_factored(Q, e, logG, ref["Q"], ref["logG"]) < 1e-11
    assert ls.rel_fro(S, ref["S"]) < 1e-11


def test_chunked_strong_decay():
    """alpha down to ~0.1 inside a chunk: every factor in the chunk form stays
    at most 1 (e^{c_i - c_j}, i > j, and e^{c_n - c_i})."""
    rng = np.random.default_rng(8)
    k, v, beta, g = tokens(rng, 128, 16, 8, x_mean=1.0)
    ref = ls.segment_pair("gdn", k, v, beta, g, want_T=False)
    Q, e, logG, S = chunked(k, v, beta, g)
    assert ls.rel_fro(S, ref["S"]) < 1e-12
    assert ls.rel_fro_factored(Q, e, logG, ref["Q"], ref["logG"]) < 1e-12


def seam_chunked(S0, q, k, v, beta, g, C=8):
    """The seam window as the tensor-core compose evaluates it: chunks of up to
    C tokens; per chunk of n tokens from the state S_0, with
    E[t][s] = prod_{s < u <= t} alpha_u and gamma_t = prod_{u <= t} alpha_u,

      Inv = (I + strictly-lower(diag(beta) K K^T) o E)^-1
      W   = Inv diag(beta gamma) K,   U~ = Inv diag(beta) V,   R = U~ - W S_0
      o_t = gamma_t S_0^T q_t + sum_{s <= t} E[t][s] (q_t . k_s) r_s
      S_n = gamma_{n-1} S_0 + Kbar^T R,   Kbar_s = E[n-1][s] k_s

    (only the products with S_0 depend on the state)."""
    S = np.array(S0, dtype=np.float64, copy=True)
    outs = []
    for c0 in range(0, len(k), C):
        K, V, Qc = k[c0:c0 + C], v[c0:c0 + C], q[c0:c0 + C]
        b, a = beta[c0:c0 + C], np.exp(g[c0:c0 + C])
        n = len(K)
        E = np.zeros((n, n))
        for t in range(n):
            for s in range(t + 1):
                E[t, s] = np.prod(a[s + 1:t + 1])
        gam = np.cumprod(a)
        Linv = np.linalg.inv(np.eye(n) + np.tril(b[:, None] * (K @ K.T) * E, -1))
        W = Linv @ ((b * gam)[:, None] * K)
        U = Linv @ (b[:, None] * V)
        R = U - W @ S
        M = np.tril((Qc @ K.T) * E)
        outs.append(gam[:, None] * (Qc @ S) + M @ R)
        S = gam[-1] * S + (E[n - 1][:, None] * K).T @ R
    return S, np.concatenate(outs)


@pytest.mark.parametrize("w", [1, 3, 8, 13, 20])
def test_seam_chunk_form_equals_token_recurrence(w):
    """The chunked seam window (chunks of 8, any window length) equals the
    oracle's token-by-token seam advance: the final state and every output."""
    rng = np.random.default_rng(300 + w)
    dk, dv = 16, 12
    k, v, beta, g = tokens(rng, w, dk, dv)
    q = rng.standard_normal((w, dk))
    S0 = rng.standard_normal((dk, dv))
    S_ref, o_ref = ls.seam_advance(S0, q, k, v, beta, g)
    S, o = seam_chunked(S0, q, k, v, beta, g)
    assert ls.rel_fro(S, S_ref) < 1e-12
    assert ls.rel_fro(o, o_ref) < 1e-12


def test_seam_chunk_form_vanishing_decay():
    """A token whose alpha underflows (log alpha = -800): gamma and E hold the
    exact zeros, and no factor of the chunk form divides by them."""
    rng = np.random.default_rng(310)
    k, v, beta, g = tokens(rng, 8, 16, 8)
    g = g.copy()
    g[5] = -800.0
    q = rng.standard_normal((8, 16))
    S0 = rng.standard_normal((16, 8))
    S_ref, o_ref = ls.seam_advance(S0, q, k, v, beta, g)
    S, o = seam_chunked(S0, q, k, v, beta, g)
    assert ls.rel_fro(S, S_ref) < 1e-12
    assert ls.rel_fro(o, o_ref) < 1e-12
