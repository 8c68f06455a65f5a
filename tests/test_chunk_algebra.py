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

The chunk form of the KDA head (per-channel gate), with its decay factors
blocked so that none exceeds 1, is checked against the oracle the same way
(``kda_chunked`` below): it is the form a tensor-core KDA build would take.
"""
import sys

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


# KDA (per-channel gate inside the delta rule) ------------------------------------
#
# S_t = (I - beta_t k_t k_t^T) diag(alpha_t) S_{t-1} + beta_t k_t v_t^T.  Within a
# chunk let c_t = g_1 + ... + g_t per key channel (all <= 0) and X_t = e^{-c_t} o S_t
# (row-wise).  Then X_t = (I - beta_t a_t b_t^T) X_{t-1} + beta_t a_t v_t^T with
# a_t = e^{-c_t} o k_t and b_t = e^{c_t} o k_t: a delta rule with distinct read
# and write keys.  Its WY form, with every decay factor written as a pairwise
# e^{c_t - c_s} (s <= t, so <= 1 and never overflowing), is
#
#   P[t][s] = sum_i k_t[i] k_s[i] e^{c_t[i] - c_s[i]}            (s < t)
#   Inv     = (I + strictly-lower(diag(beta) P))^-1
#   W = Inv diag(beta) B,  U = Inv diag(beta) V,   B_t = e^{c_t} o k_t
#   R = U - W S_0,   Kbar_s = e^{c_n - c_s} o k_s
#   S_n = diag(e^{c_n}) S_0 + Kbar^T R,   T_chunk = diag(e^{c_n}) - Kbar^T W
#   o_t = S_0^T (e^{c_t} o q_t) + sum_{s<=t} (sum_i q_t[i] k_s[i] e^{c_t[i]-c_s[i]}) r_s
#
# The tensor-core form of P splits the chunk into sub-chunks of 16: a block of
# rows t below a block of columns s takes the reference c_ref = c at the last
# token of the column block, so P = (e^{c_t - c_ref} o k_t) . (e^{c_ref - c_s} o k_s)
# is a plain product of two factors that are both <= 1; only the diagonal
# blocks need the pairwise exponent.  ``kda_chunked`` evaluates it that way.

def _pairwise(x, y, c_x, c_y, sub, inclusive):
    """sum_i x_t[i] y_s[i] e^{c_x[t][i] - c_y[s][i]} for s < t (s <= t when
    ``inclusive``), block by block as the tensor-core form takes it."""
    n = x.shape[0]
    out = np.zeros((n, n))
    for bt in range(0, n, sub):
        for bs in range(0, bt + 1, sub):
            rows, cols = slice(bt, min(bt + sub, n)), slice(bs, min(bs + sub, n))
            if bs < bt:
                ref = c_y[min(bs + sub, n) - 1]
                out[rows, cols] = (x[rows] * np.exp(c_x[rows] - ref)) @ \
                    (y[cols] * np.exp(ref - c_y[cols])).T
            else:
                blk = np.einsum("ti,si,tsi->ts", x[rows], y[cols],
                                np.exp(np.minimum(c_x[rows][:, None, :] - c_y[cols][None, :, :],
                                                  0.0)))
                out[rows, cols] = np.tril(blk, 0 if inclusive else -1)
    return np.tril(out, 0 if inclusive else -1)


def kda_chunked(k, v, beta, g, S0=None, q=None, C=64, sub=16):
    """(T, S_L, o) of a KDA unit by chunks of C tokens, from S0 (zero if None);
    o is returned when q is given."""
    L, dk = k.shape
    dv = v.shape[1]
    S = np.zeros((dk, dv)) if S0 is None else np.array(S0, np.float64)
    T = np.eye(dk)
    outs = []
    for c0 in range(0, L, C):
        K, V = k[c0:c0 + C], v[c0:c0 + C]
        b, c = beta[c0:c0 + C], np.cumsum(g[c0:c0 + C], axis=0)
        n = len(K)
        P = _pairwise(K, K, c, c, sub, inclusive=False)
        Inv = np.linalg.inv(np.eye(n) + b[:, None] * P)
        Bm = np.exp(c) * K
        W = Inv @ (b[:, None] * Bm)
        U = Inv @ (b[:, None] * V)
        R = U - W @ S
        Kbar = np.exp(c[-1] - c) * K
        if q is not None:
            Qc = q[c0:c0 + C]
            M = _pairwise(Qc, K, c, c, sub, inclusive=True)
            outs.append((np.exp(c) * Qc) @ S + M @ R)
        S = np.exp(c[-1])[:, None] * S + Kbar.T @ R
        T = (np.diag(np.exp(c[-1])) - Kbar.T @ W) @ T
    return T, S, (np.concatenate(outs) if q is not None else None)


def kda_tokens(rng, L, dk, dv, strong=False):
    k, v, beta, _ = tokens(rng, L, dk, dv)
    g = -np.logaddexp(0.0, -rng.normal(3.0, 1.0, (L, dk)))
    if strong:
        g[:, ::3] = -rng.uniform(2.0, 8.0, (L, len(range(0, dk, 3))))
    return k, v, beta, g


@pytest.mark.parametrize("L", [1, 15, 64, 100, 130])
def test_kda_chunk_form_equals_token_recurrence(L):
    """T and S(C|0) of the KDA chunk form (chunks of 64, sub-chunks of 16,
    ragged tails) equal the oracle's token recurrence."""
    rng = np.random.default_rng(400 + L)
    k, v, beta, g = kda_tokens(rng, L, 16, 12)
    ref = ls.segment_pair("kda", k, v, beta, g)
    T, S, _ = kda_chunked(k, v, beta, g)
    assert ls.rel_fro(T, ref["T"]) < 1e-11
    assert ls.rel_fro(S, ref["S"]) < 1e-11


def test_kda_chunk_form_from_a_state_with_outputs():
    """From a nonzero state, with outputs: the chunk form equals the oracle's
    token-by-token advance (the seam window of a KDA head, any length)."""
    rng = np.random.default_rng(420)
    k, v, beta, g = kda_tokens(rng, 37, 16, 12)
    q = rng.standard_normal((37, 16))
    S0 = rng.standard_normal((16, 12))
    S_ref, o_ref = ls.seam_advance(S0, q, k, v, beta, g, kind="kda")
    for C in (8, 64):
        _, S, o = kda_chunked(k, v, beta, g, S0=S0, q=q, C=C, sub=min(C, 16))
        assert ls.rel_fro(S, S_ref) < 1e-11
        assert ls.rel_fro(o, o_ref) < 1e-11


def test_kda_chunk_form_strong_decay_stays_finite():
    """Channels decaying by up to e^-8 a token: over a 64-token chunk
    e^{-c_s} would reach e^512 (beyond float64 and far beyond fp32), yet every
    factor of the blocked form stays <= 1 and the result matches the oracle."""
    rng = np.random.default_rng(430)
    k, v, beta, g = kda_tokens(rng, 128, 16, 12, strong=True)
    assert -np.cumsum(g[:64], axis=0).min() > 200.0
    ref = ls.segment_pair("kda", k, v, beta, g)
    with np.errstate(over="raise", invalid="raise"):
        T, S, _ = kda_chunked(k, v, beta, g)
    assert np.isfinite(T).all() and np.isfinite(S).all()
    assert ls.rel_fro(T, ref["T"]) < 1e-11
    assert ls.rel_fro(S, ref["S"]) < 1e-11


def _bf16(x):
    """Round to the nearest bfloat16 (ties to even), returned as float64."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = ((b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000).astype(np.uint32)
    return b.view(np.float32).astype(np.float64)


def test_kda_chunk_form_with_bf16_factors_stays_within_the_build_tolerance(monkeypatch):
    """bf16 inputs, and the two factors of every below-diagonal key-key block
    rounded to bf16 (the tensor-core operands): at dk = dv = 128 over two
    64-token chunks the pair stays within the 2e-3 relative error the builds
    are held to, with and without strongly decaying channels."""
    assert _bf16(1.0 + 2.0 ** -9) == 1.0 and _bf16(1.0 + 3 * 2.0 ** -9) == 1.0 + 2.0 ** -7
    exact = _pairwise

    def pairwise_bf16(x, y, c_x, c_y, sub, inclusive):
        n = x.shape[0]
        out = np.zeros((n, n))
        for bt in range(0, n, sub):
            for bs in range(0, bt + 1, sub):
                rows, cols = slice(bt, min(bt + sub, n)), slice(bs, min(bs + sub, n))
                if bs < bt:
                    ref = c_y[min(bs + sub, n) - 1]
                    out[rows, cols] = _bf16(x[rows] * np.exp(c_x[rows] - ref)) @ \
                        _bf16(y[cols] * np.exp(ref - c_y[cols])).T
                else:
                    out[rows, cols] = exact(x[rows], y[cols], c_x[rows], c_y[cols], sub, inclusive)
        return np.tril(out, 0 if inclusive else -1)

    for strong in (False, True):
        rng = np.random.default_rng(500 + strong)
        k, v, beta, g = kda_tokens(rng, 128, 128, 128, strong=strong)
        k, v = _bf16(k), _bf16(v)
        ref = ls.segment_pair("kda", k, v, beta, g)
        with monkeypatch.context() as m:
            m.setattr(sys.modules[__name__], "_pairwise", pairwise_bf16)
            T, S, _ = kda_chunked(k, v, beta, g)
        eT, eS = ls.rel_fro(T, ref["T"]), ls.rel_fro(S, ref["S"])
        assert eT < 2e-3 and eS < 2e-3, (strong, eT, eS)
        # and the rounding is really there: the error is far above float64's
        assert eT > 1e-6 and eS > 1e-6


# KDA in the arrangement of the tensor-core build ----------------------------------
#
# The tensor-core KDA build takes the key-key matrix of a chunk in one product
# with a single reference, the chunk start, instead of the blocked form above:
# P = (e^{c} o K)(e^{-c} o K)^T.  Every term of it is a product of two exact
# factors whose own product is k_t[i] k_s[i] e^{c_t[i] - c_s[i]} <= |k_t[i] k_s[i]|,
# so rounding errors stay relative to the terms; only e^{-c} itself can
# overflow, which bounds the chunk's decay span (the build hands units beyond
# it to the token recurrence).  The gate of each token is split into its
# largest channel m_t and the rest g_t - m_t <= 0: the rest enters the chunk
# form per channel (c' below), the largest acts as GDN's scalar decay (M), and
# the cache keeps log T = sum m, T = e^{log T} 2^exp2 Qhat.  Per chunk:
#
#   c'_t = sum_{u<=t} (g_u - m_u),  M_t = sum_{u<=t} m_u,  f_j = e^{M_n - M_j}
#   P    = (e^{c'} o K)(e^{-c'} o K)^T,   Inv = (I + strictly-lower(diag(beta) P))^-1
#   W    = Inv diag(beta) (e^{c'} o K),   Kn = e^{c'_n - c'} o K
#   Q   <- diag(e^{c'_n}) Q + Kn^T (-W Q)
#   S   <- e^{M_n} diag(e^{c'_n}) S + Kn^T (Inv diag(beta f) V - W e^{M_n} S)
#
# The state in tensor memory is pre-scaled by the next chunk's per-channel
# factor while the state operand of W X carries only the scalar one.
# ``kda_tc`` evaluates that in float64, or with every rounding the kernel makes.

KDA_SPAN_LIMIT = 64.0   # the build's bound on a chunk's per-channel decay span


def _trunc16(x):
    """Upper 16 bits of the fp32 value (bf16 by truncation), as float64."""
    b = np.asarray(x, np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return b.view(np.float32).astype(np.float64)


def _hilo(x):
    """bf16 hi + lo by truncation, as the kernel splits an fp32 operand."""
    x32 = np.asarray(x, np.float32).astype(np.float64)
    hi = _trunc16(x32)
    lo = _trunc16((x32 - hi).astype(np.float32))
    return hi, lo


def _prod3(a, b):
    """(a_h + a_l)(b_h + b_l) as three tensor-core products (lo x lo dropped)."""
    (ah, al), (bh, bl) = a, b
    return ah @ bh + ah @ bl + al @ bh


def _f16(x):
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float64)


def kda_tc(k, v, beta, g, C=64, rounded=False):
    """(log T, exp2, Qhat, S) of a KDA unit in the tensor-core build's
    arrangement; with ``rounded`` every operand is rounded as the kernel
    rounds it (hi/lo splits, fp16 state and W^T operands, fp32 elsewhere)."""
    L, dk = k.shape
    dv = v.shape[1]
    f32 = (lambda x: np.asarray(x, np.float32).astype(np.float64)) if rounded else (lambda x: x)
    Q, S = np.eye(dk), np.zeros((dk, dv))
    logT, e2, qmax = 0.0, 0, 1.0
    chunks = list(range(0, L, C))

    def decay(c0):
        gg = g[c0:c0 + C]
        m = gg.max(axis=1)
        cp = np.cumsum(gg - m[:, None], axis=0)
        M = np.cumsum(m)
        return m, cp, M

    for ci, c0 in enumerate(chunks):
        K, V, b = k[c0:c0 + C], v[c0:c0 + C], beta[c0:c0 + C]
        n = len(K)
        m, cp, M = decay(c0)
        assert -cp[-1].min() <= KDA_SPAN_LIMIT
        f = np.exp(M[-1] - M)
        Kp, Km = np.exp(cp) * K, np.exp(-cp) * K
        Kn = np.exp(cp[-1] - cp) * K
        if rounded:
            P = _prod3(_hilo(Kp), tuple(x.T for x in _hilo(Km)))
        else:
            P = Kp @ Km.T
        Lm = f32(np.tril(b[:, None] * P, -1))
        Inv = np.linalg.inv(np.eye(n) + Lm)
        BW = Inv * b[None, :]                       # B_W[t][j] = beta_j Inv[t][j]
        BU = -Inv * (b * f)[None, :]
        if rounded:
            W = _prod3(_hilo(BW), _hilo(Kp))
            Wop = _f16(W)
            BUh, BUl = _hilo(BU)
            Uterm = -(BUh @ V + BUl @ V)            # +Inv diag(beta f) V
        else:
            W, Wop, Uterm = BW @ Kp, BW @ Kp, -(BU @ V)
        # the state operands of this chunk (the previous pass wrote them)
        Qhat_op = _f16(Q) if rounded else Q
        Shat_op = np.exp(M[-1]) * S
        Shat_op = _f16(Shat_op) if rounded else Shat_op
        RQ, RS = -(Wop @ Qhat_op), -(Wop @ Shat_op - Uterm)
        if rounded:
            RQ, RS = _hilo(RQ), _hilo(RS)
            KnT = tuple(x.T for x in _hilo(Kn))
            upQ, upS = _prod3(KnT, RQ), _prod3(KnT, RS)
        else:
            upQ, upS = Kn.T @ RQ, Kn.T @ RS
        # tensor memory held the pre-scaled states
        Qtm = f32(np.exp(cp[-1])[:, None] * Q)
        Stm = f32(np.exp(M[-1]) * np.exp(cp[-1])[:, None] * S)
        Q, S = f32(Qtm + upQ), f32(Stm + upS)
        logT += M[-1]
        if ci + 1 < len(chunks):
            # power-of-two rescale of Q from the largest entry of the last pass
            _, ex = np.frexp(qmax)
            sh = 1 - int(ex)
            e2 -= sh
            Q = np.ldexp(Q, sh)
            qmax = float(np.abs(Q).max())
    return logT, e2, Q, S


@pytest.mark.parametrize("L", [1, 15, 64, 100, 130])
def test_kda_tc_arrangement_equals_token_recurrence(L):
    """The single-reference KDA arrangement (largest gate as the scalar decay,
    the rest per channel, state pre-scaled per channel) reproduces the oracle's
    T and S(C|0) in float64."""
    rng = np.random.default_rng(600 + L)
    k, v, beta, g = kda_tokens(rng, L, 16, 12)
    ref = ls.segment_pair("kda", k, v, beta, g)
    logT, e2, Q, S = kda_tc(k, v, beta, g)
    T = np.exp(logT) * np.ldexp(Q, e2)
    assert ls.rel_fro(T, ref["T"]) < 1e-11
    assert ls.rel_fro(S, ref["S"]) < 1e-11
    # log T is the sum of each token's largest gate
    assert abs(logT - g.max(axis=1).sum()) < 1e-12 * max(1.0, abs(logT))


def test_kda_tc_arrangement_mistakes_fail():
    """Planted mistakes in the arrangement: the state operand taking the
    per-channel pre-scale too, and the update keys without the per-channel
    decay, each move T or S far outside the tolerance."""
    rng = np.random.default_rng(640)
    k, v, beta, g = kda_tokens(rng, 130, 16, 12)
    g = g - rng.uniform(0.0, 0.4, g.shape)       # make the channels differ visibly
    ref = ls.segment_pair("kda", k, v, beta, g)

    def run(variant):
        L, dk = k.shape
        Q, S, logT = np.eye(dk), np.zeros((dk, v.shape[1])), 0.0
        for c0 in range(0, L, 64):
            K, V, b, gg = k[c0:c0 + 64], v[c0:c0 + 64], beta[c0:c0 + 64], g[c0:c0 + 64]
            m = gg.max(axis=1)
            cp, M = np.cumsum(gg - m[:, None], axis=0), np.cumsum(m)
            Kp, Km = np.exp(cp) * K, np.exp(-cp) * K
            Kn = K if variant == "undecayed_update_keys" else np.exp(cp[-1] - cp) * K
            Inv = np.linalg.inv(np.eye(len(K)) + np.tril(b[:, None] * (Kp @ Km.T), -1))
            W = Inv @ (b[:, None] * Kp)
            Ut = Inv @ ((b * np.exp(M[-1] - M))[:, None] * V)
            Xq, Xs = Q, np.exp(M[-1]) * S
            if variant == "prescaled_operand":
                Xq, Xs = np.exp(cp[-1])[:, None] * Xq, np.exp(cp[-1])[:, None] * Xs
            Q = np.exp(cp[-1])[:, None] * Q + Kn.T @ (-(W @ Xq))
            S = np.exp(M[-1]) * np.exp(cp[-1])[:, None] * S + Kn.T @ (Ut - W @ Xs)
            logT += M[-1]
        return np.exp(logT) * Q, S

    T, S = run(None)
    assert ls.rel_fro(T, ref["T"]) < 1e-11 and ls.rel_fro(S, ref["S"]) < 1e-11
    for variant in ("prescaled_operand", "undecayed_update_keys"):
        T, S = run(variant)
        assert max(ls.rel_fro(T, ref["T"]), ls.rel_fro(S, ref["S"])) > 1e-3, variant


@pytest.mark.parametrize("L", [512, 1500])
def test_kda_tc_rounding_stays_within_the_build_tolerance(L):
    """Every rounding point of the tensor-core KDA build simulated (bf16
    inputs; hi/lo bf16 splits of the key images, B operands and R; fp16 W^T
    and state operands; fp32 accumulators): at dk = dv = 128 the pair stays
    within the builds' 2e-3 relative error."""
    rng = np.random.default_rng(700 + L)
    k, v, beta, g = kda_tokens(rng, L, 128, 128)
    k, v = _bf16(k), _bf16(v)
    ref = ls.segment_pair("kda", k, v, beta, g)
    logT, e2, Q, S = kda_tc(k, v, beta, g, rounded=True)
    T = np.exp(logT) * np.ldexp(Q, e2)
    eT, eS = ls.rel_fro(T, ref["T"]), ls.rel_fro(S, ref["S"])
    assert eT < 2e-3 and eS < 2e-3, (eT, eS)
    assert eT > 1e-6 and eS > 1e-6


def test_kda_strong_gates_exceed_the_single_reference_span():
    """Channels decaying by e^-2..e^-8 a token take a chunk's span far past the
    single-reference bound, which is why such units go to the token
    recurrence; the workloads' gates stay far inside it."""
    rng = np.random.default_rng(430)
    _, _, _, g = kda_tokens(rng, 128, 16, 12, strong=True)
    m = g[:64].max(axis=1)
    assert -np.cumsum(g[:64] - m[:, None], axis=0)[-1].min() > KDA_SPAN_LIMIT
    _, _, _, g = kda_tokens(np.random.default_rng(431), 4096, 128, 12)
    for c0 in range(0, 4096, 64):
        gg = g[c0:c0 + 64]
        span = -np.cumsum(gg - gg.max(axis=1)[:, None], axis=0)[-1].min()
        assert span < KDA_SPAN_LIMIT / 4
