"""Pins of the float64 oracle to facts fixed outside itself.

Each test checks the oracle against something it does not compute itself: the
composition law on the pages, closed forms (RetNet, GLA, plain linear
attention), hand-expanded brute force on 1-4 tokens, the determinant of a
product of rank-1 updates, identity tokens and special structure.  The last
test plants plausible mistakes into a copy of the oracle and checks that these
pins catch every one.
"""
import json
import os

import numpy as np
import pytest

from oracle import linear_state as ls

RNG = np.random.default_rng(12345)


def gdn_tokens(rng, L, dk, dv, x_mean=-4.0, normalize=True):
    x = rng.normal(x_mean, 1.0, L)
    beta = rng.random(L)
    k = rng.standard_normal((L, dk))
    if normalize:
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((L, dv))
    g = -np.logaddexp(0.0, x)
    return k, v, beta, g


def pair_of(kind, k, v, beta, g):
    out = ls.segment_pair(kind, k, v, beta, g)
    return out["T"], out["S"]


# P1: composition law ----------------------------------------------------------

@pytest.mark.parametrize("kind", ["gdn", "scalar", "diag", "none", "token", "kda"])
def test_law_split_equals_concatenation(kind):
    rng = np.random.default_rng(1)
    dk, dv, L = 16, 12, 40
    k, v, beta, g = gdn_tokens(rng, L, dk, dv)
    if kind in ("diag", "kda"):
        g = -np.logaddexp(0.0, -rng.normal(3.0, 1.0, (L, dk)))
    if kind == "scalar":
        g = np.full(L, np.log(1 - 2 ** -6))
    full = ls.segment_pair(kind, k, v, beta, g)
    for cut in (1, 7, 20, 39):
        p1 = pair_of(kind, k[:cut], v[:cut], beta[:cut], g[:cut])
        p2 = pair_of(kind, k[cut:], v[cut:], beta[cut:], g[cut:])
        T, S = ls.compose_pair(p1, p2)
        assert np.allclose(T, full["T"], rtol=0, atol=1e-12 * max(1, np.abs(full["T"]).max()))
        assert np.allclose(S, full["S"], rtol=0, atol=1e-12 * max(1, np.abs(full["S"]).max()))
        # the same through the running-state form
        S_run = ls.compose([p1, p2], [0, 1])
        assert ls.rel_fro(S_run, full["S"]) < 1e-12


def test_law_three_segments_llm_wiki_form():
    """e_ABC = T_C (T_B e_A + e_B) + e_C and T_ABC = T_C T_B T_A."""
    rng = np.random.default_rng(2)
    k, v, beta, g = gdn_tokens(rng, 30, 8, 8)
    A = pair_of("gdn", k[:9], v[:9], beta[:9], g[:9])
    B = pair_of("gdn", k[9:20], v[9:20], beta[9:20], g[9:20])
    C = pair_of("gdn", k[20:], v[20:], beta[20:], g[20:])
    full = ls.segment_pair("gdn", k, v, beta, g)
    T_abc = C[0] @ B[0] @ A[0]
    e_abc = C[0] @ (B[0] @ A[1] + B[1]) + C[1]
    assert ls.rel_fro(T_abc, full["T"]) < 1e-12
    assert ls.rel_fro(e_abc, full["S"]) < 1e-12


def test_gdn_small_order_equals_sequential_concatenation():
    """The small gated-delta workload composed in order [2,0,3,1] equals a
    sequential run over those segments concatenated in that order."""
    from linear_attn_state_gb300 import synth
    p = synth.gdn_small()
    from oracle import schedule as sch
    body = sch.body_ranges(p.offsets, 0)
    pairs = []
    for seg in range(p.n_seg):
        u = synth.unit_inputs(p, 0, *body[seg])
        out = ls.segment_pair("gdn", u["k"], u["v"], u["beta"], u["g"])
        pairs.append((out["T"], out["S"]))
    S = ls.compose(pairs, synth.GDN_SMALL_ORDER)
    parts = [synth.unit_inputs(p, 0, *body[s]) for s in synth.GDN_SMALL_ORDER]
    cat = {key: np.concatenate([u[key] for u in parts]) for key in ("k", "v", "beta", "g")}
    S_seq = ls.run_from("gdn", np.zeros((p.dk, p.dv)), cat["k"], cat["v"], cat["beta"], cat["g"])
    assert ls.rel_fro(S, S_seq) < 1e-12
    # and the naive sum is clearly wrong here
    assert ls.rel_fro(ls.naive_add(pairs, synth.GDN_SMALL_ORDER), S_seq) > 0.05


def test_prefix_independence():
    """The pair of a segment does not depend on what came before it: running
    the segment from any prefix state equals T S_prefix + S(C|0)."""
    rng = np.random.default_rng(3)
    k, v, beta, g = gdn_tokens(rng, 25, 10, 6)
    T, S = pair_of("gdn", k, v, beta, g)
    for _ in range(3):
        S0 = rng.standard_normal((10, 6))
        assert ls.rel_fro(ls.run_from("gdn", S0, k, v, beta, g), T @ S0 + S) < 1e-12


# P2-P5: closed forms -----------------------------------------------------------

def test_retnet_closed_form():
    rng = np.random.default_rng(4)
    dk, dv = 12, 9
    gamma = 1 - 2.0 ** -7
    k1, v1, _, _ = gdn_tokens(rng, 30, dk, dv)
    k2, v2, _, _ = gdn_tokens(rng, 17, dk, dv)
    g1 = np.full(30, np.log(gamma))
    g2 = np.full(17, np.log(gamma))
    p1 = pair_of("scalar", k1, v1, None, g1)
    p2 = pair_of("scalar", k2, v2, None, g2)
    # T = gamma^L I
    assert np.allclose(p1[0], gamma ** 30 * np.eye(dk), rtol=1e-13, atol=0)
    assert np.allclose(p2[0], gamma ** 17 * np.eye(dk), rtol=1e-13, atol=0)
    # S(C|0) = sum_t gamma^(L-t) k_t v_t^T
    S_ref = sum(gamma ** (30 - 1 - t) * np.outer(k1[t], v1[t]) for t in range(30))
    assert ls.rel_fro(p1[1], S_ref) < 1e-13
    # naive - true = (1 - gamma^L2) S(C1)
    true = ls.compose([p1, p2], [0, 1])
    naive = ls.naive_add([p1, p2], [0, 1])
    assert ls.rel_fro(naive - true, (1 - gamma ** 17) * p1[1]) < 1e-12


def test_plain_linear_attention_naive_add_is_exact():
    rng = np.random.default_rng(5)
    k, v, _, _ = gdn_tokens(rng, 20, 8, 8)
    p1 = pair_of("none", k[:11], v[:11], None, None)
    p2 = pair_of("none", k[11:], v[11:], None, None)
    assert np.array_equal(p1[0], np.eye(8)) and np.array_equal(p2[0], np.eye(8))
    assert ls.rel_fro(ls.naive_add([p1, p2], [0, 1]), ls.compose([p1, p2], [0, 1])) < 1e-14
    # S = K^T V
    assert ls.rel_fro(p1[1], k[:11].T @ v[:11]) < 1e-14


def test_gla_closed_form():
    rng = np.random.default_rng(6)
    dk, dv, L = 10, 7, 33
    k, v, _, _ = gdn_tokens(rng, L, dk, dv)
    g = -np.logaddexp(0.0, -rng.normal(3.0, 1.0, (L, dk)))
    out = ls.segment_pair("diag", k, v, None, g)
    assert np.allclose(out["T"], np.diag(np.exp(g.sum(0))), rtol=1e-12, atol=0)
    # S = sum_t diag(exp(sum_{s>t} g_s)) k_t v_t^T
    S_ref = np.zeros((dk, dv))
    for t in range(L):
        S_ref += np.outer(np.exp(g[t + 1:].sum(0)) * k[t], v[t])
    assert ls.rel_fro(out["S"], S_ref) < 1e-12
    assert np.allclose(out["logG"], g.sum(0), rtol=1e-13)


def test_naive_add_slow_retnet_head_reproduces_pages(golden_dir):
    with open(os.path.join(golden_dir, "naive_add_retnet_slow_head.json")) as f:
        gold = json.load(f)
    gamma = 1.0 - 2.0 ** gold["gamma_log2_gap"]
    L2 = gold["L2"]
    rng = np.random.default_rng(7)
    dk = dv = 32
    k1, v1, _, _ = gdn_tokens(rng, 300, dk, dv)
    k2, v2, _, _ = gdn_tokens(rng, L2, dk, dv)
    p1 = pair_of("scalar", k1, v1, None, np.full(300, np.log(gamma)))
    p2 = pair_of("scalar", k2, v2, None, np.full(L2, np.log(gamma)))
    true = ls.compose([p1, p2], [0, 1])
    naive = ls.naive_add([p1, p2], [0, 1])
    err = np.linalg.norm(naive - true) / np.linalg.norm(p1[1])
    assert abs(err - (1 - gamma ** L2)) < 1e-12
    assert abs(err - gold["pages_value"]) < gold["pages_value_precision"]


# P6: brute force on 1-4 tokens ---------------------------------------------------

@pytest.mark.parametrize("dk", [1, 2, 64])
def test_brute_force_one_and_two_tokens(dk):
    rng = np.random.default_rng(10 + dk)
    dv = 3
    k, v, beta, g = gdn_tokens(rng, 2, dk, dv)
    a = np.exp(g)
    I = np.eye(dk)
    # L = 1
    out1 = ls.segment_pair("gdn", k[:1], v[:1], beta[:1], g[:1])
    A1 = a[0] * (I - beta[0] * np.outer(k[0], k[0]))
    assert np.allclose(out1["T"], A1, atol=1e-15)
    assert np.allclose(out1["S"], beta[0] * np.outer(k[0], v[0]), atol=1e-15)
    # L = 2
    out2 = ls.segment_pair("gdn", k, v, beta, g)
    A2 = a[1] * (I - beta[1] * np.outer(k[1], k[1]))
    assert np.allclose(out2["T"], A2 @ A1, atol=1e-14)
    S2 = A2 @ (beta[0] * np.outer(k[0], v[0])) + beta[1] * np.outer(k[1], v[1])
    assert np.allclose(out2["S"], S2, atol=1e-14)


def test_brute_force_scalar_key_dim():
    """dk = 1: every quantity is a scalar; T = prod alpha_t (1 - beta_t k_t^2)."""
    rng = np.random.default_rng(20)
    for L in (1, 2, 3, 4):
        k = rng.standard_normal((L, 1))       # not normalised on purpose
        v = rng.standard_normal((L, 2))
        beta = rng.random(L)
        g = -np.logaddexp(0.0, rng.normal(-4, 1, L))
        out = ls.segment_pair("gdn", k, v, beta, g)
        T = 1.0
        S = np.zeros(2)
        for t in range(L):
            a_t = np.exp(g[t]) * (1 - beta[t] * k[t, 0] ** 2)
            T = a_t * T
            S = a_t * S + beta[t] * k[t, 0] * v[t]
        assert abs(out["T"][0, 0] - T) < 1e-14
        assert np.allclose(out["S"][0], S, atol=1e-14)


def test_brute_force_three_and_four_tokens():
    rng = np.random.default_rng(21)
    dk, dv = 5, 4
    k, v, beta, g = gdn_tokens(rng, 4, dk, dv)
    I = np.eye(dk)
    A = [np.exp(g[t]) * (I - beta[t] * np.outer(k[t], k[t])) for t in range(4)]
    W = [beta[t] * np.outer(k[t], v[t]) for t in range(4)]
    out3 = ls.segment_pair("gdn", k[:3], v[:3], beta[:3], g[:3])
    assert np.allclose(out3["T"], A[2] @ A[1] @ A[0], atol=1e-14)
    assert np.allclose(out3["S"], A[2] @ A[1] @ W[0] + A[2] @ W[1] + W[2], atol=1e-14)
    out4 = ls.segment_pair("gdn", k, v, beta, g)
    assert np.allclose(out4["T"], A[3] @ A[2] @ A[1] @ A[0], atol=1e-14)
    S4 = A[3] @ A[2] @ A[1] @ W[0] + A[3] @ A[2] @ W[1] + A[3] @ W[2] + W[3]
    assert np.allclose(out4["S"], S4, atol=1e-14)


# P7: determinant; factored form ----------------------------------------------------

def test_determinant_of_delta_product():
    rng = np.random.default_rng(30)
    for L in (1, 3, 8):
        k, v, beta, g = gdn_tokens(rng, L, 16, 4)
        out = ls.segment_pair("gdn", k, v, beta, g)
        sign, logdet = np.linalg.slogdet(out["Q"])
        expect = np.prod(1 - beta * (k * k).sum(1))
        assert sign == np.sign(expect)
        assert abs(logdet - np.log(abs(expect))) < 1e-12
        # and T = exp(sum g) Q
        assert ls.rel_fro(out["T"], np.exp(g.sum()) * out["Q"]) < 1e-13
        assert abs(out["logG"] - g.sum()) < 1e-13


# P8: identity padding ----------------------------------------------------------

def test_identity_tokens_leave_pair_unchanged():
    rng = np.random.default_rng(40)
    k, v, beta, g = gdn_tokens(rng, 12, 8, 8)
    base = ls.segment_pair("gdn", k, v, beta, g)
    z8 = np.zeros((5, 8))
    for where in (0, 6, 12):
        kk = np.concatenate([k[:where], z8, k[where:]])
        vv = np.concatenate([v[:where], z8, v[where:]])
        bb = np.concatenate([beta[:where], np.zeros(5), beta[where:]])
        gg = np.concatenate([g[:where], np.zeros(5), g[where:]])
        out = ls.segment_pair("gdn", kk, vv, bb, gg)
        assert ls.rel_fro(out["T"], base["T"]) < 1e-14
        assert ls.rel_fro(out["S"], base["S"]) < 1e-14


# P9: special structure ---------------------------------------------------------

def test_zero_beta_gives_identity_and_zero_state():
    rng = np.random.default_rng(50)
    k, v, _, g = gdn_tokens(rng, 9, 8, 5)
    out = ls.segment_pair("gdn", k, v, np.zeros(9), g)
    assert np.allclose(out["Q"], np.eye(8), atol=0)
    assert np.abs(out["S"]).max() == 0.0


def test_orthonormal_keys_without_decay():
    rng = np.random.default_rng(51)
    dk, dv = 8, 3
    perm = rng.permutation(dk)[:5]
    k = np.eye(dk)[perm]
    v = rng.standard_normal((5, dv))
    beta = rng.random(5)
    out = ls.segment_pair("gdn", k, v, beta, np.zeros(5))
    diag = np.ones(dk)
    diag[perm] = 1 - beta
    assert np.allclose(out["T"], np.diag(diag), atol=1e-15)
    S_ref = sum(beta[t] * np.outer(k[t], v[t]) for t in range(5))
    assert np.allclose(out["S"], S_ref, atol=1e-15)


def test_delta_rule_without_gate_is_deltanet():
    """alpha = 1: S_t = S_{t-1} + beta_t k_t (v_t - S_{t-1}^T k_t)^T."""
    rng = np.random.default_rng(52)
    k, v, beta, _ = gdn_tokens(rng, 15, 6, 4)
    out = ls.segment_pair("gdn", k, v, beta, np.zeros(15))
    S = np.zeros((6, 4))
    for t in range(15):
        S = S + beta[t] * np.outer(k[t], v[t] - S.T @ k[t])
    assert ls.rel_fro(out["S"], S) < 1e-13


# seam window ------------------------------------------------------------------

def test_seam_one_token_by_hand():
    rng = np.random.default_rng(60)
    dk, dv = 6, 5
    S0 = rng.standard_normal((dk, dv))
    k, v, beta, g = gdn_tokens(rng, 1, dk, dv)
    q = rng.standard_normal((1, dk))
    S1, o = ls.seam_advance(S0, q, k, v, beta, g)
    a = np.exp(g[0])
    S_ref = a * (S0 - beta[0] * np.outer(k[0], k[0] @ S0)) + beta[0] * np.outer(k[0], v[0])
    assert np.allclose(S1, S_ref, atol=1e-14)
    assert np.allclose(o[0], S_ref.T @ q[0], atol=1e-14)


def test_seam_then_body_equals_full_recompute():
    """Reuse with seam windows: at each position the w seam tokens are run
    under the full prefix and then the body pair is composed; the result equals
    a sequential run over all tokens (seam + body of each segment in order)."""
    rng = np.random.default_rng(61)
    dk, dv, w = 8, 6, 3
    segs = [gdn_tokens(rng, n, dk, dv) for n in (10, 7, 12)]
    pairs = [pair_of("gdn", s[0][w:], s[1][w:], s[2][w:], s[3][w:]) for s in segs]
    order = [2, 0, 1]
    q = rng.standard_normal((3, w, dk))
    seam = dict(q=q,
                k=np.stack([segs[j][0][:w] for j in order]),
                v=np.stack([segs[j][1][:w] for j in order]),
                beta=np.stack([segs[j][2][:w] for j in order]),
                g=np.stack([segs[j][3][:w] for j in order]))
    S, o = ls.compose_with_seam(pairs, order, seam)
    cat = [np.concatenate([segs[j][i] for j in order]) for i in range(4)]
    S_seq = ls.run_from("gdn", np.zeros((dk, dv)), *cat)
    assert ls.rel_fro(S, S_seq) < 1e-12
    # the o of the first seam token of position 1 = S^T q after that token
    S_pre = ls.run_from("gdn", np.zeros((dk, dv)), *[segs[order[0]][i] for i in range(4)])
    S_t = ls.run_from("gdn", S_pre, *[segs[order[1]][i][:1] for i in range(4)])
    assert np.allclose(o[1, 0], S_t.T @ q[1, 0], atol=1e-13)


def test_factored_cache_form():
    Q = np.random.default_rng(70).standard_normal((4, 4))
    T = ls.cache_transition(Q, -3, -2.0)
    assert np.allclose(T, np.exp(-2.0) / 8.0 * Q, rtol=1e-15)
    # a device-style factorisation of the same Q: Qhat = Q 2^-e, same logG
    assert ls.rel_fro_factored(Q * 2.0 ** 5, -5, -1.5, Q, -1.5) < 1e-15
    # a wrong exponent or log-decay is visible
    assert ls.rel_fro_factored(Q * 2.0 ** 5, -4, -1.5, Q, -1.5) > 0.5
    assert ls.rel_fro_factored(Q * 2.0 ** 5, -5, -1.4, Q, -1.5) > 0.05


# Mamba2-style per-token scalar decay -------------------------------------------

def token_tokens(rng, L, dk, dv):
    """Per-token scalar gates in the Mamba2 range: g = dt * A with dt
    log-uniform in [1e-3, 1e-1] and A in [-16, -1]."""
    k, v, _, _ = gdn_tokens(rng, L, dk, dv)
    dt = np.exp(rng.uniform(np.log(1e-3), np.log(1e-1), L))
    g = dt * -rng.uniform(1.0, 16.0)
    return k, v, g


def test_token_decay_closed_form():
    """T = exp(sum g) I; S = sum_t exp(sum_{s>t} g_s) k_t v_t^T."""
    rng = np.random.default_rng(90)
    dk, dv, L = 9, 7, 37
    k, v, g = token_tokens(rng, L, dk, dv)
    out = ls.segment_pair("token", k, v, None, g)
    assert np.allclose(out["T"], np.exp(g.sum()) * np.eye(dk), rtol=1e-13, atol=0)
    S_ref = sum(np.exp(g[t + 1:].sum()) * np.outer(k[t], v[t]) for t in range(L))
    assert ls.rel_fro(out["S"], S_ref) < 1e-13
    assert out["logG"] == pytest.approx(g.sum(), rel=1e-14)


def test_token_decay_constant_gate_is_retnet():
    """A constant per-token gate is the RetNet head: T = gamma^L I and the
    closed form of the scalar family."""
    rng = np.random.default_rng(91)
    dk, dv, L = 8, 6, 25
    k, v, _ = token_tokens(rng, L, dk, dv)
    gamma = 1 - 2.0 ** -5
    out = ls.segment_pair("token", k, v, None, np.full(L, np.log(gamma)))
    assert np.allclose(out["T"], gamma ** L * np.eye(dk), rtol=1e-13, atol=0)
    S_ref = sum(gamma ** (L - 1 - t) * np.outer(k[t], v[t]) for t in range(L))
    assert ls.rel_fro(out["S"], S_ref) < 1e-13


def test_token_decay_outputs_match_the_dual_quadratic_form():
    """The state space duality of the Mamba2 paper: the recurrence's outputs
    from a zero state equal Y = (M o Q K^T) V with the 1-semiseparable mask
    M[t][s] = exp(sum_{s < r <= t} g_r) for s <= t, 0 above the diagonal."""
    rng = np.random.default_rng(92)
    dk, dv, L = 6, 5, 19
    k, v, g = token_tokens(rng, L, dk, dv)
    q = rng.standard_normal((L, dk))
    _, o = ls.seam_advance(np.zeros((dk, dv)), q, k, v, None, g, kind="token")
    cum = np.cumsum(g)
    M = np.tril(np.exp(cum[:, None] - cum[None, :]))
    assert ls.rel_fro(o, (M * (q @ k.T)) @ v) < 1e-12


# KDA: gated delta rule with a per-channel gate ------------------------------------

def kda_tokens(rng, L, dk, dv):
    k, v, beta, _ = gdn_tokens(rng, L, dk, dv)
    g = -np.logaddexp(0.0, -rng.normal(3.0, 1.0, (L, dk)))
    return k, v, beta, g


def _kda_pin_failures(segment_pair):
    """Pins of the KDA family against facts it does not compute itself; returns
    the names of those that fail."""
    fails = []
    rng = np.random.default_rng(93)
    dk, dv, L = 7, 5, 6
    k, v, beta, g = kda_tokens(rng, L, dk, dv)
    # (1) a gate equal on every channel commutes with the delta-rule factor: the
    #     family is then the gated delta rule (pinned above by brute force)
    c = g[:, 0]
    gu = np.repeat(c[:, None], dk, axis=1)
    a = segment_pair("kda", k, v, beta, gu)
    b = ls.segment_pair("gdn", k, v, beta, c)
    if not (ls.rel_fro(a["T"], b["T"]) < 1e-12 and ls.rel_fro(a["S"], b["S"]) < 1e-12):
        fails.append("uniform_gate_is_gdn")
    # (2) beta = 0: no write and no correction, only the per-channel decay
    z = segment_pair("kda", k, v, np.zeros(L), g)
    if not (np.allclose(z["T"], np.diag(np.exp(g.sum(0))), rtol=1e-13, atol=0)
            and np.abs(z["S"]).max() == 0.0):
        fails.append("zero_beta_is_decay_only")
    # (3) det T = prod_t (1 - beta_t |k_t|^2) exp(sum_i g_t[i])
    full = segment_pair("kda", k, v, beta, g)
    det_ref = np.prod(1 - beta * np.sum(k * k, axis=1)) * np.exp(g.sum())
    if not np.isclose(np.linalg.det(full["T"]), det_ref, rtol=1e-10, atol=0):
        fails.append("determinant")
    # (4) the delta rule's retrieval: for a unit key, after token t the state
    #     read at k_t is the beta-blend of the decayed old read and v_t,
    #     S_t^T k_t = (1 - beta_t) S_{t-1}^T (alpha_t o k_t) + beta_t v_t
    #     (decay first, then the correction, as the KDA paper orders them)
    for t in range(1, L):
        S_prev = segment_pair("kda", k[:t], v[:t], beta[:t], g[:t])["S"]
        S_t = segment_pair("kda", k[:t + 1], v[:t + 1], beta[:t + 1], g[:t + 1])["S"]
        lhs = S_t.T @ k[t]
        rhs = (1 - beta[t]) * (S_prev.T @ (np.exp(g[t]) * k[t])) + beta[t] * v[t]
        if not np.allclose(lhs, rhs, atol=1e-13):
            fails.append("retrieval_blend")
            break
    # (5) the composition law (pairs of a split equal the whole)
    p1 = segment_pair("kda", k[:2], v[:2], beta[:2], g[:2])
    p2 = segment_pair("kda", k[2:], v[2:], beta[2:], g[2:])
    T, S = ls.compose_pair((p1["T"], p1["S"]), (p2["T"], p2["S"]))
    if not (ls.rel_fro(T, full["T"]) < 1e-12 and ls.rel_fro(S, full["S"]) < 1e-12):
        fails.append("law")
    return fails


def test_kda_pins():
    assert _kda_pin_failures(ls.segment_pair) == []


def test_kda_no_gate_is_deltanet():
    """g = 0: S_t = S_{t-1} + beta_t k_t (v_t - S_{t-1}^T k_t)^T."""
    rng = np.random.default_rng(94)
    k, v, beta, _ = kda_tokens(rng, 13, 6, 4)
    out = ls.segment_pair("kda", k, v, beta, np.zeros((13, 6)))
    S = np.zeros((6, 4))
    for t in range(13):
        S = S + beta[t] * np.outer(k[t], v[t] - S.T @ k[t])
    assert ls.rel_fro(out["S"], S) < 1e-13


def test_kda_seam_then_body_equals_full_recompute():
    rng = np.random.default_rng(95)
    dk, dv, w = 8, 6, 3
    segs = [kda_tokens(rng, n, dk, dv) for n in (9, 6, 11)]
    pairs = [pair_of("kda", s[0][w:], s[1][w:], s[2][w:], s[3][w:]) for s in segs]
    order = [1, 2, 0]
    q = rng.standard_normal((3, w, dk))
    seam = dict(q=q, k=np.stack([segs[j][0][:w] for j in order]),
                v=np.stack([segs[j][1][:w] for j in order]),
                beta=np.stack([segs[j][2][:w] for j in order]),
                g=np.stack([segs[j][3][:w] for j in order]))
    S, o = ls.compose_with_seam(pairs, order, seam, kind="kda")
    cat = [np.concatenate([segs[j][i] for j in order]) for i in range(4)]
    assert ls.rel_fro(S, ls.run_from("kda", np.zeros((dk, dv)), *cat)) < 1e-12
    S_pre = ls.run_from("kda", np.zeros((dk, dv)), *[segs[order[0]][i] for i in range(4)])
    S_t = ls.run_from("kda", S_pre, *[segs[order[1]][i][:2] for i in range(4)])
    assert np.allclose(o[1, 1], S_t.T @ q[1, 1], atol=1e-13)


def test_kda_planted_mistakes_are_caught():
    base = ls.segment_pair

    def recur(step):
        def sp(kind, k, v, beta=None, g=None, want_T=True):
            if kind != "kda":
                return base(kind, k, v, beta, g, want_T)
            dk = k.shape[1]
            T, S = np.eye(dk), np.zeros((dk, v.shape[1]))
            for t in range(len(k)):
                T, S = step(T, S, k[t], v[t], beta[t], g[t])
            return dict(T=T, S=S)
        return sp

    def H(kt, bt):
        return np.eye(len(kt)) - bt * np.outer(kt, kt)

    swapped = recur(lambda T, S, kt, vt, bt, gt: (
        np.diag(np.exp(gt)) @ H(kt, bt) @ T,
        np.diag(np.exp(gt)) @ H(kt, bt) @ S + bt * np.outer(kt, vt)))
    no_beta_write = recur(lambda T, S, kt, vt, bt, gt: (
        H(kt, bt) @ np.diag(np.exp(gt)) @ T,
        H(kt, bt) @ np.diag(np.exp(gt)) @ S + np.outer(kt, vt)))
    gate_not_exponentiated = recur(lambda T, S, kt, vt, bt, gt: (
        H(kt, bt) @ np.diag(1 + gt) @ T,
        H(kt, bt) @ np.diag(1 + gt) @ S + bt * np.outer(kt, vt)))
    sign_flip = recur(lambda T, S, kt, vt, bt, gt: (
        (np.eye(len(kt)) + bt * np.outer(kt, kt)) @ np.diag(np.exp(gt)) @ T,
        (np.eye(len(kt)) + bt * np.outer(kt, kt)) @ np.diag(np.exp(gt)) @ S
        + bt * np.outer(kt, vt)))
    right = recur(lambda T, S, kt, vt, bt, gt: (
        H(kt, bt) @ np.diag(np.exp(gt)) @ T,
        H(kt, bt) @ np.diag(np.exp(gt)) @ S + bt * np.outer(kt, vt)))
    assert _kda_pin_failures(right) == []
    for name, m in (("swapped", swapped), ("no_beta_write", no_beta_write),
                    ("gate_not_exponentiated", gate_not_exponentiated),
                    ("sign_flip", sign_flip)):
        assert _kda_pin_failures(m), name


# planted mistakes ---------------------------------------------------------------

def _mutant_checks(segment_pair):
    """Run a compact subset of the pins against a given segment_pair; return
    the names of the pins that fail."""
    fails = []
    rng = np.random.default_rng(80)
    dk, dv = 6, 5
    k, v, beta, g = gdn_tokens(rng, 4, dk, dv)
    I = np.eye(dk)
    A = [np.exp(g[t]) * (I - beta[t] * np.outer(k[t], k[t])) for t in range(4)]
    Wt = [beta[t] * np.outer(k[t], v[t]) for t in range(4)]
    out = segment_pair("gdn", k, v, beta, g)
    if not np.allclose(out["T"], A[3] @ A[2] @ A[1] @ A[0], atol=1e-13):
        fails.append("brute_T")
    S4 = A[3] @ A[2] @ A[1] @ Wt[0] + A[3] @ A[2] @ Wt[1] + A[3] @ Wt[2] + Wt[3]
    if not np.allclose(out["S"], S4, atol=1e-13):
        fails.append("brute_S")
    gam = 1 - 2 ** -6
    o = segment_pair("scalar", k, v, None, np.full(4, np.log(gam)))
    if not np.allclose(o["T"], gam ** 4 * I, rtol=1e-12, atol=0):
        fails.append("retnet")
    return fails


def test_planted_mistakes_are_caught(monkeypatch):
    base = ls.segment_pair
    assert _mutant_checks(base) == []

    def reversed_product(kind, k, v, beta=None, g=None, want_T=True):
        out = base(kind, k, v, beta, g, want_T)
        T = np.eye(k.shape[1])
        for t in range(len(k)):
            T = T @ ls.transition(kind, k.shape[1], k[t], None if beta is None else beta[t],
                                  None if g is None else g[t])
        out["T"] = T
        return out

    def dropped_beta_write(kind, k, v, beta=None, g=None, want_T=True):
        out = base(kind, k, v, beta, g, want_T)
        S = np.zeros((k.shape[1], v.shape[1]))
        for t in range(len(k)):
            A = ls.transition(kind, k.shape[1], k[t], None if beta is None else beta[t],
                              None if g is None else g[t])
            S = A @ S + np.outer(k[t], v[t])
        out["S"] = S
        return out

    def sign_flip(kind, k, v, beta=None, g=None, want_T=True):
        return base(kind, k, v, None if beta is None else -beta, g, want_T)

    def off_by_one_decay(kind, k, v, beta=None, g=None, want_T=True):
        return base(kind, k, v, beta, None if g is None else np.roll(g, 1), want_T)

    for mutant in (reversed_product, dropped_beta_write, sign_flip, off_by_one_decay):
        assert _mutant_checks(mutant), mutant.__name__


def _seam_checks():
    """The seam pins as one function, returning the names of the ones that
    fail (an exception counts as a failure), so mutants can be run through
    them."""
    failed = []
    for name, pin in (("by_hand", test_seam_one_token_by_hand),
                      ("full_recompute", test_seam_then_body_equals_full_recompute),
                      ("square_by_hand", _seam_square_by_hand)):
        try:
            pin()
        except Exception:  # noqa: BLE001 - any failure of a pin catches the mutant
            failed.append(name)
    return failed


def _seam_square_by_hand():
    """Two seam tokens at dk = dv, expanded by hand, so a transposed read-out
    cannot hide behind a shape error."""
    rng = np.random.default_rng(62)
    d = 5
    S0 = rng.standard_normal((d, d))
    k, v, beta, g = gdn_tokens(rng, 2, d, d)
    q = rng.standard_normal((2, d))
    S, o = ls.seam_advance(S0, q, k, v, beta, g)
    ref = S0
    for t in range(2):
        ref = np.exp(g[t]) * (ref - beta[t] * np.outer(k[t], k[t] @ ref)) \
            + beta[t] * np.outer(k[t], v[t])
        assert np.allclose(o[t], ref.T @ q[t], atol=1e-13)
    assert np.allclose(S, ref, atol=1e-13)


def test_seam_planted_mistakes_are_caught(monkeypatch):
    """Mistakes planted into the oracle's seam path (on the CPU) each fail one
    of the seam pins: the read-out taken before the token's update, the read-out
    transposed, the window applied after the body instead of before it, and
    the window's decay dropped."""
    assert _seam_checks() == []
    base_adv, base_cws = ls.seam_advance, ls.compose_with_seam

    def read_before_update(S0, q, k, v, beta, g, kind="gdn"):
        S = np.array(S0, dtype=np.float64, copy=True)
        outs = []
        for t in range(len(k)):
            outs.append(S.T @ q[t])
            A = ls.transition(kind, S.shape[0], k[t], beta[t], g[t])
            S = A @ S + beta[t] * np.outer(k[t], v[t])
        return S, np.array(outs)

    def transposed_readout(S0, q, k, v, beta, g, kind="gdn"):
        S, o = base_adv(S0, q, k, v, beta, g, kind)
        S_t = np.array(S0, dtype=np.float64, copy=True)
        outs = []
        for t in range(len(k)):
            A = ls.transition(kind, S_t.shape[0], k[t], beta[t], g[t])
            S_t = A @ S_t + beta[t] * np.outer(k[t], v[t])
            outs.append(S_t @ q[t])
        return S, np.array(outs)

    def no_window_decay(S0, q, k, v, beta, g, kind="gdn"):
        return base_adv(S0, q, k, v, beta, np.zeros_like(g), kind)

    def window_after_body(pairs, order, seam, state_in=None, kind="gdn"):
        S, o_all = None, []
        for j, seg in enumerate(order):
            T, Sj = pairs[seg]
            S = (np.zeros_like(Sj) if state_in is None else np.array(state_in)) if S is None else S
            S = T @ S + Sj
            S, o = base_adv(S, seam["q"][j], seam["k"][j], seam["v"][j], seam["beta"][j],
                            seam["g"][j], kind)
            o_all.append(o)
        return S, np.array(o_all)

    for attr, mutant in (("seam_advance", read_before_update),
                         ("seam_advance", transposed_readout),
                         ("seam_advance", no_window_decay),
                         ("compose_with_seam", window_after_body)):
        with monkeypatch.context() as m:
            m.setattr(ls, attr, mutant)
            assert _seam_checks(), mutant.__name__
    assert ls.seam_advance is base_adv and ls.compose_with_seam is base_cws


def test_compose_from_a_given_state():
    """Composing from a given running state equals running the segments'
    tokens, in request order, from that state (the law applied to a prefix
    that is not cached)."""
    rng = np.random.default_rng(63)
    dk, dv = 7, 5
    segs = [gdn_tokens(rng, n, dk, dv) for n in (6, 11, 4)]
    pairs = [pair_of("gdn", *s) for s in segs]
    order = [1, 2, 0, 1]
    S0 = rng.standard_normal((dk, dv))
    cat = [np.concatenate([segs[j][i] for j in order]) for i in range(4)]
    assert ls.rel_fro(ls.compose(pairs, order, state_in=S0),
                      ls.run_from("gdn", S0, *cat)) < 1e-12
    # an empty request leaves the given state as it is
    assert np.array_equal(ls.compose(pairs, [], state_in=S0), S0)


def _compose_checks():
    """The composition pins as one function; returns the names that fail."""
    failed = []
    pins = [("law_" + kind, lambda kind=kind: test_law_split_equals_concatenation(kind))
            for kind in ("gdn", "scalar", "diag")]
    pins += [("small_order", test_gdn_small_order_equals_sequential_concatenation),
             ("given_state", test_compose_from_a_given_state),
             ("retnet", test_retnet_closed_form),
             ("factored", test_factored_cache_form)]
    for name, pin in pins:
        try:
            pin()
        except Exception:  # noqa: BLE001 - any failure of a pin catches the mutant
            failed.append(name)
    return failed


def test_compose_planted_mistakes_are_caught(monkeypatch):
    """Mistakes planted into the oracle's composition (on the CPU) each fail
    one of the composition pins: the write added before the transition, the
    transitions multiplied in the wrong order, the request order ignored, the
    given state ignored, and a sign error in the cache's exponent."""
    assert _compose_checks() == []
    base_compose = ls.compose

    def add_then_multiply(pairs, order, state_in=None):
        S = np.zeros_like(pairs[0][1]) if state_in is None else np.array(state_in, np.float64)
        for j in order:
            S = pairs[j][0] @ (S + pairs[j][1])
        return S

    def pair_product_swapped(p1, p2):
        return p1[0] @ p2[0], p2[0] @ p1[1] + p2[1]

    def order_sorted(pairs, order, state_in=None):
        return base_compose(pairs, sorted(order), state_in)

    def state_in_ignored(pairs, order, state_in=None):
        return base_compose(pairs, order, None)

    def exponent_sign(Qhat, exp2, logG):
        return np.exp(float(logG)) * np.ldexp(1.0, -int(exp2)) * np.asarray(Qhat, np.float64)

    for attr, mutant in (("compose", add_then_multiply),
                         ("compose_pair", pair_product_swapped),
                         ("compose", order_sorted),
                         ("compose", state_in_ignored),
                         ("cache_transition", exponent_sign)):
        with monkeypatch.context() as m:
            m.setattr(ls, attr, mutant)
            assert _compose_checks(), mutant.__name__
    assert ls.compose is base_compose


def _token_checks():
    """The per-token scalar decay pins as one function; returns the names that
    fail."""
    failed = []
    for name, pin in (("closed_form", test_token_decay_closed_form),
                      ("constant_gate", test_token_decay_constant_gate_is_retnet),
                      ("dual_form", test_token_decay_outputs_match_the_dual_quadratic_form)):
        try:
            pin()
        except Exception:  # noqa: BLE001 - any failure of a pin catches the mutant
            failed.append(name)
    return failed


def test_token_decay_planted_mistakes_are_caught(monkeypatch):
    """Mistakes planted into the oracle's per-token scalar decay (on the CPU)
    each fail one of its pins: the gate linearised (1 + g instead of e^g), its
    sign flipped, each token given its predecessor's gate, and the write
    decayed by its own token's gate."""
    assert _token_checks() == []
    base_tr, base_pair = ls.transition, ls.segment_pair

    def tr_mutant(fn):
        def f(kind, dk, k_t=None, beta_t=None, g_t=None):
            if kind == "token":
                return fn(float(g_t)) * np.eye(dk)
            return base_tr(kind, dk, k_t, beta_t, g_t)
        return f

    linearised = tr_mutant(lambda g: 1.0 + g)
    sign_flip = tr_mutant(lambda g: np.exp(-g))

    def previous_gate(kind, k, v, beta=None, g=None, want_T=True):
        if kind == "token":
            g = np.concatenate([[0.0], np.asarray(g)[:-1]])
        return base_pair(kind, k, v, beta, g, want_T)

    def write_decayed(kind, k, v, beta=None, g=None, want_T=True):
        out = base_pair(kind, k, v, beta, g, want_T)
        if kind == "token":
            S = np.zeros((k.shape[1], v.shape[1]))
            for t in range(len(k)):
                S = np.exp(g[t]) * (S + np.outer(k[t], v[t]))
            out["S"] = S
        return out

    for attr, mutant in (("transition", linearised), ("transition", sign_flip),
                         ("segment_pair", previous_gate), ("segment_pair", write_decayed)):
        with monkeypatch.context() as m:
            m.setattr(ls, attr, mutant)
            assert _token_checks(), (attr, mutant.__name__)
    assert ls.transition is base_tr and ls.segment_pair is base_pair


def _decay_checks():
    """The decay-only families' pins as one function; returns the names that
    fail."""
    failed = []
    pins = [("law_" + kind, lambda kind=kind: test_law_split_equals_concatenation(kind))
            for kind in ("scalar", "diag", "none")]
    pins += [("retnet", test_retnet_closed_form), ("gla", test_gla_closed_form),
             ("plain", test_plain_linear_attention_naive_add_is_exact)]
    for name, pin in pins:
        try:
            pin()
        except Exception:  # noqa: BLE001 - any failure of a pin catches the mutant
            failed.append(name)
    return failed


def test_decay_families_planted_mistakes_are_caught(monkeypatch):
    """Mistakes planted into the decay-only families (on the CPU) each fail
    one of their pins: the write decayed by its own token's gate (RetNet and
    GLA), GLA's gate taken over the value channels, and a plain linear
    attention pair whose transition is not the identity."""
    assert _decay_checks() == []
    base_pair = ls.segment_pair

    def write_decayed(family):
        def f(kind, k, v, beta=None, g=None, want_T=True):
            out = base_pair(kind, k, v, beta, g, want_T)
            if kind == family:
                S = np.zeros((k.shape[1], v.shape[1]))
                for t in range(len(k)):
                    d = np.exp(np.asarray(g[t], np.float64))
                    S = (d[:, None] if d.ndim else d) * (S + np.outer(k[t], v[t]))
                out["S"] = S
            return out
        return f

    def gla_value_side(kind, k, v, beta=None, g=None, want_T=True):
        out = base_pair(kind, k, v, beta, g, want_T)
        if kind == "diag":
            S = np.zeros((k.shape[1], v.shape[1]))
            for t in range(len(k)):
                S = S * np.exp(np.asarray(g[t]))[None, :] + np.outer(k[t], v[t])
            out["S"] = S
        return out

    def plain_scaled(kind, k, v, beta=None, g=None, want_T=True):
        out = base_pair(kind, k, v, beta, g, want_T)
        if kind == "none" and want_T:
            out["T"] = out["T"] * (1.0 - 1.0 / 64)
        return out

    for mutant in (write_decayed("scalar"), write_decayed("diag"), gla_value_side, plain_scaled):
        with monkeypatch.context() as m:
            m.setattr(ls, "segment_pair", mutant)
            assert _decay_checks(), mutant.__name__
    assert ls.segment_pair is base_pair
