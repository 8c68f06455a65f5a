"""float64 token-by-token definitions of the linear-layer caching math.

TEST INFRASTRUCTURE ONLY (see the package docstring): never called by the
library.  Nothing here is blocked, chunked, fused or reordered.

Sources (HYPIC, position-independent caching for hybrid-attention models):

* youleyou.com, "小红书联合北大上交提出HYPIC，位置无关缓存降低首token延迟3.25倍",
  linear-layer paragraph: the segment's cumulative transition T_C is the ordered
  product of the per-token transition matrices inside the segment; S(C|0) is the
  segment's final state from a zero start; both depend only on the segment's own
  tokens; the composition law is S(C1 C2) = T(C2) S(C1) + S(C2), and adding
  zero-start states without T_C is exact only for plain linear attention.
* llm-wiki.hwlabs.dev, "HYPIC: 하이브리드 어텐션 LLM 서빙에서 포지션 독립적 캐싱으로
  TTFT를 2.45배 낮추는 방법", section "세그먼트 누적 전이 연산자" (segment cumulative
  transition operator): h_out = T_S h_in + e_S, T_ABC = T_C T_B T_A,
  e_ABC = T_C (T_B e_A + e_B) + e_C.
* youleyou.com article, seam-window paragraph: the first w tokens (default 8) of
  a reused segment are not cached; at reuse the linear layer computes the
  window's own T and S on the fly, advances the running state and forwards each
  seam token's output upward.

Conventions the pages leave open, taken here (plainest reading consistent with
the law): the state S is dk x dv and LEFT-multiplied by the transition,
S_t = A_t S_{t-1} + b_t k_t v_t^T; the output of token t is o_t = S_t^T q_t,
read after token t's update; per-token transitions by head family

    gated delta (GDN):  A_t = alpha_t (I - beta_t k_t k_t^T),  b_t = beta_t
    RetNet (scalar):    A_t = gamma I,                         b_t = 1
    GLA (diagonal):     A_t = diag(alpha_t) on the key axis,   b_t = 1
    plain linear attn:  A_t = I,                               b_t = 1
    Mamba2 ("token"):   A_t = alpha_t I, alpha_t per token,    b_t = 1
    KDA:                A_t = (I - beta_t k_t k_t^T) diag(alpha_t),  b_t = beta_t

and alpha_t = exp(g_t) with g_t = log(alpha_t) the fp32 input, so the same
rounded g feeds both this oracle and the device path.

The pages only name Mamba2 and KDA among the families the method covers; their
update rules are taken from their own papers:

* Mamba2: "Transformers are SSMs: Generalized Models and Efficient Algorithms
  Through Structured State Space Duality" (Dao, Gu 2024), state space duality
  section: the SSM whose per-step transition is a scalar times the identity,
  h_t = a_t h_{t-1} + B_t x_t^T, y_t = h_t^T C_t.  Read here as k_t = B_t,
  v_t = x_t (the step size folded into the inputs by the caller), q_t = C_t,
  g_t = log a_t per token and head.
* KDA (Kimi Delta Attention): "Kimi Linear: An Expressive, Efficient Hybrid
  Linear Attention Architecture" (Kimi team 2025), KDA section: the gated delta
  rule with a per-key-channel gate, S_t = (I - beta_t k_t k_t^T) Diag(alpha_t)
  S_{t-1} + beta_t k_t v_t^T, o_t = S_t^T q_t: the decay acts first, then the
  delta-rule correction.
"""
from __future__ import annotations

import numpy as np

KINDS = ("gdn", "scalar", "diag", "none", "token", "kda")


# per-token transition ---------------------------------------------------------

def transition(kind: str, dk: int, k_t=None, beta_t=None, g_t=None) -> np.ndarray:
    """A_t as an explicit dense dk x dk float64 matrix."""
    eye = np.eye(dk)
    if kind == "gdn":
        alpha = np.exp(float(g_t))
        return alpha * (eye - float(beta_t) * np.outer(k_t, k_t))
    if kind in ("scalar", "token"):
        return np.exp(float(g_t)) * eye
    if kind == "diag":
        return np.diag(np.exp(np.asarray(g_t, dtype=np.float64)))
    if kind == "none":
        return eye
    if kind == "kda":
        H = eye - float(beta_t) * np.outer(k_t, k_t)
        return H @ np.diag(np.exp(np.asarray(g_t, dtype=np.float64)))
    raise ValueError(kind)


def write_weight(kind: str, beta_t=None) -> float:
    """b_t: beta_t for the delta rules, 1 for the decay-only families."""
    return float(beta_t) if kind in ("gdn", "kda") else 1.0


# segment pair ------------------------------------------------------------------

def segment_pair(kind: str, k, v, beta=None, g=None, want_T: bool = True):
    """(T_C, S(C|0)) of one segment by the token recurrence, plus the factored
    transition for the comparison against the device cache.

    k: [L, dk], v: [L, dv], beta: [L] (gdn, kda), g: [L] (gdn, scalar, token)
    or [L, dk] (diag, kda), all float64 copies of the exact inputs.

    Returns dict with
      T      : A_L ... A_1 (dk x dk), formed by T <- A_t T from I  (if want_T)
      S      : S_L from S_0 = 0 under S_t = A_t S_{t-1} + b_t k_t v_t^T
      logG   : sum_t g_t (gdn, scalar, token: scalar; diag, kda: per key channel
               [dk]; none: 0)
      Q      : gdn only, H_L ... H_1 with H_t = I - beta_t k_t k_t^T, so that
               T = exp(logG) * Q (decay factored out: at long L, T itself is
               far below any useful scale while Q and logG are not).
    """
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    L, dk = k.shape
    dv = v.shape[1]
    T = np.eye(dk) if want_T else None
    S = np.zeros((dk, dv))
    Q = np.eye(dk) if kind == "gdn" else None
    logG = np.zeros(dk) if kind in ("diag", "kda") else 0.0
    for t in range(L):
        if kind == "gdn":
            H = np.eye(dk) - float(beta[t]) * np.outer(k[t], k[t])
            A = np.exp(float(g[t])) * H
            Q = H @ Q
        else:
            A = transition(kind, dk, k[t], None if beta is None else beta[t],
                           None if g is None else g[t])
        if want_T:
            T = A @ T
        S = A @ S + write_weight(kind, None if beta is None else beta[t]) * np.outer(k[t], v[t])
        if kind in ("gdn", "scalar", "token"):
            logG = logG + float(g[t])
        elif kind in ("diag", "kda"):
            logG = logG + np.asarray(g[t], dtype=np.float64)
    out = dict(S=S, logG=logG)
    if want_T:
        out["T"] = T
    if Q is not None:
        out["Q"] = Q
    return out


def run_from(kind: str, S0, k, v, beta=None, g=None):
    """Final state after the tokens, starting from state S0 (full recompute)."""
    S = np.array(S0, dtype=np.float64, copy=True)
    dk = S.shape[0]
    for t in range(len(k)):
        A = transition(kind, dk, k[t], None if beta is None else beta[t],
                       None if g is None else g[t])
        S = A @ S + write_weight(kind, None if beta is None else beta[t]) * np.outer(k[t], v[t])
    return S


# composition -------------------------------------------------------------------

def compose(pairs, order, state_in=None):
    """Running state after the cached segments in ``order``:
    S <- T_j S + S_j for j in order, from ``state_in`` (zero if None).

    pairs: sequence of (T_j [dk x dk], S_j [dk x dv]) float64."""
    T0, S0 = pairs[order[0]] if len(order) else pairs[0]
    S = np.zeros_like(S0, dtype=np.float64) if state_in is None else \
        np.array(state_in, dtype=np.float64, copy=True)
    for j in order:
        T, Sj = pairs[j]
        S = T @ S + Sj
    return S


def compose_pair(p1, p2):
    """(T, S) of the concatenation C1 C2 from the two cached pairs:
    T(C1 C2) = T(C2) T(C1),  S(C1 C2) = T(C2) S(C1) + S(C2)."""
    T1, S1 = p1
    T2, S2 = p2
    return T2 @ T1, T2 @ S1 + S2


def naive_add(pairs, order):
    """The strawman the pages reject: sum of zero-start final states."""
    S = None
    for j in order:
        S = pairs[j][1].copy() if S is None else S + pairs[j][1]
    return S


def cache_transition(Qhat, exp2, logG):
    """T from the device cache's factored form T = e^logG * 2^exp2 * Qhat
    (gdn), evaluated in float64."""
    return np.exp(float(logG)) * np.ldexp(1.0, int(exp2)) * np.asarray(Qhat, np.float64)


# seam window -------------------------------------------------------------------

def seam_advance(S0, q, k, v, beta, g, kind: str = "gdn"):
    """Advance the running state through seam-window tokens of one head, token
    by token, emitting o_t = S_t^T q_t after each update (gated delta unless
    ``kind`` names another family).

    S0: [dk, dv]; q, k: [w, dk]; v: [w, dv]; beta: [w] (delta rules, else
    None); g: [w] or [w, dk] (per-channel gates).  Returns (S_w, o [w, dv])."""
    S = np.array(S0, dtype=np.float64, copy=True)
    dk = S.shape[0]
    outs = []
    for t in range(len(k)):
        b = None if beta is None else beta[t]
        A = transition(kind, dk, k[t], b, None if g is None else g[t])
        S = A @ S + write_weight(kind, b) * np.outer(k[t], v[t])
        outs.append(S.T @ np.asarray(q[t], dtype=np.float64))
    return S, np.array(outs).reshape(len(k), S.shape[1])


def compose_with_seam(pairs, order, seam, state_in=None, kind: str = "gdn"):
    """Reuse path for one (request, stream): at every position j the w seam
    tokens of that position advance the state (emitting o), then the cached
    body pair of segment order[j] is composed: S <- T S + S_body.

    seam: dict of float64 arrays q, k [P, w, dk], v [P, w, dv], beta [P, w]
    (delta rules), g [P, w] or [P, w, dk] (None without decay) (P = len(order)).
    Returns (S_final, o [P, w, dv])."""
    S = None
    o_all = []
    for j, seg in enumerate(order):
        T, Sj = pairs[seg]
        if S is None:
            S = np.zeros_like(Sj) if state_in is None else np.array(state_in, np.float64)
        beta, g = seam.get("beta"), seam.get("g")
        S, o = seam_advance(S, seam["q"][j], seam["k"][j], seam["v"][j],
                            None if beta is None else beta[j], None if g is None else g[j], kind)
        o_all.append(o)
        S = T @ S + Sj
    return S, np.array(o_all)


# error metric ------------------------------------------------------------------

def rel_fro(x, ref) -> float:
    """||x - ref||_F / ||ref||_F in float64 (0 when both are zero)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0.0:
        return 0.0 if num == 0.0 else float("inf")
    return float(num / den)


def rel_fro_factored(Qhat, exp2, logG, Q_ref, logG_ref) -> float:
    """Relative error of a factored device transition against the oracle's
    factored one: || e^(logG - logG_ref) 2^exp2 Qhat - Q_ref ||_F / ||Q_ref||_F."""
    scale = np.exp(float(logG) - float(logG_ref)) * np.ldexp(1.0, int(exp2))
    return rel_fro(scale * np.asarray(Qhat, np.float64), Q_ref)
