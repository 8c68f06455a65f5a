"""Seeded synthetic inputs for the linear-layer caching path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no transition, state, composition or schedule).  It is the
one module that both the CUDA path's tests/bench and the float64 oracle read.

Workload shapes follow the HYPIC pages' description of prompts built from
tens to hundreds of independent segments, usually longer than 512 tokens,
32k-128k tokens in total (youleyou.com HYPIC article, opening and seam-window
paragraphs).  The public datasets the pages evaluate on are not used; these
draws stand in for them and take only their shape.

Recipe (numpy PCG64 ``default_rng(seed)``; draws in float64, then one cast to
the dtype the library reads, torch round-to-nearest-even):

* draw order: decay logits x, beta, k, v, q (a draw a workload does not use is
  skipped);
* gated-delta heads: x ~ N(-4, 1), g = log(alpha) = -softplus(x) (float64,
  then fp32); beta ~ U(0, 1) fp32; k ~ N(0, 1) then L2-normalised in float64;
  v ~ N(0, 1); q ~ N(0, 1) (normalised only where the workload says so);
* RetNet heads: per-head constant gamma_h = 1 - 2^(-5-h), passed as fp32
  log(gamma_h);
* GLA heads: per (token, head, key channel) alpha = sigmoid(z), z ~ N(3, 1), so
  g = -softplus(-z).
* Mamba2-style heads (per-token scalar decay): per head A_h ~ -U(1, 16), per
  (token, head) step dt = exp(U(ln 1e-3, ln 1e-1)), g = dt * A_h (the ranges of
  the Mamba2 paper's initialisation); k L2-normalised, v ~ N(0, 1).
* KDA heads: beta ~ U(0, 1), k L2-normalised, v ~ N(0, 1) and the GLA gate per
  (token, head, key channel).

Tokens are packed varlen: ``[N_tok, n_streams, d]`` row-major, with int64
``offsets[n_seg + 1]``.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

# The five workloads (sizes) -------------------------------------------------
GDN_SMALL = dict(n_seg=4, seg_len=256, n_streams=1, d=64, seed=1000)
DECAY_HEADS = dict(n_seg=16, seg_len=512, n_retnet=8, n_gla=8, d=128, seed=1001)
GDN_LAYER = dict(n_seg=64, seg_len=1024, n_streams=16, d=128, seed=1002)
REUSE = dict(n_req=32, n_pos=128, w=8, n_streams=16, d=128, seed=1003)
COLD_LONG = dict(total=131072, mean_len=1024.0, sigma=0.8, lo=128, hi=8192,
                 n_layers=30, n_heads=16, d=128, seed=1004)
SLOW_REUSE = dict(n_seg=8, seg_len=256, n_req=4, n_pos=8, w=8, n_streams=16,
                  d=128, seed=1005)
TOKEN_KDA_HEADS = dict(n_seg=16, seg_len=512, n_token=8, n_kda=8, d=128, seed=1006)

_BLOCK = 1 << 22  # elements per float64 draw block (32 MiB)


def softplus64(x: np.ndarray) -> np.ndarray:
    """log(1 + e^x) in float64, without overflow."""
    return np.logaddexp(0.0, x)


def _draw(rng, kind: str, shape, *, normalize=False, loc=0.0, scale=1.0):
    """Draw ``shape`` float64 values in row blocks (same stream as one draw)."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.float64)
    if out.size == 0:
        return out
    flat = out.reshape(shape[0], -1)
    per_row = flat.shape[1]
    rows = max(1, _BLOCK // max(per_row, 1))
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        n = (r1 - r0, per_row)
        if kind == "normal":
            blk = rng.standard_normal(n)
            if scale != 1.0 or loc != 0.0:
                blk = blk * scale + loc
        elif kind == "uniform":
            blk = rng.random(n)
        else:
            raise ValueError(kind)
        flat[r0:r1] = blk
    if normalize:
        out /= np.linalg.norm(out, axis=-1, keepdims=True)
    return out


def _cast(a: np.ndarray, dtype: torch.dtype) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype)


def offsets_of(lengths) -> np.ndarray:
    lengths = np.asarray(lengths, dtype=np.int64)
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    off[1:] = np.cumsum(lengths)
    return off


@dataclass
class Packed:
    """One build call's inputs: packed tokens for ``n_streams`` streams."""
    kind: str                   # "gdn" | "scalar" | "diag" | "none" | "token" | "kda"
    offsets: np.ndarray         # int64 [n_seg + 1]
    k: torch.Tensor             # [N_tok, S, dk] bf16 or fp32
    v: torch.Tensor             # [N_tok, S, dv]
    beta: Optional[torch.Tensor] = None       # [N_tok, S] fp32 (gdn, kda)
    log_alpha: Optional[torch.Tensor] = None  # gdn, token [N,S]; diag, kda [N,S,dk]; scalar [S]
    q: Optional[torch.Tensor] = None          # [N_tok, S, dk] (unused by build)
    seam_w: int = 0
    meta: dict = field(default_factory=dict)

    @property
    def n_seg(self):
        return len(self.offsets) - 1

    @property
    def n_streams(self):
        return self.k.shape[1]

    @property
    def dk(self):
        return self.k.shape[2]

    @property
    def dv(self):
        return self.v.shape[2]


def gdn_packed(lengths, n_streams, dk, dv, seed, dtype=torch.bfloat16,
               x_mean=-4.0, with_q=False, q_normalize=False, seam_w=0) -> Packed:
    """Gated-delta heads over segments of the given lengths."""
    rng = np.random.default_rng(seed)
    off = offsets_of(lengths)
    n = int(off[-1])
    x = _draw(rng, "normal", (n, n_streams), loc=x_mean)
    beta = _draw(rng, "uniform", (n, n_streams))
    k = _draw(rng, "normal", (n, n_streams, dk), normalize=True)
    v = _draw(rng, "normal", (n, n_streams, dv))
    q = None
    if with_q:
        q = _cast(_draw(rng, "normal", (n, n_streams, dk), normalize=q_normalize), dtype)
    g = -softplus64(x)
    return Packed("gdn", off, _cast(k, dtype), _cast(v, dtype),
                  _cast(beta, torch.float32), _cast(g, torch.float32), q,
                  seam_w=seam_w, meta=dict(seed=seed, x_mean=x_mean))


def token_packed(lengths, n_streams, dk, dv, seed, dtype=torch.bfloat16) -> Packed:
    """Mamba2-style heads (per-token scalar decay) over segments of the given
    lengths.  Draw order: A, dt, k, v."""
    rng = np.random.default_rng(seed)
    off = offsets_of(lengths)
    n = int(off[-1])
    A = -(1.0 + 15.0 * _draw(rng, "uniform", (1, n_streams)))
    dt = np.exp(np.log(1e-3) + (np.log(1e-1) - np.log(1e-3)) *
                _draw(rng, "uniform", (n, n_streams)))
    k = _draw(rng, "normal", (n, n_streams, dk), normalize=True)
    v = _draw(rng, "normal", (n, n_streams, dv))
    return Packed("token", off, _cast(k, dtype), _cast(v, dtype), None,
                  _cast(dt * A, torch.float32), meta=dict(seed=seed))


def kda_packed(lengths, n_streams, dk, dv, seed, dtype=torch.bfloat16, z_mean=3.0) -> Packed:
    """KDA heads over segments of the given lengths.  Draw order: z, beta, k, v."""
    rng = np.random.default_rng(seed)
    off = offsets_of(lengths)
    n = int(off[-1])
    z = _draw(rng, "normal", (n, n_streams, dk), loc=z_mean)
    beta = _draw(rng, "uniform", (n, n_streams))
    k = _draw(rng, "normal", (n, n_streams, dk), normalize=True)
    v = _draw(rng, "normal", (n, n_streams, dv))
    return Packed("kda", off, _cast(k, dtype), _cast(v, dtype), _cast(beta, torch.float32),
                  _cast(-softplus64(-z), torch.float32), meta=dict(seed=seed, z_mean=z_mean))


def gdn_small() -> Packed:
    """Single gated-delta head, dk=dv=64, fp32, 4 segments x 256 tokens."""
    c = GDN_SMALL
    return gdn_packed([c["seg_len"]] * c["n_seg"], c["n_streams"], c["d"], c["d"],
                      c["seed"], dtype=torch.float32, with_q=True, q_normalize=True)


GDN_SMALL_ORDER = [2, 0, 3, 1]


def decay_heads():
    """8 RetNet heads + 8 GLA heads, dk=dv=128, bf16, 16 segments x 512 tokens.

    Returns (retnet Packed, gla Packed); each is one build call of 8 streams.
    """
    c = DECAY_HEADS
    rng = np.random.default_rng(c["seed"])
    lengths = [c["seg_len"]] * c["n_seg"]
    off = offsets_of(lengths)
    n, d = int(off[-1]), c["d"]
    nr, ng = c["n_retnet"], c["n_gla"]
    z = _draw(rng, "normal", (n, ng, d), loc=3.0)
    k = _draw(rng, "normal", (n, nr + ng, d), normalize=True)
    v = _draw(rng, "normal", (n, nr + ng, d))
    gamma = 1.0 - np.exp2(-5.0 - np.arange(nr, dtype=np.float64))
    retnet = Packed("scalar", off, _cast(k[:, :nr], torch.bfloat16),
                    _cast(v[:, :nr], torch.bfloat16), None,
                    _cast(np.log(gamma), torch.float32),
                    meta=dict(seed=c["seed"], gamma=gamma))
    gla = Packed("diag", off, _cast(k[:, nr:], torch.bfloat16),
                 _cast(v[:, nr:], torch.bfloat16), None,
                 _cast(-softplus64(-z), torch.float32), meta=dict(seed=c["seed"]))
    return retnet, gla


def token_kda_heads():
    """8 Mamba2-style heads (per-token scalar decay) + 8 KDA heads, dk=dv=128,
    bf16, 16 segments x 512 tokens; one build call of 8 streams each."""
    c = TOKEN_KDA_HEADS
    lengths = [c["seg_len"]] * c["n_seg"]
    tok = token_packed(lengths, c["n_token"], c["d"], c["d"], c["seed"])
    kda = kda_packed(lengths, c["n_kda"], c["d"], c["d"], c["seed"] + 1)
    return tok, kda


def gdn_layer(n_seg=None, seg_len=None, n_streams=None, seed=None, seam_w=0) -> Packed:
    """One hybrid-model linear layer: 16 GDN heads, dk=dv=128, bf16, 64 x 1024."""
    c = dict(GDN_LAYER)
    for key, val in (("n_seg", n_seg), ("seg_len", seg_len),
                     ("n_streams", n_streams), ("seed", seed)):
        if val is not None:
            c[key] = val
    return gdn_packed([c["seg_len"]] * c["n_seg"], c["n_streams"], c["d"], c["d"],
                      c["seed"], seam_w=seam_w)


@dataclass
class ReuseBatch:
    """Per-request segment orders and the seam-window tokens of each position."""
    order: torch.Tensor        # int32 [n_req, n_pos] in [0, n_seg)
    q: torch.Tensor            # [n_req, n_pos, w, S, dk] bf16
    k: torch.Tensor            # [n_req, n_pos, w, S, dk] bf16
    v: torch.Tensor            # [n_req, n_pos, w, S, dv] bf16
    beta: Optional[torch.Tensor]        # [n_req, n_pos, w, S] fp32 (delta rules)
    log_alpha: Optional[torch.Tensor]   # [n_req, n_pos, w, S] fp32 (layout by family)
    w: int
    n_seg: int


def reuse_batch(n_req=None, n_pos=None, n_seg=64, w=None, n_streams=None, d=None,
                seed=None, x_mean=-4.0, dtype=torch.bfloat16) -> ReuseBatch:
    """Reuse path: each request composes n_pos cached pairs in a seeded random
    order (independent permutations of 0..n_seg-1, concatenated until n_pos),
    with w fresh seam tokens per position; q ~ N(0,1) not normalised."""
    c = dict(REUSE)
    for key, val in (("n_req", n_req), ("n_pos", n_pos), ("w", w),
                     ("n_streams", n_streams), ("d", d), ("seed", seed)):
        if val is not None:
            c[key] = val
    rng = np.random.default_rng(c["seed"])
    R, P, W, S, D = c["n_req"], c["n_pos"], c["w"], c["n_streams"], c["d"]
    order = np.empty((R, P), dtype=np.int32)
    for r in range(R):
        perms = []
        while sum(len(p) for p in perms) < P:
            perms.append(rng.permutation(n_seg))
        order[r] = np.concatenate(perms)[:P]
    x = _draw(rng, "normal", (R, P, W, S), loc=x_mean)
    beta = _draw(rng, "uniform", (R, P, W, S))
    k = _draw(rng, "normal", (R, P, W, S, D), normalize=True)
    v = _draw(rng, "normal", (R, P, W, S, D))
    q = _draw(rng, "normal", (R, P, W, S, D))
    return ReuseBatch(torch.from_numpy(order), _cast(q, dtype), _cast(k, dtype),
                      _cast(v, dtype), _cast(beta, torch.float32),
                      _cast(-softplus64(x), torch.float32), W, n_seg)


def seam_batch(kind, n_req, n_pos, n_seg, w, n_streams, d, seed, dtype=torch.bfloat16) -> ReuseBatch:
    """Reuse requests for a head family: seeded orders (as reuse_batch) and w
    fresh seam tokens per position.  Gate layouts follow the build inputs:
    gated delta and Mamba2-style one log-decay per token, GLA and KDA one per
    key channel, RetNet one per stream; beta for the delta rules only.  Draw
    order: order, gates, beta, k, v, q."""
    rng = np.random.default_rng(seed)
    R, P, W, S, D = n_req, n_pos, w, n_streams, d
    order = np.empty((R, P), dtype=np.int32)
    for r in range(R):
        perms = []
        while sum(len(x) for x in perms) < P:
            perms.append(rng.permutation(n_seg))
        order[r] = np.concatenate(perms)[:P]
    g = None
    if kind == "gdn":
        g = -softplus64(_draw(rng, "normal", (R, P, W, S), loc=-4.0))
    elif kind == "token":
        A = -(1.0 + 15.0 * _draw(rng, "uniform", (1, S)))
        dt = np.exp(np.log(1e-3) + (np.log(1e-1) - np.log(1e-3)) *
                    _draw(rng, "uniform", (R * P * W, S)))
        g = (dt * A).reshape(R, P, W, S)
    elif kind == "scalar":
        g = np.log(1.0 - np.exp2(-5.0 - np.arange(S, dtype=np.float64) % 8))
    elif kind in ("diag", "kda"):
        g = -softplus64(-_draw(rng, "normal", (R, P, W, S, D), loc=3.0))
    beta = _draw(rng, "uniform", (R, P, W, S)) if kind in ("gdn", "kda") else None
    k = _draw(rng, "normal", (R, P, W, S, D), normalize=True)
    v = _draw(rng, "normal", (R, P, W, S, D))
    q = _draw(rng, "normal", (R, P, W, S, D))
    return ReuseBatch(torch.from_numpy(order), _cast(q, dtype), _cast(k, dtype), _cast(v, dtype),
                      None if beta is None else _cast(beta, torch.float32),
                      None if g is None else _cast(g, torch.float32), W, n_seg)


def slow_reuse():
    """Compose on weighty transitions: x ~ N(-9, 1) (alpha ~ 0.9999), 256-token
    segments, 8 positions, so the T*S term dominates the composed state.

    Returns (Packed build inputs, ReuseBatch)."""
    c = SLOW_REUSE
    pk = gdn_packed([c["seg_len"]] * c["n_seg"], c["n_streams"], c["d"], c["d"],
                    c["seed"], x_mean=-9.0)
    rb = reuse_batch(n_req=c["n_req"], n_pos=c["n_pos"], n_seg=c["n_seg"], w=c["w"],
                     n_streams=c["n_streams"], d=c["d"], seed=c["seed"] + 100,
                     x_mean=-9.0)
    return pk, rb


def cold_long_lengths(total=None, seed=None) -> np.ndarray:
    """Segment lengths for the cold long prompt.

    lognormal with arithmetic mean 1024 and sigma 0.8 (mu = ln 1024 - sigma^2/2),
    L = clip(rint(x), 128, 8192); when fewer than 128 tokens would remain after a
    segment, that segment takes the remainder (so the last may exceed 8192)."""
    c = COLD_LONG
    total = c["total"] if total is None else total
    rng = np.random.default_rng(c["seed"] if seed is None else seed)
    mu = np.log(c["mean_len"]) - 0.5 * c["sigma"] ** 2
    out, rem = [], total
    while rem > 0:
        x = rng.lognormal(mu, c["sigma"])
        L = int(np.clip(np.rint(x), c["lo"], c["hi"]))
        if rem - L < c["lo"]:
            L = rem
        out.append(L)
        rem -= L
    return np.asarray(out, dtype=np.int64)


def cold_long_device(device, n_layers=None, n_heads=None, total=None, seed=None,
                     dtype=torch.bfloat16) -> Packed:
    """Cold long prompt drawn on the device (32 GB of K/V would not fit a host
    upload): a torch.Generator on ``device`` seeded with ``seed``; per layer,
    draw x, beta, k, v in that order (k L2-normalised in fp32, then cast)."""
    c = COLD_LONG
    L_ = c["n_layers"] if n_layers is None else n_layers
    H = c["n_heads"] if n_heads is None else n_heads
    seed = c["seed"] if seed is None else seed
    lengths = cold_long_lengths(total=total, seed=seed)
    off = offsets_of(lengths)
    n, d, S = int(off[-1]), c["d"], L_ * H
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    k = torch.empty((n, S, d), dtype=dtype, device=device)
    v = torch.empty((n, S, d), dtype=dtype, device=device)
    beta = torch.empty((n, S), dtype=torch.float32, device=device)
    g = torch.empty((n, S), dtype=torch.float32, device=device)
    for layer in range(L_):
        sl = slice(layer * H, (layer + 1) * H)
        x = torch.randn((n, H), generator=gen, device=device, dtype=torch.float32) - 4.0
        g[:, sl] = -torch.nn.functional.softplus(x)
        beta[:, sl] = torch.rand((n, H), generator=gen, device=device, dtype=torch.float32)
        kk = torch.randn((n, H, d), generator=gen, device=device, dtype=torch.float32)
        kk = kk / kk.norm(dim=-1, keepdim=True)
        k[:, sl] = kk.to(dtype)
        del kk
        v[:, sl] = torch.randn((n, H, d), generator=gen, device=device,
                               dtype=torch.float32).to(dtype)
    return Packed("gdn", off, k, v, beta, g, meta=dict(seed=seed, lengths=lengths))


def cold_long_order(n_seg, seed=None) -> np.ndarray:
    """The random request order the cold prompt is composed in."""
    rng = np.random.default_rng((COLD_LONG["seed"] if seed is None else seed) + 7)
    return rng.permutation(n_seg).astype(np.int32)


# float64 views for the oracle -------------------------------------------------

def f64(t: Optional[torch.Tensor]) -> Optional[np.ndarray]:
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


def unit_inputs(p: Packed, stream: int, a: int, b: int):
    """float64 copies of stream ``stream``'s tokens [a, b) (a unit's body: the
    caller supplies the range, e.g. from the oracle's body ranges)."""
    a, b = int(a), int(b)
    out = dict(kind=p.kind,
               k=f64(p.k[a:b, stream]), v=f64(p.v[a:b, stream]))
    if p.kind in ("gdn", "kda"):
        out["beta"] = f64(p.beta[a:b, stream])
        out["g"] = f64(p.log_alpha[a:b, stream])
    elif p.kind in ("diag", "token"):
        out["g"] = f64(p.log_alpha[a:b, stream])
    elif p.kind == "scalar":
        out["g"] = np.full(b - a, float(p.log_alpha[stream]), dtype=np.float64)
    return out
