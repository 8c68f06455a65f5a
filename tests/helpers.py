"""Shared test helpers: run the oracle on sampled units and compare with the
device cache.  Imports the oracle (test infrastructure) and the seeded inputs;
never the other way round."""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np
import torch

from linear_attn_state_gb300 import synth
from oracle import linear_state as ls
from oracle import schedule as sch

BUILD_TOL = 2e-3     # relative Frobenius, T_C and S(C|0) from bf16 inputs
COMPOSE_TOL = 1e-4   # relative Frobenius, compose on fp32 caches
SEAM_TOL = 1e-4      # relative Frobenius, seam outputs and state


def body_range(p: synth.Packed, seg: int, seam_w=None):
    """Token range of a unit's body, by the oracle's seam-window rule."""
    w = p.seam_w if seam_w is None else seam_w
    return sch.body_ranges(p.offsets[seg:seg + 2], w)[0]


def oracle_unit(p: synth.Packed, seg: int, stream: int, seam_w=None):
    u = synth.unit_inputs(p, stream, *body_range(p, seg, seam_w))
    # KDA's T has no closed factored form in the oracle: form it explicitly
    return ls.segment_pair(u["kind"], u["k"], u["v"], u.get("beta"), u.get("g"),
                           want_T=(u["kind"] == "kda"))


def _oracle_job(job):
    kind, k, v, beta, g = job
    return ls.segment_pair(kind, k, v, beta, g, want_T=(kind == "kda"))


def oracle_units_parallel(p: synth.Packed, units, seam_w=None):
    """The oracle's pair of each (segment, stream) in ``units``, computed in a
    spawn process pool over the host cores (one BLAS thread each), longest
    units first; returns the results in the order of ``units``."""
    jobs = []
    for seg, s in units:
        u = synth.unit_inputs(p, s, *body_range(p, seg, seam_w))
        jobs.append((u["kind"], u["k"], u["v"], u.get("beta"), u.get("g")))
    order = sorted(range(len(jobs)), key=lambda i: -len(jobs[i][1]))
    n = max(1, min(len(jobs), len(os.sched_getaffinity(0))))
    prev = os.environ.get("OPENBLAS_NUM_THREADS")
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            res = pool.map(_oracle_job, [jobs[i] for i in order], chunksize=1)
    finally:
        if prev is None:
            os.environ.pop("OPENBLAS_NUM_THREADS", None)
        else:
            os.environ["OPENBLAS_NUM_THREADS"] = prev
    out = [None] * len(jobs)
    for i, r in zip(order, res):
        out[i] = r
    return out


def record(kind, **kw):
    """Appends one measured error to the file named by HYPIC_ERR_REPORT (if set)."""
    import json
    import os
    path = os.environ.get("HYPIC_ERR_REPORT")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(kind=kind, **kw)) + "\n")


def unit_errors(p: synth.Packed, cache, seg: int, stream: int, ref=None, seam_w=None):
    """(T error, S error) of one device unit against the oracle."""
    if ref is None:
        ref = oracle_unit(p, seg, stream, seam_w)
    S_dev = cache.S[seg, stream].double().cpu().numpy()
    eS = ls.rel_fro(S_dev, ref["S"])
    if p.kind == "gdn":
        eT = ls.rel_fro_factored(cache.Qhat[seg, stream].double().cpu().numpy(),
                                 int(cache.exp2[seg, stream]), float(cache.log_T[seg, stream]),
                                 ref["Q"], ref["logG"])
    elif p.kind == "kda":
        T_dev = ls.cache_transition(cache.Qhat[seg, stream].double().cpu().numpy(),
                                    int(cache.exp2[seg, stream]), float(cache.log_T[seg, stream]))
        eT = ls.rel_fro(T_dev, ref["T"])
    elif p.kind == "diag":
        lt = cache.log_T[seg, stream].double().cpu().numpy()
        eT = float(np.max(np.abs(np.expm1(lt - np.asarray(ref["logG"])))))
    else:
        lt = float(cache.log_T[seg, stream])
        eT = abs(np.expm1(lt - float(ref["logG"])))
    L = int(p.offsets[seg + 1] - p.offsets[seg])
    record("build", family=p.kind, dtype=str(p.k.dtype), d=p.dk, L=L, eT=eT, eS=eS)
    return eT, eS


def oracle_cache_fp32(p: synth.Packed, streams, device="cuda"):
    """A device cache whose entries for ``streams`` are the oracle's pairs
    rounded to fp32 in the cache layout (other streams: identity pairs).
    Used to feed compose the same fp32 inputs on both sides."""
    from linear_attn_state_gb300.hypic import Cache
    c = Cache.empty(p.kind, p.n_seg, p.n_streams, p.dk, p.dv, device="cpu")
    c.S.zero_()
    c.log_T.zero_()
    if c.Qhat is not None:
        c.Qhat.zero_()
        c.Qhat += torch.eye(p.dk)
        c.exp2.zero_()
    for s in streams:
        for seg in range(p.n_seg):
            ref = oracle_unit(p, seg, s)
            c.S[seg, s] = torch.from_numpy(ref["S"]).float()
            if p.kind in ("gdn", "kda"):
                # gdn: T = e^logG Q; kda: T itself, with log T = 0
                Q, lg = (ref["Q"], float(ref["logG"])) if p.kind == "gdn" else (ref["T"], 0.0)
                m = np.abs(Q).max()
                e = int(np.floor(np.log2(m))) if m > 0 else 0
                c.Qhat[seg, s] = torch.from_numpy(np.ldexp(Q, -e)).float()
                c.exp2[seg, s] = e
                c.log_T[seg, s] = lg
            elif p.kind == "diag":
                c.log_T[seg, s] = torch.from_numpy(np.asarray(ref["logG"])).float()
            else:
                c.log_T[seg, s] = float(ref["logG"])
    for name in ("S", "log_T", "Qhat", "exp2"):
        t = getattr(c, name)
        if t is not None:
            setattr(c, name, t.to(device))
    return c


def cache_pairs_f64(cache, stream):
    """float64 (T, S) pairs of one stream from an fp32 cache (host copy)."""
    pairs = []
    for seg in range(cache.n_seg):
        S = cache.S[seg, stream].double().cpu().numpy()
        if cache.kind in ("gdn", "kda"):
            T = ls.cache_transition(cache.Qhat[seg, stream].double().cpu().numpy(),
                                    int(cache.exp2[seg, stream]),
                                    float(cache.log_T[seg, stream]))
        elif cache.kind == "diag":
            T = np.diag(np.exp(cache.log_T[seg, stream].double().cpu().numpy()))
        else:
            T = np.exp(float(cache.log_T[seg, stream])) * np.eye(cache.dk)
        pairs.append((T, S))
    return pairs


def seam_f64(rb, r, stream):
    """float64 seam inputs of request r, stream s: arrays [P, w, ...] (a
    per-stream gate is repeated over the window's tokens)."""
    f = lambda t: None if t is None else t[r, :, :, stream].double().cpu().numpy()
    P, w = rb.q.shape[1], rb.q.shape[2]
    g = rb.log_alpha
    if g is not None and g.dim() == 1:
        g = np.full((P, w), float(g[stream]))
    else:
        g = f(g)
    return dict(q=f(rb.q), k=f(rb.k), v=f(rb.v), beta=f(rb.beta), g=g)


def to_dev(p: synth.Packed, device="cuda") -> synth.Packed:
    import dataclasses
    mv = lambda t: None if t is None else t.to(device).contiguous()
    return dataclasses.replace(p, k=mv(p.k), v=mv(p.v), beta=mv(p.beta),
                               log_alpha=mv(p.log_alpha), q=mv(p.q))
