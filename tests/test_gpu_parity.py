"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Tolerances (relative Frobenius, max over the units compared): 2e-3 for T_C and
S(C|0) built from bf16 inputs; 1e-4 for compose on fp32 caches and for seam
outputs/states (fp32 state, exact inputs); the LPT order and offsets are
bit-exact.  Compose is fed the oracle's own pairs rounded to the fp32 cache
layout, so no oracle input ever comes from the device.
"""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

from linear_attn_state_gb300 import build as hbuild
from linear_attn_state_gb300 import hypic as H
from linear_attn_state_gb300 import synth
from oracle import linear_state as ls
from oracle import schedule as sch
from tests.helpers import (BUILD_TOL, COMPOSE_TOL, SEAM_TOL, cache_pairs_f64, oracle_cache_fp32,
                           oracle_unit, oracle_units_parallel, seam_f64, to_dev, unit_errors)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    hbuild.build()
    return H.lib()


def run_build(p: synth.Packed, seam_w=None, **kw):
    d = to_dev(p)
    return H.hypic_segment_build(p.kind, p.offsets, d.k, d.v, d.beta, d.log_alpha,
                                 seam_w=p.seam_w if seam_w is None else seam_w,
                                 check_status=True, **kw)


def decay_packed(kind, lengths, n_streams, d, dtype, seed):
    if kind == "token":
        return synth.token_packed(lengths, n_streams, d, d, seed, dtype=dtype)
    if kind == "kda":
        return synth.kda_packed(lengths, n_streams, d, d, seed, dtype=dtype)
    base = synth.gdn_packed(lengths, n_streams, d, d, seed, dtype=dtype)
    n = int(base.offsets[-1])
    rng = np.random.default_rng(seed + 1)
    if kind == "scalar":
        la = torch.from_numpy(np.log(1 - 2.0 ** (-5 - np.arange(n_streams) % 8))).float()
    elif kind == "diag":
        z = rng.normal(3.0, 1.0, (n, n_streams, d))
        la = torch.from_numpy(-np.logaddexp(0.0, -z)).float()
    else:
        la = None
    return dataclasses.replace(base, kind=kind, beta=None, log_alpha=la)


RAGGED = [0, 1, 63, 64, 65, 130]


@pytest.mark.parametrize("kind", ["gdn", "scalar", "diag", "none", "token", "kda"])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("d", [64, 128])
def test_small_ragged_segments(kind, dtype, d):
    """Segments of 0, 1, 63, 64, 65, 130 tokens (empty, single token, chunk
    edges, ragged tails) on 2 streams, packed varlen."""
    seed = 7 + d + (dtype == torch.float32)
    if kind == "gdn":
        p = synth.gdn_packed(RAGGED, 2, d, d, seed, dtype=dtype)
    else:
        p = decay_packed(kind, RAGGED, 2, d, dtype, seed)
    cache = run_build(p)
    tol = BUILD_TOL if dtype == torch.bfloat16 else 1e-4
    for seg in range(p.n_seg):
        for s in range(2):
            eT, eS = unit_errors(p, cache, seg, s)
            assert eT <= tol and eS <= tol, (seg, s, eT, eS)
    if kind in ("gdn", "kda"):
        # the empty segment holds the identity pair
        assert torch.equal(cache.Qhat[0, 0].cpu(), torch.eye(d))
        assert int(cache.exp2[0, 0]) == 0 and float(cache.log_T[0, 0]) == 0.0
        assert float(cache.S[0, 0].abs().max()) == 0.0


@pytest.mark.parametrize("kind,d", [("gdn", 64), ("gdn", 128), ("kda", 128)])
def test_seam_window_skipped_in_build(kind, d):
    """A seam window of 8 tokens: the 5- and 8-token segments leave empty bodies
    (identity pairs), the others build from their ninth token on."""
    make = synth.gdn_packed if kind == "gdn" else synth.kda_packed
    p = make([5, 8, 40, 100], 3, d, d, 31)
    cache = run_build(p, seam_w=8)
    for seg in range(4):
        for s in range(3):
            eT, eS = unit_errors(p, cache, seg, s, seam_w=8)
            assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, eT, eS)
    for seg in (0, 1):
        assert torch.equal(cache.Qhat[seg, 0].cpu(), torch.eye(d))
        assert int(cache.exp2[seg, 0]) == 0 and float(cache.log_T[seg, 0]) == 0.0
        assert float(cache.S[seg, 0].abs().max()) == 0.0


def test_gdn_small_workload():
    """Single GDN head, dk=dv=64, fp32: build 4 x 256 and compose [2,0,3,1]."""
    p = synth.gdn_small()
    cache = run_build(p)
    refs = [oracle_unit(p, seg, 0) for seg in range(4)]
    for seg in range(4):
        eT, eS = unit_errors(p, cache, seg, 0, ref=refs[seg])
        assert eT <= BUILD_TOL and eS <= BUILD_TOL
    order = torch.tensor([synth.GDN_SMALL_ORDER], dtype=torch.int32, device="cuda")
    # end to end: device build + device compose vs oracle build + oracle compose
    state, _ = H.hypic_compose(cache, order, check_status=True)
    pairs = [(np.exp(r["logG"]) * r["Q"], r["S"]) for r in refs]
    S_ref = ls.compose(pairs, synth.GDN_SMALL_ORDER)
    assert ls.rel_fro(state[0, 0].double().cpu().numpy(), S_ref) <= BUILD_TOL
    # compose alone on identical fp32 caches
    oc = oracle_cache_fp32(p, [0])
    state2, _ = H.hypic_compose(oc, order, check_status=True)
    S2 = ls.compose(cache_pairs_f64(oc, 0), synth.GDN_SMALL_ORDER)
    assert ls.rel_fro(state2[0, 0].double().cpu().numpy(), S2) <= COMPOSE_TOL


def test_decay_heads_workload():
    """8 RetNet + 8 GLA heads, 16 x 512, bf16: every unit against the oracle,
    the RetNet closed form, and the naive-add error on the slowest head."""
    retnet, gla = synth.decay_heads()
    for p in (retnet, gla):
        cache = run_build(p)
        for seg in range(p.n_seg):
            for s in range(p.n_streams):
                eT, eS = unit_errors(p, cache, seg, s)
                assert eT <= BUILD_TOL and eS <= BUILD_TOL, (p.kind, seg, s, eT, eS)
        if p.kind == "scalar":
            gamma = p.meta["gamma"]
            lt = cache.log_T.double().cpu().numpy()
            assert np.allclose(lt, 512 * np.log(gamma)[None, :], rtol=1e-6, atol=0)
            # naive add vs compose for two consecutive segments on head 7
            order = torch.tensor([[0, 1]], dtype=torch.int32, device="cuda")
            true, _ = H.hypic_compose(cache, order, check_status=True)
            S1 = cache.S[0, 7].double()
            naive = (S1 + cache.S[1, 7].double()).cpu().numpy()
            err = np.linalg.norm(naive - true[0, 7].double().cpu().numpy()) / float(S1.norm())
            closed = 1 - gamma[7] ** 512
            assert abs(err - closed) <= 1e-3 * closed
            assert err >= 0.05


@pytest.mark.parametrize("n_streams", [8, 6])
def test_token_decay_tensor_core_and_fallback(n_streams):
    """Mamba2-style per-token decay, dk=dv=128, bf16: 8 streams take the
    tensor-core build (gate boxes of 4 streams), 6 streams the recurrence;
    ragged and multi-chunk segments, every unit against the oracle."""
    p = synth.token_packed(RAGGED + [512, 777], n_streams, 128, 128, seed=400 + n_streams)
    cache = run_build(p)
    for seg in range(p.n_seg):
        for s in range(n_streams):
            eT, eS = unit_errors(p, cache, seg, s)
            assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, eT, eS)
    assert float(cache.log_T[0].abs().max()) == 0.0 and float(cache.S[0].abs().max()) == 0.0


def test_token_kda_heads_workload():
    """8 Mamba2-style + 8 KDA heads, 16 x 512, bf16: every Mamba2-style unit
    and one KDA unit of every segment against the oracle; the KDA build is
    deterministic."""
    tok, kda = synth.token_kda_heads()
    cache = run_build(tok)
    for seg in range(tok.n_seg):
        for s in range(tok.n_streams):
            eT, eS = unit_errors(tok, cache, seg, s)
            assert eT <= BUILD_TOL and eS <= BUILD_TOL, ("token", seg, s, eT, eS)
    cache = run_build(kda)
    # one KDA unit of every segment (streams cycling), through the process pool
    units = [(seg, seg % kda.n_streams) for seg in range(kda.n_seg)] + [(15, 7), (6, 3)]
    for (seg, s), ref in zip(units, oracle_units_parallel(kda, units)):
        eT, eS = unit_errors(kda, cache, seg, s, ref=ref)
        assert eT <= BUILD_TOL and eS <= BUILD_TOL, ("kda", seg, s, eT, eS)
    again = run_build(kda)
    assert torch.equal(cache.S, again.S) and torch.equal(cache.Qhat, again.Qhat)


def assert_every_log_T(cache, offsets, log_alpha):
    """Every unit of a gated-delta cache: log T is the sum of the log-decays
    over the unit's body (T = Gamma 2^e Qhat, Gamma the product of the alphas),
    so a unit built over the wrong token range or stream shows.  float64 prefix
    sums of the same fp32 draws on one side; on the other fp32 sums of 64-token
    chunks carried in float64 (at most 129 chunks of |g| < 1 here)."""
    g = log_alpha.to(cache.log_T.device).double()
    off = torch.as_tensor(np.asarray(offsets.cpu() if torch.is_tensor(offsets) else offsets),
                          dtype=torch.int64).to(g.device)
    cs = torch.cat([torch.zeros_like(g[:1]), torch.cumsum(g, dim=0)])
    want = cs[off[1:]] - cs[off[:-1]]
    err = (cache.log_T.double() - want).abs() - 1e-5 * want.abs()
    assert float(err.max()) <= 2e-3, float(err.max())


def test_gdn_layer_sampled_units_and_determinism():
    """16 GDN heads, dk=dv=128, bf16, 64 x 1024: 32 units vs the oracle (the
    first and last of both corners and seeded draws covering every stream), and
    two runs are bitwise equal."""
    p = synth.gdn_layer()
    cache = run_build(p)
    rng = np.random.default_rng(0)
    units = [(0, 0), (63, 15), (31, 7), (0, 15), (63, 0)]
    units += [(int(rng.integers(64)), s % 16) for s in range(27)]
    refs = oracle_units_parallel(p, units)
    for (seg, s), ref in zip(units, refs):
        eT, eS = unit_errors(p, cache, seg, s, ref=ref)
        assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, eT, eS)
    assert_every_log_T(cache, p.offsets, p.log_alpha)
    again = run_build(p)
    assert torch.equal(cache.S, again.S) and torch.equal(cache.Qhat, again.Qhat)
    assert torch.equal(cache.exp2, again.exp2) and torch.equal(cache.log_T, again.log_T)


def test_reuse_path_sampled_requests():
    """32 requests x 128 positions x 16 streams, w=8 seam tokens per position,
    on the layer's cache: one stream's cache built by the oracle (fp32), the
    device composes every request; every third request vs the oracle."""
    p = synth.gdn_layer()
    rb = synth.reuse_batch()
    s_star = 5
    oc = oracle_cache_fp32(p, [s_star])
    dev = lambda t: t.cuda().contiguous()
    seam = (dev(rb.q), dev(rb.k), dev(rb.v), dev(rb.beta), dev(rb.log_alpha))
    state, o = H.hypic_compose(oc, dev(rb.order), seam=seam, check_status=True)
    pairs = cache_pairs_f64(oc, s_star)
    for r in range(0, 32, 3):
        order = rb.order[r].tolist()
        S_ref, o_ref = ls.compose_with_seam(pairs, order, seam_f64(rb, r, s_star))
        assert ls.rel_fro(state[r, s_star].double().cpu().numpy(), S_ref) <= COMPOSE_TOL, r
        assert ls.rel_fro(o[r, :, :, s_star].double().cpu().numpy(), o_ref) <= SEAM_TOL, r


def test_slow_decay_compose_weighty_transitions():
    """alpha ~ 0.9999, 256-token segments: T S dominates the composed state, so
    compose precision is visible (naive addition is far off)."""
    p, rb = synth.slow_reuse()
    s_star = 3
    oc = oracle_cache_fp32(p, [s_star])
    dev = lambda t: t.cuda().contiguous()
    seam = (dev(rb.q), dev(rb.k), dev(rb.v), dev(rb.beta), dev(rb.log_alpha))
    state, o = H.hypic_compose(oc, dev(rb.order), seam=seam, check_status=True)
    pairs = cache_pairs_f64(oc, s_star)
    for r in range(rb.order.shape[0]):
        order = rb.order[r].tolist()
        S_ref, o_ref = ls.compose_with_seam(pairs, order, seam_f64(rb, r, s_star))
        assert ls.rel_fro(state[r, s_star].double().cpu().numpy(), S_ref) <= COMPOSE_TOL
        assert ls.rel_fro(o[r, :, :, s_star].double().cpu().numpy(), o_ref) <= SEAM_TOL
        assert ls.rel_fro(ls.naive_add(pairs, order), ls.compose(pairs, order)) > 1e-2
    # and the device build of these slow-decay segments
    cache = run_build(p)
    for seg in (0, 7):
        eT, eS = unit_errors(p, cache, seg, s_star)
        assert eT <= BUILD_TOL and eS <= BUILD_TOL


def test_seam_advance_standalone():
    rng = np.random.default_rng(3)
    R, S, D, w = 3, 4, 128, 8
    rb = synth.reuse_batch(n_req=R, n_pos=1, n_seg=1, w=w, n_streams=S, d=D, seed=77)
    state0 = torch.from_numpy(rng.standard_normal((R, S, D, D))).float()
    state = state0.cuda()
    dev = lambda t: t.cuda().contiguous()
    o = H.hypic_seam_advance(state, dev(rb.q), dev(rb.k), dev(rb.v), dev(rb.beta),
                             dev(rb.log_alpha), check_status=True)
    for r in range(R):
        for s in range(S):
            sm = seam_f64(rb, r, s)
            S_ref, o_ref = ls.seam_advance(state0[r, s].double().numpy(), sm["q"][0], sm["k"][0],
                                           sm["v"][0], sm["beta"][0], sm["g"][0])
            assert ls.rel_fro(state[r, s].double().cpu().numpy(), S_ref) <= SEAM_TOL
            assert ls.rel_fro(o[r, 0, :, s].double().cpu().numpy(), o_ref) <= SEAM_TOL


def test_compose_state_in_and_decay_kinds():
    """Compose from a given state, for every transition family, on identical
    fp32 caches (oracle-built)."""
    rng = np.random.default_rng(5)
    for kind in ("gdn", "scalar", "diag", "none", "token", "kda"):
        if kind == "gdn":
            p = synth.gdn_packed([30, 50, 20], 2, 64, 64, 41)
        else:
            p = decay_packed(kind, [30, 50, 20], 2, 64, torch.bfloat16, 41)
        oc = oracle_cache_fp32(p, [0, 1])
        order = torch.tensor([[2, 0, 1, 1], [1, 2, 2, 0]], dtype=torch.int32, device="cuda")
        s_in = torch.from_numpy(rng.standard_normal((2, 2, 64, 64))).float().cuda()
        out, _ = H.hypic_compose(oc, order, state_in=s_in, check_status=True)
        for r in range(2):
            for s in range(2):
                ref = ls.compose(cache_pairs_f64(oc, s), order[r].tolist(),
                                 state_in=s_in[r, s].double().cpu().numpy())
                assert ls.rel_fro(out[r, s].double().cpu().numpy(), ref) <= COMPOSE_TOL, kind


def test_device_detected_errors():
    p = synth.gdn_packed([10, 20], 1, 64, 64, 3)
    d = to_dev(p)
    cache = H.hypic_segment_build("gdn", p.offsets, d.k, d.v, d.beta, d.log_alpha)
    order = torch.tensor([[0, 2]], dtype=torch.int32, device="cuda")
    ws = H.workspace(4096)
    H.hypic_compose(cache, order, ws=ws)
    assert H.hypic_read_device_status(ws) == 4  # HYPIC_ERR_INDEX
    H.hypic_compose(cache, order[:, :1], ws=ws)
    assert H.hypic_read_device_status(ws) == 0
    # a device offsets copy that disagrees with the validated host copy
    bad = torch.tensor([0, 25, 10], dtype=torch.int64, device="cuda")
    ws2 = H.workspace(1 << 16)
    H.hypic_segment_build("gdn", p.offsets, d.k, d.v, d.beta, d.log_alpha, ws=ws2, d_offsets=bad)
    assert H.hypic_read_device_status(ws2) == 3  # HYPIC_ERR_OFFSETS


def test_empty_calls():
    p = synth.gdn_packed([], 2, 64, 64, 1)
    d = to_dev(p)
    cache = H.hypic_segment_build("gdn", p.offsets, d.k, d.v, d.beta, d.log_alpha,
                                  check_status=True)
    assert cache.S.numel() == 0
    c2 = run_build(synth.gdn_packed([4], 1, 64, 64, 2))
    out, _ = H.hypic_compose(c2, torch.zeros((0, 3), dtype=torch.int32, device="cuda"))
    assert out.shape[0] == 0


# The build's work list in its workspace: 16-byte items after the 256-byte
# header, in the order the persistent kernel takes them.
WORK_ITEM = np.dtype([("tok_start", "<i8"), ("len", "<i4"), ("unit", "<i4")])


def device_work_list(ws, n_items):
    raw = ws[256:256 + 16 * n_items].cpu().numpy()
    return raw.view(WORK_ITEM)


def assert_work_list_is_lpt(ws, offsets, seam_w, n_streams, order=None):
    """The device work list equals, item by item, the oracle's LPT order with
    each item's body range (bit-exact)."""
    if order is None:
        order, _ = sch.lpt_schedule(list(offsets), seam_w, n_streams, 1)
    body = sch.body_ranges(list(offsets), seam_w)
    got = device_work_list(ws, len(order))
    want_unit = np.asarray(order, dtype=np.int64)
    seg = want_unit // n_streams
    want_start = np.asarray([body[i][0] for i in seg], dtype=np.int64)
    want_len = np.asarray([body[i][1] - body[i][0] for i in seg], dtype=np.int64)
    assert np.array_equal(got["unit"].astype(np.int64), want_unit)
    assert np.array_equal(got["tok_start"], want_start)
    assert np.array_equal(got["len"].astype(np.int64), want_len)


def device_gdn_inputs(n_tok, n_streams, seed):
    """Seeded device draws in the gated-delta layout (for checks that do not
    compare values with the oracle)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    k = torch.nn.functional.normalize(torch.randn(n_tok, n_streams, 128, device="cuda",
                                                  generator=g), dim=-1).to(torch.bfloat16)
    v = torch.randn(n_tok, n_streams, 128, device="cuda", generator=g).to(torch.bfloat16)
    beta = torch.rand(n_tok, n_streams, device="cuda", generator=g)
    la = -torch.nn.functional.softplus(torch.randn(n_tok, n_streams, device="cuda",
                                                   generator=g) - 4.0)
    return k, v, beta, la.contiguous()


@pytest.mark.parametrize("seam_w", [0, 8])
def test_device_work_list_is_the_lpt_schedule(seam_w, golden_dir):
    """The LPT work list the build ranks on the device (the cold prompt's 134
    lognormal segments x 3 streams with and without a seam window, and the four
    hand-worked golden cases) equals the oracle's order and body ranges bit for
    bit; for the golden cases also the order worked out by hand."""
    import json
    import os
    lengths = synth.cold_long_lengths()
    off = np.asarray(sch.offsets_from_lengths(lengths), dtype=np.int64)
    k, v, beta, la = device_gdn_inputs(int(off[-1]), 3, 77)
    ws = H.workspace(1 << 20)
    H.hypic_segment_build("gdn", off, k, v, beta, la, seam_w=seam_w, ws=ws, check_status=True)
    assert_work_list_is_lpt(ws, off, seam_w, 3)
    with open(os.path.join(golden_dir, "lpt_hand_example.json")) as f:
        gold = json.load(f)
    cases = [gold] + [gold[k] for k in ("second_case", "third_case", "fourth_case")]
    for c in cases:
        off = np.asarray(sch.offsets_from_lengths(c["lengths"]), dtype=np.int64)
        S = int(c["n_streams"])
        k, v, beta, la = device_gdn_inputs(int(off[-1]), S, 78)
        H.hypic_segment_build("gdn", off, k, v, beta, la, seam_w=int(c["seam_w"]), ws=ws,
                              check_status=True)
        assert_work_list_is_lpt(ws, off, int(c["seam_w"]), S)
        assert_work_list_is_lpt(ws, off, int(c["seam_w"]), S, order=c["order"])


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_index_order_builds_the_same_cache(kind):
    """With the segment-index order the device work list is the units in index
    order (same body ranges), and the cached pairs are bitwise those of the LPT
    build: the order only changes which CTA takes which unit when."""
    lengths = synth.cold_long_lengths()[:40]
    off = np.asarray(sch.offsets_from_lengths(lengths), dtype=np.int64)
    S = 3
    k, v, beta, la = device_gdn_inputs(int(off[-1]), S, 91)
    if kind == "kda":
        la = -0.1 * torch.rand(la.shape[0], S, k.shape[-1], device="cuda",
                               generator=torch.Generator(device="cuda").manual_seed(92))
    ws = H.workspace(1 << 20)
    lpt = H.hypic_segment_build(kind, off, k, v, beta, la, seam_w=8, ws=ws, check_status=True)
    assert H.hypic_set_build_order(H.ORDER_INDEX) == H.ORDER_LPT
    try:
        idx = H.hypic_segment_build(kind, off, k, v, beta, la, seam_w=8, ws=ws,
                                    check_status=True)
        assert_work_list_is_lpt(ws, off, 8, S, order=list(range(len(lengths) * S)))
    finally:
        assert H.hypic_set_build_order(H.ORDER_LPT) == H.ORDER_INDEX
    torch.cuda.synchronize()
    assert torch.equal(idx.S, lpt.S)
    assert torch.equal(idx.Qhat, lpt.Qhat)
    assert torch.equal(idx.log_T, lpt.log_T)
    assert torch.equal(idx.exp2, lpt.exp2)


def test_cold_long_prompt_sampled_units():
    """131,072 tokens, lognormal segments, 30 layers x 16 GDN heads (480
    streams), drawn on the device; LPT build (its work list checked bit for bit
    against the oracle's schedule); one unit of every segment plus the longest
    segment's outer streams, the shortest segment and seeded draws vs the
    oracle."""
    p = synth.cold_long_device("cuda")
    d_off = torch.from_numpy(p.offsets).cuda()
    ws = H.workspace(256 + 16 * p.n_seg * p.n_streams)
    cache = H.hypic_segment_build("gdn", p.offsets, p.k, p.v, p.beta, p.log_alpha,
                                  d_offsets=d_off, ws=ws, check_status=True)
    assert_work_list_is_lpt(ws, p.offsets, 0, p.n_streams)
    lengths = np.diff(p.offsets)
    rng = np.random.default_rng(11)
    # one unit of every segment (stream seg mod 480), the longest segment's
    # first and last stream, and seeded draws
    units = [(seg, seg % p.n_streams) for seg in range(p.n_seg)]
    units += [(int(np.argmax(lengths)), 0), (int(np.argmax(lengths)), 479),
              (int(np.argmin(lengths)), 17)]
    units += [(int(rng.integers(p.n_seg)), int(rng.integers(480))) for _ in range(3)]
    refs = oracle_units_parallel(p, units)
    for (seg, s), ref in zip(units, refs):
        eT, eS = unit_errors(p, cache, seg, s, ref=ref)
        assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, int(lengths[seg]), eT, eS)
    assert_every_log_T(cache, d_off, p.log_alpha)
    del cache, p
    torch.cuda.empty_cache()


def test_compose_at_cold_long_shape():
    """Compose of a seeded random order over 128+ cached pairs x 480 streams on
    a synthetic fp32 cache (random Qhat, exp2, log_T, S drawn on the device);
    every 32nd stream (and two more) vs the oracle on the same fp32 values."""
    from linear_attn_state_gb300.hypic import Cache
    n_seg = len(synth.cold_long_lengths())
    S, D = 480, 128
    g = torch.Generator(device="cuda")
    g.manual_seed(2024)
    c = Cache.empty("gdn", n_seg, S, D, D)
    c.Qhat.copy_(torch.rand(c.Qhat.shape, generator=g, device="cuda") * 2 - 1)
    c.Qhat.mul_(1.0 / 16)
    c.exp2.copy_(torch.randint(-3, 2, c.exp2.shape, generator=g, device="cuda", dtype=torch.int32))
    c.log_T.copy_(-torch.rand(c.log_T.shape, generator=g, device="cuda") * 2)
    c.S.copy_(torch.randn(c.S.shape, generator=g, device="cuda"))
    order = torch.from_numpy(synth.cold_long_order(n_seg)).view(1, -1).cuda()
    out, _ = H.hypic_compose(c, order, check_status=True)
    for s in list(range(0, S, 32)) + [123, 479]:
        ref = ls.compose(cache_pairs_f64(c, s), order[0].tolist())
        assert ls.rel_fro(out[0, s].double().cpu().numpy(), ref) <= COMPOSE_TOL, s


@pytest.mark.parametrize("kind", ["gdn", "kda"])
def test_bounded_wait_reports_timeout_and_recovers(kind):
    """Every bounded device wait set to give up without polling
    (HYPIC_SPIN_EXPIRE_NOW): the build kernel's first wait runs out, the kernel
    records HYPIC_ERR_DEVICE_TIMEOUT, drains its own copies and MMAs in flight,
    frees its tensor memory and returns (for KDA the rebuild launch that follows
    sees the status and returns too); the context stays usable and a normal
    build then succeeds.  The same for a limit of one poll, where a wait may also
    be satisfied on its first poll."""
    make = synth.gdn_packed if kind == "gdn" else synth.kda_packed
    p = make([300, 200, 100], 4, 128, 128, 5)
    d = to_dev(p)
    ws = H.workspace(1 << 16)
    for limit, allowed in ((H.SPIN_EXPIRE_NOW, (9,)), (1, (0, 9))):
        prev = H.hypic_set_spin_limit(limit)
        try:
            H.hypic_segment_build(kind, p.offsets, d.k, d.v, d.beta, d.log_alpha, ws=ws)
            st = H.hypic_read_device_status(ws)
        finally:
            H.hypic_set_spin_limit(0)
        assert st in allowed, (limit, st)
        cache = H.hypic_segment_build(kind, p.offsets, d.k, d.v, d.beta, d.log_alpha, ws=ws)
        assert H.hypic_read_device_status(ws) == 0
        for seg in range(3):
            eT, eS = unit_errors(p, cache, seg, 1)
            assert eT <= BUILD_TOL and eS <= BUILD_TOL


def test_longest_segments():
    """Bodies at the cold prompt's clip maximum (8192) and just above it (8319,
    a last segment that absorbed a short remainder): the error of T grows with
    the number of chunks, so these are the hardest units for the tolerance."""
    p = synth.gdn_packed([8192, 8319], 2, 128, 128, seed=8192)
    cache = run_build(p)
    for seg in range(2):
        for s in range(2):
            eT, eS = unit_errors(p, cache, seg, s)
            assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, eT, eS)


@pytest.mark.parametrize("rows", [[[2, 7, 0, 1], [1, 0, -1, 2]], [[2, 7, 0, 1]]])
def test_compose_skips_out_of_range_positions(rows):
    """An order index outside [0, n_seg) is reported (HYPIC_ERR_INDEX) and that
    position is skipped; the other positions compose as usual (dk = dv = 128),
    with operand copies (2 x 4 positions of 3 pairs) and with the in-kernel
    conversion shared by the state warps (1 x 4)."""
    p = synth.gdn_packed([70, 40, 90], 2, 128, 128, 61)
    oc = oracle_cache_fp32(p, [0, 1])
    order = torch.tensor(rows, dtype=torch.int32, device="cuda")
    ws = H.compose_workspace(oc, *order.shape)
    out, _ = H.hypic_compose(oc, order, ws=ws)
    assert H.hypic_read_device_status(ws) == 4
    for r, row in enumerate(rows):
        kept = [x for x in row if 0 <= x < 3]
        for s in range(2):
            ref = ls.compose(cache_pairs_f64(oc, s), kept)
            assert ls.rel_fro(out[r, s].double().cpu().numpy(), ref) <= COMPOSE_TOL


@pytest.mark.gpu
@pytest.mark.parametrize("max_group_tokens", [5000, 700, 1 << 30])
def test_host_input_build_matches_device_build(max_group_tokens):
    """Build from page-locked host inputs (segment groups copied on a second
    stream while the previous group builds) writes exactly the cache the
    device-input build writes (groups of 4 segments, single segments longer
    than the group size, and one group)."""
    cases = [("gdn", synth.gdn_layer())]
    ret, gla = synth.decay_heads()
    tok, kda = synth.token_kda_heads()
    cases += [("scalar", ret), ("diag", gla), ("token", tok), ("kda", kda)]
    copy_stream = torch.cuda.Stream()
    for kind, p in cases:
        dev = lambda t: None if t is None else t.cuda().contiguous()
        pin = lambda t: None if t is None else t.contiguous().pin_memory()
        ref = H.hypic_segment_build(kind, p.offsets, dev(p.k), dev(p.v), dev(p.beta),
                                    dev(p.log_alpha), check_status=True)
        d_off = torch.from_numpy(np.asarray(p.offsets, dtype=np.int64)).cuda()
        cache = H.Cache.empty(kind, p.n_seg, p.n_streams, 128, 128, device="cuda")
        H.hypic_segment_build_host(kind, p.offsets, pin(p.k), pin(p.v), pin(p.beta),
                                   pin(p.log_alpha), d_off, cache, max_group_tokens,
                                   copy_stream=copy_stream, check_status=True)
        torch.cuda.synchronize()
        assert torch.equal(cache.S, ref.S), kind
        assert torch.equal(cache.log_T, ref.log_T), kind
        if kind in ("gdn", "kda"):
            assert torch.equal(cache.Qhat, ref.Qhat) and torch.equal(cache.exp2, ref.exp2)


@pytest.mark.gpu
def test_split_build_long_segments():
    """Split build: bodies cut into pieces (1000 tokens: ragged pieces, not chunk
    multiples), built as pairs and composed, against the oracle on the hardest
    units (8192 and 8319 tokens), with a seam window of 8 and a segment whose
    body is a single short piece."""
    p = synth.gdn_packed([8200, 100, 8327], 2, 128, 128, seed=8193, seam_w=8)
    dev = lambda t: t.cuda().contiguous()
    cache = H.hypic_segment_build_split("gdn", p.offsets, dev(p.k), dev(p.v), dev(p.beta),
                                        dev(p.log_alpha), piece_tokens=1000, seam_w=8,
                                        check_status=True)
    for seg in range(3):
        for s in range(2):
            eT, eS = unit_errors(p, cache, seg, s, seam_w=8)
            assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, eT, eS)


@pytest.mark.gpu
@pytest.mark.parametrize("lengths,S,w,P", [([8200, 100, 8327], 2, 8, 1000),
                                           ([0, 1, 9, 64, 1000, 2047, 300], 3, 8, 300)])
def test_split_build_work_list_is_the_lpt_of_its_pieces(lengths, S, w, P):
    """The split build cuts the bodies into pieces (the oracle's split rule:
    seam windows as pieces of their own, bodies in pieces of at most P tokens)
    and builds them under the LPT order; its work list, read back from the
    scratch's build workspace, equals the oracle's LPT order of the pieces and
    their token ranges bit for bit, and the values match the oracle."""
    off = np.asarray(sch.offsets_from_lengths(lengths), dtype=np.int64)
    poff, body = sch.split_pieces(list(off), w, P)
    p = synth.gdn_packed(lengths, S, 128, 128, seed=7000 + P, seam_w=w)
    d = to_dev(p)
    a, keep = H.build_args("gdn", p.offsets, d.k, d.v, d.beta, d.log_alpha, seam_w=w)
    scratch = H.workspace(H.lib().hypic_build_split_scratch_bytes(ctypes.byref(a), P))
    del keep
    cache = H.hypic_segment_build_split("gdn", p.offsets, d.k, d.v, d.beta, d.log_alpha,
                                        piece_tokens=P, seam_w=w, scratch=scratch,
                                        check_status=True)
    assert_work_list_is_lpt(scratch, poff, 0, S)
    for seg in range(len(lengths)):
        eT, eS = unit_errors(p, cache, seg, S - 1, seam_w=w)
        assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, eT, eS)


@pytest.mark.gpu
def test_split_build_decay_families():
    """Split build of the RetNet and GLA heads (512-token segments in 3 pieces)
    equals the oracle like the unsplit build."""
    retnet, gla = synth.decay_heads()
    tok, kda = synth.token_kda_heads()
    dev = lambda t: None if t is None else t.cuda().contiguous()
    for p in (retnet, gla, tok, kda):
        cache = H.hypic_segment_build_split(p.kind, p.offsets, dev(p.k), dev(p.v), dev(p.beta),
                                            dev(p.log_alpha), piece_tokens=200, check_status=True)
        for seg in (0, 7, 15):
            for s in (0, 7):
                eT, eS = unit_errors(p, cache, seg, s)
                assert eT <= BUILD_TOL and eS <= BUILD_TOL, (p.kind, seg, s, eT, eS)


@pytest.mark.gpu
def test_kda_long_segments_unsplit_and_split():
    """KDA bodies of 3000 tokens (47 chunks of the factored T) built whole and
    split into 700-token pieces, with a seam window of 8, against the oracle."""
    p = synth.kda_packed([3008, 100, 2999], 2, 128, 128, seed=3000)
    p = dataclasses.replace(p, seam_w=8)
    dev = lambda t: t.cuda().contiguous()
    whole = run_build(p)
    split = H.hypic_segment_build_split("kda", p.offsets, dev(p.k), dev(p.v), dev(p.beta),
                                        dev(p.log_alpha), piece_tokens=700, seam_w=8,
                                        check_status=True)
    for seg, s in ((0, 0), (1, 1), (2, 1)):
        ref = oracle_unit(p, seg, s)
        for cache in (whole, split):
            eT, eS = unit_errors(p, cache, seg, s, ref=ref)
            assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, eT, eS)


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["gdn", "scalar", "diag", "none", "token", "kda"])
@pytest.mark.parametrize("d", [64, 128])
def test_compose_with_seam_every_family(kind, d):
    """Compose with the seam window of every position, for each head family: the
    seam tokens advance the state with the family's own transitions, then the
    cached pair is composed (oracle-built fp32 cache; 3 requests x 5 positions,
    w = 8)."""
    if kind == "gdn":
        p = synth.gdn_packed([40, 70, 25], 2, d, d, 71)
    else:
        p = decay_packed(kind, [40, 70, 25], 2, d, torch.bfloat16, 71)
    oc = oracle_cache_fp32(p, [0, 1])
    rb = synth.seam_batch(kind, 3, 5, 3, 8, 2, d, seed=72)
    dev = lambda t: None if t is None else t.cuda().contiguous()
    seam = (dev(rb.q), dev(rb.k), dev(rb.v), dev(rb.beta), dev(rb.log_alpha))
    state, o = H.hypic_compose(oc, dev(rb.order), seam=seam, check_status=True)
    for s in range(2):
        pairs = cache_pairs_f64(oc, s)
        for r in range(3):
            S_ref, o_ref = ls.compose_with_seam(pairs, rb.order[r].tolist(), seam_f64(rb, r, s),
                                                kind=kind)
            assert ls.rel_fro(state[r, s].double().cpu().numpy(), S_ref) <= COMPOSE_TOL, (kind, r, s)
            assert ls.rel_fro(o[r, :, :, s].double().cpu().numpy(), o_ref) <= SEAM_TOL, (kind, r, s)


@pytest.mark.gpu
@pytest.mark.parametrize("kind", ["scalar", "diag", "none", "token", "kda"])
def test_seam_advance_standalone_families(kind):
    rng = np.random.default_rng(9)
    R, S, D, w = 2, 4, 128, 8
    rb = synth.seam_batch(kind, R, 1, 1, w, S, D, seed=90)
    state0 = torch.from_numpy(rng.standard_normal((R, S, D, D))).float()
    state = state0.cuda()
    dev = lambda t: None if t is None else t.cuda().contiguous()
    o = H.hypic_seam_advance(state, dev(rb.q), dev(rb.k), dev(rb.v), dev(rb.beta),
                             dev(rb.log_alpha), check_status=True, kind=kind)
    for r in range(R):
        for s in range(S):
            sm = seam_f64(rb, r, s)
            S_ref, o_ref = ls.seam_advance(state0[r, s].double().numpy(), sm["q"][0], sm["k"][0],
                                           sm["v"][0], None if sm["beta"] is None else sm["beta"][0],
                                           None if sm["g"] is None else sm["g"][0], kind=kind)
            assert ls.rel_fro(state[r, s].double().cpu().numpy(), S_ref) <= SEAM_TOL
            assert ls.rel_fro(o[r, 0, :, s].double().cpu().numpy(), o_ref) <= SEAM_TOL


@pytest.mark.gpu
def test_seam_outputs_in_bf16():
    """o_t written as bf16 (round to nearest even) equals the fp32 outputs
    rounded by torch, bit for bit, on the tensor-core compose (gated delta,
    dk = 128) and on the CUDA-core path (KDA); the states are unchanged."""
    dev = lambda t: None if t is None else t.cuda().contiguous()
    for kind, d in (("gdn", 128), ("kda", 128), ("scalar", 64)):
        if kind == "gdn":
            p = synth.gdn_packed([40, 70, 25], 2, d, d, 81)
        else:
            p = decay_packed(kind, [40, 70, 25], 2, d, torch.bfloat16, 81)
        oc = oracle_cache_fp32(p, [0, 1])
        rb = synth.seam_batch(kind, 3, 5, 3, 8, 2, d, seed=82)
        seam = (dev(rb.q), dev(rb.k), dev(rb.v), dev(rb.beta), dev(rb.log_alpha))
        s32, o32 = H.hypic_compose(oc, dev(rb.order), seam=seam, check_status=True)
        s16, o16 = H.hypic_compose(oc, dev(rb.order), seam=seam, check_status=True,
                                   o_dtype=torch.bfloat16)
        assert o16.dtype == torch.bfloat16
        assert torch.equal(o16, o32.to(torch.bfloat16)), kind
        assert torch.equal(s16, s32), kind


@pytest.mark.gpu
@pytest.mark.parametrize("w,dtype", [(1, torch.bfloat16), (3, torch.bfloat16),
                                     (16, torch.bfloat16), (20, torch.bfloat16),
                                     (8, torch.float32), (12, torch.float32)])
def test_compose_seam_window_lengths(w, dtype):
    """Seam windows from 1 to 20 tokens in bf16 and fp32 on the tensor-core
    compose (chunks of 8 tokens), with operand copies of Qhat (2 requests x 4
    positions of 3 pairs) and with the in-kernel conversion (1 x 4); against
    the oracle (gated delta, dk = dv = 128)."""
    p = synth.gdn_packed([50, 90, 30], 2, 128, 128, 91)
    oc = oracle_cache_fp32(p, [0, 1])
    for n_req in (2, 1):
        rb = synth.reuse_batch(n_req=n_req, n_pos=4, n_seg=3, w=w, n_streams=2, d=128,
                               seed=92, dtype=dtype)
        dev = lambda t: t.cuda().contiguous()
        seam = (dev(rb.q), dev(rb.k), dev(rb.v), dev(rb.beta), dev(rb.log_alpha))
        state, o = H.hypic_compose(oc, dev(rb.order), seam=seam, check_status=True)
        for s in range(2):
            pairs = cache_pairs_f64(oc, s)
            for r in range(n_req):
                S_ref, o_ref = ls.compose_with_seam(pairs, rb.order[r].tolist(),
                                                    seam_f64(rb, r, s))
                assert ls.rel_fro(state[r, s].double().cpu().numpy(), S_ref) <= COMPOSE_TOL, \
                    (w, n_req, r, s)
                assert ls.rel_fro(o[r, :, :, s].double().cpu().numpy(), o_ref) <= SEAM_TOL, \
                    (w, n_req, r, s)


@pytest.mark.gpu
def test_compose_operand_copy_path_matches_in_kernel_converter():
    """The gated-delta compose at dk = 128 converts each pair's Qhat in the
    kernel when pairs are used about once (a power-of-two scale per row of
    Qhat), and from operand copies made once per call when they are reused
    (n_req * n_pos >= 2 n_seg; one scale per pair).  Both split Qhat into fp16
    hi + lo exactly up to 22 bits, so one request's chain agrees between the
    two paths to ~1e-6, with and without a seam window, and matches the oracle."""
    p = synth.gdn_packed([90, 60, 120, 45], 2, 128, 128, 101)
    oc = oracle_cache_fp32(p, [0, 1])
    rb = synth.seam_batch("gdn", 2, 4, 4, 8, 2, 128, seed=102)
    dev = lambda t: None if t is None else t.cuda().contiguous()
    one = lambda t: dev(t[:1])
    order2 = dev(rb.order)                      # 2 x 4 positions of 4 pairs: operand copies
    order1 = one(rb.order)                      # 1 x 4: the in-kernel converter
    cs = oc.struct()
    assert H.lib().hypic_compose_workspace_bytes(ctypes.byref(cs), 2, 4, 0) > \
        H.lib().hypic_compose_workspace_bytes(ctypes.byref(cs), 1, 4, 0)
    s2, _ = H.hypic_compose(oc, order2, check_status=True)
    s1, _ = H.hypic_compose(oc, order1, check_status=True)
    close = lambda a, b: ls.rel_fro(a.double().cpu().numpy(), b.double().cpu().numpy()) <= 1e-5
    assert close(s1[0], s2[0])
    seam2 = tuple(dev(t) for t in (rb.q, rb.k, rb.v, rb.beta, rb.log_alpha))
    seam1 = tuple(one(t) for t in (rb.q, rb.k, rb.v, rb.beta, rb.log_alpha))
    t2, o2 = H.hypic_compose(oc, order2, seam=seam2, check_status=True)
    t1, o1 = H.hypic_compose(oc, order1, seam=seam1, check_status=True)
    assert close(t1[0], t2[0]) and close(o1[0], o2[0])
    for s in range(2):
        S_ref, o_ref = ls.compose_with_seam(cache_pairs_f64(oc, s), rb.order[0].tolist(),
                                            seam_f64(rb, 0, s))
        assert ls.rel_fro(t1[0, s].double().cpu().numpy(), S_ref) <= COMPOSE_TOL
        assert ls.rel_fro(o1[0, :, :, s].double().cpu().numpy(), o_ref) <= SEAM_TOL


@pytest.mark.gpu
def test_compose_seam_strong_and_vanishing_decay():
    """Seam chunks under strong decay: log alpha four times the usual draws
    (alpha down to ~1e-2 a token) and, on one token, log alpha = -200, where
    alpha underflows to zero in fp32.  The chunk form divides by no decay
    product, so states and outputs still match the token-serial oracle."""
    p = synth.gdn_packed([90, 60, 120], 2, 128, 128, 111)
    oc = oracle_cache_fp32(p, [0, 1])
    rb = synth.seam_batch("gdn", 3, 4, 3, 8, 2, 128, seed=112)
    g = rb.log_alpha.clone() * 4.0
    g[1, 2, 5, :] = -200.0
    dev = lambda t: None if t is None else t.cuda().contiguous()
    seam = (dev(rb.q), dev(rb.k), dev(rb.v), dev(rb.beta), dev(g))
    state, o = H.hypic_compose(oc, dev(rb.order), seam=seam, check_status=True)
    rb2 = dataclasses.replace(rb, log_alpha=g)
    for s in range(2):
        pairs = cache_pairs_f64(oc, s)
        for r in range(3):
            S_ref, o_ref = ls.compose_with_seam(pairs, rb.order[r].tolist(), seam_f64(rb2, r, s))
            assert ls.rel_fro(state[r, s].double().cpu().numpy(), S_ref) <= COMPOSE_TOL, (r, s)
            assert ls.rel_fro(o[r, :, :, s].double().cpu().numpy(), o_ref) <= SEAM_TOL, (r, s)


@pytest.mark.gpu
def test_kda_strong_gates_rebuilt_by_the_recurrence():
    """KDA heads where every other channel of stream 1 decays by e^-1..e^-6 a
    token: the chunks' decay spans lie far past the tensor-core build's
    single-reference bound (checked on the inputs), so those units are rebuilt
    by the token recurrence, while stream 0 (ordinary gates) stays on the tensor
    cores; every unit against the oracle, and the build is deterministic."""
    p = synth.kda_packed([200, 64, 130, 1, 0, 77], 2, 128, 128, seed=910)
    g = p.log_alpha.clone()
    rng = np.random.default_rng(911)
    strong = torch.from_numpy(-rng.uniform(1.0, 6.0, (g.shape[0], 64))).float()
    g[:, 1, ::2] = strong
    p = dataclasses.replace(p, log_alpha=g)
    for seg, limit in ((0, 64.0), (2, 64.0)):
        a = int(p.offsets[seg])
        gg = g[a:a + 64, 1].double().numpy()
        assert -np.cumsum(gg - gg.max(axis=1, keepdims=True), axis=0)[-1].min() > limit
        gg = g[a:a + 64, 0].double().numpy()
        assert -np.cumsum(gg - gg.max(axis=1, keepdims=True), axis=0)[-1].min() < limit / 4
    cache = run_build(p)
    for seg in range(p.n_seg):
        for s in range(2):
            eT, eS = unit_errors(p, cache, seg, s)
            assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, eT, eS)
    again = run_build(p)
    assert torch.equal(cache.S, again.S) and torch.equal(cache.Qhat, again.Qhat)
    assert torch.equal(cache.exp2, again.exp2) and torch.equal(cache.log_T, again.log_T)
    # no unit keeps the rebuild marker
    assert int(cache.exp2.min()) > -(1 << 30)


@pytest.mark.gpu
def test_kda_large_spans_within_the_bound_stay_on_the_tensor_cores():
    """KDA heads whose channels decay by up to e^-0.9 a token relative to the
    largest gate: a chunk's per-channel decay span reaches 30-60 nats, inside
    the tensor-core build's single-reference bound, so the key images carry
    factors up to e^60 through the products; every unit against the oracle and
    no unit handed to the token recurrence."""
    p = synth.kda_packed([130, 64, 200], 2, 128, 128, seed=920)
    g = p.log_alpha.clone()
    rng = np.random.default_rng(921)
    g[:, :, 1::2] = torch.from_numpy(-rng.uniform(0.3, 0.9, (g.shape[0], 2, 64))).float()
    p = dataclasses.replace(p, log_alpha=g)
    spans = []
    for seg in range(p.n_seg):
        for s in range(2):
            a, b = int(p.offsets[seg]), int(p.offsets[seg + 1])
            for c0 in range(a, b, 64):
                gg = g[c0:min(c0 + 64, b), s].double().numpy()
                spans.append(-np.cumsum(gg - gg.max(axis=1, keepdims=True), axis=0)[-1].min())
    assert 30.0 < max(spans) < 64.0
    cache = run_build(p)
    assert int(cache.exp2.min()) > -(1 << 30)
    for seg in range(p.n_seg):
        for s in range(2):
            eT, eS = unit_errors(p, cache, seg, s)
            assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, eT, eS)
