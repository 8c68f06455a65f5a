"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, its host-only functions are bit-exact against the oracle's
integer logic, and invalid arguments are rejected before any launch."""
import ctypes
import os
import re

import numpy as np
import pytest

from linear_attn_state_gb300 import build as hbuild
from linear_attn_state_gb300 import hypic as H
from linear_attn_state_gb300 import synth
from oracle import schedule as sch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    hbuild.build()
    return H.lib()


def declared_functions():
    with open(os.path.join(ROOT, "include", "hypic.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hypic_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(H.EXPORTS)
    assert L.hypic_version() >= 100
    assert L.hypic_status_str(0) == b"HYPIC_OK"
    assert L.hypic_status_str(9) == b"HYPIC_ERR_DEVICE_TIMEOUT"


def test_offsets_bit_exact(L):
    rng = np.random.default_rng(0)
    for n in (0, 1, 5, 300):
        lengths = rng.integers(0, 5000, n)
        assert list(H.hypic_offsets_from_lengths(lengths)) == sch.offsets_from_lengths(lengths)
    with pytest.raises(H.HypicError):
        H.hypic_offsets_from_lengths([3, -1])


def _check_lpt(off, w, S, m):
    order, worker = H.hypic_lpt_schedule(off, w, S, m)
    o_ref, w_ref = sch.lpt_schedule(list(off), w, S, m)
    assert order.tolist() == o_ref
    assert worker.tolist() == w_ref


def test_lpt_bit_exact_hand_and_random(L):
    _check_lpt([0, 3, 8, 10, 13, 15], 0, 1, 2)
    _check_lpt([0, 10, 14, 23], 3, 2, 3)
    _check_lpt([0, 4, 8], 0, 2, 3)      # equal costs across segments and streams
    _check_lpt([0, 2, 6], 5, 1, 2)      # bodies emptied by the seam window
    rng = np.random.default_rng(1)
    for _ in range(20):
        n = int(rng.integers(1, 40))
        lengths = rng.integers(0, 50, n)
        off = sch.offsets_from_lengths(lengths)
        _check_lpt(off, int(rng.integers(0, 10)), int(rng.integers(1, 5)), int(rng.integers(1, 9)))


@pytest.mark.parametrize("m", [1, 8, 152, 304])
def test_lpt_bit_exact_workloads(L, m):
    off = synth.offsets_of([1024] * 64)
    _check_lpt(off, 0, 16, m)
    off4 = synth.offsets_of(synth.cold_long_lengths())
    _check_lpt(off4, 0, 480, m)
    _check_lpt(off4, 8, 480, m)


def torch_cuda_available():
    import torch
    return torch.cuda.is_available()


def _fake(n):
    return ctypes.c_void_p(0x10000 + 256 * n)


def _args(**kw):
    off = np.array([0, 4, 9], dtype=np.int64)
    d = dict(n_seg=2, seam_w=0, n_streams=1, dk=64, dv=64, kind=0, in_dtype=0, reserved0=0,
             n_tok=9, h_offsets=off.ctypes.data_as(ctypes.c_void_p), d_offsets=_fake(1),
             k=_fake(2), v=_fake(3), beta=_fake(4), log_alpha=_fake(5))
    d.update(kw)
    a = H.BuildArgs(**d)
    return a, off


def _cache(**kw):
    d = dict(n_seg=2, n_streams=1, dk=64, dv=64, kind=0, reserved0=0, Qhat=_fake(6),
             exp2=_fake(7), log_T=_fake(8), S=_fake(9))
    d.update(kw)
    return H.CacheStruct(**d)


def _build(L, a, c, ws=_fake(10), ws_bytes=1 << 20):
    return L.hypic_segment_build(ctypes.byref(a), ctypes.byref(c), ws, ws_bytes, None)


def test_build_argument_validation(L):
    a, off = _args()
    c = _cache()
    assert L.hypic_segment_build(None, ctypes.byref(c), _fake(10), 1 << 20, None) == 1
    assert _build(L, *_args(dk=96, dv=96)[:1], c) == 2
    assert _build(L, _args(dk=64, dv=128)[0], c) == 2
    assert _build(L, _args(kind=7)[0], c) == 5
    assert _build(L, _args(in_dtype=3)[0], c) == 5
    assert _build(L, _args(beta=None)[0], c) == 1
    assert _build(L, _args(d_offsets=None)[0], c) == 1
    bad = np.array([0, 5, 4], dtype=np.int64)
    assert _build(L, _args(h_offsets=bad.ctypes.data_as(ctypes.c_void_p), n_tok=4)[0], c) == 3
    first = np.array([1, 4, 9], dtype=np.int64)
    assert _build(L, _args(h_offsets=first.ctypes.data_as(ctypes.c_void_p))[0], c) == 3
    assert _build(L, _args(n_tok=10)[0], c) == 3
    # a token count past the device's 32-bit token coordinates
    assert _build(L, _args(n_tok=(1 << 31))[0], c) == 2
    # arrays the kernels read with TMA or 16-byte vector loads start on 16 bytes
    odd = lambda n, b: ctypes.c_void_p(0x10000 + 256 * n + b)
    assert _build(L, _args(k=odd(2, 2))[0], c) == 2
    assert _build(L, _args(v=odd(3, 8))[0], c) == 2
    assert _build(L, a, _cache(S=odd(9, 4))) == 2
    assert _build(L, a, _cache(Qhat=odd(6, 12))) == 2
    kda = dict(kind=5, log_alpha=odd(5, 4))
    assert _build(L, _args(**kda)[0], _cache(kind=5)) == 2
    if not torch_cuda_available():
        # a scalar gate array is read per element: 4-byte alignment is enough
        assert _build(L, _args(log_alpha=odd(5, 4))[0], c) in (7, 8)
        assert _build(L, _args(**dict(kda, log_alpha=_fake(5)))[0], _cache(kind=5)) in (7, 8)
    assert L.hypic_segment_build_static_ws(ctypes.byref(_args(k=odd(2, 2))[0]), ctypes.byref(c),
                                           None, None) == 2
    assert _build(L, a, _cache(n_seg=3)) == 2
    assert _build(L, a, _cache(Qhat=None)) == 1
    assert _build(L, a, c, ws=None) == 6
    assert _build(L, a, c, ws=ctypes.c_void_p(0x10008)) == 6
    assert _build(L, a, c, ws_bytes=16) == 6
    # all host checks pass: the next step needs a device.  Only on a host
    # without a GPU (the fake pointers must never reach a kernel): the library
    # reports a CUDA error or a wrong arch, and still never aborts.
    import torch
    if not torch.cuda.is_available():
        assert _build(L, a, c) in (7, 8)


def test_compose_and_seam_validation(L):
    c = _cache()
    order = _fake(11)
    P = ctypes.POINTER
    assert L.hypic_compose(None, order, 1, 1, None, _fake(12), None, _fake(10), 4096, None) == 1
    assert L.hypic_compose(ctypes.byref(_cache(dk=32, dv=32)), order, 1, 1, None, _fake(12),
                           None, _fake(10), 4096, None) == 2
    assert L.hypic_compose(ctypes.byref(c), order, -1, 1, None, _fake(12), None, _fake(10),
                           4096, None) == 2
    assert L.hypic_compose(ctypes.byref(c), None, 1, 1, None, _fake(12), None, _fake(10),
                           4096, None) == 1
    assert L.hypic_compose(ctypes.byref(c), order, 1, 1, None, _fake(12), None, _fake(10),
                           16, None) == 6
    seam = H.SeamArgs(0, 0, _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), _fake(6))
    assert L.hypic_compose(ctypes.byref(c), order, 1, 1, None, _fake(12), ctypes.byref(seam),
                           _fake(10), 4096, None) == 2
    seam.w = 8
    seam.q = None
    assert L.hypic_compose(ctypes.byref(c), order, 1, 1, None, _fake(12), ctypes.byref(seam),
                           _fake(10), 4096, None) == 1
    seam.q = _fake(1)
    assert L.hypic_compose(ctypes.byref(_cache(kind=1)), order, 1, 1, None, _fake(12),
                           ctypes.byref(seam), _fake(10), 4096, None) == 5
    assert L.hypic_seam_advance(ctypes.byref(seam), 1, 1, 64, 64, None, _fake(10), 4096,
                                None) == 1
    assert L.hypic_seam_advance(ctypes.byref(seam), 1, 1, 64, 128, _fake(12), _fake(10), 4096,
                                None) == 2
    assert L.hypic_seam_advance(None, 1, 1, 64, 64, _fake(12), _fake(10), 4096, None) == 1
    # 16-byte boundaries: cache arrays, states, seam tokens
    odd = lambda n, b: ctypes.c_void_p(0x10000 + 256 * n + b)
    assert L.hypic_compose(ctypes.byref(c), order, 1, 1, None, odd(12, 4), None, _fake(10),
                           4096, None) == 2
    assert L.hypic_compose(ctypes.byref(c), order, 1, 1, odd(13, 8), _fake(12), None,
                           _fake(10), 4096, None) == 2
    assert L.hypic_compose(ctypes.byref(_cache(S=odd(9, 4))), order, 1, 1, None, _fake(12),
                           None, _fake(10), 4096, None) == 2
    seam.k = odd(2, 2)
    assert L.hypic_compose(ctypes.byref(c), order, 1, 1, None, _fake(12), ctypes.byref(seam),
                           _fake(10), 4096, None) == 2
    assert L.hypic_seam_advance(ctypes.byref(seam), 1, 1, 64, 64, _fake(12), _fake(10), 4096,
                                None) == 2
    seam.k = _fake(2)
    assert L.hypic_seam_advance(ctypes.byref(seam), 1, 1, 64, 64, odd(12, 4), _fake(10), 4096,
                                None) == 2


def test_compose_workspace_bytes(L):
    """The compose workspace: a 256-byte header; for a gated-delta (or KDA)
    cache at dk = dv = 128, one 16,896-byte seam chunk record per (request,
    position, 8-token chunk, stream), and, when the positions reuse each pair
    twice or more on average, a 64 KB operand copy of every pair's Qhat plus
    4 bytes each, every part rounded up to 256 bytes; a compose given less is
    refused before launch."""
    rec, up = 16896, (lambda x: -(-x // 256) * 256)
    ws = lambda c, *a: L.hypic_compose_workspace_bytes(ctypes.byref(c), *a)
    assert L.hypic_compose_workspace_bytes(None, 1, 1, 0) == 0
    small = _cache(n_seg=64, n_streams=4, dk=64, dv=64)          # dk = 64: CUDA-core compose
    assert ws(small, 32, 128, 8) == 256
    big = _cache(n_seg=64, n_streams=4, dk=128, dv=128)
    ops = up(64 * 4 * 65536) + up(64 * 4 * 4)
    assert ws(big, 0, 128, 8) == 256
    assert ws(big, 1, 64, 0) == 256                               # each pair used once
    assert ws(big, 1, 128, 0) == 256 + ops                        # twice on average
    for w, nch in ((1, 1), (8, 1), (9, 2), (16, 2), (20, 3)):
        assert ws(big, 2, 3, w) == 256 + up(2 * 3 * nch * 4 * rec)
        assert ws(big, 2, 64, w) == 256 + up(2 * 64 * nch * 4 * rec) + ops
    assert ws(_cache(n_seg=64, n_streams=4, dk=128, dv=128, kind=1), 2, 64, 8) == 256
    assert ws(_cache(n_seg=64, n_streams=4, dk=128, dv=128, kind=5), 2, 64, 8) == \
        256 + up(2 * 64 * 4 * rec) + ops
    seam = H.SeamArgs(8, 0, _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), _fake(6))
    c = _cache(n_streams=2, dk=128, dv=128)
    need = ws(c, 1, 1, 8)
    assert need == 256 + up(2 * rec)
    assert L.hypic_compose(ctypes.byref(c), _fake(11), 1, 1, None, _fake(12), ctypes.byref(seam),
                           _fake(10), need - 256, None) == 6
    assert L.hypic_compose(ctypes.byref(c), _fake(11), 1, 1, None, _fake(12), None, _fake(10),
                           256, None) != 6


def test_new_family_validation(L):
    """Mamba2-style per-token decay (kind 4) and KDA (kind 5): their required
    inputs and cache fields, and the seam, which only the gated-delta cache
    takes, are checked before any launch."""
    c4 = _cache(kind=4, Qhat=None, exp2=None)
    c5 = _cache(kind=5)
    assert _build(L, _args(kind=4, log_alpha=None)[0], c4) == 1      # gate missing
    assert _build(L, _args(kind=5, beta=None)[0], c5) == 1           # beta missing
    assert _build(L, _args(kind=5, log_alpha=None)[0], c5) == 1
    assert _build(L, _args(kind=5)[0], _cache(kind=5, Qhat=None)) == 1   # KDA caches Qhat
    assert _build(L, _args(kind=4)[0], c5) == 2                      # kind mismatch
    assert _build(L, _args(kind=6)[0], _cache(kind=6)) == 5
    # the seam tokens' family must be the cache's; each family's inputs are checked
    seam = H.SeamArgs(8, 0, _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), _fake(6))
    for kind in (4, 5):
        assert L.hypic_compose(ctypes.byref(_cache(kind=kind)), _fake(11), 1, 1, None, _fake(12),
                               ctypes.byref(seam), _fake(10), 4096, None) == 5
    no_beta = H.SeamArgs(8, 0, _fake(1), _fake(2), _fake(3), None, _fake(5), _fake(6), 5, 0)
    assert L.hypic_compose(ctypes.byref(c5), _fake(11), 1, 1, None, _fake(12),
                           ctypes.byref(no_beta), _fake(10), 4096, None) == 1
    no_gate = H.SeamArgs(8, 0, _fake(1), _fake(2), _fake(3), None, None, _fake(6), 4, 0)
    assert L.hypic_seam_advance(ctypes.byref(no_gate), 1, 1, 64, 64, _fake(12), _fake(10), 4096,
                                None) == 1
    bad_kind = H.SeamArgs(8, 0, _fake(1), _fake(2), _fake(3), _fake(4), _fake(5), _fake(6), 7, 0)
    assert L.hypic_seam_advance(ctypes.byref(bad_kind), 1, 1, 64, 64, _fake(12), _fake(10), 4096,
                                None) == 5
    assert L.hypic_compose(ctypes.byref(_cache(kind=5, exp2=None)), _fake(11), 1, 1, None,
                           _fake(12), None, _fake(10), 4096, None) == 1
    import torch
    if not torch.cuda.is_available():
        assert _build(L, _args(kind=4, beta=None)[0], c4) in (7, 8)
        assert _build(L, _args(kind=5)[0], c5) in (7, 8)
        ok = H.SeamArgs(8, 0, _fake(1), _fake(2), _fake(3), None, None, _fake(6), 3, 0)
        assert L.hypic_seam_advance(ctypes.byref(ok), 1, 1, 64, 64, _fake(12), _fake(10), 4096,
                                    None) in (7, 8)


def test_host_stage_bytes_per_family():
    """Staging per token: beta for the delta rules, one gate per stream
    (GDN, Mamba2-style) or dk gates (GLA, KDA)."""
    import torch
    off = np.array([0, 300], dtype=np.int64)
    up = lambda x: (x + 255) // 256 * 256
    f = H.lib().hypic_build_host_stage_bytes
    T, S, d = 300, 4, 128
    kv = 2 * up(T * S * d * 2)
    expect = {"gdn": kv + 2 * up(T * S * 4), "token": kv + up(T * S * 4),
              "diag": kv + up(T * S * d * 4), "kda": kv + up(T * S * 4) + up(T * S * d * 4),
              "none": kv, "scalar": kv + up(S * 4)}
    for kind, half in expect.items():
        a = H.BuildArgs(1, 0, S, d, d, H.KIND[kind], H.DTYPE[torch.bfloat16], 0, T,
                        off.ctypes.data_as(ctypes.c_void_p), ctypes.c_void_p(1),
                        ctypes.c_void_p(1), ctypes.c_void_p(1), ctypes.c_void_p(1),
                        ctypes.c_void_p(1))
        assert f(ctypes.byref(a), 1 << 20) == 2 * half, kind


def test_spin_limit_roundtrip(L):
    prev = L.hypic_set_spin_limit(5)
    assert L.hypic_set_spin_limit(0) == 5
    # the expire-now hook reads back as itself
    assert L.hypic_set_spin_limit(0xFFFFFFFF) != 0xFFFFFFFF
    assert L.hypic_set_spin_limit(prev) == 0xFFFFFFFF
    assert L.hypic_set_spin_limit(prev) == prev


def test_build_order_roundtrip(L):
    """The build order is LPT unless set; an unknown order is refused (-1) and
    leaves the setting as it was."""
    assert L.hypic_set_build_order(H.ORDER_INDEX) == H.ORDER_LPT
    assert L.hypic_set_build_order(7) == -1
    assert L.hypic_set_build_order(-1) == -1
    assert L.hypic_set_build_order(H.ORDER_LPT) == H.ORDER_INDEX
    assert L.hypic_set_build_order(H.ORDER_LPT) == H.ORDER_LPT


def test_host_build_stage_bytes_follows_segment_groups():
    """Staging for a host-input build: two halves sized for the largest group of
    consecutive segments within the token limit (a longer segment alone)."""
    import ctypes
    off = np.array([0, 100, 250, 400, 1400, 1500], dtype=np.int64)
    import torch
    a = H.BuildArgs(5, 0, 3, 128, 128, H.KIND["gdn"], H.DTYPE[torch.bfloat16], 0, 1500,
                    off.ctypes.data_as(ctypes.c_void_p), ctypes.c_void_p(1), ctypes.c_void_p(1),
                    ctypes.c_void_p(1), ctypes.c_void_p(1), ctypes.c_void_p(1))
    f = H.lib().hypic_build_host_stage_bytes
    up = lambda x: (x + 255) // 256 * 256
    def half(T, S=3):   # k, v bf16, beta, log_alpha fp32
        return up(T * S * 128 * 2) * 2 + up(T * S * 4) * 2
    # groups within 400 tokens: [0,400) then the 1000-token segment alone, then [1400,1500)
    assert f(ctypes.byref(a), 400) == 2 * half(1000)
    assert f(ctypes.byref(a), 1 << 20) == 2 * half(1500)
    assert f(ctypes.byref(a), 0) == 0


def test_split_scratch_bytes():
    """Scratch of a split build: positive for valid args, growing with the
    number of pieces, 0 for a non-positive piece size."""
    import torch
    off = np.array([0, 5000, 5100, 9000], dtype=np.int64)
    a = H.BuildArgs(3, 8, 2, 128, 128, H.KIND["gdn"], H.DTYPE[torch.bfloat16], 0, 9000,
                    off.ctypes.data_as(ctypes.c_void_p), ctypes.c_void_p(1), ctypes.c_void_p(1),
                    ctypes.c_void_p(1), ctypes.c_void_p(1), ctypes.c_void_p(1))
    f = H.lib().hypic_build_split_scratch_bytes
    big, small = f(ctypes.byref(a), 4096), f(ctypes.byref(a), 500)
    assert 0 < big < small
    assert f(ctypes.byref(a), 0) == 0


def test_build_workspace_bytes_is_header_plus_work_list(L):
    """A build's workspace: the 256-byte header (status word, queue) and the
    16-byte work item of every (segment, stream), rounded up to 256 bytes;
    invalid arguments ask for nothing."""
    import ctypes
    import torch
    for n_seg, S in ((0, 1), (3, 2), (64, 16), (134, 480)):
        off = np.arange(n_seg + 1, dtype=np.int64) * 7
        k = torch.zeros((int(off[-1]), S, 128), dtype=torch.bfloat16)
        a, keep = H.build_args("gdn", off, k, k, None, None)
        items = 16 * n_seg * S
        assert L.hypic_build_workspace_bytes(ctypes.byref(a)) == 256 + (items + 255) // 256 * 256
        a.n_streams = 0
        assert L.hypic_build_workspace_bytes(ctypes.byref(a)) == 0
        del keep
    assert L.hypic_build_workspace_bytes(None) == 0
