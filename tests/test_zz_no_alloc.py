"""The allocation-free build entry point.

hypic_segment_build_static_ws serves callers that cannot allocate device
memory when they build (for example a serving loop that must not let cudaMalloc
synchronise the device mid-request, or a framework whose allocator owns all
device memory): its scratch is a fixed array inside the library instead of a
caller-provided workspace.  It runs the same deterministic kernels as
hypic_segment_build, so this test calls it through the C ABI twice in a row and
requires each result to equal the ordinary entry point's bit for bit, and checks
two units against the oracle.  It sits in a file pytest collects last and
passes alone in a fresh process as well as after the other tests.
"""
import ctypes

import pytest
import torch

from linear_attn_state_gb300 import build as hbuild
from linear_attn_state_gb300 import hypic as H
from linear_attn_state_gb300 import synth
from tests.helpers import BUILD_TOL, unit_errors

pytestmark = pytest.mark.gpu


def test_static_workspace_build_matches_ordinary_build():
    assert torch.cuda.is_available()
    hbuild.build()
    L = H.lib()
    p = synth.gdn_packed([300, 64, 1, 0, 190], 6, 128, 128, seed=909, seam_w=8)
    dev = lambda t: t.cuda().contiguous()
    k, v, beta, la = dev(p.k), dev(p.v), dev(p.beta), dev(p.log_alpha)
    ref = H.hypic_segment_build("gdn", p.offsets, k, v, beta, la, seam_w=8, check_status=True)
    a, keep = H.build_args("gdn", p.offsets, k, v, beta, la, seam_w=8)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):
        out = H.Cache.empty("gdn", p.n_seg, p.n_streams, 128, 128)
        for t in (out.S, out.Qhat, out.log_T):
            t.fill_(float("nan"))
        out.exp2.fill_(-12345)
        cs = out.struct()
        st = ctypes.c_int32(-1)
        rc = L.hypic_segment_build_static_ws(ctypes.byref(a), ctypes.byref(cs), stream,
                                             ctypes.byref(st))
        assert rc == 0 and st.value == 0
        for name in ("S", "Qhat", "exp2", "log_T"):
            assert torch.equal(getattr(out, name), getattr(ref, name)), name
        for seg, s in ((0, 0), (4, 5)):
            eT, eS = unit_errors(p, out, seg, s)
            assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, eT, eS)
    del keep


def test_static_workspace_at_the_maximum_item_count():
    """Exactly HYPIC_STATIC_WS_MAX_ITEMS work items (131,072 one-token segments x
    2 streams, dk = dv = 64): the fixed array holds the whole work list, the
    device ranks 131,072 segments, and the result equals the ordinary build
    bit for bit; two units against the oracle."""
    hbuild.build()
    L = H.lib()
    n_seg, S = 262144 // 2, 2
    p = synth.gdn_packed([1] * n_seg, S, 64, 64, seed=262144)
    dev = lambda t: t.cuda().contiguous()
    k, v, beta, la = dev(p.k), dev(p.v), dev(p.beta), dev(p.log_alpha)
    ref = H.hypic_segment_build("gdn", p.offsets, k, v, beta, la, check_status=True)
    a, keep = H.build_args("gdn", p.offsets, k, v, beta, la)
    out = H.Cache.empty("gdn", n_seg, S, 64, 64)
    cs = out.struct()
    st = ctypes.c_int32(-1)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.hypic_segment_build_static_ws(ctypes.byref(a), ctypes.byref(cs), stream, ctypes.byref(st))
    assert rc == 0 and st.value == 0
    for name in ("S", "Qhat", "exp2", "log_T"):
        assert torch.equal(getattr(out, name), getattr(ref, name)), name
    for seg, s in ((0, 0), (n_seg - 1, 1)):
        eT, eS = unit_errors(p, out, seg, s)
        assert eT <= BUILD_TOL and eS <= BUILD_TOL, (seg, s, eT, eS)
    del keep, ref, out
    torch.cuda.empty_cache()


def test_static_workspace_rejects_too_many_items():
    """More work items than the fixed array holds: rejected before any launch."""
    import numpy as np
    hbuild.build()
    L = H.lib()
    n_seg = 262144 // 2 + 1          # x 2 streams = one item over the maximum
    off = np.zeros(n_seg + 1, dtype=np.int64)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: rejected before any launch
    a = H.BuildArgs(n_seg, 0, 2, 128, 128, 0, 0, 0, 0, off.ctypes.data_as(ctypes.c_void_p),
                    fake, fake, fake, fake, fake)
    c = H.CacheStruct(n_seg, 2, 128, 128, 0, 0, fake, fake, fake, fake)
    assert L.hypic_segment_build_static_ws(ctypes.byref(a), ctypes.byref(c), None, None) == 6


def test_static_workspace_checks_arguments_before_the_size_limit():
    """A missing cache is reported as HYPIC_ERR_NULL even when the item count is
    also over the limit: the ordinary build's checks run first."""
    import numpy as np
    hbuild.build()
    L = H.lib()
    n_seg = 262144 // 2 + 1
    off = np.zeros(n_seg + 1, dtype=np.int64)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced
    a = H.BuildArgs(n_seg, 0, 2, 128, 128, 0, 0, 0, 0, off.ctypes.data_as(ctypes.c_void_p),
                    fake, fake, fake, fake, fake)
    assert L.hypic_segment_build_static_ws(ctypes.byref(a), None, None, None) == 1
