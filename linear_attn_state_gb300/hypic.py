"""Thin ctypes binding of libhypic.so (include/hypic.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  torch tensors supply device memory and the current CUDA stream; the
functions below pass their data pointers through the C ABI and raise on any
non-OK status.  There is no fallback: if the library is not built, importing
a compute entry point raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libhypic.so")

HYPIC_OK = 0
SPIN_EXPIRE_NOW = 0xFFFFFFFF   # hypic_set_spin_limit: every bounded wait gives up at once
STATUS = {0: "HYPIC_OK", 1: "HYPIC_ERR_NULL", 2: "HYPIC_ERR_SHAPE", 3: "HYPIC_ERR_OFFSETS",
          4: "HYPIC_ERR_INDEX", 5: "HYPIC_ERR_DTYPE", 6: "HYPIC_ERR_WORKSPACE",
          7: "HYPIC_ERR_ARCH", 8: "HYPIC_ERR_CUDA", 9: "HYPIC_ERR_DEVICE_TIMEOUT"}
KIND = {"gdn": 0, "scalar": 1, "diag": 2, "none": 3, "token": 4, "kda": 5}
FACTORED = ("gdn", "kda")   # caches holding T = exp(log_T) 2^exp2 Qhat
DTYPE = {torch.bfloat16: 0, torch.float32: 1}

EXPORTS = ("hypic_build_workspace_bytes", "hypic_segment_build", "hypic_compose_workspace_bytes",
           "hypic_compose", "hypic_seam_advance", "hypic_lpt_schedule",
           "hypic_offsets_from_lengths", "hypic_read_device_status", "hypic_set_spin_limit",
           "hypic_set_build_order",
           "hypic_status_str", "hypic_version", "hypic_segment_build_static_ws",
           "hypic_build_host_stage_bytes", "hypic_segment_build_host",
           "hypic_build_split_scratch_bytes", "hypic_segment_build_split")


class HypicError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


class BuildArgs(ctypes.Structure):
    _fields_ = [("n_seg", ctypes.c_int32), ("seam_w", ctypes.c_int32),
                ("n_streams", ctypes.c_int32), ("dk", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("kind", ctypes.c_int32), ("in_dtype", ctypes.c_int32),
                ("reserved0", ctypes.c_int32), ("n_tok", ctypes.c_int64),
                ("h_offsets", ctypes.c_void_p), ("d_offsets", ctypes.c_void_p),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("beta", ctypes.c_void_p),
                ("log_alpha", ctypes.c_void_p)]


class CacheStruct(ctypes.Structure):
    _fields_ = [("n_seg", ctypes.c_int32), ("n_streams", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("kind", ctypes.c_int32),
                ("reserved0", ctypes.c_int32), ("Qhat", ctypes.c_void_p),
                ("exp2", ctypes.c_void_p), ("log_T", ctypes.c_void_p), ("S", ctypes.c_void_p)]


class SeamArgs(ctypes.Structure):
    _fields_ = [("w", ctypes.c_int32), ("in_dtype", ctypes.c_int32), ("q", ctypes.c_void_p),
                ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("beta", ctypes.c_void_p),
                ("log_alpha", ctypes.c_void_p), ("out_o", ctypes.c_void_p),
                ("kind", ctypes.c_int32), ("o_bf16", ctypes.c_int32)]


_lib = None


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is not built: run linear_attn_state_gb300.build.build()")
        L = ctypes.CDLL(_LIB_PATH)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        sig = {
            "hypic_build_workspace_bytes": (SZ, [ctypes.POINTER(BuildArgs)]),
            "hypic_segment_build": (I32, [ctypes.POINTER(BuildArgs), ctypes.POINTER(CacheStruct),
                                          P, SZ, P]),
            "hypic_compose_workspace_bytes": (SZ, [ctypes.POINTER(CacheStruct), I32, I32, I32]),
            "hypic_compose": (I32, [ctypes.POINTER(CacheStruct), P, I32, I32, P, P,
                                    ctypes.POINTER(SeamArgs), P, SZ, P]),
            "hypic_seam_advance": (I32, [ctypes.POINTER(SeamArgs), I32, I32, I32, I32, P, P, SZ,
                                         P]),
            "hypic_lpt_schedule": (I32, [P, I32, I32, I32, I32, P, P]),
            "hypic_offsets_from_lengths": (I32, [P, I32, P]),
            "hypic_read_device_status": (I32, [P, P, ctypes.POINTER(I32)]),
            "hypic_set_spin_limit": (ctypes.c_uint32, [ctypes.c_uint32]),
            "hypic_set_build_order": (I32, [I32]),
            "hypic_status_str": (ctypes.c_char_p, [I32]),
            "hypic_version": (I32, []),
            "hypic_segment_build_static_ws": (I32, [ctypes.POINTER(BuildArgs),
                                                    ctypes.POINTER(CacheStruct), P,
                                                    ctypes.POINTER(I32)]),
            "hypic_build_host_stage_bytes": (SZ, [ctypes.POINTER(BuildArgs), I64]),
            "hypic_segment_build_host": (I32, [ctypes.POINTER(BuildArgs),
                                               ctypes.POINTER(CacheStruct), I64, P, SZ, P, SZ,
                                               P, P]),
            "hypic_build_split_scratch_bytes": (SZ, [ctypes.POINTER(BuildArgs), I64]),
            "hypic_segment_build_split": (I32, [ctypes.POINTER(BuildArgs),
                                                ctypes.POINTER(CacheStruct), I64, P, SZ, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check(st: int, where: str):
    if st != HYPIC_OK:
        raise HypicError(st, where)


# host-only helpers ------------------------------------------------------------

def hypic_offsets_from_lengths(lengths) -> np.ndarray:
    ln = np.ascontiguousarray(np.asarray(lengths, dtype=np.int64))
    out = np.zeros(len(ln) + 1, dtype=np.int64)
    _check(lib().hypic_offsets_from_lengths(ln.ctypes.data_as(ctypes.c_void_p), len(ln),
                                            out.ctypes.data_as(ctypes.c_void_p)),
           "hypic_offsets_from_lengths")
    return out


def hypic_lpt_schedule(offsets, seam_w: int, n_streams: int, n_workers: int):
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    n_seg = len(off) - 1
    order = np.zeros(n_seg * n_streams, dtype=np.int32)
    worker = np.zeros(n_seg * n_streams, dtype=np.int32)
    _check(lib().hypic_lpt_schedule(off.ctypes.data_as(ctypes.c_void_p), n_seg, seam_w,
                                    n_streams, n_workers, order.ctypes.data_as(ctypes.c_void_p),
                                    worker.ctypes.data_as(ctypes.c_void_p)),
           "hypic_lpt_schedule")
    return order, worker


def hypic_set_spin_limit(limit: int) -> int:
    return int(lib().hypic_set_spin_limit(int(limit)))


ORDER_LPT, ORDER_INDEX = 0, 1   # hypic_set_build_order


def hypic_set_build_order(order: int) -> int:
    return int(lib().hypic_set_build_order(int(order)))


def hypic_read_device_status(ws: torch.Tensor, stream=None) -> int:
    out = ctypes.c_int32(-1)
    _check(lib().hypic_read_device_status(_ptr(ws), _stream_ptr(stream), ctypes.byref(out)),
           "hypic_read_device_status")
    return int(out.value)


# cache ------------------------------------------------------------------------

@dataclass
class Cache:
    """Device tensors of a (T_C, S(C|0)) cache (layouts of include/hypic.h)."""
    kind: str
    n_seg: int
    n_streams: int
    dk: int
    dv: int
    S: torch.Tensor
    log_T: torch.Tensor
    Qhat: Optional[torch.Tensor] = None
    exp2: Optional[torch.Tensor] = None

    @staticmethod
    def empty(kind, n_seg, n_streams, dk, dv, device="cuda"):
        S = torch.empty((n_seg, n_streams, dk, dv), dtype=torch.float32, device=device)
        lt_shape = (n_seg, n_streams, dk) if kind == "diag" else (n_seg, n_streams)
        log_T = torch.empty(lt_shape, dtype=torch.float32, device=device)
        Qhat = exp2 = None
        if kind in FACTORED:
            Qhat = torch.empty((n_seg, n_streams, dk, dk), dtype=torch.float32, device=device)
            exp2 = torch.empty((n_seg, n_streams), dtype=torch.int32, device=device)
        return Cache(kind, n_seg, n_streams, dk, dv, S, log_T, Qhat, exp2)

    def struct(self) -> CacheStruct:
        return CacheStruct(self.n_seg, self.n_streams, self.dk, self.dv, KIND[self.kind], 0,
                           _ptr(self.Qhat), _ptr(self.exp2), _ptr(self.log_T), _ptr(self.S))


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned device buffer of at least ``nbytes`` bytes."""
    t = torch.empty(max(int(nbytes), 256) + 256, dtype=torch.uint8, device=device)
    off = (-t.data_ptr()) % 256
    return t[off:off + max(int(nbytes), 256)]


# compute entry points ---------------------------------------------------------

def build_args(kind, offsets, k, v, beta=None, log_alpha=None, seam_w=0, d_offsets=None):
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.int64))
    if d_offsets is None:
        d_offsets = torch.from_numpy(off).to(k.device)
    a = BuildArgs(len(off) - 1, int(seam_w), k.shape[1], k.shape[2], v.shape[2], KIND[kind],
                  DTYPE[k.dtype], 0, int(off[-1]), off.ctypes.data_as(ctypes.c_void_p),
                  _ptr(d_offsets), _ptr(k), _ptr(v), _ptr(beta), _ptr(log_alpha))
    return a, (off, d_offsets)  # keep the buffers alive with the struct


def hypic_segment_build(kind, offsets, k, v, beta=None, log_alpha=None, seam_w=0,
                        cache: Optional[Cache] = None, ws: Optional[torch.Tensor] = None,
                        d_offsets=None, stream=None, check_status=False) -> Cache:
    """(T_C, S(C|0)) of every (segment, stream) body; see hypic_segment_build in
    include/hypic.h for layouts.  Tensors must be contiguous on the device.
    ``d_offsets``: the offsets already on the device (int64); when omitted they
    are uploaded on every call, a copy from pageable memory that waits for the
    stream's earlier work."""
    for t in (k, v, beta, log_alpha):
        assert t is None or t.is_contiguous()
    a, keep = build_args(kind, offsets, k, v, beta, log_alpha, seam_w, d_offsets)
    if cache is None:
        cache = Cache.empty(kind, a.n_seg, a.n_streams, a.dk, a.dv, device=k.device)
    need = lib().hypic_build_workspace_bytes(ctypes.byref(a))
    if ws is None:
        ws = workspace(need, device=k.device)
    cs = cache.struct()
    _check(lib().hypic_segment_build(ctypes.byref(a), ctypes.byref(cs), _ptr(ws), ws.numel(),
                                     _stream_ptr(stream)), "hypic_segment_build")
    if check_status:
        _check(hypic_read_device_status(ws, stream), "hypic_segment_build (device)")
    del keep
    return cache


def hypic_segment_build_host(kind, offsets, k, v, beta, log_alpha, d_offsets, cache: Cache,
                             max_group_tokens: int, stage: Optional[torch.Tensor] = None,
                             ws: Optional[torch.Tensor] = None, stream=None, copy_stream=None,
                             check_status=False) -> Cache:
    """Build from host-resident k, v, beta, log_alpha (page-locked CPU tensors),
    copying consecutive-segment groups of at most ``max_group_tokens`` tokens on
    ``copy_stream`` while the previous group builds on ``stream``; see
    hypic_segment_build_host in include/hypic.h.  ``d_offsets`` are the offsets
    on the device; the cache is on the device."""
    for t in (k, v, beta, log_alpha):
        assert t is None or (t.is_contiguous() and t.device.type == "cpu")
    a, keep = build_args(kind, offsets, k, v, beta, log_alpha, 0, d_offsets)
    dev = cache.S.device
    need = lib().hypic_build_host_stage_bytes(ctypes.byref(a), int(max_group_tokens))
    if stage is None:
        stage = workspace(need, device=dev)
    if ws is None:
        ws = workspace(lib().hypic_build_workspace_bytes(ctypes.byref(a)), device=dev)
    cs = cache.struct()
    st = _stream_ptr(stream)
    cp = st if copy_stream is None else ctypes.c_void_p(copy_stream.cuda_stream)
    _check(lib().hypic_segment_build_host(ctypes.byref(a), ctypes.byref(cs), int(max_group_tokens),
                                          _ptr(stage), stage.numel(), _ptr(ws), ws.numel(), st, cp),
           "hypic_segment_build_host")
    if check_status:
        _check(hypic_read_device_status(ws, stream), "hypic_segment_build_host (device)")
    del keep
    return cache


def hypic_segment_build_split(kind, offsets, k, v, beta=None, log_alpha=None, piece_tokens=1024,
                              seam_w=0, cache: Optional[Cache] = None,
                              scratch: Optional[torch.Tensor] = None, d_offsets=None, stream=None,
                              check_status=False) -> Cache:
    """The same pairs as hypic_segment_build, with every segment body cut into
    pieces of at most ``piece_tokens`` tokens built in parallel and composed;
    see hypic_segment_build_split in include/hypic.h."""
    for t in (k, v, beta, log_alpha):
        assert t is None or t.is_contiguous()
    a, keep = build_args(kind, offsets, k, v, beta, log_alpha, seam_w, d_offsets)
    if cache is None:
        cache = Cache.empty(kind, a.n_seg, a.n_streams, a.dk, a.dv, device=k.device)
    need = lib().hypic_build_split_scratch_bytes(ctypes.byref(a), int(piece_tokens))
    if scratch is None:
        scratch = workspace(need, device=k.device)
    cs = cache.struct()
    _check(lib().hypic_segment_build_split(ctypes.byref(a), ctypes.byref(cs), int(piece_tokens),
                                           _ptr(scratch), scratch.numel(), _stream_ptr(stream)),
           "hypic_segment_build_split")
    if check_status:
        _check(hypic_read_device_status(scratch, stream), "hypic_segment_build_split (device)")
    del keep
    return cache


def seam_struct(q, k, v, beta, log_alpha, out_o, kind="gdn") -> SeamArgs:
    for t in (q, k, v, beta, log_alpha, out_o):
        assert t is None or t.is_contiguous()
    return SeamArgs(k.shape[2], DTYPE[k.dtype], _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                    _ptr(log_alpha), _ptr(out_o), KIND[kind],
                    1 if out_o.dtype == torch.bfloat16 else 0)


def compose_workspace(cache: "Cache", n_req: int, n_pos: int, seam_w: int = 0) -> torch.Tensor:
    """Workspace for hypic_compose of ``cache`` over n_req x n_pos positions with
    a seam window of seam_w tokens (0: none), on the cache's device."""
    cs = cache.struct()
    return workspace(lib().hypic_compose_workspace_bytes(ctypes.byref(cs), n_req, n_pos, seam_w),
                     device=cache.S.device)


def hypic_compose(cache: Cache, order: torch.Tensor, state_in=None, state_out=None, seam=None,
                  ws=None, stream=None, check_status=False, o_dtype=torch.float32):
    """Compose cached pairs in request order.  ``order`` int32 [n_req, n_pos]
    on the device; ``seam`` is None or a tuple (q, k, v, beta, log_alpha)
    shaped [n_req, n_pos, w, S, d] / [n_req, n_pos, w, S] (layouts by family in
    include/hypic.h), advanced with the cache's family.
    Returns (state_out [n_req, S, dk, dv], o or None)."""
    n_req, n_pos = order.shape
    dev = order.device
    if state_out is None:
        state_out = torch.empty((n_req, cache.n_streams, cache.dk, cache.dv),
                                dtype=torch.float32, device=dev)
    o = None
    sp = None
    if seam is not None:
        q, k, v, beta, la = seam
        o = torch.empty(tuple(v.shape[:4]) + (cache.dv,), dtype=o_dtype, device=dev)
        sp = seam_struct(q, k, v, beta, la, o, cache.kind)
    if ws is None:
        ws = compose_workspace(cache, n_req, n_pos, sp.w if sp is not None else 0)
    cs = cache.struct()
    _check(lib().hypic_compose(ctypes.byref(cs), _ptr(order.contiguous()), n_req, n_pos,
                               _ptr(state_in), _ptr(state_out),
                               ctypes.byref(sp) if sp is not None else None, _ptr(ws),
                               ws.numel(), _stream_ptr(stream)), "hypic_compose")
    if check_status:
        _check(hypic_read_device_status(ws, stream), "hypic_compose (device)")
    return state_out, o


def hypic_seam_advance(state: torch.Tensor, q, k, v, beta, log_alpha, ws=None, stream=None,
                       check_status=False, kind="gdn", o_dtype=torch.float32):
    """Advance ``state`` [n_req, S, dk, dv] in place through one seam window per
    request (q, k, v [n_req, 1, w, S, d]; beta, log_alpha [n_req, 1, w, S], or
    the layouts of ``kind`` in include/hypic.h).  Returns o [n_req, 1, w, S, dv]."""
    n_req, n_streams, dk, dv = state.shape
    o = torch.empty(tuple(v.shape[:4]) + (dv,), dtype=o_dtype, device=state.device)
    sp = seam_struct(q, k, v, beta, log_alpha, o, kind)
    if ws is None:
        ws = workspace(256, device=state.device)
    _check(lib().hypic_seam_advance(ctypes.byref(sp), n_req, n_streams, dk, dv, _ptr(state),
                                    _ptr(ws), ws.numel(), _stream_ptr(stream)),
           "hypic_seam_advance")
    if check_status:
        _check(hypic_read_device_status(ws, stream), "hypic_seam_advance (device)")
    return o
