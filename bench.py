"""Benchmark of the linear-layer caching hot path on GB300.

One step = one pass of the whole path over one batch of synthetic input:

* ``cold_long`` (default): a 131,072-token prompt cut into lognormal segments
  (mean 1024, sigma 0.8, clipped to [128, 8192]) for a 30-layer x 16-head
  gated-delta stack, dk = dv = 128, bf16: segment build of every
  (segment, stream) pair under the LPT work order, then compose of the
  segments in a seeded random request order (one request, 480 streams).
* ``layer_reuse``: one 16-head layer, 64 x 1024-token segments built, then 32
  requests compose 128 cached pairs each with w = 8 seam tokens per position.

value = prompt tokens per second of the whole step (N_tok / step time, summed
over ranks).  Inputs are resident in HBM and larger than L2 (no flush needed).
``e2e`` repeats the step through the public API with inputs in pinned host
memory: the host->device copy of the step's inputs and the device->host read
of the composed states are inside the timed region.

``--impl reference`` times the float64 CPU oracle on a bounded sample of the
same workload on the host cores (the pages publish no runnable reference).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("segment-build tokens/s for (T_C,S) at dk=dv=128; compose µs/request; "
          "% roofline")


# ---------------------------------------------------------------- CPU oracle leg

def _oracle_unit_job(job):
    """One (k, v, beta, g) unit through the float64 oracle; returns seconds."""
    os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
    import numpy as np  # noqa: F401
    from oracle import linear_state as ls
    k, v, beta, g = job
    t = time.perf_counter()
    ls.segment_pair("gdn", k, v, beta, g, want_T=False)
    return time.perf_counter() - t


def oracle_sample(n_units=None, unit_len=256, seconds=15.0, cores=None):
    """Times the oracle's gated-delta build on seeded 128-dim units with a
    spawn pool over the host cores; returns (token-streams/s, cores, desc,
    token-streams/s of one pool process, i.e. one core)."""
    import numpy as np
    from linear_attn_state_gb300 import synth
    cores = cores or len(os.sched_getaffinity(0))
    # one unit's time in this process sizes the sample
    p = synth.gdn_packed([unit_len], 1, 128, 128, seed=99)
    u = synth.unit_inputs(p, 0, 0, unit_len)
    t1 = _oracle_unit_job((u["k"], u["v"], u["beta"], u["g"]))
    if n_units is None:
        n_units = max(cores, int(seconds * cores / max(t1, 1e-3)))
        n_units = int(np.ceil(n_units / cores) * cores)
    pk = synth.gdn_packed([unit_len] * n_units, 1, 128, 128, seed=100)
    jobs = []
    for i in range(n_units):
        uu = synth.unit_inputs(pk, 0, i * unit_len, (i + 1) * unit_len)
        jobs.append((uu["k"], uu["v"], uu["beta"], uu["g"]))
    ctx = mp.get_context("spawn")
    env_prev = os.environ.get("OPENBLAS_NUM_THREADS")
    os.environ["OPENBLAS_NUM_THREADS"] = "1"
    t0 = time.perf_counter()
    with ctx.Pool(cores) as pool:
        per_unit = pool.map(_oracle_unit_job, jobs)
    wall = time.perf_counter() - t0
    if env_prev is None:
        os.environ.pop("OPENBLAS_NUM_THREADS", None)
    rate = n_units * unit_len / wall
    desc = (f"{n_units} gated-delta units x {unit_len} tokens (dk=dv=128), float64 "
            f"explicit-transition oracle, {cores} spawn processes, {wall:.1f} s wall")
    # single-core figure: each pool process runs one BLAS thread on one core
    rate1 = unit_len / (sum(per_unit) / len(per_unit))
    return rate, cores, desc, rate1


# ---------------------------------------------------------------- clocks

class Clocks:
    """nvidia-smi sampling during the timed region."""

    def __init__(self):
        self.proc = None
        # raw samples: HYPIC_CLOCKS_DIR if set (to keep them), else the temp dir
        d = os.environ.get("HYPIC_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(d, f"hypic_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
            idx = os.environ.get("LOCAL_RANK", "0")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", idx, f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower() in ("active", "1"):
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- workloads

def build_flops(n_tok_streams, dk=128, dv=128, C=64):
    """Algorithmic FLOPs of the chunked gated-delta build per token-stream:
    4 dk (dk + dv) + 2 C (2 dk + dv)."""
    return n_tok_streams * (4 * dk * (dk + dv) + 2 * C * (2 * dk + dv))


def source_hash(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "linear_attn_state_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# the source files each measured kernel is compiled from
KERNEL_SOURCES = {"gdn_tc.cu": ("gdn_tc.cu", "chunk_tc.cuh", "tc_ptx.cuh")}


def measured_traffic(kernel_file, units_per_launch):
    """DRAM bytes per launch from a committed ncu summary, when it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[kernel_file]
        if e["source_hash"] != source_hash(*KERNEL_SOURCES.get(kernel_file, (kernel_file,))):
            return None
        return e["bytes_per_unit"] * units_per_launch
    except Exception:
        return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


def cold_long_config(n_tok, n_seg, n_streams, n_layers):
    return {"workload": "cold_long: 131072-token prompt, lognormal segments "
                        f"(mean 1024, sigma 0.8, [128, 8192]), {n_layers} layers x 16 GDN "
                        "heads, dk=dv=128, bf16; LPT build + compose of a random order",
            "n_tok": n_tok, "n_seg": n_seg, "n_streams": n_streams,
            "dk": 128, "dv": 128, "global_batch": 1, "seq_len": n_tok,
            "l2": f"inputs ({n_tok * n_streams * 520 / 1e9:.1f} GB) larger than L2; no flush"}


def layer_reuse_config(n_tok):
    return {"workload": "layer_reuse: 16 GDN heads, 64 x 1024 tokens built; then 32 "
                        "requests x 128 cached pairs with w=8 seam tokens",
            "n_tok": n_tok, "dk": 128, "dv": 128, "global_batch": 32,
            "seq_len": n_tok, "l2": "inputs larger than L2; no flush"}


def workload_config(workload, n_layers, world):
    """The config of rank 0's workload, from the host-side draws alone (the
    segment lengths), as the device arm reports it."""
    from linear_attn_state_gb300 import synth
    if workload == "cold_long":
        lengths = synth.cold_long_lengths()
        c = cold_long_config(int(sum(lengths)), len(lengths), 16 * n_layers, n_layers)
    else:
        g = synth.GDN_LAYER
        c = layer_reuse_config(g["n_seg"] * g["seg_len"])
    return dict(c, parallelism=f"replicas{world}")


class ColdLong:
    name = "cold_long"

    def __init__(self, dev, seed_offset=0, n_layers=30):
        import torch
        from linear_attn_state_gb300 import synth
        self.p = synth.cold_long_device(dev, n_layers=n_layers,
                                        seed=synth.COLD_LONG["seed"] + seed_offset)
        self.n_tok = int(self.p.offsets[-1])
        self.S = self.p.n_streams
        self.order = torch.from_numpy(synth.cold_long_order(self.p.n_seg)).view(1, -1).to(dev)
        self.d_off = torch.from_numpy(self.p.offsets).to(dev)
        self.config = cold_long_config(self.n_tok, self.p.n_seg, self.S, n_layers)


class LayerReuse:
    name = "layer_reuse"

    def __init__(self, dev, seed_offset=0):
        import torch
        from linear_attn_state_gb300 import synth
        import dataclasses
        p = synth.gdn_layer(seed=synth.GDN_LAYER["seed"] + seed_offset)
        mv = lambda t: t.to(dev).contiguous()
        self.p = dataclasses.replace(p, k=mv(p.k), v=mv(p.v), beta=mv(p.beta),
                                     log_alpha=mv(p.log_alpha))
        rb = synth.reuse_batch()
        self.rb = rb
        dv = lambda t: t.to(dev).contiguous()
        self.seam = tuple(dv(t) for t in (rb.q, rb.k, rb.v, rb.beta, rb.log_alpha))
        self.order = dv(rb.order)
        self.n_tok = int(self.p.offsets[-1])
        self.S = self.p.n_streams
        self.d_off = torch.from_numpy(self.p.offsets).to(dev)
        self.config = layer_reuse_config(self.n_tok)


# ---------------------------------------------------------------- multi-rank host logic
# One process per GPU; each rank builds and composes its own seeded replica of
# the workload (independent units, no data-path collective).  The only
# cross-rank steps are the barriers around the timed region and the max of the
# step time.

def replica_seed_offset(rank):
    """Seed offset of a rank's replica: rank r draws the workload with seed + r."""
    return int(rank)


def reduce_max(value, world, device=None):
    """Max over ranks of a per-rank time (the slowest rank sets the step time)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world, n_tok_per_rank, ms_step):
    """Whole-job prompt tokens/s: every rank processed n_tok_per_rank tokens
    (of all its streams) per step of ms_step (max over ranks)."""
    return world * n_tok_per_rank / (ms_step / 1e3)


def emit(out, rank):
    """The single JSON line, printed by rank 0 only; returns the line (or None)."""
    if rank != 0:
        return None
    line = json.dumps(out)
    print(line, flush=True)
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="hypic", choices=["hypic", "reference"])
    ap.add_argument("--workload", default="cold_long", choices=["cold_long", "layer_reuse"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-reuse", action="store_true")
    ap.add_argument("--layers", type=int, default=30,
                    help="layers of the cold long stack (30; fewer only to profile a smaller case)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args)
        return

    # the CPU oracle leg runs first, before any CUDA call (spawn pool)
    cpu = None
    if rank == 0 and not args.no_cpu:
        rate, cores, desc, rate1 = oracle_sample(seconds=4.0)
        streams = 16 * args.layers if args.workload == "cold_long" else 16
        cpu = {"value": rate / streams, "unit": "tokens/s",
               "cores": cores, "kind": "oracle",
               "single_core_value": round(rate1 / streams, 3),
               "sample": desc + "; converted to prompt tokens/s of the stack "
                                "(token-streams/s / streams)"}
        if args.workload == "cold_long":
            # extrapolated, not measured: the whole prompt at the sampled rate
            cpu["extrapolated_prompt_s"] = round(131072 / cpu["value"], 1)

    import torch
    import torch.distributed as dist
    from linear_attn_state_gb300 import build as hbuild
    from linear_attn_state_gb300 import hypic as H

    hbuild.build()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    off = replica_seed_offset(rank)
    W = ColdLong(dev, off, args.layers) if args.workload == "cold_long" else LayerReuse(dev, off)
    p = W.p
    stream = torch.cuda.current_stream()
    cache = H.Cache.empty("gdn", p.n_seg, p.n_streams, 128, 128, device=dev)
    from ctypes import byref
    a, keep = H.build_args("gdn", p.offsets, p.k, p.v, p.beta, p.log_alpha, 0, W.d_off)
    ws_b = H.workspace(H.lib().hypic_build_workspace_bytes(byref(a)), device=dev)
    n_req, n_pos = W.order.shape
    seam = getattr(W, "seam", None)
    ws_c = H.compose_workspace(cache, n_req, n_pos, seam[1].shape[2] if seam else 0)
    state = torch.empty((n_req, W.S, 128, 128), dtype=torch.float32, device=dev)

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        step_build(H, p, cache, ws_b, W)
        if ev is not None:
            ev[1].record(stream)
        H.hypic_compose(cache, W.order, state_out=state, seam=seam, ws=ws_c)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    assert H.hypic_read_device_status(ws_b) == 0 and H.hypic_read_device_status(ws_c) == 0

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = Clocks()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    build_ms = [e[0].elapsed_time(e[1]) for e in evs]
    comp_ms = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms = reduce_max(total_ms, world, dev)
    if world > 1:
        dist.barrier()
    ms_step = total_ms / args.steps
    value = job_throughput(world, W.n_tok, ms_step)

    # roofline of the dominant kernel (the build launch).  The burst bf16 peak
    # applies unless the clocks sampled during the timed region show the power
    # cap (then the sustained one); both fractions are reported.
    pk, src = peaks()
    b_ms = statistics.mean(build_ms)
    flops = build_flops(W.n_tok * W.S)
    achieved = flops / (b_ms / 1e3) / 1e12
    capped = "sw_power_cap" in clk.get("reasons", [])
    burst = pk.get("bf16_tflops")
    sustained = pk.get("bf16_tflops_sustained", burst)
    peak = sustained if capped else burst
    units = W.n_tok * W.S
    n_pairs = p.n_seg * W.S
    # algorithmic bytes of the build: k, v (bf16), beta, g (fp32) in; the cached
    # pair (Qhat, S fp32, exponent, log T) out
    build_bytes = units * 520 + n_pairs * 131080
    roof = {"kernel": "hypic_segment_build (gated delta, bf16)", "bound": "tensor",
            "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "peak_source": f"{src} bf16 dense {'sustained (power cap seen)' if capped else 'burst'}",
            "frac_of_burst": round(achieved / burst, 4),
            "frac_of_sustained": round(achieved / sustained, 4),
            "traffic": measured_traffic("gdn_tc.cu", units),
            "algorithmic_flops_per_launch": flops,
            "algorithmic_bytes_per_launch": build_bytes,
            "hbm_frac": round(build_bytes / (b_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)}
    c_ms = statistics.mean(comp_ms)
    # compose: every position reads one cached pair; the states are written once
    comp_bytes = n_req * n_pos * W.S * 131080 + n_req * W.S * 128 * 128 * 4
    compose_roof = {"algorithmic_bytes": comp_bytes,
                    "algorithmic_gb_per_s": round(comp_bytes / (c_ms / 1e3) / 1e9, 1),
                    "hbm_frac": round(comp_bytes / (c_ms / 1e3) / 1e9 / pk["hbm_gbs"], 4)}

    lpt = None
    if rank == 0 and args.workload == "cold_long":
        n = max(3, min(args.steps, 5))
        lpt = lpt_gain(H, torch, stream, lambda: step_build(H, p, cache, ws_b, W), n)
        lpt["one_layer"] = one_layer_lpt_gain(H, torch, stream, p, W, n)
    e2e = None
    if not args.no_e2e and rank == 0:
        e2e = run_e2e(W, H, torch, dev, cache, ws_b, ws_c, state, seam, args)
    reuse = None
    if rank == 0 and args.workload == "cold_long" and not args.no_reuse:
        del W.p, cache
        torch.cuda.empty_cache()
        reuse = reuse_path(H, torch, dev, max(3, min(args.steps, 10)), args.warmup, pk["hbm_gbs"],
                           pk["bf16_tflops"])
    decay = None
    if rank == 0 and not args.no_reuse:
        decay = decay_build(H, torch, dev, max(3, min(args.steps, 10)), args.warmup, pk["hbm_gbs"])

    if rank == 0:
        out = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
               "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": dict(W.config, parallelism=f"replicas{world}"),
               "build_ms": round(b_ms, 4),
               "build_token_streams_per_s": round(units / (b_ms / 1e3), 1),
               "compose_us_per_request": round(c_ms * 1e3 / n_req, 2),
               "compose_roofline": compose_roof,
               "roofline": roof, "clocks": clk,
               # per step: work-list prepare, the build, the compose; with seam
               # windows also the chunk records and the operand copies of Qhat
               "gpu_launches": (5 if seam else 3) * args.steps,
               "lpt_gain": lpt, "reuse_path": reuse, "decay_build": decay,
               "e2e": e2e, "cpu_baseline": cpu}
        emit(out, rank)
    if world > 1:
        dist.destroy_process_group()


def step_build(H, p, cache, ws_b, W):
    H.hypic_segment_build("gdn", p.offsets, p.k, p.v, p.beta, p.log_alpha, cache=cache,
                          ws=ws_b, d_offsets=W.d_off)


def lpt_gain(H, torch, stream, build, steps):
    """The build alone with its units taken in segment-index order and in the
    default longest-first (LPT) order, interleaved on the same inputs (larger
    than L2), outside the timed region: what the LPT order gains on this
    length mix.  The cached pairs are the same either way."""
    ms = {H.ORDER_INDEX: [], H.ORDER_LPT: []}
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    try:
        for i in range(2 * steps + 2):
            order = H.ORDER_INDEX if i % 2 == 0 else H.ORDER_LPT
            H.hypic_set_build_order(order)
            ev[0].record(stream)
            build()
            ev[1].record(stream)
            torch.cuda.synchronize()
            if i >= 2:   # the first pair warms the index order up
                ms[order].append(ev[0].elapsed_time(ev[1]))
    finally:
        H.hypic_set_build_order(H.ORDER_LPT)
    idx, lpt = statistics.median(ms[H.ORDER_INDEX]), statistics.median(ms[H.ORDER_LPT])
    return {"index_order_build_ms": round(idx, 4), "lpt_build_ms": round(lpt, 4),
            "speedup": round(idx / lpt, 4), "builds_each": steps}


def one_layer_lpt_gain(H, torch, stream, p, W, steps):
    """The same comparison on one 16-head layer of the prompt (134 segments x
    16 streams = about 14 units per CTA), where the order decides the tail."""
    from ctypes import byref
    k, v = p.k[:, :16].contiguous(), p.v[:, :16].contiguous()
    beta, la = p.beta[:, :16].contiguous(), p.log_alpha[:, :16].contiguous()
    cache = H.Cache.empty("gdn", p.n_seg, 16, 128, 128, device=k.device)
    a, keep = H.build_args("gdn", p.offsets, k, v, beta, la, 0, W.d_off)
    ws = H.workspace(H.lib().hypic_build_workspace_bytes(byref(a)), device=k.device)

    def build():
        H.hypic_segment_build("gdn", p.offsets, k, v, beta, la, cache=cache, ws=ws,
                              d_offsets=W.d_off)
    out = lpt_gain(H, torch, stream, build, steps)
    out["workload"] = "one layer: 134 segments x 16 streams (1.1 GB of inputs)"
    del keep
    return out


def run_e2e(W, H, torch, dev, cache, ws_b, ws_c, state, seam, args):
    """Same step through the public API with host inputs: k, v, beta, log_alpha
    in page-locked host memory, built by hypic_segment_build_host (consecutive-
    segment groups copied on a second stream while the previous group builds),
    then compose and the D2H read of the composed states."""
    p = W.p
    try:
        host = []
        for t in (p.k, p.v, p.beta, p.log_alpha):
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            host.append(h)
    except RuntimeError as e:
        return {"unavailable": f"pinned host copy failed: {e}"[:200]}
    out_host = torch.empty(state.shape, dtype=state.dtype).pin_memory()
    stream = torch.cuda.current_stream()
    copy_stream = torch.cuda.Stream()
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = out_host.numel() * out_host.element_size()
    group = 16384
    a, keep = H.build_args("gdn", p.offsets, p.k, p.v, p.beta, p.log_alpha, 0, W.d_off)
    stage = H.workspace(H.lib().hypic_build_host_stage_bytes(a, group), device=dev)
    del keep

    def step():
        H.hypic_segment_build_host("gdn", p.offsets, host[0], host[1], host[2], host[3], W.d_off,
                                   cache, group, stage=stage, ws=ws_b, copy_stream=copy_stream)
        H.hypic_compose(cache, W.order, state_out=state, seam=seam, ws=ws_c)
        out_host.copy_(state, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        step()
    torch.cuda.synchronize()
    n = max(1, min(args.steps, 5))
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(n):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    del host, stage
    return {"value": round(W.n_tok / (ms / 1e3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 3),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "path": "hypic_segment_build_host (16384-token segment groups, copies overlapped "
                    "with the build) + hypic_compose + D2H of the states"}


def reuse_path(H, torch, dev, steps, warmup, hbm_gbs, bf16_tflops):
    """Reuse path measured beside the main workload: the 16-head layer's cache
    (64 x 1024-token segments) built (the build timed too: inputs of 545 MB,
    larger than L2), then 32 requests compose 128 cached pairs each with w = 8
    seam tokens per position (compose + seam timed)."""
    import dataclasses
    from linear_attn_state_gb300 import synth
    p = synth.gdn_layer()
    mv = lambda t: t.to(dev).contiguous()
    p = dataclasses.replace(p, k=mv(p.k), v=mv(p.v), beta=mv(p.beta), log_alpha=mv(p.log_alpha))
    cache = H.hypic_segment_build("gdn", p.offsets, p.k, p.v, p.beta, p.log_alpha,
                                  check_status=True)
    d_off = torch.as_tensor(p.offsets, dtype=torch.int64).to(dev)
    from ctypes import byref
    a, keep = H.build_args("gdn", p.offsets, p.k, p.v, p.beta, p.log_alpha, 0, d_off)
    ws_b = H.workspace(H.lib().hypic_build_workspace_bytes(byref(a)), device=dev)
    del keep
    stream = torch.cuda.current_stream()

    def build():
        H.hypic_segment_build("gdn", p.offsets, p.k, p.v, p.beta, p.log_alpha, cache=cache,
                              ws=ws_b, d_offsets=d_off)
    for _ in range(max(1, warmup)):
        build()
    torch.cuda.synchronize()
    assert H.hypic_read_device_status(ws_b) == 0
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(stream)
    for _ in range(steps):
        build()
    b1.record(stream)
    torch.cuda.synchronize()
    b_ms = b0.elapsed_time(b1) / steps
    units = int(p.offsets[-1]) * p.n_streams
    flops = build_flops(units)
    layer_build = {"workload": "one 16-head gated-delta layer: 64 segments x 1024 tokens",
                   "ms": round(b_ms, 4),
                   "token_streams_per_s": round(units / (b_ms / 1e3), 1),
                   "prompt_tokens_per_s": round(int(p.offsets[-1]) / (b_ms / 1e3), 1),
                   "achieved_tflops": round(flops / (b_ms / 1e3) / 1e12, 2),
                   "frac_of_burst": round(flops / (b_ms / 1e3) / 1e12 / bf16_tflops, 4)}
    rb = synth.reuse_batch()
    seam = tuple(mv(t) for t in (rb.q, rb.k, rb.v, rb.beta, rb.log_alpha))
    order = mv(rb.order)
    n_req, n_pos = order.shape
    state = torch.empty((n_req, p.n_streams, 128, 128), dtype=torch.float32, device=dev)
    ws = H.compose_workspace(cache, n_req, n_pos, rb.w)
    for _ in range(max(1, warmup)):
        H.hypic_compose(cache, order, state_out=state, seam=seam, ws=ws)
    torch.cuda.synchronize()
    assert H.hypic_read_device_status(ws) == 0
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(steps):
        H.hypic_compose(cache, order, state_out=state, seam=seam, ws=ws)
    t1.record(stream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / steps
    S, w = p.n_streams, rb.w
    token_streams = n_req * n_pos * w * S
    nbytes = (n_req * n_pos * S * 131080 + token_streams * (3 * 128 * 2 + 8 + 128 * 4)
              + n_req * S * 128 * 128 * 4)
    return {"workload": "reuse: 16-head layer cache (64 x 1024 tokens); 32 requests x 128 cached "
                        "pairs, w=8 seam tokens per position, bf16 seam inputs",
            "compose_us_per_request": round(ms * 1e3 / n_req, 2), "ms": round(ms, 4),
            "algorithmic_gb_per_s": round(nbytes / (ms / 1e3) / 1e9, 1),
            "hbm_frac": round(nbytes / (ms / 1e3) / 1e9 / hbm_gbs, 4),
            "algorithmic_bytes": nbytes, "layer_build": layer_build}


def decay_build(H, torch, dev, steps, warmup, hbm_gbs):
    """Builds of the other families measured beside the main workload: 128
    segments x 512 tokens x 16 streams each of RetNet (scalar gamma), GLA
    (per-channel decay), Mamba2-style (per-token scalar decay) and KDA (gated
    delta rule with a per-channel gate), dk = dv = 128, bf16 (seeded device
    draws).  Algorithmic bytes = k, v (+ gates, beta) in, the cached pairs out;
    the decay-only builds are HBM-bound, KDA's is the chunked tensor-core build
    (bound by its CUDA-core share: gate scans, key images, the 64x64 inverse)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(1001)
    n_seg, L, S = 128, 512, 16
    N = n_seg * L
    offs = [i * L for i in range(n_seg + 1)]
    k = torch.nn.functional.normalize(torch.randn(N, S, 128, device=dev, generator=gen), dim=-1)
    k = k.to(torch.bfloat16)
    v = torch.randn(N, S, 128, device=dev, generator=gen).to(torch.bfloat16)
    out = {"workload": "decay build: 128 segments x 512 tokens x 16 streams, dk=dv=128, bf16"}
    ws = H.workspace(1 << 20, device=dev)
    d_off = torch.tensor(offs, dtype=torch.int64, device=dev)   # offsets uploaded once
    beta = None
    for kind in ("scalar", "diag", "token", "kda"):
        if kind == "scalar":
            g = torch.log1p(-torch.exp2(-5.0 - torch.arange(S, device=dev, dtype=torch.float64) % 8))
            g = g.float().contiguous()
        elif kind == "token":
            A = -(1.0 + 15.0 * torch.rand(1, S, device=dev, generator=gen))
            dt = torch.exp(torch.empty(N, S, device=dev).uniform_(math.log(1e-3), math.log(1e-1),
                                                                   generator=gen))
            g = (dt * A).contiguous()
        else:
            z = torch.randn(N, S, 128, device=dev, generator=gen) + 3.0
            g = (-torch.nn.functional.softplus(-z)).contiguous()
        if kind == "kda":
            beta = torch.rand(N, S, device=dev, generator=gen)
        cache = H.Cache.empty(kind, n_seg, S, 128, 128, device=dev)
        for _ in range(max(1, warmup)):
            H.hypic_segment_build(kind, offs, k, v, beta, g, cache=cache, ws=ws, d_offsets=d_off)
        torch.cuda.synchronize()
        assert H.hypic_read_device_status(ws) == 0
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            H.hypic_segment_build(kind, offs, k, v, beta, g, cache=cache, ws=ws, d_offsets=d_off)
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        # in: k, v (+ gates, beta); out: S, log T (+ Qhat, exponents)
        nbytes = N * S * 2 * 128 * 2 + n_seg * S * 128 * 128 * 4
        if kind == "diag":
            nbytes += N * S * 128 * 4 + n_seg * S * 128 * 4
        elif kind == "token":
            nbytes += N * S * 4 + n_seg * S * 4
        elif kind == "kda":
            nbytes += N * S * 128 * 4 + N * S * 4 + n_seg * S * (128 * 128 * 4 + 8)
        else:
            nbytes += n_seg * S * 4
        gbs = nbytes / (ms / 1e3) / 1e9
        name = {"scalar": "retnet", "diag": "gla", "token": "mamba2", "kda": "kda"}[kind]
        out[name] = {
            "ms": round(ms, 4), "tokens_per_s": round(N * S / (ms / 1e3), 1),
            "algorithmic_bytes": nbytes, "algorithmic_gb_per_s": round(gbs, 1),
            "hbm_frac": round(gbs / hbm_gbs, 4)}
        del cache, g
    return out


def run_reference(args):
    """The float64 CPU oracle as the reference arm: each step a bounded sample
    of the workload's gated-delta units on the host cores."""
    rates = []
    desc = ""
    cores = len(os.sched_getaffinity(0))
    total = args.warmup + args.steps
    sec = max(2.0, min(20.0, 150.0 / max(total, 1)))
    for i in range(total):
        rate, cores, desc, _ = oracle_sample(seconds=sec, cores=cores)
        if i >= args.warmup:
            rates.append(rate)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    config = workload_config(args.workload, args.layers, world)
    streams = config.get("n_streams", 16)
    n_tok = config["n_tok"]
    value = statistics.mean(rates) / streams
    ms = n_tok / value * 1e3
    out = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": "tokens/s",
           "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 1), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": config,
           "note": "float64 oracle on host cores; each step times a bounded sample of "
                   "gated-delta units and extrapolates to the workload",
           "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cores,
                            "kind": "oracle", "sample": desc},
           "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


if __name__ == "__main__":
    main()
