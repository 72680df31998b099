#!/usr/bin/env python
"""Throughput of one step of the A2ATS hot path on GB300.

A step is one pass of the whole path over one batch of cached keys, each
stage one C-ABI call of liba2ats.so: windowed RoPE of the cache with the
retrieval split (proxy query) in one pass and the H-weighted assignment of
the retrieval rows on one stream, the plain nearest-centroid assignment of
every row on another, then the retrieval rows' codes copied over.  The
calibration (query second moment and Cholesky factor) is a one-off per layer
on the pages: it runs once before the timed steps, and its own time is
reported beside them, except on the long-context workload, whose steps
recompute it every time.  The codebook side of the assignments (centroids
transformed by L, their norms and 16-bit planes) depends only on the
codebook and L, so the timed steps reuse what the first step built; a step
that rebuilds it is timed separately and reported too.

Default workload: one attention layer of a Llama-3.2-3B-shaped model
(8 KV heads x 32768 cached keys x d=128, bf16; K=1024 centroids per head;
H from 8192 calibration queries per head; window 512; retrieval fraction
0.05), seeded synthetic data.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is keys assigned per second over all
ranks with the inputs resident on the GPU, the step replayed as one captured
CUDA graph (A2ATSStep.capture; the stage table and the contraction's roofline
come from a pass of eager calls before it).  Each of the K timed steps is
timed by its own CUDA events after an L2 flush; untimed replays between them
keep the timed region long enough for the clock sampler.  `e2e` repeats the
measurement through the public API (one captured step per device input set,
replayed) with each step's cache copied in from pinned host memory (beside
the previous step) and its codes and split copied back inside the timed
region; the codebook, a per-layer constant, is copied in once.  The reference
arm (`--impl reference`) times the fp64 CPU oracle on this machine's host
cores on a bounded sample of the same workload.  Under torchrun each rank
runs an independent replica of the workload (weak scaling, no data-path
collective).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "keys assigned/sec (windowed RoPE + H-weighted VQ argmin); % of roofline"

# DRAM bytes (read + write) of one stored-order contraction launch on the
# default workload, from an ncu capture of this kernel (the summary under
# profiles/ names the command).  It holds only for the contraction source it
# was taken on (the first 16 hex digits of the sha256 of csrc/assign_tc.cu);
# for any other source the bench reports null.
TC_TRAFFIC = {"llama32_3b_layer": ("658832b0770f7b11", 87563264)}
DEFAULT_WORKLOAD = "llama32_3b_layer"
L2_FLUSH_BYTES = 256 << 20
# the timed region lasts at least this long (untimed replays between the
# timed steps), so that the 100 ms clock sampler sees it under load
MIN_TIMED_REGION_S = 0.6


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--path", choices=["step", "hweighted", "attention", "dequantize",
                                       "subvector", "calibrate", "rope"],
                   default="step",
                   help="hweighted: time the H-weighted rule over every key of the cache "
                        "(L from the workload's calibration, windowed RoPE fused); "
                        "rope: time the windowed RoPE of the whole cache on its own; "
                        "attention: time the code-based attention scores and top tokens; "
                        "dequantize: time the reconstruction of the keys from their codes "
                        "(both steps after the path); calibrate: time one layer's codebook "
                        "calibration (H, L, z = k L, k-means++, back to key space) instead "
                        "of the step")
    p.add_argument("--subvector-composed", action="store_true",
                   help="--path subvector: code the sub-vectors with the composed assignment "
                        "calls instead of the sub-vector kernel")
    p.add_argument("--calib-tokens", type=int, default=4096,
                   help="calibration keys per head for --path calibrate")
    p.add_argument("--lloyd", type=int, default=10,
                   help="Lloyd rounds after the k-means++ seeding for --path calibrate")
    p.add_argument("--batch", type=int, default=0,
                   help="sequences of the decode workload's batch (0: the workload's own); "
                        "a smaller batch is for profiler captures")
    p.add_argument("--separate-split", action="store_true",
                   help="run RoPE and the split on the second stream beside a separate "
                        "plain-VQ call, instead of the fused call (same outputs)")
    return p.parse_args()


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return rank, local, world


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class Clocks:
    """nvidia-smi sampled every 100 ms while the timed region runs."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        self.gpu = vis.split(",")[local_rank] if vis else str(local_rank)
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.25)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        with open(self.file.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def _tc_traffic(workload: str):
    import hashlib
    entry = TC_TRAFFIC.get(workload)
    if entry is None:
        return None
    src = os.path.join(ROOT, "query_aware_vq_gb300", "csrc", "assign_tc.cu")
    with open(src, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:16]
    return entry[1] if digest == entry[0] else None


def _inputs(w, rank):
    # each rank its own batch of sequences; the codebook and the calibration
    # inputs are the layer's, shared by every rank
    keys = synth.keys(w, batch_offset=rank * w.B)
    cb = synth.codebook(w)
    queries = synth.queries(w) if (w.M and not w.h_given) else None
    hg = synth.given_h(w) if w.h_given else None
    return keys, cb, queries, hg


def _work(w, count):
    """Algorithmic work of each stage for one step (bytes or flops)."""
    s = {"f32": 4, "bf16": 2, "f16": 2}[w.dtype]
    keys = w.B * w.H * w.N
    n_ret = int(count.sum())
    return {
        "second_moment": ("tensor", 2.0 * w.H * w.M * w.d * w.d),
        "cholesky": ("alu", w.H * w.d ** 3 / 3.0),
        "windowed_rope": ("hbm", keys * w.d * 2.0 * s),
        "retrieval_split": ("hbm", keys * (w.d * s + 4.0)),
        # one read of the keys, the rotated keys written, the scores written
        # and read back by the select, the split written
        "rope_and_split": ("hbm", keys * (2.0 * w.d * s + 12.0)),
        "assign_retrieval": ("tensor", n_ret * (2.0 * w.d * w.K + 2.0 * w.d * w.d)),
        # the bulk rule runs over every row; the retrieval rows' codes are
        # copied over it afterwards
        "assign_bulk": ("tensor", keys * 2.0 * w.d * w.K),
        "route": ("hbm", n_ret * 12.0),
        # the fused call: RoPE, split and the bulk rule over every row; its
        # work is dominated by the contraction
        "rope_split_bulk": ("tensor", keys * 2.0 * w.d * w.K),
    }


def run_ours(a):
    import query_aware_vq_gb300 as q
    from query_aware_vq_gb300.pipeline import A2ATSStep

    rank, local, world = _dist()
    torch.cuda.set_device(local)
    w = synth.WORKLOADS[a.workload]
    keys, cb, queries, hg = _inputs(w, rank)
    dt = synth.DTYPES[w.dtype]
    step = A2ATSStep(w.B, w.H, w.N, w.d, w.K, dt, window=w.W, fraction=w.fraction,
                     rope_base=w.rope_base, far_offset=w.far_offset, M=w.M, ridge=w.ridge,
                     beta=w.betas[-1], fused=not a.separate_split)
    kd, cd = keys.cuda(), cb.cuda()
    qd = queries.cuda() if queries is not None else None
    hd = hg.cuda() if hg is not None else None
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    # the calibration: inside every step, or once ahead (timed on its own)
    calib_ms = None
    if qd is None and hd is None:
        kw, calib_mode = {}, "none (cosine blend)"
    elif w.calibrate_in_step:
        kw, calib_mode = dict(queries=qd, h_given=hd), "inside every step"
    else:
        calib_mode = "once before the timed steps (H, L reused)"
        cal_ev = []
        for _ in range(max(a.warmup, 3)):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            step.calibrate(queries=qd, h_given=hd)
            e1.record(stream)
            cal_ev.append((e0, e1))
        torch.cuda.synchronize()
        calib_ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in cal_ev)
        kw = dict(calibrated=True)

    # the codebook side of the assignments (transform by L, norms, planes) is
    # built by the first step and reused after it: the codebook and L are
    # per-layer constants.  A step that rebuilds it is timed on its own.
    rebuild_ev = []
    for i in range(max(a.warmup, 3)):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step(kd, cd, **kw)
        e1.record(stream)
        rebuild_ev.append((e0, e1))
    torch.cuda.synchronize()
    rebuild_ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in rebuild_ev)
    kw = dict(kw, reuse_codebook=True)
    for _ in range(a.warmup):
        step(kd, cd, **kw)
        flush.zero_()
    torch.cuda.synchronize()

    # ---- a profiling pass (eager calls): per-stage CUDA events, the
    # library's own timing of the stored-order contraction, and the number of
    # kernel launches per step
    events = {}
    launches0 = q.kernel_launches()
    q.set_kernel_timing(True)
    q.timed_kernels_ms()
    for _ in range(a.steps):
        step(kd, cd, events=events, **kw)
        flush.zero_()
    torch.cuda.synchronize()
    launches_per_step = (q.kernel_launches() - launches0) / a.steps
    tc_ms, tc_launches = q.timed_kernels_ms()
    q.set_kernel_timing(False)
    stage_ms = {k: sum(e0.elapsed_time(e1) for e0, e1 in v) / len(v) for k, v in events.items()}

    # ---- the step as one CUDA graph (both streams), replayed K times; eager
    # calls if the capture is refused
    try:
        graph = step.capture(kd, cd, **kw)
        run_step = graph.replay
        launch_mode = "CUDA graph of one step, replayed"
    except Exception as ex:  # noqa: BLE001
        torch.cuda.synchronize()
        run_step = lambda: step(kd, cd, **kw)  # noqa: E731
        launch_mode = f"eager calls (graph capture refused: {type(ex).__name__})"
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0.record(stream)
    for _ in range(a.warmup):
        run_step()
    w1.record(stream)
    torch.cuda.synchronize()
    flush.zero_()
    replay_ms = w0.elapsed_time(w1) / max(a.warmup, 1)

    # ---- timed region: K steps on resident inputs, each timed by its own
    # events, the L2 flushed before each.  Untimed replays between the timed
    # steps keep the GPU loaded for at least MIN_TIMED_REGION_S, so the
    # clock sampler sees the clocks the steps ran at.
    pad = max(0, int(MIN_TIMED_REGION_S * 1e3 / (a.steps * max(replay_ms, 1e-3))) - 1)
    step_ev = []
    clocks = Clocks(local)
    clocks.start()
    _barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for _ in range(a.steps):
        for _ in range(pad):
            run_step()
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_step()
        e1.record(stream)
        step_ev.append((e0, e1))
    torch.cuda.synchronize()
    _barrier(world)
    t_wall = time.perf_counter() - t_wall
    launches = int(round(launches_per_step * a.steps))
    launches_region = int(round(launches_per_step * a.steps * (pad + 1)))
    clk = clocks.stop()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in step_ev]
    ms = sum(step_ms) / len(step_ms)
    ms = _max_over_ranks(ms, world)
    keys_per_step = w.B * w.H * w.N
    value = world * keys_per_step / (ms * 1e-3)

    # ---- roofline of the dominant kernel: the tensor-core contraction over
    # the keys in stored order (every key outside the RoPE window), timed by
    # the library's CUDA events on the launching stream
    hbm, bf16, src = _peaks()
    work = _work(w, step.count.cpu())
    if tc_launches > 0:
        per_launch = tc_ms / tc_launches
        far_rows = w.B * w.H * max(w.N - max(w.W, 0), 0)
        amount = far_rows * 2.0 * w.d * w.K
        achieved = amount / (per_launch * 1e-3) / 1e12
        roof = {"kernel": "assign_tc_kernel (stored-order pass, bulk rows)", "bound": "tensor",
                "achieved": round(achieved, 3), "peak": bf16, "unit": "TFLOP/s",
                "frac": round(achieved / bf16, 5), "traffic": _tc_traffic(w.name),
                "flop_per_launch": amount, "ms_per_launch": round(per_launch, 5),
                "launches": tc_launches, "peak_source": f"{src} (bf16_tflops, burst)"}
    else:
        dom = max(stage_ms, key=stage_ms.get)
        bound, amount = work[dom]
        sec = stage_ms[dom] * 1e-3
        if bound == "hbm":
            achieved, peak, unit = amount / sec / 1e9, hbm, "GB/s"
        else:
            achieved, peak, unit = amount / sec / 1e12, bf16, "TFLOP/s"
            bound = "tensor"
        roof = {"kernel": dom, "bound": bound, "achieved": round(achieved, 3), "peak": peak,
                "unit": unit, "frac": round(achieved / peak, 5), "traffic": None,
                "peak_source": f"{src} ({'hbm_gbs' if unit == 'GB/s' else 'bf16_tflops'})"}
    stages = {}
    for k, v in stage_ms.items():
        b, amt = work[k]
        entry = {"ms": round(v, 4)}
        if b == "hbm":
            entry["GB/s"] = round(amt / (v * 1e-3) / 1e9, 1)
        else:
            entry["TFLOP/s"] = round(amt / (v * 1e-3) / 1e12, 3)
        stages[k] = entry

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs from pinned host memory and reads its outputs back;
    # the steps run as a pipeline, the copy of step i + 1's inputs (on a copy
    # stream, into the second of two device input sets) beside step i, the
    # way a serving loop feeds a layer.  The single-step latency (copy in,
    # step, copy out, synchronise) is reported beside it.
    e2e = None
    if not a.no_e2e:
        hk = keys.pin_memory()
        hc = cb.pin_memory()
        # per-step inputs: the cache, plus the calibration inputs when the
        # step recomputes H and L.  The codebook is a per-layer constant: it
        # is copied in once, before the timed steps, and the steps reuse the
        # codebook side built from it.
        per_step = "queries" in kw
        hq = queries.pin_memory() if (per_step and queries is not None) else None
        hh = hg.pin_memory() if (per_step and hg is not None) else None
        out_codes = torch.empty(step.codes.shape, dtype=torch.int32).pin_memory()
        out_perm = torch.empty(step.perm.shape, dtype=torch.int32).pin_memory()
        out_count = torch.empty(step.count.shape, dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in (hk, hq, hh) if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in (out_codes, out_perm, out_count))
        cd.copy_(hc)
        host = [hk, None, hq, hh]
        dev_sets = [[kd, cd, qd if hq is not None else None, hd if hh is not None else None]]
        dev_sets.append([None if t is None else torch.empty_like(t) for t in dev_sets[0]])
        dev_sets[1][1] = cd  # one resident codebook

        def step_kw(dset):
            k2 = dict(kw)
            if per_step:
                k2["queries"], k2["h_given"] = dset[2], dset[3]
            return k2

        def copy_in(dset, on):
            with torch.cuda.stream(on):
                for dst, src in zip(dset, host):
                    if src is not None:
                        dst.copy_(src, non_blocking=True)

        def copy_out(on):
            with torch.cuda.stream(on):
                out_codes.copy_(step.codes, non_blocking=True)
                out_perm.copy_(step.perm, non_blocking=True)
                out_count.copy_(step.count, non_blocking=True)

        # the latency of one step, alone: copy in, step, copy out
        lat_ms = []
        for i in range(a.warmup + a.steps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            copy_in(dev_sets[0], stream)
            step(dev_sets[0][0], dev_sets[0][1], **step_kw(dev_sets[0]))
            copy_out(stream)
            e1.record(stream)
            e1.synchronize()
            if i >= a.warmup:
                lat_ms.append(e0.elapsed_time(e1))
        lat = _max_over_ranks(sum(lat_ms) / len(lat_ms), world)

        # the pipeline: one captured step per input set
        try:
            runs = []
            for dset in dev_sets:
                copy_in(dset, stream)
                g = step.capture(dset[0], dset[1], **step_kw(dset))
                runs.append(g.replay)
            e2e_launch = "CUDA graph per input set"
        except Exception as ex:  # noqa: BLE001
            torch.cuda.synchronize()
            runs = [lambda dset=dset: step(dset[0], dset[1], **step_kw(dset)) for dset in dev_sets]
            e2e_launch = f"eager calls (graph capture refused: {type(ex).__name__})"
        cstream = torch.cuda.Stream()
        ready = [torch.cuda.Event(), torch.cuda.Event()]
        free = [torch.cuda.Event(), torch.cuda.Event()]
        for ev in free:
            ev.record(stream)

        def prefetch(s_):
            cstream.wait_event(free[s_])
            copy_in(dev_sets[s_], cstream)
            ready[s_].record(cstream)

        def pipeline(n):
            prefetch(0)
            for i in range(n):
                s_ = i % 2
                if i + 1 < n:
                    prefetch(1 - s_)
                stream.wait_event(ready[s_])
                runs[s_]()
                free[s_].record(stream)
                copy_out(stream)

        pipeline(max(a.warmup, 3))
        torch.cuda.synchronize()
        _barrier(world)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pipeline(a.steps)   # the last step waits for the last copy, so e1 follows every copy
        e1.record(stream)
        e1.synchronize()
        em = _max_over_ranks(e0.elapsed_time(e1) / a.steps, world)
        e2e = {"value": world * keys_per_step / (em * 1e-3), "unit": "keys/s",
               "ms_per_step": round(em, 4), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "mode": "pipelined: inputs of step i + 1 copied in beside step i (two device "
                       "input sets, together larger than L2; no flush)",
               "launch": e2e_launch,
               "latency_ms_per_step": round(lat, 4),
               "latency_keys_per_s": world * keys_per_step / (lat * 1e-3)}

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_baseline(w, keys, cb, queries, hg)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; correlated-Gaussian keys with outlier channels, "
                    "queries and codebooks from the same generator; no model weights)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "K": w.K,
                       "M": w.M, "window": w.W, "fraction": w.fraction, "storage": w.dtype,
                       "l2": "flushed between steps (256 MB write)",
                       "calibration": calib_mode,
                       "calibration_ms": None if calib_ms is None else round(calib_ms, 4),
                       "codebook_side": "built once, reused by every timed step",
                       "launch": launch_mode,
                       "composition": ("RoPE and split on the second stream, plain VQ apart"
                                       if a.separate_split else
                                       "one call for RoPE, split and plain VQ; the retrieval "
                                       "rule on the second stream"),
                       "ms_per_step_rebuilding_codebook_side": round(rebuild_ms, 4),
                       "parallelism": f"replicas x{world} (independent batches)"},
            "roofline": roof, "stages": stages, "cpu_baseline": cpu, "clocks": clk,
            "e2e": e2e, "gpu_launches": launches_region, "wall_s_timed": round(t_wall, 3),
            "timed_region": {"timed_steps": a.steps, "untimed_replays_between_timed_steps": pad,
                             "gpu_launches_in_timed_steps": launches},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_decode(a):
    """The decode-streaming workload: each step appends one key per (sequence,
    head), re-rotates and re-splits every cached key, and assigns the new keys
    (cosine blend, proxy query = the new key).  The cache (several GB) is far
    larger than L2, so nothing is flushed between steps.  `value` counts the
    cached keys each step processes (re-rotated and ranked); the new keys per
    second are reported beside it."""
    import query_aware_vq_gb300 as q
    from query_aware_vq_gb300.pipeline import A2ATSDecodeStep

    rank, local, world = _dist()
    torch.cuda.set_device(local)
    w = synth.WORKLOADS[a.workload]
    if a.batch > 0:
        w = synth.scaled(w, B=a.batch)
    total = min(a.warmup + a.steps, w.decode_steps)
    warm = min(a.warmup, max(total - 1, 0))
    steps = total - warm
    lens0 = synth.decode_lengths(w)
    keys = synth.keys(synth.scaled(w, N=int(lens0.max())))
    cache = torch.zeros((w.B, w.H, w.N, w.d), dtype=synth.DTYPES[w.dtype], device="cuda")
    cache[:, :, :keys.shape[2]] = keys.cuda()
    del keys
    lengths = torch.from_numpy(lens0).cuda()
    cb = synth.codebook(w).cuda()
    new = [synth.decode_new_keys(w, s) for s in range(total)]
    new_d = [t.cuda() for t in new]
    step = A2ATSDecodeStep(w.B, w.H, w.N, w.d, w.K, synth.DTYPES[w.dtype], window=w.W,
                           fraction=w.fraction, rope_base=w.rope_base, beta=w.betas[0])
    stream = torch.cuda.current_stream()
    # the codebook side (decoded centroids and norms) is built by the first
    # step and reused by the others, as for the default workload
    for s in range(warm):
        step(cache, lengths, new_d[s], cb, reuse_codebook=s > 0)
    torch.cuda.synchronize()
    cached = [int(lengths.sum()) + w.B * (i + 1) for i in range(steps)]  # after each append
    events, step_ev = {}, []
    clocks = Clocks(local)
    clocks.start()
    _barrier(world)
    torch.cuda.synchronize()
    launches0 = q.kernel_launches()
    for i in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step(cache, lengths, new_d[warm + i], cb, events=events, reuse_codebook=warm + i > 0)
        e1.record(stream)
        step_ev.append((e0, e1))
    torch.cuda.synchronize()
    _barrier(world)
    launches = q.kernel_launches() - launches0
    clk = clocks.stop()
    ms = _max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in step_ev) / steps, world)
    keys_per_step = w.H * sum(cached) / steps
    value = world * keys_per_step / (ms * 1e-3)
    stage_ms = {k: sum(e0.elapsed_time(e1) for e0, e1 in v) / len(v) for k, v in events.items()}
    hbm, _, src = _peaks()
    s_el = {"f32": 4, "bf16": 2, "f16": 2}[w.dtype]
    amount = keys_per_step * (2.0 * w.d * s_el + 12.0)
    achieved = amount / (stage_ms["rope_and_split"] * 1e-3) / 1e9
    roof = {"kernel": "cosine_score_kernel + select_kernel (re-rotation and split of the cache)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
            "frac": round(achieved / hbm, 5), "traffic": None,
            "bytes_per_step": amount, "peak_source": f"{src} (hbm_gbs)"}
    # end to end: the new keys from pinned host memory, their codes back
    e2e = None
    if not a.no_e2e:
        hnew = [t.pin_memory() for t in new[warm:]]
        out = torch.empty((w.B, w.H), dtype=torch.int32).pin_memory()
        staged = torch.empty_like(new_d[0])
        e2e_ms = []
        room = w.N - int(lengths.max())
        n_e2e = min(steps, room)
        e2e_warm = min(3, max(n_e2e - 1, 0))
        for i in range(n_e2e):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            staged.copy_(hnew[i], non_blocking=True)
            step(cache, lengths, staged, cb, reuse_codebook=True)
            idx = (lengths.long() - 1).view(w.B, 1, 1).expand(w.B, w.H, 1)
            out.copy_(step.codes.gather(2, idx).squeeze(2), non_blocking=True)
            e1.record(stream)
            e1.synchronize()
            if i >= e2e_warm:
                e2e_ms.append(e0.elapsed_time(e1))
        if e2e_ms:
            em = _max_over_ranks(sum(e2e_ms) / len(e2e_ms), world)
            e2e = {"value": world * keys_per_step / (em * 1e-3), "unit": "keys/s",
                   "ms_per_step": round(em, 4),
                   "h2d_bytes_per_step": staged.numel() * staged.element_size(),
                   "d2h_bytes_per_step": out.numel() * out.element_size()}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "keys/s", "n_gpus": world,
            "steps": steps, "warmup": warm, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; correlated-Gaussian keys with outlier channels; no model "
                    "weights)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "Ncap": w.N, "d": w.d, "K": w.K,
                       "window": w.W, "fraction": w.fraction, "beta": w.betas[0],
                       "storage": w.dtype, "l2": "inputs larger than L2 (no flush)",
                       "value_counts": "cached keys re-rotated and ranked per second",
                       "new_keys_per_s": world * w.B * w.H / (ms * 1e-3),
                       "parallelism": f"replicas x{world} (independent batches)"},
            "roofline": roof,
            "stages": {k: {"ms": round(v, 4)} for k, v in stage_ms.items()},
            "cpu_baseline": None, "clocks": clk, "e2e": e2e, "gpu_launches": launches,
        }
        print(json.dumps(line), flush=True)


def _oracle_sample(w, keys, cb, queries, hg, rows: int, h: int, nthreads=None):
    """One bounded sample of the workload on the oracle: the first `rows`
    keys of head h (as a sequence of that length) through the whole step,
    on nthreads host threads (None: the oracle's default)."""
    import oracle
    n = min(rows, w.N)
    k = keys[0, h, :n]
    L = None
    if queries is not None:
        hm = oracle.query_second_moment(queries[h], w.ridge)
        L, _ = oracle.cholesky(hm.astype(np.float32).astype(np.float64))
    elif hg is not None:
        L, _ = oracle.cholesky(hg[h].double().numpy())
    t0 = time.perf_counter()
    oracle.pipeline_step(k, n - 1, cb[h], w.W, w.far_offset, w.rope_base, w.fraction, l=L,
                         beta=w.betas[-1], nthreads=nthreads)
    return n, time.perf_counter() - t0


def cpu_baseline(w, keys, cb, queries, hg, rows: int = 8192, reps: int = 2):
    n_done, t = 0, 0.0
    for r in range(reps):
        n, dt = _oracle_sample(w, keys, cb, queries, hg, rows, r % w.H)
        n_done += n
        t += dt
    import oracle
    n1, t1 = _oracle_sample(w, keys, cb, queries, hg, rows // 4, 0, nthreads=1)
    return {"value": n_done / t, "unit": "keys/s", "cores": oracle.default_threads(),
            "kind": "oracle",
            "sample": f"{reps} x the first {rows} keys of one head as a whole sequence "
                      f"(all stages; calibration of L excluded from the time), fp64 C",
            "single_thread": {"value": n1 / t1, "unit": "keys/s", "cores": 1,
                              "sample": f"the first {rows // 4} keys of head 0, one thread"}}


def run_reference(a):
    rank, local, world = _dist()
    if rank != 0:
        return
    w = synth.WORKLOADS[a.workload]
    keys, cb, queries, hg = _inputs(w, rank)
    rows = 4096
    for i in range(a.warmup):
        _oracle_sample(w, keys, cb, queries, hg, rows, i % w.H)
    t, n_done, per = 0.0, 0, []
    for i in range(a.steps):
        n, dt = _oracle_sample(w, keys, cb, queries, hg, rows, i % w.H)
        t += dt
        n_done += n
        per.append(dt)
    value = n_done / t
    import oracle
    line = {
        "metric": METRIC, "value": value, "unit": "keys/s", "impl": "reference",
        "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": round(1e3 * t / a.steps, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded, same generator)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "K": w.K},
        "cpu_baseline": {"value": value, "unit": "keys/s", "cores": oracle.default_threads(),
                         "kind": "oracle",
                         "sample": f"each step: the first {rows} keys of one head as a whole "
                                   "sequence through every stage, fp64 C oracle"},
        "e2e": {"value": value, "unit": "keys/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_attention(a):
    """The code-based attention scores of the decode query with every cached
    key (far keys through the codes the one-call step wrote, window keys
    exactly) and the top tokens by them, on the workload's keys; the newest
    key of each (b, h) is the query.  The codes are computed once, before
    the timed calls; L2 is flushed between calls."""
    import query_aware_vq_gb300 as q

    rank, local, world = _dist()
    torch.cuda.set_device(local)
    w = synth.WORKLOADS[a.workload]
    keys, cb, _, _ = _inputs(w, rank)
    kd, cd = keys.cuda(), cb.cuda()
    rope = dict(window=w.W, rope_base=w.rope_base)
    _, _, _, codes = q.a2ats_rope_split_plain_assign(kd, cd, None, w.fraction, rope=rope)
    qd = kd[:, :, -1, :].contiguous()
    lib = q.library()
    ws = torch.empty(lib.a2ats_code_attention_topk_workspace_size(w.B, w.H, w.N, w.d, w.K),
                     dtype=torch.uint8, device="cuda")
    scores = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device="cuda")
    perm = torch.empty((w.B, w.H, w.N), dtype=torch.int32, device="cuda")
    count = torch.empty((w.B, w.H), dtype=torch.int32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def call():
        q.a2ats_code_attention_topk(kd, codes, cd, qd, w.fraction, rope=rope, far_b=2048,
                                    scores=scores, perm=perm, count=count, workspace=ws)

    for _ in range(max(a.warmup, 3)):
        call()
        flush.zero_()
    torch.cuda.synchronize()
    launches0 = q.kernel_launches()
    evs = []
    clocks = Clocks(local)
    clocks.start()
    _barrier(world)
    torch.cuda.synchronize()
    for _ in range(a.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        evs.append((e0, e1))
        flush.zero_()
    torch.cuda.synchronize()
    _barrier(world)
    clk = clocks.stop()
    ms = _max_over_ranks(sum(x.elapsed_time(y) for x, y in evs) / a.steps, world)
    keys_per_call = w.B * w.H * w.N
    hbm, _, src = _peaks()
    # per key: its code read, its score written, read by the select, its
    # slot of perm written (the window keys' extra reads are left out)
    bytes_per_call = keys_per_call * 16.0
    achieved = bytes_per_call / (ms * 1e-3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "keys scored/sec (code-based attention scores + top tokens)",
            "value": world * keys_per_call / (ms * 1e-3), "unit": "keys/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; the workload's keys and codebook; no model weights)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "K": w.K,
                       "window": w.W, "far_b": 2048, "fraction": w.fraction,
                       "l2": "flushed between calls (256 MB write)"},
            "roofline": {"kernel": "query table + far-row gather + window rows + select",
                         "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm,
                         "unit": "GB/s", "frac": round(achieved / hbm, 4), "traffic": None,
                         "bytes_per_call": bytes_per_call,
                         "peak_source": f"{src} (hbm_gbs)"},
            "clocks": clk,
            "gpu_launches": int(round((q.kernel_launches() - launches0) / a.steps)) * a.steps,
        }), flush=True)


def run_dequantize(a):
    """The keys reconstructed from the codes the one-call step writes
    (codebook[h, code] per row), on the workload's cache; L2 flushed between
    calls.  HBM-bound: a 4-byte code read and a d-element row written per
    key (the codebook stays in L2)."""
    import query_aware_vq_gb300 as q

    rank, local, world = _dist()
    torch.cuda.set_device(local)
    w = synth.WORKLOADS[a.workload]
    keys, cb, _, _ = _inputs(w, rank)
    kd, cd = keys.cuda(), cb.cuda()
    rope = dict(window=w.W, rope_base=w.rope_base)
    _, _, _, codes = q.a2ats_rope_split_plain_assign(kd, cd, None, w.fraction, rope=rope)
    out = torch.empty_like(kd)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(a.warmup, 3)):
        q.a2ats_dequantize(codes, cd, out=out)
        flush.zero_()
    torch.cuda.synchronize()
    launches0 = q.kernel_launches()
    evs = []
    clocks = Clocks(local)
    clocks.start()
    _barrier(world)
    torch.cuda.synchronize()
    for _ in range(a.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        q.a2ats_dequantize(codes, cd, out=out)
        e1.record(stream)
        evs.append((e0, e1))
        flush.zero_()
    torch.cuda.synchronize()
    _barrier(world)
    clk = clocks.stop()
    ms = _max_over_ranks(sum(x.elapsed_time(y) for x, y in evs) / a.steps, world)
    keys_per_call = w.B * w.H * w.N
    esize = out.element_size()
    bytes_per_call = keys_per_call * (4.0 + w.d * esize)
    hbm, _, src = _peaks()
    achieved = bytes_per_call / (ms * 1e-3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "keys reconstructed/sec (dequantisation from codes)",
            "value": world * keys_per_call / (ms * 1e-3), "unit": "keys/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded; the workload's keys and codebook)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d, "K": w.K,
                       "l2": "flushed between calls (256 MB write)"},
            "roofline": {"kernel": "dequantize_kernel", "bound": "hbm",
                         "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4), "traffic": None,
                         "bytes_per_call": bytes_per_call, "peak_source": f"{src} (hbm_gbs)"},
            "clocks": clk,
            "gpu_launches": int(round((q.kernel_launches() - launches0) / a.steps)) * a.steps,
        }), flush=True)


def run_rope(a):
    """The windowed RoPE of every valid cached key on its own (API page,
    a2ats_windowed_rope; the per-step re-rotation of the deploy-preview
    page), 16-bit keys in and out.  HBM-bound: a row read and a row written
    per key.  The decode workload's cache (its lengths) is far larger than
    L2; smaller caches are flushed from L2 between calls."""
    import query_aware_vq_gb300 as q

    rank, local, world = _dist()
    torch.cuda.set_device(local)
    w = synth.WORKLOADS[a.workload]
    if a.batch > 0:
        w = synth.scaled(w, B=a.batch)
    if w.decode_steps:
        lens0 = synth.decode_lengths(w)
        keys = synth.keys(synth.scaled(w, N=int(lens0.max())))
        kd = torch.zeros((w.B, w.H, w.N, w.d), dtype=synth.DTYPES[w.dtype], device="cuda")
        kd[:, :, :keys.shape[2]] = keys.cuda()
        del keys
        lengths = torch.from_numpy(lens0).cuda()
        valid = w.H * int(lens0.sum())
    else:
        keys, _, _, _ = _inputs(w, rank)
        kd = keys.cuda()
        lengths = None
        valid = w.B * w.H * w.N
    out = torch.empty_like(kd)
    rope = dict(window=w.W, far_offset=w.far_offset, rope_base=w.rope_base)
    flush_needed = valid * w.d * kd.element_size() * 2 < 4 * L2_FLUSH_BYTES
    flush = torch.empty(L2_FLUSH_BYTES if flush_needed else 1, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(a.warmup, 3)):
        q.a2ats_windowed_rope(kd, lengths=lengths, out=out, **rope)
        flush.zero_()
    torch.cuda.synchronize()
    launches0 = q.kernel_launches()
    evs = []
    clocks = Clocks(local)
    clocks.start()
    _barrier(world)
    torch.cuda.synchronize()
    for _ in range(a.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        q.a2ats_windowed_rope(kd, lengths=lengths, out=out, **rope)
        e1.record(stream)
        evs.append((e0, e1))
        flush.zero_()
    torch.cuda.synchronize()
    _barrier(world)
    clk = clocks.stop()
    ms = _max_over_ranks(sum(x.elapsed_time(y) for x, y in evs) / a.steps, world)
    bytes_per_call = valid * w.d * (kd.element_size() + out.element_size())
    hbm, _, src = _peaks()
    achieved = bytes_per_call / (ms * 1e-3) / 1e9
    if rank == 0:
        print(json.dumps({
            "metric": "keys rotated/sec (windowed RoPE of the cache)",
            "value": world * valid / (ms * 1e-3), "unit": "keys/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded; the workload's keys)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "window": w.W, "valid_keys": valid,
                       "l2": "flushed between calls (256 MB write)" if flush_needed
                             else "inputs larger than L2 (no flush)"},
            "roofline": {"kernel": "windowed_rope_bh_kernel", "bound": "hbm",
                         "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                         "frac": round(achieved / hbm, 4), "traffic": None,
                         "bytes_per_call": bytes_per_call, "peak_source": f"{src} (hbm_gbs)"},
            "clocks": clk,
            "gpu_launches": int(round((q.kernel_launches() - launches0) / a.steps)) * a.steps,
        }), flush=True)


def run_hweighted(a):
    """The H-weighted rule (API page, a2ats_h_weighted_assignment, Eq. 14-18)
    over every key of the workload's cache, with L from the workload's own
    calibration and the windowed RoPE fused: every key outside the window
    goes through the tensor-core pass over the stored keys against the
    three 16-bit planes of c L L^T (exact products), the window rows through
    the two-plane compact pass, the rows the bound cannot certify through the
    exact path.  L2 flushed between calls.  The roofline is that of the pass
    over the stored keys, from the library's CUDA events on its stream, at
    2 d K + 2 d^2 algorithmic flops per key (z = k L and the distances)."""
    import query_aware_vq_gb300 as q

    rank, local, world = _dist()
    torch.cuda.set_device(local)
    w = synth.WORKLOADS[a.workload]
    keys, cb, queries, hg = _inputs(w, rank)
    kd, cd = keys.cuda(), cb.cuda()
    if hg is not None:
        hm = hg.cuda()
    else:
        qd = queries.cuda() if queries is not None else None
        if qd is None:
            raise SystemExit("the workload has no calibration queries or H")
        hm = q.a2ats_query_second_moment(qd, w.ridge)
    L, info = q.a2ats_cholesky_factor(hm)
    torch.cuda.synchronize()
    if int(info.max()) != 0:
        raise SystemExit("H is not positive definite")
    rope = dict(window=w.W, far_offset=w.far_offset, rope_base=w.rope_base)
    lib = q.library()
    B, H, N, d, K = w.B, w.H, w.N, w.d, w.K
    ws = torch.empty(lib.a2ats_h_weighted_assign_workspace_size(B, H, N, d, K),
                     dtype=torch.uint8, device="cuda")
    codes = torch.empty((B, H, N), dtype=torch.int32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for i in range(max(a.warmup, 3)):
        q.a2ats_h_weighted_assign(kd, cd, L, rope=rope, codes=codes, workspace=ws, reuse=i > 0)
        flush.zero_()
    torch.cuda.synchronize()
    launches0 = q.kernel_launches()
    q.set_kernel_timing(True)
    q.timed_kernels_ms()
    evs = []
    clocks = Clocks(local)
    clocks.start()
    _barrier(world)
    torch.cuda.synchronize()
    for _ in range(a.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        q.a2ats_h_weighted_assign(kd, cd, L, rope=rope, codes=codes, workspace=ws, reuse=True)
        e1.record(stream)
        evs.append((e0, e1))
        flush.zero_()
    torch.cuda.synchronize()
    _barrier(world)
    clk = clocks.stop()
    tc_ms, tc_launches = q.timed_kernels_ms()
    q.set_kernel_timing(False)
    ms = _max_over_ranks(sum(x.elapsed_time(y) for x, y in evs) / a.steps, world)
    keys_per_call = B * H * N
    far_rows = B * H * max(N - max(w.W, 0), 0)
    flop = far_rows * (2.0 * d * K + 2.0 * d * d)
    per_launch = tc_ms / max(tc_launches, 1)
    achieved = flop / (per_launch * 1e-3) / 1e12
    _, bf16, src = _peaks()
    if rank == 0:
        print(json.dumps({
            "metric": "keys assigned/sec (windowed RoPE + H-weighted VQ argmin, every key)",
            "value": world * keys_per_call / (ms * 1e-3), "unit": "keys/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; the workload's keys, codebook and calibration)",
            "config": {"workload": w.name, "B": B, "H": H, "N": N, "d": d, "K": K,
                       "window": w.W, "rows": "all", "storage": w.dtype,
                       "codebook_side": "built by the first call, reused",
                       "l2": "flushed between calls (256 MB write)"},
            "roofline": {"kernel": "assign_tc_kernel (stored-order pass, H-weighted planes)",
                         "bound": "tensor", "achieved": round(achieved, 3), "peak": bf16,
                         "unit": "TFLOP/s", "frac": round(achieved / bf16, 5), "traffic": None,
                         "flop_per_launch": flop, "ms_per_launch": round(per_launch, 5),
                         "launches": tc_launches, "peak_source": f"{src} (bf16_tflops, burst)"},
            "clocks": clk,
            "gpu_launches": int(round((q.kernel_launches() - launches0) / a.steps)) * a.steps,
        }), flush=True)


def run_subvector(a):
    """The pages' wrapper defaults on the workload's cache: sub-vector VQ at
    sub_dim = 8 with 2^8 centroids for keys (H-weighted retrieval tokens,
    8 x 8 factor) and values (plain); L2 flushed between steps."""
    import query_aware_vq_gb300 as q
    from query_aware_vq_gb300.pipeline import A2ATSSubvectorStep

    rank, local, world = _dist()
    torch.cuda.set_device(local)
    w = synth.WORKLOADS[a.workload]
    s, K = 8, 256
    keys, _, _, _ = _inputs(w, rank)
    kd = keys.cuda()
    vd = synth.gaussian((w.B, w.H, w.N, w.d), seed=7000 + rank, dtype="f32").cuda()
    ck = synth.gaussian((w.H, K, s), seed=7100, dtype="f32").cuda()
    cv = synth.gaussian((w.H, K, s), seed=7200, dtype="f32").cuda()
    Qd = synth.gaussian((w.H, 8192, s), seed=7300, dtype="f32").cuda()
    L, _ = q.a2ats_cholesky_factor(q.a2ats_query_second_moment(Qd, 1e-4))
    step = A2ATSSubvectorStep(w.B, w.H, w.N, w.d, s, K, synth.DTYPES[w.dtype], window=w.W,
                              fraction=w.fraction, rope_base=w.rope_base,
                              dedicated=not a.subvector_composed)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(a.warmup, 3)):
        step(kd, vd, ck, cv, L)
        flush.zero_()
    torch.cuda.synchronize()
    launches0 = q.kernel_launches()
    evs = []
    clocks = Clocks(local)
    clocks.start()
    _barrier(world)
    torch.cuda.synchronize()
    for _ in range(a.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step(kd, vd, ck, cv, L)
        e1.record(stream)
        evs.append((e0, e1))
        flush.zero_()
    torch.cuda.synchronize()
    _barrier(world)
    clk = clocks.stop()
    ms = _max_over_ranks(sum(x.elapsed_time(y) for x, y in evs) / a.steps, world)
    keys_per_step = w.B * w.H * w.N
    if rank == 0:
        print(json.dumps({
            "metric": "tokens quantised/sec (sub-vector VQ of keys and values)",
            "value": world * keys_per_step / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded; the workload's keys, Gaussian values and tables)",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "sub_dim": s, "K": K, "window": w.W, "fraction": w.fraction,
                       "assignment": "composed calls" if a.subvector_composed
                       else "sub-vector kernel",
                       "l2": "flushed between steps (256 MB write)"},
            "clocks": clk,
            "gpu_launches": int(round((q.kernel_launches() - launches0) / a.steps)) * a.steps,
        }), flush=True)


def run_calibrate(a):
    """One layer's codebook calibration in Cholesky space: H from the
    workload's calibration queries, L = chol(H), z = k L for the calibration
    keys, k-means++ seeding and Lloyd rounds on z, and the codebook back in
    key space.  Inputs resident; L2 flushed between calibrations."""
    import query_aware_vq_gb300 as q

    rank, local, world = _dist()
    torch.cuda.set_device(local)
    w = synth.scaled(synth.WORKLOADS[a.workload], N=a.calib_tokens)
    keys = synth.keys(w, batch_offset=rank * w.B)[0].cuda()  # [H, n, d]
    Qd = synth.queries(w).cuda()
    u = torch.from_numpy(np.random.default_rng(5000 + rank).random((w.H, w.K))).cuda()
    H_, n, d = keys.shape
    z = torch.empty((H_, n, d), dtype=torch.float32, device="cuda")
    cz = torch.empty((H_, w.K, d), dtype=torch.float32, device="cuda")
    c = torch.empty_like(cz)
    codes = torch.empty((H_, n), dtype=torch.int32, device="cuda")
    obj = torch.empty((H_, a.lloyd + 1), dtype=torch.float64, device="cuda")

    def calibrate():
        hm = q.a2ats_query_second_moment(Qd, w.ridge)
        L, _ = q.a2ats_cholesky_factor(hm)
        q.a2ats_cholesky_rows(keys, L, out=z)
        q.a2ats_kmeanspp(z, w.K, u, a.lloyd, centroids=cz, codes=codes, objective=obj)
        q.a2ats_cholesky_solve_rows(cz, L, out=c)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    for _ in range(max(a.warmup, 3)):
        calibrate()
        flush.zero_()
    torch.cuda.synchronize()
    launches0 = q.kernel_launches()
    evs = []
    clocks = Clocks(local)
    clocks.start()
    _barrier(world)
    torch.cuda.synchronize()
    for _ in range(a.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        calibrate()
        e1.record(stream)
        evs.append((e0, e1))
        flush.zero_()
    torch.cuda.synchronize()
    _barrier(world)
    clk = clocks.stop()
    ms = _max_over_ranks(sum(x.elapsed_time(y) for x, y in evs) / a.steps, world)
    if rank == 0:
        print(json.dumps({
            "metric": "codebook calibrations/sec (one layer: H, L, z = k L, k-means++, "
                      "Lloyd rounds, key-space codebook)",
            "value": world / (ms * 1e-3), "unit": "layers/s", "n_gpus": world,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32+f64",
            "data": "synthetic (seeded; the workload's keys and queries, uniform draws)",
            "config": {"workload": w.name, "H": w.H, "tokens": n, "d": d, "K": w.K,
                       "M": w.M, "lloyd_rounds": a.lloyd,
                       "l2": "flushed between calibrations (256 MB write)"},
            "objective_last": float(obj[:, -1].sum().item()),
            "clocks": clk,
            "gpu_launches": int(round((q.kernel_launches() - launches0) / a.steps)) * a.steps,
        }), flush=True)


if __name__ == "__main__":
    args = _args()
    if args.impl == "reference":
        run_reference(args)
    elif args.path == "hweighted":
        run_hweighted(args)
    elif args.path == "attention":
        run_attention(args)
    elif args.path == "dequantize":
        run_dequantize(args)
    elif args.path == "subvector":
        run_subvector(args)
    elif args.path == "calibrate":
        run_calibrate(args)
    elif args.path == "rope":
        run_rope(args)
    elif synth.WORKLOADS[args.workload].decode_steps:
        run_decode(args)
    else:
        run_ours(args)
