#!/usr/bin/env python
"""Benchmark of the Skip-Softmax (BLASST) attention forward on GB300.

One step = one call of ``blasst_attn_fwd`` (the whole hot path: Q K^T for every
tile pair, the per-tile skip test, softmax and P V for kept tiles, epilogue) on
the Wan-shaped self-attention workload: B=1, H=40, Sq=Sk=32760 (a 21 x 30 x 52
latent grid, cells 3 x 6 x 6), d=128, bf16, seeded synthetic clustered inputs.

The JSON line reports dense-equivalent TFLOPS (4 B H Sq Sk d / time) at the
headline factor, with ms/call, the skip fraction and executed TFLOPS for every
factor of the workload's sweep, the tensor-core roofline of the kernel, the
end-to-end number through the C ABI with host buffers, and the CPU oracle's
throughput on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--factor F]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "ms/call and dense-equiv TFLOPS vs skip fraction, bf16 d=128, S=32760, 1×GB300"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one headline launch, from an
# ncu capture (see profiles/), keyed by a hash of the kernel sources it was taken on: a
# kernel that has changed since reports null.
KERNEL_SOURCES = ["softmax_threshold_tile_gb300/csrc/blasst_fwd.cu", "softmax_threshold_tile_gb300/csrc/sm103_ptx.cuh"]
NCU_TRAFFIC = {
    "265a36ec00c0eed3": {"workload": "wan_32760", "factor": 32.0, "bytes": 1008250112 + 322755328},
    "f126bb95c3f763e9": {"workload": "wan_32760", "factor": 32.0, "bytes": 1007854848 + 322692096},
    "d55dd674df77d3f0": {"workload": "wan_32760", "factor": 32.0, "bytes": 1008416512 + 322506496},
    "2fc024e7b09c30be": {"workload": "wan_32760", "factor": 32.0, "bytes": 1007930880 + 320723200},
}
UNIT = "TFLOPS (dense-equivalent)"
TILE = 128


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="wan_32760", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--factor", type=float, default=None, help="headline factor (default: largest of the sweep)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--heads-per-group", type=int, default=0,
                    help="largest head group of the end-to-end host-buffer call (0: H / 5)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the max_prob, packed-document and FP8 timings")
    ap.add_argument("--cpu-units", type=int, default=48, help="query tiles in the CPU oracle sample")
    return ap.parse_args()


def workload_factors(w):
    if w.curve is not None:
        a, b, ts = w.curve
        return [0.0] + [a * math.exp(b * t) for t in ts]
    return list(w.factors)


def dense_flops(w):
    return 4.0 * w.B * w.H * w.S * w.S * w.d


def executed_flops(w, mask):
    """2 r c d per QK^T tile pair, plus the same for P V on kept pairs (r, c = valid rows / keys)."""
    nQ, nK = mask.shape[-2], mask.shape[-1]
    r = np.minimum(TILE, w.S - TILE * np.arange(nQ)).astype(np.float64)
    c = np.minimum(TILE, w.S - TILE * np.arange(nK)).astype(np.float64)
    rc = np.outer(r, c)
    kept = 1.0 - mask.reshape(-1, nQ, nK).astype(np.float64)
    return float((2.0 * w.d * rc[None] * (1.0 + kept)).sum())


def sample_units(w, n):
    """The first query tiles of the first and last head (batch 0): a bounded CPU sample."""
    per_head = max(1, n // 2)
    heads = (0, w.H - 1) if w.H > 1 else (0,)
    nQ = -(-w.S // TILE)
    return np.array([(0, h, t) for h in heads for t in range(min(per_head, nQ))], dtype=np.int32)


def kernel_source_hash():
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, factor):
    rec = NCU_TRAFFIC.get(kernel_source_hash())
    if rec and rec["workload"] == workload and rec["factor"] == factor:
        return rec["bytes"]
    return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "of measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 1700.0, "of fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(backend: str = "nccl"):
    """(world, rank, local_rank) from the torchrun environment; one process per GPU."""
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cuda"):
    """The largest per-rank value (the job's time is the slowest rank's)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms_max: float) -> float:
    """Weak scaling: every rank processes units_per_rank in its own time; the job's rate is all
    ranks' units over the slowest rank's time (per second)."""
    return world * units_per_rank / (ms_max * 1e-3)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the CPU baseline."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def cpu_oracle_rate(w, q, k, v, factor, n_units, threads, units=None):
    """Dense-equivalent TFLOPS of the CPU oracle on a bounded sample of query tiles (all query
    tiles of the workload when `units` is "all")."""
    import oracle
    if units is None:
        units = sample_units(w, n_units)
    elif isinstance(units, str):
        units = oracle.all_units(w.B, w.H, w.S)
    scale = 1.0 / math.sqrt(w.d)
    t0 = time.perf_counter()
    oracle.skip_softmax_attn(q, k, v, scale, factor, units=units, threads=threads)
    dt = time.perf_counter() - t0
    flops = sum(4.0 * min(TILE, w.S - TILE * int(t)) * w.S * w.d for _, _, t in units)
    return flops / dt / 1e12, dt, units


def run_reference(args, w):
    """The reference arm: the CPU oracle, as it stands, timed on the host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    q, k, v = synth.make_qkv(w)
    factor = args.factor if args.factor is not None else max(workload_factors(w))
    threads = os.cpu_count() or 1
    n_units = max(1, min(threads, 8))
    units = sample_units(w, n_units)
    scale = 1.0 / math.sqrt(w.d)
    for _ in range(args.warmup):
        oracle.skip_softmax_attn(q, k, v, scale, factor, units=units[:1], threads=1)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.skip_softmax_attn(q, k, v, scale, factor, units=units, threads=threads)
        times.append(time.perf_counter() - t0)
    flops = sum(4.0 * min(TILE, w.S - TILE * int(t)) * w.S * w.d for _, _, t in units)
    value = flops * args.steps / sum(times) / 1e12
    sample = (f"{len(units)} query tiles of {w.name} (batch 0, heads 0 and {w.H - 1}, first tiles) "
              f"per step at factor {factor:g}, fp64 scalar C oracle; rate extrapolated to the whole "
              f"call from {len(units)} of {w.B * w.H * (-(-w.S // TILE))} query tiles")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded clustered video-DiT token grid)",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "S": w.S, "d": w.d, "factor": factor,
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "cpu_model": cpu_model(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def time_calls(blasst, stream, args_fn, n):
    import torch
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(n):
            args_fn()
        end.record(stream)
    end.synchronize()
    return start.elapsed_time(end) / n  # ms per call


def run_ours(args, w):
    import torch

    import softmax_threshold_tile_gb300 as blasst

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    blasst.build_library()
    blasst.load_library()
    factors = workload_factors(w)
    head_factor = args.factor if args.factor is not None else max(factors)

    q, k, v = synth.make_qkv(w)
    qd, kd, vd = (torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16) for x in (q, k, v))
    B, S, H, d = w.B, w.S, w.H, w.d
    nQ = -(-S // TILE)
    od = torch.empty_like(qd)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    counts = torch.empty((B * H,), dtype=torch.int32, device="cuda")
    mask = torch.empty((B, H, nQ, nQ), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    scale = 1.0 / math.sqrt(d)

    def call(f, with_mask=False):
        st = blasst.blasst_attn_fwd(qd, kd, vd, od, lse, B, H, S, S, d, scale, f, stream.cuda_stream,
                                    counts, mask if with_mask else None)
        if st != blasst.BLASST_OK:
            raise blasst.BlasstError(st, "blasst_attn_fwd")

    def mask_of(f):
        with torch.cuda.stream(stream):
            call(f, True)
        stream.synchronize()
        return mask.cpu().numpy()

    peak_burst, _, peak_src = measured_peaks()
    dense = dense_flops(w)

    # ---- factor sweep (ms/call and TFLOPS vs skip fraction); not the contract's timed region
    sweep = []
    if not args.no_sweep:
        n_sweep = max(3, args.steps // 2)
        for f in factors:
            m = mask_of(f)
            for _ in range(args.warmup):
                call(f)
            ms = time_calls(blasst, stream, lambda: call(f), n_sweep)
            skip = float(m.mean())
            ex = executed_flops(w, m)
            entry = {"factor": f, "lambda": f / S, "skip_fraction": skip, "ms": ms,
                     "exec_tflops": ex / ms / 1e9, "dense_equiv_tflops": dense / ms / 1e9,
                     "tensor_frac": ex / ms / 1e9 / peak_burst}
            if B > 1:
                entry["skip_fraction_per_batch"] = [round(float(x), 4) for x in m.reshape(B, -1).mean(1)]
            if w.gamma_range is not None:  # per-head structure: report the spread over heads
                per_head = m.reshape(B, H, -1).mean(2).ravel()
                entry["skip_fraction_per_head"] = {"min": float(per_head.min()), "median": float(np.median(per_head)),
                                                   "max": float(per_head.max())}
            sweep.append(entry)
        base = next((s["ms"] for s in sweep if s["factor"] == 0.0), None)
        for s in sweep:
            s["speedup_vs_dense"] = base / s["ms"] if base else None
            s["bound"] = 1.0 / (1.0 - s["skip_fraction"] / 2.0)

    # ---- the extended entry point: max_prob overhead and packed documents (not the timed region)
    extras = None
    if not args.no_extras and w.B == 1:
        n_x = max(3, args.steps // 2)
        mp = torch.empty((B, H, S), dtype=torch.float32, device="cuda")

        def call_mp(f):
            st = blasst.blasst_attn_fwd_ex(qd, kd, vd, od, lse, mp, B, H, S, S, d, scale, f, stream.cuda_stream,
                                           counts, None)
            if st != blasst.BLASST_OK:
                raise blasst.BlasstError(st, "blasst_attn_fwd_ex")

        for _ in range(args.warmup):
            call_mp(head_factor)
        ms_mp = time_calls(blasst, stream, lambda: call_mp(head_factor), n_x)
        ms_plain = time_calls(blasst, stream, lambda: call(head_factor), n_x)
        # Packed documents: the same tokens cut into documents of decreasing length, each
        # attending to itself (lambda = factor / longest document).
        lens = [S // 2]
        while sum(lens) + lens[-1] // 2 < S and lens[-1] >= 2048:
            lens.append(lens[-1] // 2)
        lens.append(S - sum(lens))
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device="cuda")
        q3, k3, v3, o3 = (t.view(S, H, d) for t in (qd, kd, vd, od))
        lse3 = torch.empty((H, S), dtype=torch.float32, device="cuda")
        cnt3 = torch.empty((len(lens) * H,), dtype=torch.int32, device="cuda")

        def call_varlen(f):
            st = blasst.blasst_attn_fwd_ex(q3, k3, v3, o3, lse3, None, len(lens), H, S, S, d, scale, f,
                                           stream.cuda_stream, cnt3, None, cu, cu, max(lens), max(lens))
            if st != blasst.BLASST_OK:
                raise blasst.BlasstError(st, "blasst_attn_fwd_ex")

        vl = {"doc_lengths": lens}
        packed_dense = 4.0 * H * d * sum(L * L for L in lens)
        for f in (0.0, head_factor):
            for _ in range(args.warmup):
                call_varlen(f)
            ms_v = time_calls(blasst, stream, lambda: call_varlen(f), n_x)
            stream.synchronize()
            skipped = int(cnt3.sum().item())
            pairs = sum((-(-L // TILE)) ** 2 for L in lens) * H
            vl[f"factor_{f:g}"] = {"ms": ms_v, "dense_equiv_tflops": packed_dense / ms_v / 1e9,
                                   "skip_fraction": skipped / pairs}
        # FP8 score product: per-tensor e4m3 q / k (quantised on the device by torch: input
        # preparation only), v and P . V in bf16.
        fp8 = None
        if hasattr(torch, "float8_e4m3fn"):
            dq = float(qd.float().abs().max()) / 448.0
            dk = float(kd.float().abs().max()) / 448.0
            q8 = (qd.float() / dq).to(torch.float8_e4m3fn)
            k8 = (kd.float() / dk).to(torch.float8_e4m3fn)

            def call_fp8(f):
                st = blasst.blasst_attn_fwd_ex(q8, k8, vd, od, lse, None, B, H, S, S, d, scale, f,
                                               stream.cuda_stream, counts, None, qk_format=blasst.BLASST_QK_E4M3,
                                               q_descale=dq, k_descale=dk)
                if st != blasst.BLASST_OK:
                    raise blasst.BlasstError(st, "blasst_attn_fwd_ex")

            fp8 = {}
            for f in (0.0, head_factor):
                for _ in range(args.warmup):
                    call_fp8(f)
                ms_8 = time_calls(blasst, stream, lambda: call_fp8(f), n_x)
                stream.synchronize()
                fp8[f"factor_{f:g}"] = {"ms": ms_8, "dense_equiv_tflops": dense / ms_8 / 1e9,
                                        "skip_fraction": int(counts.sum().item()) / (B * H * nQ * nQ)}
            del q8, k8
        extras = {"max_prob": {"ms_with": ms_mp, "ms_without": ms_plain, "overhead": ms_mp / ms_plain - 1.0,
                               "factor": head_factor},
                  "varlen": vl, "fp8_qk": fp8}

    # ---- the timed region: K calls at the headline factor
    m = mask_of(head_factor)
    skip = float(m.mean())
    ex = executed_flops(w, m)
    for _ in range(args.warmup):
        call(head_factor)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        start.record(stream)
        for _ in range(args.steps):
            call(head_factor)
        end.record(stream)
        end.synchronize()
    torch.cuda.synchronize()
    barrier(world)
    ms_local = start.elapsed_time(end) / args.steps
    ms = max_over_ranks(ms_local, world)
    # host cost of one call (argument checks, cached tensor descriptors, launch), enqueue only
    n_h = max(3, args.steps)
    t_h = time.perf_counter()
    for _ in range(n_h):
        call(head_factor)
    host_us = (time.perf_counter() - t_h) * 1e6 / n_h
    torch.cuda.synchronize()
    value = job_throughput(dense, world, ms) / 1e12
    achieved = ex / (ms_local * 1e-3) / 1e12

    # ---- end to end through the C ABI with host buffers (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e:
        # End to end through the host-buffer C entry point: pinned host q / k / v in, host o / lse
        # out, the copies overlapped with the kernels by head group inside the call.
        qh, kh, vh = (torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).pin_memory() for x in (q, k, v))
        oh = torch.empty(od.shape, dtype=torch.bfloat16).pin_memory()
        lh = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
        hpg = args.heads_per_group or max(1, H // 5)
        ws_bytes = blasst.blasst_host_workspace_bytes(B, H, S, S, hpg)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        n_e2e = max(3, min(args.steps, 10))

        def e2e_step():
            st = blasst.blasst_attn_fwd_host(qh, kh, vh, oh, lh, B, H, S, S, d, scale, head_factor, ws, ws_bytes,
                                             hpg, stream.cuda_stream)
            if st != blasst.BLASST_OK:
                raise blasst.BlasstError(st, "blasst_attn_fwd_host")

        e2e_step()
        stream.synchronize()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        stream.synchronize()
        e2e_ms = (time.perf_counter() - t0) * 1e3 / n_e2e
        e2e_ms = max_over_ranks(e2e_ms, world)
        h2d_bytes = int(3 * q.nbytes)
        d2h_bytes = int(oh.numel() * 2 + lh.numel() * 4)
        # Diagnosis (outside the timed steps): each step again on its own, followed by plain
        # contiguous copies of the same bytes in each direction, so that a step that ran slow can
        # be told apart as host-link bound (the probe copies slow too) or not.
        step_ms, h2d_gbs, d2h_gbs = [], [], []
        probe_in = torch.empty(h2d_bytes, dtype=torch.uint8, device="cuda")
        probe_src = torch.empty(h2d_bytes, dtype=torch.uint8).pin_memory()
        probe_out = torch.empty(d2h_bytes, dtype=torch.uint8).pin_memory()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        for _ in range(n_e2e):
            t1 = time.perf_counter()
            e2e_step()
            stream.synchronize()
            step_ms.append((time.perf_counter() - t1) * 1e3)
            with torch.cuda.stream(stream):
                ev[0].record(stream)
                probe_in.copy_(probe_src, non_blocking=True)
                ev[1].record(stream)
                probe_out.copy_(probe_in[:d2h_bytes], non_blocking=True)
                ev[2].record(stream)
            ev[2].synchronize()
            h2d_gbs.append(h2d_bytes / (ev[0].elapsed_time(ev[1]) * 1e-3) / 1e9)
            d2h_gbs.append(d2h_bytes / (ev[1].elapsed_time(ev[2]) * 1e-3) / 1e9)
        del probe_in, probe_src, probe_out
        e2e = {"value": job_throughput(dense, world, e2e_ms) / 1e12, "unit": UNIT, "ms_per_step": e2e_ms,
               "steps": n_e2e, "api": "blasst_attn_fwd_host", "heads_per_group": hpg,
               "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
               "diagnosis": {"step_ms": [round(x, 3) for x in step_ms],
                             "h2d_probe_gbs": [round(x, 1) for x in h2d_gbs],
                             "d2h_probe_gbs": [round(x, 1) for x in d2h_gbs],
                             "kernel_ms": ms_local,
                             "note": "each step re-run alone, then one contiguous pinned copy of the step's "
                                     "input bytes H2D and output bytes D2H (CUDA events)"}}
        del ws

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        threads = min(os.cpu_count() or 1, args.cpu_units)
        n_all = w.B * w.H * nQ
        rate, dt, units = cpu_oracle_rate(w, q, k, v, head_factor, args.cpu_units, threads)
        # the same oracle on one core, on a smaller sample (query tiles are independent, so the
        # rate does not depend on the sample's size)
        n1 = max(1, min(4, args.cpu_units))
        rate1, dt1, units1 = cpu_oracle_rate(w, q, k, v, head_factor, n1, 1)
        # and on one core over a whole call of the smallest workload (every query tile)
        wt = synth.WORKLOADS["tiny_1024"]
        qt_, kt_, vt_ = synth.make_qkv(wt)
        ft = max(workload_factors(wt))
        rate_t, dt_t, units_t = cpu_oracle_rate(wt, qt_, kt_, vt_, ft, 0, 1, units="all")
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "cpu_model": cpu_model(), "kind": "oracle",
               "sample": f"{len(units)} query tiles (batch 0, heads 0 and {w.H - 1}, first tiles) of "
                         f"{w.name} at factor {head_factor:g}, {threads} threads; {dt:.1f} s wall; rate "
                         f"extrapolated to the whole call from {len(units)} of {n_all} query tiles",
               "single_core": {"value": rate1, "unit": UNIT, "cores": 1,
                               "sample": f"{len(units1)} query tiles of the same sample; {dt1:.1f} s wall; "
                                         f"extrapolated from {len(units1)} of {n_all} query tiles"},
               "single_core_full_call": {"value": rate_t, "unit": UNIT, "cores": 1, "workload": wt.name,
                                         "factor": ft, "s": dt_t,
                                         "sample": f"the whole {wt.name} call ({len(units_t)} query tiles), "
                                                   f"not extrapolated"}}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded clustered video-DiT token grid; replicas per GPU)",
            "config": {"workload": w.name, "B": B, "H": H, "S": S, "d": d, "factor": head_factor,
                       "lambda": head_factor / S, "skip_fraction": skip,
                       "exec_tflops": achieved,
                       "l2": f"inputs {3 * q.nbytes / 1e9:.2f} GB > 129 MB L2; no flush"},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                         "frac": achieved / peak_burst, "traffic": ncu_traffic(w.name, head_factor),
                         "algorithmic_bytes": 4 * B * H * S * d * 2 + 4 * B * H * S,
                         "kernel": "blasst_fwd_sm103a", "peak_source": f"bf16 burst {peak_src}"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "host_enqueue_us_per_call": host_us,
            "clocks": clocks.summary(),
            "sweep": sweep,
            "extras": extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def main():
    args = parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
