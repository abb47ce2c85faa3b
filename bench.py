#!/usr/bin/env python3
"""Benchmark: THD causal attention TFLOPS, forward and forward+backward, on GB300.

One step = one pass of the whole hot path over one synthetic packed batch:
metadata validation + pad detection + per-rank partition + schedule (one
planner launch), the fused ring-decomposed forward (thd_attn_fwd), and the
backward (thd_attn_bwd: the planner, the Delta preprocess, the
query-stationary dQ kernel, the key-stationary dK/dV kernel).  Inputs are resident in HBM before the timed
region; L2 is flushed (256 MiB write) between timed steps, outside the
events.  Each step is timed with CUDA events on the launching stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config packed]
    python bench.py --impl reference ...   # the CPU fp64 oracle on host cores
    python bench.py --a2a 4 ...            # the same step through the emulated Ulysses layer (cp 4);
                                           # --a2a 2: hierarchical a2a+p2p sizes [2, 2]
    python bench.py --hbm-kernels          # LSE merge, tail-zero and A2A move vs the HBM copy peak

Under torchrun each rank runs its own replica of the workload (weak scaling,
no collective on the data path); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "THD causal attn TFLOPS fwd & fwd+bwd, 1 GB300; % of BF16 tensor peak"
UNIT = "TFLOPS"


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default="packed", help="tiny|packed|padded|long|fwdbwd (or C1..C5)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fwd-only", action="store_true", help="time the forward alone as the step")
    ap.add_argument("--hbm-kernels", action="store_true",
                    help="time the HBM-bound kernels (LSE merge, gradient tail-zero, A2A move) against the copy peak")
    ap.add_argument("--a2a", type=int, default=0,
                    help="a2a group size: time the step through the emulated Ulysses (a2a = cp) or hierarchical "
                         "a2a+p2p layer (thd_attn_fwd_a2a / thd_attn_bwd_a2a on per-rank shards)")
    return ap.parse_args()


def _kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu capture of this kernel on
    this workload (profiles/traffic.txt), or None when there is none or the
    kernel's source changed since the counters were taken."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.txt")) as f:
            rec = json.load(f).get(kernel)
    except Exception:
        return None
    if not rec or rec.get("workload") != workload:
        return None
    cs = os.path.join(ROOT, "packed_sequence_context_gb300", "csrc")
    h = hashlib.sha256()
    for name in (kernel.split("_")[0] + ".cu", "common.cuh", "ptx.cuh"):
        with open(os.path.join(cs, name), "rb") as f:
            h.update(f.read())
    if h.hexdigest()[:16] != rec.get("source_sha"):
        return None
    return rec.get("bytes_per_launch")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), float(p["hbm_gbs"]), "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.index)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- CPU oracle leg
def _oracle_item(args):
    """One (sequence, head) fwd+bwd of the oracle; runs in a spawned worker."""
    q, k, v, do, scale = args
    from oracle import thd_oracle as orc
    import numpy as np
    L = q.shape[0]
    cu = np.array([0, L], np.int32)
    t0 = time.perf_counter()
    orc.attn_fwd(q, k, v, cu, cu, softmax_scale=scale)
    orc.attn_bwd(q, k, v, do, cu, cu, softmax_scale=scale)
    return time.perf_counter() - t0


def _oracle_items(w, t, heads):
    G = w.Hq // w.Hkv
    items = []
    for b in range(w.B):
        off = int(w.cu_seqlens_padded[b])
        L = w.lengths[b]
        if L == 0:
            continue
        for h in heads:
            sl = slice(off, off + L)
            items.append((t["q"][sl, h:h + 1].float().numpy(), t["k"][sl, h // G:h // G + 1].float().numpy(),
                          t["v"][sl, h // G:h // G + 1].float().numpy(), t["do"][sl, h:h + 1].float().numpy(),
                          w.softmax_scale))
    return items


def _sample_flops(w, heads):
    from packed_sequence_context_gb300 import inputs
    _, both = inputs.algorithmic_flops(w.lengths, 1, w.D)
    return both * len(heads)


def _spawn_pool(n):
    import multiprocessing as mp
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    return mp.get_context("spawn").Pool(n)


def cpu_baseline(w, t, target_s=15.0):
    """Time the oracle (as it stands) on a bounded sample of the workload:
    fwd+bwd of query heads 0, 1, 2, ... over every sequence, adding batches of
    heads until about `target_s` seconds of host time (or the whole workload)."""
    cores = os.cpu_count() or 1
    n_seq = max(1, sum(1 for L in w.lengths if L))
    per_batch = max(1, cores // n_seq)
    done, spent = 0, 0.0
    with _spawn_pool(cores) as pool:
        while done < w.Hq and spent < target_s:
            heads = list(range(done, min(w.Hq, done + per_batch)))
            items = _oracle_items(w, t, heads)
            t0 = time.perf_counter()
            pool.map(_oracle_item, items)
            spent += time.perf_counter() - t0
            done += len(heads)
    flops = _sample_flops(w, list(range(done)))
    scope = "all" if done == w.Hq else f"0..{done - 1} of {w.Hq}"
    return {"value": flops / spent / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd of query heads {scope} over all {w.B} sequences of the "
                      f"'{w.name}' workload ({spent:.1f} s, process pool of {cores}, one BLAS thread each)",
            "seconds": spent}


# ----------------------------------------------------------------- reference arm
def run_reference(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from packed_sequence_context_gb300 import inputs
    w = inputs.make_workload(a.config)
    t = inputs.make_tensors(w, with_grad=True)
    cores = os.cpu_count() or 1
    fwd_only = a.fwd_only
    with _spawn_pool(cores) as pool:
        times = []
        for i in range(a.warmup + a.steps):
            h = i % w.Hq
            items = _oracle_items(w, t, [h])
            t0 = time.perf_counter()
            pool.map(_oracle_item, items)
            dt = time.perf_counter() - t0
            if i >= a.warmup:
                times.append(dt)
    flops = _sample_flops(w, [0])
    mean = sum(times) / len(times)
    value = flops / mean / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sequences": w.B, "tokens": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                       "cp_size": w.cp_size, "causal": True, "step": "fwd+bwd" if not fwd_only else "fwd",
                       "sample": "one query head (rotating) over all sequences per step"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": "fp64 oracle fwd+bwd, one query head over all sequences per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- replicas
def slowest_rank_ms(ms: float, world: int, device) -> float:
    """The step time of the slowest replica: an all-reduce MAX of each rank's
    mean step time (the only collective of a run; none on the data path)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_tflops(step_flops: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank runs its own replica of the step, so
    the job does world x step_flops in the slowest rank's step time."""
    return step_flops * world / (ms_max * 1e-3) / 1e12


# ----------------------------------------------------------------- GPU arm
def run_ours(a):
    import torch
    import torch.distributed as dist

    from packed_sequence_context_gb300 import inputs
    from packed_sequence_context_gb300 import thd_attn as T

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    T.lib()
    peak, peak_sus, hbm, peak_kind = _peaks()

    w = inputs.make_workload(a.config)
    t = inputs.make_tensors(w, with_grad=True)
    # the CPU leg runs first, before this process touches the GPU with work
    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_baseline(w, t)

    dev = torch.device("cuda", local)
    q, k, v, do = (t[x].to(dev) for x in ("q", "k", "v", "do"))
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    cu_pad = torch.from_numpy(w.cu_seqlens_padded).to(dev)
    B, Tq = w.B, w.T
    o = torch.empty_like(q)
    lse = torch.empty((w.Hq, Tq), dtype=torch.float32, device=dev)
    dq = torch.empty((w.dq_rows, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    dk = torch.empty((w.dkv_rows, w.Hkv, w.D), dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    wsf = torch.empty(T.thd_workspace_size(B, Tq, Tq, w.Hq, w.Hkv, w.D, w.cp_size, 0), dtype=torch.uint8, device=dev)
    wsb = torch.empty(T.thd_workspace_size(B, Tq, Tq, w.Hq, w.Hkv, w.D, w.cp_size, 1), dtype=torch.uint8, device=dev)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    def fwd():
        rc = T.thd_attn_fwd(q, k, v, o, lse, cu, cu, cu_pad, cu_pad, B, Tq, Tq, w.Hq, w.Hkv, w.D, 1,
                            w.softmax_scale, w.cp_size, -1, wsf, wsf.numel(), st, sptr)
        assert rc == 0, T.thd_status_string(rc)

    def bwd():
        rc = T.thd_attn_bwd(q, k, v, o, lse, do, dq, dk, dv, w.dq_rows, w.dkv_rows, cu, cu, cu_pad, cu_pad, B, Tq,
                            Tq, w.Hq, w.Hkv, w.D, 1, w.softmax_scale, w.cp_size, -1, wsb, wsb.numel(), st, sptr)
        assert rc == 0, T.thd_status_string(rc)

    def step():
        fwd()
        if not a.fwd_only:
            bwd()

    def timed(fn, n, kernel_id):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        T.thd_profile_enable(kernel_id, n)
        n0 = T.thd_launch_count()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for e0, e1 in evs:
            flush_buf.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        launches = T.thd_launch_count() - n0
        kms = T.thd_profile_read(n)
        T.thd_profile_enable(0, 0)
        return [e0.elapsed_time(e1) for e0, e1 in evs], kms, launches

    fwd_flops, both_flops = inputs.algorithmic_flops(w.lengths, w.Hq, w.D)
    step_flops = fwd_flops if a.fwd_only else both_flops
    for _ in range(max(a.warmup, 3)):
        flush_buf.zero_()
        step()
    torch.cuda.synchronize()
    assert int(st.item()) == 0, T.thd_status_string(int(st.item()))

    main_kernel = T.THD_KERNEL_FWD if a.fwd_only else T.THD_KERNEL_BWD
    with ClockSampler(local) as clk:
        times, kms, launches = timed(step, a.steps, main_kernel)
        fwd_times, fwd_kms, _ = timed(fwd, a.steps, T.THD_KERNEL_FWD)
        dq_kms = None
        if not a.fwd_only:
            _, dq_kms, _ = timed(bwd, max(3, min(a.steps, 20)), T.THD_KERNEL_BWD_DQ)
    assert int(st.item()) == 0, T.thd_status_string(int(st.item()))

    ms = sum(times) / len(times)
    ms_max = slowest_rank_ms(ms, world, dev)
    value = weak_scaling_tflops(step_flops, world, ms_max)
    fwd_ms = sum(fwd_times) / len(fwd_times)
    fwd_tflops = fwd_flops / (fwd_ms * 1e-3) / 1e12

    # algorithmic work of the dominant kernel: the forward's two matmuls, or
    # the dK/dV kernel's four (S^T, dP^T, dV, dK: twice the forward)
    main_flops = fwd_flops if a.fwd_only else 2.0 * fwd_flops
    kavg = sum(kms) / len(kms) if kms else float("nan")
    achieved = main_flops / (kavg * 1e-3) / 1e12
    fk = sum(fwd_kms) / len(fwd_kms) if fwd_kms else float("nan")
    fwd_kernel_tflops = fwd_flops / (fk * 1e-3) / 1e12

    e2e = None
    if not a.no_e2e:
        e2e = e2e_measure(a, w, t, dev, stream, step_flops)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "sequences": w.B, "tokens": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                       "cp_size": w.cp_size, "causal": True, "step": "fwd" if a.fwd_only else "fwd+bwd",
                       "grad_rows": w.dq_rows, "l2": "flushed between timed steps (256 MiB write)",
                       "parallelism": f"replicas x{world}"},
            "fwd_tflops": fwd_tflops, "fwd_ms": fwd_ms, "fwd_frac_of_peak": fwd_tflops / peak,
            "roofline": {"bound": "tensor", "kernel": "bwd_kernel" if not a.fwd_only else "fwd_kernel",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "peak_kind": f"bf16 burst ({peak_kind})", "frac_of_sustained": achieved / peak_sus,
                         "kernel_ms": kavg,
                         "traffic": _kernel_traffic("fwd_kernel" if a.fwd_only else "bwd_kernel", w.name)},
            "fwd_roofline": {"bound": "tensor", "kernel": "fwd_kernel", "achieved": fwd_kernel_tflops, "peak": peak,
                             "unit": "TFLOP/s", "frac": fwd_kernel_tflops / peak, "kernel_ms": fk,
                             "traffic": _kernel_traffic("fwd_kernel", w.name)},
            "dq_roofline": None if not dq_kms else {
                "bound": "tensor", "kernel": "dq_kernel", "unit": "TFLOP/s", "peak": peak,
                "kernel_ms": sum(dq_kms) / len(dq_kms),
                # executed: S, dP (recomputed) and dQ, 1.5x the forward's matmuls; of these only dQ
                # (0.5x) counts toward the algorithmic backward
                "achieved": 1.5 * fwd_flops / (sum(dq_kms) / len(dq_kms) * 1e-3) / 1e12,
                "frac": 1.5 * fwd_flops / (sum(dq_kms) / len(dq_kms) * 1e-3) / 1e12 / peak,
                "flops": "executed (S and dP recomputed)"},
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "e2e": e2e,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_a2a(a):
    """The fwd+bwd step through the emulated A2A / hierarchical layer: inputs
    and outputs are per-rank shards; the layout moves (a2a_kernel) run inside
    the step.  One GPU; prints one JSON line with the step's TFLOPS and the
    moves' HBM roofline."""
    import torch

    from packed_sequence_context_gb300 import inputs
    from packed_sequence_context_gb300 import thd_attn as T

    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        raise SystemExit("--a2a runs on one GPU")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    T.lib()
    peak, _, hbm, _ = _peaks()
    w = inputs.make_workload(a.config)
    t = inputs.make_tensors(w, with_grad=True)
    dev = torch.device("cuda", 0)
    cp, A = w.cp_size, a.a2a
    B, Tn, Hq, Hkv, D = w.B, w.T, w.Hq, w.Hkv, w.D
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    cup = torch.from_numpy(w.cu_seqlens_padded).to(dev)
    # per-rank shards of the synthetic tensors, made with the library's own move
    # (with a2a 1 the single member's layout is the global tensor)
    sh = {}
    for x in ("q", "k", "v", "do"):
        sh[x], st0 = T.cp_a2a(t[x].to(dev)[None], cup, cp_size=cp, a2a_size=1, direction=T.THD_A2A_TO_SHARDS)
        T.check_status(st0)
    o = torch.empty_like(sh["q"])
    lse = torch.empty((Hq, Tn), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(sh["q"]), torch.empty_like(sh["k"]), torch.empty_like(sh["v"])
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    wsf = torch.empty(T.thd_a2a_workspace_size(B, Tn, Hq, Hkv, D, cp, A, 0), dtype=torch.uint8, device=dev)
    wsb = torch.empty(T.thd_a2a_workspace_size(B, Tn, Hq, Hkv, D, cp, A, 1), dtype=torch.uint8, device=dev)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream

    def fwd():
        assert T.thd_attn_fwd_a2a(sh["q"], sh["k"], sh["v"], o, lse, cu, cup, B, Tn, Hq, Hkv, D, 1, w.softmax_scale,
                                  cp, A, wsf, wsf.numel(), st, sptr) == 0

    def step():
        fwd()
        assert T.thd_attn_bwd_a2a(sh["q"], sh["k"], sh["v"], o, lse, sh["do"], dq, dk, dv, cu, cup, B, Tn, Hq, Hkv,
                                  D, 1, w.softmax_scale, cp, A, wsb, wsb.numel(), st, sptr) == 0

    def timed(fn, n, kernel_id=0, per_step=0):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        T.thd_profile_enable(kernel_id, n * per_step)
        n0 = T.thd_launch_count()
        torch.cuda.synchronize()
        for e0, e1 in evs:
            flush_buf.zero_()
            e0.record(stream)
            fn()
            e1.record(stream)
        torch.cuda.synchronize()
        launches = T.thd_launch_count() - n0
        kms = T.thd_profile_read(n * per_step) if kernel_id else []
        T.thd_profile_enable(0, 0)
        return [e0.elapsed_time(e1) for e0, e1 in evs], kms, launches

    fwd_flops, both_flops = inputs.algorithmic_flops(w.lengths, Hq, D)
    for _ in range(max(a.warmup, 3)):
        flush_buf.zero_()
        step()
    torch.cuda.synchronize()
    T.check_status(st)
    with ClockSampler(0) as clk:
        times, kms, launches = timed(step, a.steps, T.THD_KERNEL_A2A, 4)
        fwd_times, _, _ = timed(fwd, a.steps)
    T.check_status(st)
    ms = sum(times) / len(times)
    fwd_ms = sum(fwd_times) / len(fwd_times)
    move_bytes = a2a_step_bytes(Tn, Hq, Hkv, D)
    move_ms = sum(kms) / a.steps
    gbs = move_bytes / (move_ms * 1e-3) / 1e9
    mode = "a2a" if A == cp else ("p2p" if A == 1 else "a2a+p2p")
    line = {
        "metric": METRIC, "value": both_flops / (ms * 1e-3) / 1e12, "unit": UNIT, "n_gpus": 1, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": w.name, "sequences": B, "tokens": Tn, "Hq": Hq, "Hkv": Hkv, "D": D, "cp_size": cp,
                   "cp_comm": mode, "hierarchical_sizes": [A, cp // A], "causal": True, "step": "fwd+bwd",
                   "inputs": "per-rank shards", "l2": "flushed between timed steps (256 MiB write)"},
        "fwd_tflops": fwd_flops / (fwd_ms * 1e-3) / 1e12, "fwd_ms": fwd_ms,
        "a2a_roofline": {"bound": "hbm", "kernel": "a2a_kernel", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "ms_per_step": move_ms, "share_of_step": move_ms / ms,
                         "bytes_per_step": move_bytes, "launches_per_step": 4, "traffic": None},
        "gpu_launches": launches,
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- HBM-bound kernels
def merge_bytes(T: int, H: int, D: int) -> int:
    """thd_lse_merge, per launch: reads O and lse of both sides (fp32), writes
    the merged O and lse."""
    return 3 * T * H * (4 * D + 4)


def tail_zero_bytes(dq_rows: int, dkv_rows: int, end_q: int, end_kv: int, Hq: int, Hkv: int, D: int) -> int:
    """thd_grad_tail_zero, per launch: bf16 zeros written to the slack rows of
    dQ, dK and dV (nothing read)."""
    return 2 * D * ((dq_rows - end_q) * Hq + 2 * (dkv_rows - end_kv) * Hkv)


def a2a_move_bytes(T: int, H: int, D: int) -> int:
    """thd_cp_a2a, per launch and tensor: every bf16 element read once and written once."""
    return 2 * 2 * T * H * D


def a2a_step_bytes(T: int, Hq: int, Hkv: int, D: int) -> int:
    """The moves of one fwd+bwd step through the emulated A2A layer: forward q,
    k, v in and O out; backward q, k, v, O, dO in and dQ, dK, dV out."""
    fwd_in, fwd_out = (Hq, Hkv, Hkv), (Hq,)
    bwd_in, bwd_out = (Hq, Hkv, Hkv, Hq, Hq), (Hq, Hkv, Hkv)
    return sum(a2a_move_bytes(T, H, D) for H in fwd_in + fwd_out + bwd_in + bwd_out)


def run_hbm_kernels(a):
    """One JSON line per HBM-bound kernel: algorithmic bytes per launch over the
    mean duration of `steps` launches (after `warmup`), taken with the
    library's profiling hook (CUDA events recorded on the launching stream
    right around the kernel), L2 flushed between launches, against the
    measured copy peak."""
    import torch

    from packed_sequence_context_gb300 import inputs
    from packed_sequence_context_gb300 import thd_attn as T

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    T.lib()
    _, _, hbm, peak_kind = _peaks()
    dev = torch.device("cuda", 0)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)

    def time_it(fn, kernel_id):
        for _ in range(max(a.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        T.thd_profile_enable(kernel_id, a.steps)
        for _ in range(a.steps):
            flush_buf.zero_()
            fn()
        torch.cuda.synchronize()
        kms = T.thd_profile_read(a.steps)
        T.thd_profile_enable(0, 0)
        assert len(kms) == a.steps, (kernel_id, len(kms))
        return sum(kms) / len(kms)

    def line(kernel, workload, nbytes, ms, extra):
        gbs = nbytes / (ms * 1e-3) / 1e9
        print(json.dumps({"kernel": kernel, "workload": workload, "bound": "hbm", "achieved": gbs, "peak": hbm,
                          "unit": "GB/s", "frac": gbs / hbm, "peak_kind": f"copy ({peak_kind})",
                          "bytes_per_launch": nbytes, "ms": ms, "steps": a.steps, **extra}), flush=True)

    # LSE merge: two fp32 partials of the packed workload's shape (finite lse on every row)
    w = inputs.make_workload("packed")
    Tn, H, D = w.T, w.Hq, w.D
    g = torch.Generator(device=dev).manual_seed(11)
    o_acc = torch.randn((Tn, H, D), generator=g, device=dev)
    o_part = torch.randn((Tn, H, D), generator=g, device=dev)
    l_acc = torch.randn((H, Tn), generator=g, device=dev)
    l_part = torch.randn((H, Tn), generator=g, device=dev)
    ms = time_it(lambda: T.lse_merge(o_acc, l_acc, o_part, l_part), T.THD_KERNEL_LSE_MERGE)
    line("lse_merge_kernel", "packed (fp32 partials)", merge_bytes(Tn, H, D), ms, {})

    # gradient tail-zero: the fwdbwd workload's dQ/dK/dV buffers, 10% slack past the last sequence
    w = inputs.make_workload("fwdbwd")
    dq = torch.empty((w.dq_rows, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    dk = torch.empty((w.dkv_rows, w.Hkv, w.D), dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    cup = torch.from_numpy(w.cu_seqlens_padded).to(dev)
    ms = time_it(lambda: T.grad_tail_zero(dq, dk, dv, cup, cup), T.THD_KERNEL_TAIL_ZERO)
    end = int(w.cu_seqlens_padded[-1])
    line("tail_zero_kernel", "fwdbwd (dQ/dK/dV slack rows)",
         tail_zero_bytes(w.dq_rows, w.dkv_rows, end, end, w.Hq, w.Hkv, w.D), ms,
         {"slack_rows": w.dq_rows - end})

    # A2A move of one tensor: the packed workload's q shards -> Ulysses member layout (cp 4, a2a 4)
    w = inputs.make_workload("packed")
    x = torch.randn((w.cp_size, w.T // w.cp_size, w.Hq, w.D), generator=g, device=dev).to(torch.bfloat16)
    y = torch.empty((w.cp_size, w.T, w.Hq // w.cp_size, w.D), dtype=torch.bfloat16, device=dev)
    cup = torch.from_numpy(w.cu_seqlens_padded).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ms = time_it(lambda: T.cp_a2a(x, cup, cp_size=w.cp_size, a2a_size=w.cp_size, direction=T.THD_A2A_TO_GROUPS,
                                  out=y, dev_status=st), T.THD_KERNEL_A2A)
    T.check_status(st)
    line("a2a_kernel", "packed (q, shards -> Ulysses members)", a2a_move_bytes(w.T, w.Hq, w.D), ms, {})
    return 0


def e2e_measure(a, w, t, dev, stream, step_flops):
    """Same metric through the public API with host buffers: pinned H2D of the
    step's inputs and metadata, the calls, and D2H of O, lse, dQ, dK, dV."""
    import torch

    from packed_sequence_context_gb300 import thd_attn as T

    host = {x: t[x].pin_memory() for x in ("q", "k", "v", "do")}
    cu_h = torch.from_numpy(w.cu_seqlens).pin_memory()
    cup_h = torch.from_numpy(w.cu_seqlens_padded).pin_memory()
    dev_in = {x: torch.empty_like(host[x], device=dev) for x in host}
    cu_d = torch.empty_like(cu_h, device=dev)
    cup_d = torch.empty_like(cup_h, device=dev)
    outs = None
    h2d = sum(x.numel() * x.element_size() for x in host.values()) + 2 * cu_h.numel() * 4
    n = max(3, min(a.steps, 20))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n + 2)]
    host_out = None
    times = []
    for i, (e0, e1) in enumerate(evs):
        e0.record(stream)
        for x in host:
            dev_in[x].copy_(host[x], non_blocking=True)
        cu_d.copy_(cu_h, non_blocking=True)
        cup_d.copy_(cup_h, non_blocking=True)
        o, lse, st = T.attn_fwd(dev_in["q"], dev_in["k"], dev_in["v"], cu_d, cu_d, cup_d, cup_d,
                                cp_size=w.cp_size, softmax_scale=w.softmax_scale)
        res = [o, lse]
        if not a.fwd_only:
            dq, dk, dv, st2 = T.attn_bwd(dev_in["q"], dev_in["k"], dev_in["v"], o, lse, dev_in["do"], cu_d, cu_d,
                                         cup_d, cup_d, cp_size=w.cp_size, softmax_scale=w.softmax_scale,
                                         dq_rows=w.dq_rows, dkv_rows=w.dkv_rows)
            res += [dq, dk, dv]
        if host_out is None:
            host_out = [torch.empty(r.shape, dtype=r.dtype, pin_memory=True) for r in res]
        for hd, r in zip(host_out, res):
            hd.copy_(r, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
        if i >= 2:
            times.append(e0.elapsed_time(e1))
    d2h = sum(x.numel() * x.element_size() for x in host_out)
    ms = sum(times) / len(times)
    return {"value": step_flops / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}


def main():
    a = _args()
    from packed_sequence_context_gb300.inputs import CONFIG_ALIASES
    a.config = CONFIG_ALIASES.get(a.config, a.config)
    if a.impl == "reference":
        return run_reference(a)
    if a.hbm_kernels:
        return run_hbm_kernels(a)
    if a.a2a:
        return run_a2a(a)
    return run_ours(a)


if __name__ == "__main__":
    sys.exit(main())
