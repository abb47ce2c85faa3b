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
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="long", help="tiny|packed|padded|long|fwdbwd (or C1..C5)")
    ap.add_argument("--lengths", default=None,
                    help="comma-separated sequence lengths replacing the named workload's (its heads, head "
                         "dimension, cp size and padding rule kept), e.g. a smaller case of the same kernels "
                         "for a profiler capture; the workload is then named config[lengths]")
    ap.add_argument("--no-extras", action="store_true",
                    help="time only the named workload (no per_config, HBM-kernel, ring or ABBA keys)")
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


def _workload(a):
    """The named workload, or its --lengths variant (named config[lengths])."""
    from packed_sequence_context_gb300 import inputs
    if not a.lengths:
        return inputs.make_workload(a.config)
    L = [int(x) for x in a.lengths.split(",") if x.strip()]
    w = inputs.make_workload(a.config, lengths=L)
    w.name = f"{a.config}[{','.join(str(x) for x in L)}]"
    return w


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
    src = {"fwd_dual_kernel": "fwd_dual.cu"}.get(kernel, kernel.split("_")[0] + ".cu")
    for name in (src, "common.cuh", "ptx.cuh", "sched.cuh"):
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


# The CPU legs time the oracle on whole sequences up to this length; a longer
# sequence is sampled as the same problem on its first ORACLE_PREFIX tokens
# (a 131072-token sequence would take the fp64 oracle hours per head).  The
# cpu_baseline leg cuts at CPU_BASELINE_PREFIX, so that its sample of the
# single-sequence workload holds 10-30 s of host work; the reference arm keeps
# its steps at a few seconds each.
ORACLE_PREFIX = 4096
CPU_BASELINE_PREFIX = 8192


def _sample_lengths(w, prefix=ORACLE_PREFIX):
    return [min(int(L), prefix) for L in w.lengths if L]


def _oracle_items(w, t, heads, prefix=ORACLE_PREFIX):
    G = w.Hq // w.Hkv
    items = []
    for b in range(w.B):
        off = int(w.cu_seqlens_padded[b])
        L = min(int(w.lengths[b]), prefix)
        if L == 0:
            continue
        for h in heads:
            sl = slice(off, off + L)
            items.append((t["q"][sl, h:h + 1].float().numpy(), t["k"][sl, h // G:h // G + 1].float().numpy(),
                          t["v"][sl, h // G:h // G + 1].float().numpy(), t["do"][sl, h:h + 1].float().numpy(),
                          w.softmax_scale))
    return items


def _sample_flops(w, heads, prefix=ORACLE_PREFIX):
    from packed_sequence_context_gb300 import inputs
    _, both = inputs.algorithmic_flops(_sample_lengths(w, prefix), 1, w.D)
    return both * len(heads)


def _sample_scope(w, prefix=ORACLE_PREFIX):
    cut = [L for L in w.lengths if L > prefix]
    if not cut:
        return f"all {w.B} sequences whole"
    return (f"{w.B} sequences, the {len(cut)} longer than {prefix} tokens cut to their first {prefix} "
            f"(the same causal problem on fewer tokens)")


def _spawn_pool(n):
    import multiprocessing as mp
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[k] = "1"
    return mp.get_context("spawn").Pool(n)


def cpu_baseline(w, t, target_s=15.0, prefix=CPU_BASELINE_PREFIX):
    """Time the oracle (as it stands) on a bounded sample of the workload:
    fwd+bwd of query heads 0, 1, 2, ... over every sequence (long sequences
    cut to `prefix` tokens), adding batches of heads until about `target_s`
    seconds of host time (or the whole workload)."""
    cores = os.cpu_count() or 1
    n_seq = max(1, sum(1 for L in w.lengths if L))
    per_batch = max(1, cores // n_seq)
    done, spent = 0, 0.0
    with _spawn_pool(cores) as pool:
        while done < w.Hq and spent < target_s:
            heads = list(range(done, min(w.Hq, done + per_batch)))
            items = _oracle_items(w, t, heads, prefix)
            t0 = time.perf_counter()
            pool.map(_oracle_item, items)
            spent += time.perf_counter() - t0
            done += len(heads)
    flops = _sample_flops(w, list(range(done)), prefix)
    scope = "all" if done == w.Hq else f"0..{done - 1} of {w.Hq}"
    return {"value": flops / spent / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"fp64 oracle fwd+bwd of query heads {scope} on the '{w.name}' workload: "
                      f"{_sample_scope(w, prefix)} ({spent:.1f} s, process pool of {cores}, one BLAS thread each); "
                      f"TFLOPS counted on the sample's own valid pairs",
            "seconds": spent}


# ----------------------------------------------------------------- reference arm
def run_reference(a):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from packed_sequence_context_gb300 import inputs
    w = _workload(a)
    t = inputs.make_tensors(w, with_grad=True)
    cores = os.cpu_count() or 1
    n_seq = max(1, sum(1 for L in w.lengths if L))
    nh = max(1, min(w.Hq, cores // n_seq))   # query heads per step: one pool's worth of work
    with _spawn_pool(cores) as pool:
        times = []
        for i in range(a.warmup + a.steps):
            heads = [(i * nh + j) % w.Hq for j in range(nh)]
            items = _oracle_items(w, t, heads)
            t0 = time.perf_counter()
            pool.map(_oracle_item, items)
            dt = time.perf_counter() - t0
            if i >= a.warmup:
                times.append(dt)
    flops = _sample_flops(w, list(range(nh)))
    mean = sum(times) / len(times)
    value = flops / mean / 1e12
    sample = (f"fp64 oracle fwd+bwd of {nh} query head(s) per step (rotating) on the '{w.name}' workload: "
              f"{_sample_scope(w)}")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus,
            "steps": a.steps, "warmup": a.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sequences": w.B, "tokens": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                       "cp_size": w.cp_size, "causal": True, "step": "fwd+bwd", "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
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
class Case:
    """One synthetic workload resident in HBM, with the library calls of one
    fwd+bwd step bound to its buffers (inputs are never re-created inside a
    timed region)."""

    def __init__(self, w, t, dev, stream):
        import torch
        from packed_sequence_context_gb300 import thd_attn as T
        self.T, self.w, self.stream = T, w, stream
        self.q, self.k, self.v, self.do = (t[x].to(dev) for x in ("q", "k", "v", "do"))
        self.cu = torch.from_numpy(w.cu_seqlens).to(dev)
        self.cu_pad = torch.from_numpy(w.cu_seqlens_padded).to(dev)   # separately allocated
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((w.Hq, w.T), dtype=torch.float32, device=dev)
        self.dq = torch.empty((w.dq_rows, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
        self.dk = torch.empty((w.dkv_rows, w.Hkv, w.D), dtype=torch.bfloat16, device=dev)
        self.dv = torch.empty_like(self.dk)
        self.st = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = lambda b: torch.empty(max(256, T.thd_workspace_size(w.B, w.T, w.T, w.Hq, w.Hkv, w.D, w.cp_size, b)),
                                   dtype=torch.uint8, device=dev)
        self.wsf, self.wsb = ws(0), ws(1)
        self.fwd_flops, self.both_flops = algorithmic_flops(w)

    def fwd(self, pad_flag=-1, cu_pad=None):
        w, T = self.w, self.T
        cp = self.cu_pad if cu_pad is None else cu_pad
        rc = T.thd_attn_fwd(self.q, self.k, self.v, self.o, self.lse, self.cu, self.cu, cp, cp, w.B, w.T, w.T, w.Hq,
                            w.Hkv, w.D, 1, w.softmax_scale, w.cp_size, pad_flag, self.wsf, self.wsf.numel(), self.st,
                            self.stream.cuda_stream)
        assert rc == 0, T.thd_status_string(rc)

    def bwd(self, pad_flag=-1, cu_pad=None):
        w, T = self.w, self.T
        cp = self.cu_pad if cu_pad is None else cu_pad
        rc = T.thd_attn_bwd(self.q, self.k, self.v, self.o, self.lse, self.do, self.dq, self.dk, self.dv, w.dq_rows,
                            w.dkv_rows, self.cu, self.cu, cp, cp, w.B, w.T, w.T, w.Hq, w.Hkv, w.D, 1, w.softmax_scale,
                            w.cp_size, pad_flag, self.wsb, self.wsb.numel(), self.st, self.stream.cuda_stream)
        assert rc == 0, T.thd_status_string(rc)

    def step(self, pad_flag=-1, cu_pad=None):
        self.fwd(pad_flag, cu_pad)
        self.bwd(pad_flag, cu_pad)

    def check(self):
        code = int(self.st.item())
        assert code == 0, self.T.thd_status_string(code)


def algorithmic_flops(w):
    from packed_sequence_context_gb300 import inputs
    return inputs.algorithmic_flops(w.lengths, w.Hq, w.D)


def timed(fn, n, stream, flush_buf, kernel_id=0, records_per_call=1, world=1):
    """n calls of fn, L2 flushed (256 MiB write) before each, outside the
    events; per call the CUDA-event time on `stream`; with kernel_id, the
    library hook's per-launch times of that kernel.  Returns (ms list,
    kernel ms list, launches of the library in the timed calls)."""
    import torch
    from packed_sequence_context_gb300 import thd_attn as T
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    T.thd_profile_enable(kernel_id, n * records_per_call)
    n0 = T.thd_launch_count()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    for e0, e1 in evs:
        flush_buf.zero_()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    launches = T.thd_launch_count() - n0
    kms = T.thd_profile_read(n * records_per_call) if kernel_id else []
    T.thd_profile_enable(0, 0)
    return [e0.elapsed_time(e1) for e0, e1 in evs], kms, launches


def _mean(x):
    return sum(x) / len(x) if x else float("nan")


def fwd_kernel_name(w) -> str:
    """The forward kernel the library runs on this workload: the single-item
    kernel when sequences average >= 16384 rows of K/V buffer, else the
    two-item one (the rule in csrc/api.cu)."""
    return "fwd_kernel" if int(w.cu_seqlens_padded[-1]) >= 16384 * len(w.lengths) else "fwd_dual_kernel"


def tensor_roofline(kernel, flops, kms, peak, peak_sus, peak_kind, workload, executed=False):
    """The kernel's achieved TFLOP/s: its work per launch over the mean
    per-launch CUDA-event time (library hook), against the bf16 peak."""
    k = _mean(kms)
    ach = flops / (k * 1e-3) / 1e12
    r = {"bound": "tensor", "kernel": kernel, "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
         "peak_kind": f"bf16 burst ({peak_kind})", "frac_of_sustained": ach / peak_sus, "kernel_ms": k,
         "traffic": _kernel_traffic(kernel, workload)}
    if executed:
        r["flops"] = "executed (S and dP recomputed: 1.5x the forward's matmuls, 0.5x algorithmic)"
    return r


def measure_case(c, steps, warmup, stream, flush_buf, peaks, world=1):
    """fwd+bwd steps, forward-only calls and backward-only calls of one
    workload; TFLOPS on algorithmic work and the three attention kernels'
    rooflines."""
    from packed_sequence_context_gb300 import thd_attn as T
    peak, peak_sus, _, peak_kind = peaks
    for _ in range(max(warmup, 3)):
        flush_buf.zero_()
        c.step()
    c.check()
    both, kms, launches = timed(c.step, steps, stream, flush_buf, T.THD_KERNEL_BWD, 1, world)
    fwd, fkms, _ = timed(c.fwd, steps, stream, flush_buf, T.THD_KERNEL_FWD, 1, world)
    _, dkms, _ = timed(c.bwd, max(3, min(steps, 20)), stream, flush_buf, T.THD_KERNEL_BWD_DQ, 1, world)
    c.check()
    name = c.w.name
    return {
        "ms_fwdbwd": _mean(both), "ms_fwd": _mean(fwd), "launches_per_step": launches / steps,
        "fwdbwd_tflops": c.both_flops / (_mean(both) * 1e-3) / 1e12,
        "fwd_tflops": c.fwd_flops / (_mean(fwd) * 1e-3) / 1e12,
        "roofline": tensor_roofline("bwd_kernel", 2.0 * c.fwd_flops, kms, peak, peak_sus, peak_kind, name),
        "fwd_roofline": tensor_roofline(fwd_kernel_name(c.w), c.fwd_flops, fkms, peak, peak_sus, peak_kind, name),
        "dq_roofline": tensor_roofline("dq_kernel", 1.5 * c.fwd_flops, dkms, peak, peak_sus, peak_kind, name,
                                       executed=True),
        "_times": both,
    }


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
    peaks = _peaks()
    peak, peak_sus, hbm, peak_kind = peaks

    w = _workload(a)
    t = inputs.make_tensors(w, with_grad=True)
    # the CPU leg runs first, before this process touches the GPU with work
    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        cpu = cpu_baseline(w, t)

    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    c = Case(w, t, dev, stream)
    step = c.fwd if a.fwd_only else c.step
    step_flops = c.fwd_flops if a.fwd_only else c.both_flops
    for _ in range(max(a.warmup, 3)):
        flush_buf.zero_()
        step()
    torch.cuda.synchronize()
    c.check()

    main_kernel = T.THD_KERNEL_FWD if a.fwd_only else T.THD_KERNEL_BWD
    with ClockSampler(local) as clk:
        times, kms, launches = timed(step, a.steps, stream, flush_buf, main_kernel, 1, world)
        fwd_times, fwd_kms, _ = timed(c.fwd, a.steps, stream, flush_buf, T.THD_KERNEL_FWD, 1, world)
        dq_kms = []
        if not a.fwd_only:
            _, dq_kms, _ = timed(c.bwd, max(3, min(a.steps, 20)), stream, flush_buf, T.THD_KERNEL_BWD_DQ, 1, world)
    c.check()

    ms = _mean(times)
    ms_max = slowest_rank_ms(ms, world, dev)
    value = weak_scaling_tflops(step_flops, world, ms_max)
    fwd_ms = _mean(fwd_times)
    fwd_tflops = c.fwd_flops / (fwd_ms * 1e-3) / 1e12
    fwd_roof = tensor_roofline(fwd_kernel_name(w), c.fwd_flops, fwd_kms, peak, peak_sus, peak_kind, w.name)
    if a.fwd_only:
        roof = fwd_roof
    else:
        # the dominant kernel: dK/dV, four matmuls per tile pair (S^T, dP^T, dV, dK: twice the forward's)
        roof = tensor_roofline("bwd_kernel", 2.0 * c.fwd_flops, kms, peak, peak_sus, peak_kind, w.name)
    dq_roof = None if not dq_kms else tensor_roofline("dq_kernel", 1.5 * c.fwd_flops, dq_kms, peak, peak_sus,
                                                      peak_kind, w.name, executed=True)

    e2e = None
    if not a.no_e2e:
        e2e = e2e_measure(a, w, t, dev, stream, step_flops)

    extras = {}
    if rank == 0 and world == 1 and not a.no_extras and not a.fwd_only:
        del c
        torch.cuda.empty_cache()
        extras = bench_extras(a.config, dev, stream, flush_buf, peaks)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
            "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": w.name, "sequences": w.B, "tokens": w.T, "Hq": w.Hq, "Hkv": w.Hkv, "D": w.D,
                       "cp_size": w.cp_size, "causal": True, "step": "fwd" if a.fwd_only else "fwd+bwd",
                       "grad_rows": w.dq_rows, "l2": "flushed between timed steps (256 MiB write)",
                       "parallelism": f"replicas x{world}"},
            "frac_of_peak": value / world / peak,
            "fwd_tflops": fwd_tflops, "fwd_ms": fwd_ms, "fwd_frac_of_peak": fwd_tflops / peak,
            "roofline": roof,
            "fwd_roofline": fwd_roof,
            "dq_roofline": dq_roof,
            "gpu_launches": launches,
            "clocks": clk.summary(),
            "cpu_baseline": cpu,
            "e2e": e2e,
            **extras,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def bench_extras(main_config, dev, stream, flush_buf, peaks, steps=20, warmup=3):
    """The other measured workloads and kernels, timed after the main line
    (one GPU, rank 0): per_config (every other named workload's fwd and
    fwd+bwd TFLOPS with the three kernels' rooflines), the HBM-bound kernels
    against the copy peak, the materialised ring with bf16 partials, and the
    four-arm ABBA timing of value-equal padded metadata."""
    import torch
    from packed_sequence_context_gb300 import inputs

    out = {"per_config": {}}
    for name in ("fwdbwd", "padded", "packed"):
        if name == main_config:
            continue
        w = inputs.make_workload(name)
        c = Case(w, inputs.make_tensors(w, with_grad=True), dev, stream)
        r = measure_case(c, steps, warmup, stream, flush_buf, peaks)
        r.pop("_times")
        r.update({"tokens": w.T, "sequences": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "cp_size": w.cp_size,
                  "fwd_frac_of_peak": r["fwd_tflops"] / peaks[0], "fwdbwd_frac_of_peak": r["fwdbwd_tflops"] / peaks[0],
                  "steps": steps})
        out["per_config"][name] = r
        del c
        torch.cuda.empty_cache()
    out["hbm_kernels"] = hbm_kernel_lines(dev, stream, flush_buf, peaks, steps, warmup)
    out["ring_bf16"] = ring_bf16_line(dev, stream, flush_buf, peaks, steps, warmup)
    out["regression_arms"] = abba_arms(dev, stream, flush_buf, steps=5, rounds=3)
    return out


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
    w = _workload(a)
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
def merge_bytes(T: int, H: int, D: int, part_bytes: int = 4) -> int:
    """thd_lse_merge (part_bytes 4) / thd_lse_merge_bf16 (2), per launch: reads
    the fp32 accumulator's O and lse and the partial's O (part_bytes per
    element) and lse, writes the merged O and lse."""
    return T * H * (2 * (4 * D + 4) + part_bytes * D + 4)


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


def hbm_line(kernel, workload, nbytes, kms, peaks, extra=None):
    _, _, hbm, peak_kind = peaks
    ms = _mean(kms)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"kernel": kernel, "workload": workload, "bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
            "frac": gbs / hbm, "peak_kind": f"copy ({peak_kind})", "bytes_per_launch": nbytes, "kernel_ms": ms,
            "launches": len(kms), **(extra or {})}


def hbm_kernel_lines(dev, stream, flush_buf, peaks, steps=20, warmup=3):
    """The HBM-bound kernels, each on its own buffers: algorithmic bytes per
    launch over the library hook's per-launch CUDA-event time (L2 flushed
    between launches), against the measured copy peak."""
    import torch
    from packed_sequence_context_gb300 import inputs
    from packed_sequence_context_gb300 import thd_attn as T

    def run(fn, kernel_id):
        for _ in range(warmup):
            fn()
        _, kms, _ = timed(fn, steps, stream, flush_buf, kernel_id)
        assert len(kms) == steps, (kernel_id, len(kms))
        return kms

    lines = {}
    g = torch.Generator(device=dev).manual_seed(11)
    # LSE merge: two partials of the packed workload's shape (finite lse on every row)
    w = inputs.make_workload("packed")
    Tn, H, D = w.T, w.Hq, w.D
    o_acc = torch.randn((Tn, H, D), generator=g, device=dev)
    l_acc = torch.randn((H, Tn), generator=g, device=dev)
    l_part = torch.randn((H, Tn), generator=g, device=dev)
    o_part = torch.randn((Tn, H, D), generator=g, device=dev)
    kms = run(lambda: T.lse_merge(o_acc, l_acc, o_part, l_part), T.THD_KERNEL_LSE_MERGE)
    lines["lse_merge"] = hbm_line("lse_merge_kernel<float>", "packed (fp32 partials)", merge_bytes(Tn, H, D), kms,
                                  peaks)
    o_part16 = o_part.to(torch.bfloat16)
    del o_part
    kms = run(lambda: T.lse_merge_bf16(o_acc, l_acc, o_part16, l_part), T.THD_KERNEL_LSE_MERGE)
    lines["lse_merge_bf16"] = hbm_line("lse_merge_kernel<bf16>", "packed (bf16 partial into fp32)",
                                       merge_bytes(Tn, H, D, part_bytes=2), kms, peaks)
    del o_acc, o_part16
    # gradient tail-zero: the fwdbwd workload's dQ/dK/dV buffers, 10% slack past the last sequence
    w = inputs.make_workload("fwdbwd")
    dq = torch.empty((w.dq_rows, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    dk = torch.empty((w.dkv_rows, w.Hkv, w.D), dtype=torch.bfloat16, device=dev)
    dv = torch.empty_like(dk)
    cup = torch.from_numpy(w.cu_seqlens_padded).to(dev)
    kms = run(lambda: T.grad_tail_zero(dq, dk, dv, cup, cup), T.THD_KERNEL_TAIL_ZERO)
    end = int(w.cu_seqlens_padded[-1])
    lines["tail_zero"] = hbm_line("tail_zero_kernel", "fwdbwd (dQ/dK/dV slack rows)",
                                  tail_zero_bytes(w.dq_rows, w.dkv_rows, end, end, w.Hq, w.Hkv, w.D), kms, peaks,
                                  {"slack_rows": w.dq_rows - end})
    # no tail (the buffer ends at the last sequence): the host flag launches nothing
    n0 = T.thd_launch_count()
    T.grad_tail_zero(dq[:end], dk[:end], dv[:end], cup, cup, host_knows_no_tail=True)
    lines["tail_zero"]["launches_when_host_knows_no_tail"] = T.thd_launch_count() - n0
    del dq, dk, dv
    torch.cuda.empty_cache()
    return lines


def ring_bf16_line(dev, stream, flush_buf, peaks, steps=20, warmup=3):
    """The materialised ring on the packed workload: every ring step's
    partial written in bf16 (thd_attn_fwd_step_bf16) and merged into an fp32
    accumulator (thd_lse_merge_bf16), cp_size steps per forward."""
    import torch
    from packed_sequence_context_gb300 import inputs
    from packed_sequence_context_gb300 import thd_attn as T

    w = inputs.make_workload("packed")
    t = inputs.make_tensors(w)
    q, k, v = (t[x].to(dev) for x in ("q", "k", "v"))
    cu = torch.from_numpy(w.cu_seqlens).to(dev)
    cup = torch.from_numpy(w.cu_seqlens_padded).to(dev)
    o_part = torch.empty((w.T, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    l_part = torch.empty((w.Hq, w.T), dtype=torch.float32, device=dev)
    o_acc = torch.empty((w.T, w.Hq, w.D), dtype=torch.float32, device=dev)
    l_acc = torch.empty((w.Hq, w.T), dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(T.thd_workspace_size(w.B, w.T, w.T, w.Hq, w.Hkv, w.D, w.cp_size, 0), dtype=torch.uint8,
                     device=dev)

    def ring():
        o_acc.zero_()
        l_acc.fill_(float("-inf"))
        for i in range(w.cp_size):
            rc = T.thd_attn_fwd_step_bf16(q, k, v, o_part, l_part, cu, cu, cup, cup, w.B, w.T, w.T, w.Hq, w.Hkv,
                                          w.D, 1, w.softmax_scale, w.cp_size, -1, i, ws, ws.numel(), st,
                                          stream.cuda_stream)
            assert rc == 0
            T.lse_merge_bf16(o_acc, l_acc, o_part, l_part)

    for _ in range(warmup):
        ring()
    times, kms, launches = timed(ring, steps, stream, flush_buf, T.THD_KERNEL_LSE_MERGE, w.cp_size)
    assert int(st.item()) == 0
    fwd_flops, _ = algorithmic_flops(w)
    ms = _mean(times)
    return {"workload": w.name, "cp_size": w.cp_size, "ms_per_forward": ms,
            "fwd_tflops": fwd_flops / (ms * 1e-3) / 1e12, "launches_per_forward": launches / steps,
            "merge": hbm_line("lse_merge_kernel<bf16>", "packed ring step (bf16 partial into fp32)",
                              merge_bytes(w.T, w.Hq, w.D, part_bytes=2), kms, peaks),
            "note": "each forward also clears the fp32 accumulator (two torch fills, inside the events)"}


def abba_arms(dev, stream, flush_buf, steps=5, rounds=3):
    """The value-equal padded-metadata case of the pages' regression report,
    timed in ABBA order on the packed workload's fwd+bwd step: arms
    pad_between_seqs -1 with cu_seqlens_padded the same pointer as
    cu_seqlens, -1 with a value-equal clone, 0, and 1.  Per arm: mean ms per
    step, library launches per step, and whether O, dQ, dK, dV equal the first
    arm's bit for bit."""
    import torch
    from packed_sequence_context_gb300 import inputs
    from packed_sequence_context_gb300 import thd_attn as T

    w = inputs.make_workload("packed")
    c = Case(w, inputs.make_tensors(w, with_grad=True), dev, stream)
    arms = {"auto_same_pointer": (-1, c.cu), "auto_value_equal_clone": (-1, c.cu_pad),
            "flag_0_no_padding": (0, c.cu_pad), "flag_1_padding": (1, c.cu_pad)}
    names = list(arms)
    for n in names:
        c.step(*arms[n])
    torch.cuda.synchronize()
    c.check()
    order = (names + names[::-1]) * rounds
    acc = {n: [] for n in names}
    launches = {n: [] for n in names}
    ref = None
    same = {n: True for n in names}
    for n in order:
        ts, _, nl = timed(lambda: c.step(*arms[n]), steps, stream, flush_buf)
        acc[n].extend(ts)
        launches[n].append(nl / steps)
        outs = [c.o.clone(), c.dq.clone(), c.dk.clone(), c.dv.clone()]
        if ref is None:
            ref = outs
        same[n] = same[n] and all(torch.equal(x, y) for x, y in zip(ref, outs))
    c.check()
    return {"workload": w.name, "order": "ABCD DCBA x" + str(rounds), "steps_per_visit": steps,
            "arms": {n: {"ms_per_step": _mean(acc[n]), "launches_per_step": _mean(launches[n]),
                         "bit_identical_to_first_arm": same[n]} for n in names}}


def run_hbm_kernels(a):
    """One JSON line per HBM-bound kernel (the same lines the default run
    adds under hbm_kernels)."""
    import torch
    from packed_sequence_context_gb300 import thd_attn as T

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    T.lib()
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    for name, line in hbm_kernel_lines(dev, stream, flush_buf, _peaks(), a.steps, max(a.warmup, 3)).items():
        print(json.dumps({"name": name, **line}), flush=True)
    return 0


def _split_copy(dst, src, streams, after):
    """dst.copy_(src) as one slice per copy stream (dimension 0), each slice
    started after the event `after`; returns the events that mark them done.
    Several host<->device copies in flight use several copy engines.  A
    device source is recorded on the copy streams, so that its memory is not
    handed to a later allocation before the copy has read it."""
    import torch
    n = len(streams)
    rows = src.shape[0]
    done = []
    for j, cs in enumerate(streams):
        lo, hi = rows * j // n, rows * (j + 1) // n
        if lo == hi:
            continue
        cs.wait_event(after)
        with torch.cuda.stream(cs):
            dst[lo:hi].copy_(src[lo:hi], non_blocking=True)
        if src.is_cuda:
            src.record_stream(cs)
        ev = torch.cuda.Event()
        ev.record(cs)
        done.append(ev)
    return done


def e2e_measure(a, w, t, dev, stream, step_flops):
    """Same metric through the public API with host buffers: every step, the
    pinned H2D of its inputs and metadata, the calls, and the D2H of O, lse,
    dQ, dK, dV, all inside the timed region.  Copies run on four copy
    streams, one slice of each tensor per stream.

    The value is a pipelined run of K steps, the way a training loop feeds
    the library: two device input buffers, step i+1's inputs uploaded while
    step i computes (once step i-1, the buffer's last reader, is done), step
    i's outputs downloaded while step i+1 computes; the events open before
    the first upload and close after the last download.  `serial` is the
    same step with each step's copies and calls alone between its events
    (inputs before the forward, dO during it, O and lse during the backward,
    gradients after it)."""
    import torch

    from packed_sequence_context_gb300 import thd_attn as T

    host = {x: t[x].pin_memory() for x in ("q", "k", "v", "do")}
    cu_h = torch.from_numpy(w.cu_seqlens).pin_memory()
    cup_h = torch.from_numpy(w.cu_seqlens_padded).pin_memory()
    bufs = []
    for _ in range(2):
        b = {x: torch.empty_like(host[x], device=dev) for x in host}
        b["cu"] = torch.empty_like(cu_h, device=dev)
        b["cup"] = torch.empty_like(cup_h, device=dev)
        bufs.append(b)
    copy_streams = [torch.cuda.Stream(device=dev) for _ in range(4)]
    h2d = sum(x.numel() * x.element_size() for x in host.values()) + 2 * cu_h.numel() * 4
    n = max(3, min(a.steps, 20))
    out_shapes = [((w.T, w.Hq, w.D), torch.bfloat16), ((w.Hq, w.T), torch.float32)]
    if not a.fwd_only:
        out_shapes += [((w.dq_rows, w.Hq, w.D), torch.bfloat16), ((w.dkv_rows, w.Hkv, w.D), torch.bfloat16),
                       ((w.dkv_rows, w.Hkv, w.D), torch.bfloat16)]
    host_out = [torch.empty(shape, dtype=dt, pin_memory=True) for shape, dt in out_shapes]
    d2h_bytes = sum(x.numel() * x.element_size() for x in host_out)

    def wait_all(events):
        for ev in events:
            stream.wait_event(ev)

    def upload(b, after):
        """H2D of one step's inputs into buffer b; returns (q/k/v/metadata events, dO events)."""
        ev = []
        with torch.cuda.stream(copy_streams[0]):
            copy_streams[0].wait_event(after)
            b["cu"].copy_(cu_h, non_blocking=True)
            b["cup"].copy_(cup_h, non_blocking=True)
            e = torch.cuda.Event()
            e.record(copy_streams[0])
            ev.append(e)
        for x in ("q", "k", "v"):
            ev += _split_copy(b[x], host[x], copy_streams, after)
        do_ev = [] if a.fwd_only else _split_copy(b["do"], host["do"], copy_streams, after)
        return ev, do_ev

    def compute(b, in_ev, do_ev):
        """The calls on the compute stream, then the D2H of their results;
        returns (the event after the step's last call, the D2H events)."""
        wait_all(in_ev)
        o, lse, st = T.attn_fwd(b["q"], b["k"], b["v"], b["cu"], b["cu"], b["cup"], b["cup"],
                                cp_size=w.cp_size, softmax_scale=w.softmax_scale)
        fwd_done = torch.cuda.Event()
        fwd_done.record(stream)
        d2h = _split_copy(host_out[0], o, copy_streams, fwd_done) + \
            _split_copy(host_out[1], lse, copy_streams, fwd_done)
        last = fwd_done
        if not a.fwd_only:
            wait_all(do_ev)
            dq, dk, dv, st2 = T.attn_bwd(b["q"], b["k"], b["v"], o, lse, b["do"], b["cu"], b["cu"], b["cup"],
                                         b["cup"], cp_size=w.cp_size, softmax_scale=w.softmax_scale,
                                         dq_rows=w.dq_rows, dkv_rows=w.dkv_rows)
            last = torch.cuda.Event()
            last.record(stream)
            for hd, r in zip(host_out[2:], (dq, dk, dv)):
                d2h += _split_copy(hd, r, copy_streams, last)
        return last, d2h

    # serial: each step alone between its events
    serial = []
    for i in range(n + 2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        in_ev, do_ev = upload(bufs[0], e0)
        _, d2h = compute(bufs[0], in_ev, do_ev)
        wait_all(d2h)
        e1.record(stream)
        stream.synchronize()
        if i >= 2:
            serial.append(e0.elapsed_time(e1))

    # pipelined: n steps in flight through two input buffers
    def pipelined(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        pending = [upload(bufs[0], e0)]
        done, d2h_all = [], []
        for i in range(steps):
            if i + 1 < steps:   # the next step's buffer is free once step i-1 is done
                pending.append(upload(bufs[(i + 1) % 2], done[i - 1] if i >= 1 else e0))
            last, d2h = compute(bufs[i % 2], *pending[i])
            done.append(last)
            d2h_all += d2h
        wait_all(d2h_all)
        e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) / steps

    pipelined(3)   # warm-up
    ms = pipelined(n)
    ms_serial = sum(serial) / len(serial)
    return {"value": step_flops / (ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h_bytes),
            "steps": n,
            "copies": ("pipelined: step i+1's inputs uploaded and step i-1's outputs downloaded while step i "
                       "computes (two device input buffers, 4 copy streams, one slice each per tensor); the "
                       "events open before the first upload and close after the last download"),
            "serial": {"value": step_flops / (ms_serial * 1e-3) / 1e12, "ms_per_step": ms_serial,
                       "copies": "each step alone: q/k/v before the forward, dO during it, O and lse during "
                                 "the backward, dQ/dK/dV after it"}}


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
