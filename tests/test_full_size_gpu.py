"""Full-size parity: the packed, padded (GQA) and fwdbwd workloads run
forward and backward through the C ABI in the bench's launch configuration
(cp_size of the workload, padding decided from values, gradient buffers with
the workload's slack), and every valid row of every head of O, lse, dQ, dK
and dV is compared with the CPU fp64 oracle (a process pool over
(sequence, kv-head group)).  The 131072-token workload is compared on the
forward's full rows of two query heads (every row of heads 0 and 17, in
blocks of query rows).  Bars as in oracle_pool: lse within 1e-3; O and the
gradients within 2e-2 beyond their own bf16 rounding, and raw within 2e-2
wherever |ref| < 2; rows without a valid token exactly 0 / -inf."""

import os

import numpy as np
import pytest
import torch

import oracle_pool as op
from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T
from thd_testutil import device_inputs

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib(thd_lib):
    return thd_lib


def _report(name, stats):
    parts = []
    for k, s in stats.items():
        if isinstance(s, dict):
            parts.append(f"{k}: max {s['max_abs']:.3e} at |ref| {s['ref_at_max']:.2f}, beyond bf16 rounding "
                         f"{s['excess']:.3e}, raw where |ref|<{op.RAW_BAR_BELOW:g} {s['raw_small']:.3e}, "
                         f"{s['n_over']} of {s['n']} over {op.TOL:g}")
        else:
            parts.append(f"{k}: max {s:.3e}")
    print(f"[{name}] " + "; ".join(parts), flush=True)


def _assert(stats):
    for k, s in stats.items():
        if k == "lse":
            assert s <= op.LSE_TOL, f"lse max-abs {s:.3e}"
        else:
            assert s["excess"] <= op.TOL, f"{k}: {s}"
            assert s["raw_small"] <= op.TOL, f"{k}: {s}"


@pytest.mark.parametrize("name", ["packed", "padded", "fwdbwd"])
def test_full_size_fwd_bwd_every_row_every_head(name):
    w = inputs.make_workload(name)
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"], cp_size=w.cp_size,
                            softmax_scale=w.softmax_scale)
    dq, dk, dv, st2 = T.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], d["cu"], d["cu_pad"],
                                 d["cu_pad"], cp_size=w.cp_size, softmax_scale=w.softmax_scale, dq_rows=w.dq_rows,
                                 dkv_rows=w.dkv_rows)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    # rows without a valid token, and the slack rows, exactly 0 / -inf
    inv = ~inputs.valid_row_mask(w)
    invt = torch.from_numpy(inv).cuda()
    if inv.any():
        assert torch.all(o[invt] == 0) and torch.all(torch.isneginf(lse[:, invt]))
        for g in (dq, dk, dv):
            assert torch.all(g[:w.T][invt] == 0)
    for g in (dq, dk, dv):
        assert torch.all(g[w.T:] == 0)
    store = op.Store()
    try:
        for k_, x in (("q", t["q"]), ("k", t["k"]), ("v", t["v"]), ("do", t["do"]), ("o", o), ("lse", lse),
                      ("dq", dq[:w.T]), ("dk", dk[:w.T]), ("dv", dv[:w.T])):
            store.put(k_, x.float().cpu().numpy() if x.is_cuda else x.float().numpy())
        G = w.Hq // w.Hkv
        specs = [{"root": ROOT, "dir": store.dir, "off": int(w.cu_seqlens_padded[b]), "L": int(w.lengths[b]),
                  "kv_heads": [hk], "G": G, "scale": w.softmax_scale, "bwd": True}
                 for b in range(w.B) if w.lengths[b] > 0 for hk in range(w.Hkv)]
        # longest first, so the pool's tail is short
        specs.sort(key=lambda s: -s["L"])
        res = op.run(op._worker_seq, specs)
    finally:
        store.close()
    stats = {}
    for r in res:
        for k_ in ("o", "dq", "dk", "dv"):
            stats[k_] = op.merge_stats(stats.get(k_), r[k_])
        stats["lse"] = max(stats.get("lse", 0.0), r["lse"])
    _report(name, stats)
    _assert(stats)


def test_long_forward_every_row_of_two_heads():
    w = inputs.make_workload("long")
    t = inputs.make_tensors(w, with_grad=False)
    d = device_inputs(w, t)
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"], cp_size=w.cp_size,
                            softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    heads = [0, 17]
    G = w.Hq // w.Hkv
    store = op.Store()
    try:
        store.put("q", t["q"][:, heads].float().numpy())
        store.put("k", t["k"][:, [h // G for h in heads]].float().numpy())
        store.put("v", t["v"][:, [h // G for h in heads]].float().numpy())
        store.put("o", o[:, heads].float().cpu().numpy())
        store.put("lse", lse[heads].cpu().numpy())
        L, blk = w.lengths[0], 4096
        # in the stored arrays head j of `heads` reads kv column j (G = 1 there)
        specs = [{"root": ROOT, "dir": store.dir, "off": 0, "i0": i0, "i1": min(L, i0 + blk), "h": j, "G": 1,
                  "scale": w.softmax_scale} for j in range(len(heads)) for i0 in range(0, L, blk)]
        specs.sort(key=lambda s: -s["i1"])
        res = op.run(op._worker_rows, specs)
    finally:
        store.close()
    stats = {}
    for r in res:
        stats["o"] = op.merge_stats(stats.get("o"), r["o"])
        stats["lse"] = max(stats.get("lse", 0.0), r["lse"])
    _report("long, heads 0 and 17", stats)
    _assert(stats)


@pytest.mark.parametrize("bf16", [True, False])
def test_materialised_ring_full_packed_every_row(bf16):
    """The ring with its per-step partials materialised: cp_size launches of
    thd_attn_fwd_step_bf16 (or the fp32 thd_attn_fwd_step), each merged into an
    fp32 accumulator by thd_lse_merge_bf16 (thd_lse_merge), against the
    oracle's emulated ring on every valid row of every head of the packed
    workload."""
    w = inputs.make_workload("packed")
    t = inputs.make_tensors(w)
    d = device_inputs(w, t)
    acc_o = torch.zeros((w.T, w.Hq, w.D), dtype=torch.float32, device="cuda")
    acc_l = torch.full((w.Hq, w.T), float("-inf"), dtype=torch.float32, device="cuda")
    for i in range(w.cp_size):
        kw = dict(step=i, cp_size=w.cp_size, softmax_scale=w.softmax_scale)
        if bf16:
            o, l, st = T.attn_fwd_step_bf16(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"], **kw)
            assert o.dtype == torch.bfloat16
            T.lse_merge_bf16(acc_o, acc_l, o, l)
        else:
            o, l, st = T.attn_fwd_step(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"], **kw)
            T.lse_merge(acc_o, acc_l, o, l)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
    store = op.Store()
    try:
        for k_, x in (("q", t["q"]), ("k", t["k"]), ("v", t["v"])):
            store.put(k_, x.float().numpy())
        store.put("o", acc_o.cpu().numpy())
        store.put("lse", acc_l.cpu().numpy())
        G = w.Hq // w.Hkv
        specs = [{"root": ROOT, "dir": store.dir, "off": int(w.cu_seqlens_padded[b]), "L": int(w.lengths[b]),
                  "P": int(w.cu_seqlens_padded[b + 1] - w.cu_seqlens_padded[b]), "h": h, "G": G,
                  "cp": w.cp_size, "scale": w.softmax_scale}
                 for b in range(w.B) if w.lengths[b] > 0 for h in range(w.Hq)]
        specs.sort(key=lambda s: -s["L"])
        res = op.run(op._worker_ring, specs)
    finally:
        store.close()
    stats = {"o": None, "lse": 0.0}
    for r in res:
        stats["o"] = op.merge_stats(stats["o"], r["o"])
        stats["lse"] = max(stats["lse"], r["lse"])
    _report(f"packed ring, {'bf16' if bf16 else 'fp32'} partials", stats)
    _assert(stats)
    if not bf16:   # fp32 partials: the raw bar holds on every element
        assert stats["o"]["n_over"] == 0
