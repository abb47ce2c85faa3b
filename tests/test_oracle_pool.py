"""CPU checks of the full-size comparison plumbing (oracle_pool): a worker
given the oracle's own results as the "device" results reports errors at
float32 rounding only, a planted mistake in one gradient element is found,
and the query-row blocks of the long-sequence check reproduce the whole
sequence's forward."""

import os

import numpy as np

import oracle_pool as op
from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _store(w, t, res):
    s = op.Store()
    for k, x in t.items():
        s.put(k, x.float().numpy())
    for k, x in res.items():
        s.put(k, x)
    return s


def test_worker_finds_nothing_in_exact_results_and_a_planted_mistake():
    w = inputs.make_workload("custom", 5, lengths=[40, 72], Hq=4, Hkv=2, D=16, cp_size=2)
    t = inputs.make_tensors(w, with_grad=True)
    qn, kn, vn, don = (t[x].float().numpy() for x in ("q", "k", "v", "do"))
    O, lse = orc.attn_fwd(qn, kn, vn, w.cu_seqlens, w.cu_seqlens, softmax_scale=w.softmax_scale)
    dq, dk, dv = orc.attn_bwd(qn, kn, vn, don, w.cu_seqlens, w.cu_seqlens, softmax_scale=w.softmax_scale)
    dk_bad = dk.copy()
    dk_bad[50, 1, 3] += 0.05   # sequence 1, kv head 1
    for planted in (False, True):
        s = _store(w, t, {"o": O, "lse": lse, "dq": dq, "dk": dk_bad if planted else dk, "dv": dv})
        try:
            specs = [{"root": ROOT, "dir": s.dir, "off": int(w.cu_seqlens_padded[b]), "L": w.lengths[b],
                      "kv_heads": [hk], "G": 2, "scale": w.softmax_scale, "bwd": True}
                     for b in range(w.B) for hk in range(w.Hkv)]
            res = op.run(op._worker_seq, specs, n=2)
        finally:
            s.close()
        worst = {k: max(r[k]["max_abs"] for r in res) for k in ("o", "dq", "dk", "dv")}
        if planted:
            assert worst["dk"] > 0.04 and max(r["dk"]["n_over"] for r in res) == 1
            assert max(r["dk"]["excess"] for r in res) > op.TOL
        else:
            assert max(worst.values()) < 1e-5, worst
            assert max(r["lse"] for r in res) < 1e-5


def test_row_blocks_reproduce_the_whole_forward():
    w = inputs.make_workload("custom", 6, lengths=[300], Hq=2, Hkv=1, D=16, cp_size=1)
    t = inputs.make_tensors(w)
    qn, kn, vn = (t[x].float().numpy() for x in ("q", "k", "v"))
    O, lse = orc.attn_fwd(qn, kn, vn, w.cu_seqlens, w.cu_seqlens, softmax_scale=w.softmax_scale)
    s = _store(w, t, {"o": O, "lse": lse})
    try:
        specs = [{"root": ROOT, "dir": s.dir, "off": 0, "i0": i0, "i1": min(300, i0 + 64), "h": h, "G": 2,
                  "scale": w.softmax_scale} for h in range(2) for i0 in range(0, 300, 64)]
        res = op.run(op._worker_rows, specs, n=2)
    finally:
        s.close()
    assert max(r["o"]["max_abs"] for r in res) < 1e-5
    assert max(r["lse"] for r in res) < 1e-5


def test_bar_counts_rounding_of_large_values():
    ref = np.array([0.5, 9.0, -12.3, 1.9])
    got = ref + np.array([0.015, 0.04, -0.03, 0.019])
    s = op.compare(got, ref)
    assert s["n_over"] == 2 and s["raw_small"] <= op.TOL and s["excess"] <= op.TOL
    s = op.compare(ref + np.array([0.0, 0.0, 0.0, 0.021]), ref)
    assert s["raw_small"] > op.TOL   # |ref| < 2 keeps the raw bar


def test_ring_worker_reproduces_unsplit_attention():
    """The ring worker compares the oracle's emulated ring with the device
    result; given unsplit attention as the "device" result it reports only
    rounding (the ring equals plain attention), padded sequences included."""
    w = inputs.make_workload("custom", 7, lengths=[60, 96], pad_to=16, Hq=2, Hkv=1, D=16, cp_size=2)
    t = inputs.make_tensors(w)
    qn, kn, vn = (t[x].float().numpy() for x in ("q", "k", "v"))
    O, lse = orc.attn_fwd(qn, kn, vn, w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded, w.cu_seqlens_padded,
                          softmax_scale=w.softmax_scale)
    s = _store(w, t, {"o": O, "lse": lse})
    try:
        specs = [{"root": ROOT, "dir": s.dir, "off": int(w.cu_seqlens_padded[b]), "L": w.lengths[b],
                  "P": int(w.cu_seqlens_padded[b + 1] - w.cu_seqlens_padded[b]), "h": h, "G": 2, "cp": 2,
                  "scale": w.softmax_scale} for b in range(w.B) for h in range(2)]
        res = op.run(op._worker_ring, specs, n=2)
    finally:
        s.close()
    assert max(r["o"]["max_abs"] for r in res) < 1e-5
    assert max(r["lse"] for r in res) < 1e-5
