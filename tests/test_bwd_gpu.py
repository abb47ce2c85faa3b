"""GPU parity of the backward path (thd_attn_bwd) against the CPU fp64
oracle, through the C-ABI binding.  Bar: max-abs <= 2e-2 on dQ/dK/dV over
valid rows; every row without a valid token, including the slack rows past
the last sequence, exactly 0."""

import numpy as np
import pytest
import torch

from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T
from thd_testutil import O_TOL, device_inputs, f64, rounding_aware_excess

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(thd_lib):
    return thd_lib


def _custom(lengths, cp, Hq=2, Hkv=2, D=64, pad_to=0, seed=0, slack=0.0):
    return inputs.make_workload("custom", seed, lengths=lengths, pad_to=pad_to, Hq=Hq, Hkv=Hkv, D=D, cp_size=cp,
                                grad_slack=slack)


def _run(w, d, causal=True, canary=7.0, pad_flag=-1, cu_pad="default"):
    cp = d["cu_pad"] if isinstance(cu_pad, str) else cu_pad
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], cp, cp, cp_size=w.cp_size, causal=causal,
                            softmax_scale=w.softmax_scale, pad_between_seqs=pad_flag)
    dq = torch.full((w.dq_rows, w.Hq, w.D), canary, dtype=torch.bfloat16, device="cuda")
    dk = torch.full((w.dkv_rows, w.Hkv, w.D), canary, dtype=torch.bfloat16, device="cuda")
    dv = torch.full_like(dk, canary)
    dq, dk, dv, st2 = T.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], d["cu"], cp, cp,
                                 cp_size=w.cp_size, causal=causal, softmax_scale=w.softmax_scale,
                                 pad_between_seqs=pad_flag, dq_rows=w.dq_rows, dkv_rows=w.dkv_rows, dq=dq, dk=dk,
                                 dv=dv)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0, (int(st.item()), int(st2.item()))
    return o, lse, dq, dk, dv


def _assert_bwd_close(w, t, dq, dk, dv, causal=True, rounding_aware=False):
    """max-abs <= O_TOL on valid rows.  With rounding_aware, the bar applies to
    the error beyond the bf16 rounding of the result (half an ulp of the
    reference value), used for GQA stress cases whose summed dK/dV reach
    magnitudes where that rounding alone is 0.016-0.031."""
    ref = orc.attn_bwd(*(t[x].float().numpy() for x in ("q", "k", "v", "do")), w.cu_seqlens, w.cu_seqlens,
                       w.cu_seqlens_padded, w.cu_seqlens_padded, causal=causal, softmax_scale=w.softmax_scale,
                       dq_rows=w.dq_rows, dkv_rows=w.dkv_rows)
    valid = np.zeros(w.dq_rows, bool)
    valid[:w.T] = inputs.valid_row_mask(w)
    errs = []
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = f64(got)
        e = float(np.abs(g[valid] - r[valid]).max()) if valid.any() else 0.0
        worst = float(np.abs(r[valid]).max()) if valid.any() else 0.0
        if rounding_aware:
            ex = rounding_aware_excess(g[valid], r[valid]) if valid.any() else 0.0
            assert ex <= O_TOL, f"{name} max-abs {e:.3e}, beyond bf16 rounding {ex:.3e} (largest |ref| {worst:.2f})"
        else:
            assert e <= O_TOL, f"{name} max-abs {e:.3e} (largest |ref| {worst:.2f})"
        assert np.all(g[~valid] == 0), f"{name}: rows without a valid token must be 0"
        errs.append(e)
    return errs


def test_tiny_workload_backward_matches_oracle():
    w = inputs.make_workload("tiny")
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    _, _, dq, dk, dv = _run(w, d)
    _assert_bwd_close(w, t, dq, dk, dv)


CASES = [
    ([8, 16, 24], 1, 2, 1, 64, 0),
    ([4, 252, 8, 132], 2, 2, 2, 64, 0),
    ([512, 1024, 264], 4, 4, 2, 128, 0),
    ([600, 16, 1000], 4, 4, 4, 128, 64),
    ([130, 3, 257, 0, 61], 2, 6, 2, 64, 16),
    ([1536, 24], 3, 2, 1, 128, 0),
    ([2048], 8, 2, 2, 128, 0),
    ([96, 160, 2000], 8, 4, 1, 64, 0),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_custom_cases_backward_match_oracle(case):
    lengths, cp, Hq, Hkv, D, pad_to = CASES[case]
    w = _custom(lengths, cp, Hq, Hkv, D, pad_to, seed=20 + case, slack=0.05 * (case % 3))
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    _, _, dq, dk, dv = _run(w, d)
    _assert_bwd_close(w, t, dq, dk, dv, rounding_aware=Hq > Hkv)


@pytest.mark.parametrize("case", [1, 3])
def test_non_causal_backward_matches_oracle(case):
    lengths, cp, Hq, Hkv, D, pad_to = CASES[case]
    w = _custom(lengths, cp, Hq, Hkv, D, pad_to, seed=40 + case)
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    _, _, dq, dk, dv = _run(w, d, causal=False)
    _assert_bwd_close(w, t, dq, dk, dv, causal=False)


def test_value_equal_padded_metadata_backward():
    """[P2]: every way of saying 'no padding' takes the same path, and every
    gradient is summed in a fixed order, so all of dQ, dK, dV are bit-identical."""
    w = inputs.make_workload("tiny")
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    _, _, dq0, dk0, dv0 = _run(w, d, cu_pad=None)
    for flag, cp in ((-1, d["cu_pad"]), (0, d["cu_pad"]), (1, d["cu_pad"]), (-1, d["cu"])):
        _, _, dq, dk, dv = _run(w, d, pad_flag=flag, cu_pad=cp)
        assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
        assert torch.equal(dq, dq0)


def test_slack_rows_are_tail_zeroed():
    w = _custom([128, 256], 2, 2, 2, 64, slack=0.25)
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    _, _, dq, dk, dv = _run(w, d, canary=5.0)
    for g in (dq, dk, dv):
        assert torch.all(g[w.T:] == 0)


def _sub_problem(w, t, b, heads):
    """Slice sequence b (its valid rows) out of a workload for the oracle."""
    off = int(w.cu_seqlens_padded[b])
    L = w.lengths[b]
    sl = slice(off, off + L)
    G = w.Hq // w.Hkv
    kv_heads = sorted({h // G for h in heads})
    q_heads = [hk * G + j for hk in kv_heads for j in range(G)]
    qq = t["q"][sl][:, q_heads].float().numpy()
    dd = t["do"][sl][:, q_heads].float().numpy()
    kk = t["k"][sl][:, kv_heads].float().numpy()
    vv = t["v"][sl][:, kv_heads].float().numpy()
    return sl, q_heads, kv_heads, qq, kk, vv, dd, L


@pytest.mark.parametrize("name,heads,n_seq", [("fwdbwd", [3], 4), ("padded", [9], 3), ("packed", [2], 3)])
def test_full_size_backward_sampled(name, heads, n_seq):
    """Full-size workloads in the bench's launch configuration; the oracle
    recomputes whole sequences (the shortest few plus one mid-length) for
    one query-head group."""
    w = inputs.make_workload(name)
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    _, _, dq, dk, dv = _run(w, d)
    order = np.argsort(w.lengths)
    pick = list(order[:n_seq - 1]) + [order[len(order) // 2]]
    worst = 0.0
    for b in pick:
        sl, q_heads, kv_heads, qq, kk, vv, dd, L = _sub_problem(w, t, int(b), heads)
        cu = np.array([0, L], np.int32)
        rq, rk, rv = orc.attn_bwd(qq, kk, vv, dd, cu, cu, softmax_scale=w.softmax_scale)
        gq = dq[sl][:, q_heads].float().cpu().numpy()
        gk = dk[sl][:, kv_heads].float().cpu().numpy()
        gv = dv[sl][:, kv_heads].float().cpu().numpy()
        for g, r in ((gq, rq), (gk, rk), (gv, rv)):
            worst = max(worst, float(np.abs(g - r).max()))
    assert worst <= O_TOL, f"sampled gradient max-abs {worst:.3e}"
    inv = torch.from_numpy(~inputs.valid_row_mask(w)).cuda()
    for g in (dq, dk, dv):
        assert torch.all(g[w.T:] == 0)
        if inv.any():
            assert torch.all(g[:w.T][inv] == 0)
        assert torch.isfinite(g.float()).all()


def test_backward_bit_reproducible_over_repeats():
    """dK/dV accumulate in TMEM over the key tile's query steps and dQ over
    the query tile's key tiles, each in a fixed order (no atomics): repeated
    calls agree bit for bit; a pipeline race between the MMA, producer and
    compute roles shows up here as run-to-run differences."""
    w = inputs.make_workload("packed")
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    o, lse, dq0, dk0, dv0 = _run(w, d)
    for _ in range(10):
        dq, dk, dv, st = T.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], d["cu"], d["cu_pad"],
                                    d["cu_pad"], cp_size=w.cp_size, softmax_scale=w.softmax_scale)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert torch.equal(dk, dk0) and torch.equal(dv, dv0)
        assert torch.equal(dq, dq0)
