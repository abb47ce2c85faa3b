"""GPU parity of bottom-right causal attention (T_q != T_kv, query i sees
key j iff j <= i + L_kv - L_q) through the C ABI: forward, backward and the
materialised ring steps against the CPU fp64 oracle's BOTTOM_RIGHT mode,
with fewer queries than keys, more queries than keys (the first
L_q - L_kv queries see no key: O = 0, lse = -inf, zero gradients), ragged
and padded sequences, GQA, and cp_size 1 to 4."""

import numpy as np
import pytest
import torch

from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T
from thd_testutil import LSE_TOL, O_TOL, assert_within_bar, f64

pytestmark = pytest.mark.gpu
BR = orc.BOTTOM_RIGHT

CASES = [
    # L_q, L_kv, cp, Hq, Hkv, D, pad_to
    ([100, 300, 17], [500, 300, 90], 2, 2, 2, 64, 16),
    ([1000, 40], [130, 700], 4, 4, 2, 128, 64),
    ([257, 0, 600], [64, 128, 2048], 1, 4, 1, 128, 8),
    ([384, 129], [2000, 1500], 3, 2, 1, 64, 48),
]


@pytest.fixture(scope="module", autouse=True, params=[T.THD_FWD_KERNEL_SINGLE, T.THD_FWD_KERNEL_DUAL],
                ids=["single", "dual"])
def _lib(thd_lib, request):
    """Every test of this module runs once per forward kernel (the
    single-item kernel the library picks for long sequences, and the
    two-item one it picks for shorter ones)."""
    assert T.thd_test_select_fwd_kernel(request.param) == T.THD_OK
    yield thd_lib
    T.thd_test_select_fwd_kernel(0)


def _case(i, grad=True):
    Lq, Lk, cp, Hq, Hkv, D, pad = CASES[i]
    c = inputs.make_cross(Lq, Lk, pad_to=pad, Hq=Hq, Hkv=Hkv, D=D, cp_size=cp, seed=60 + i, with_grad=grad)
    d = {k: (torch.from_numpy(v).cuda() if isinstance(v, np.ndarray) else v.cuda())
         for k, v in c.items() if k not in ("L_q", "L_kv")}
    return c, d, cp, 1.0 / np.sqrt(D)


def _valid_q(c):
    m = np.zeros(int(c["cu_q_pad"][-1]), bool)
    for b, n in enumerate(c["L_q"]):
        m[int(c["cu_q_pad"][b]):int(c["cu_q_pad"][b]) + n] = True
    return m


@pytest.mark.parametrize("case", range(len(CASES)))
def test_bottom_right_forward_and_backward_match_oracle(case):
    c, d, cp, scale = _case(case)
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu_q"], d["cu_kv"], d["cu_q_pad"], d["cu_kv_pad"],
                            cp_size=cp, causal=T.THD_CAUSAL_BOTTOM_RIGHT, softmax_scale=scale)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, T.thd_status_string(int(st.item()))
    args = (c["cu_q"], c["cu_kv"], c["cu_q_pad"], c["cu_kv_pad"])
    qn, kn, vn, don = (c[x].float().numpy() for x in ("q", "k", "v", "do"))
    O_ref, l_ref = orc.attn_fwd(qn, kn, vn, *args, causal=BR, softmax_scale=scale)
    og, lg = f64(o), f64(lse)
    valid = _valid_q(c)
    seen = valid & np.isfinite(l_ref).all(axis=0)        # rows that see at least one key
    assert np.abs(og[valid] - O_ref[valid]).max() <= O_TOL
    assert np.abs(lg[:, seen] - l_ref[:, seen]).max() <= LSE_TOL
    assert np.all(og[~seen] == 0) and np.all(np.isneginf(lg[:, ~seen]))
    if case in (1, 2):
        assert (valid & ~seen).any(), "the case has queries that see no key"
    dq, dk, dv, st2 = T.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu_q"], d["cu_kv"], d["cu_q_pad"],
                                 d["cu_kv_pad"], cp_size=cp, causal=T.THD_CAUSAL_BOTTOM_RIGHT, softmax_scale=scale)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = orc.attn_bwd(qn, kn, vn, don, *args, causal=BR, softmax_scale=scale)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        gg = f64(g)
        assert np.isfinite(gg).all(), name
        assert_within_bar(name, gg, r)
    assert np.all(f64(dq)[~seen] == 0)


@pytest.mark.parametrize("case", [0, 1, 3])
def test_bottom_right_ring_steps_match_the_oracle_ring(case):
    """Each ring step's materialised partial equals the oracle's positional-
    mask ring partial, and merging them gives the fused forward."""
    c, d, cp, scale = _case(case, grad=False)
    qn, kn, vn = (c[x].float().numpy() for x in ("q", "k", "v"))
    args = (c["cu_q"], c["cu_kv"], c["cu_q_pad"], c["cu_kv_pad"])
    O_ref, l_ref, parts = orc.cp_ring_fwd_masked(qn, kn, vn, *args, cp, causal=BR, softmax_scale=scale,
                                                 return_partials=True)
    valid = _valid_q(c)
    acc_o = torch.zeros((int(c["cu_q_pad"][-1]),) + tuple(d["q"].shape[1:]), device="cuda")
    acc_l = torch.full((d["q"].shape[1], acc_o.shape[0]), float("-inf"), device="cuda")
    for i in range(cp):
        o, l, st = T.attn_fwd_step(d["q"], d["k"], d["v"], d["cu_q"], d["cu_kv"], d["cu_q_pad"], d["cu_kv_pad"],
                                   step=i, cp_size=cp, causal=T.THD_CAUSAL_BOTTOM_RIGHT, softmax_scale=scale)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        Oi, li = parts[i]
        og, lg = f64(o), f64(l)
        assert np.abs(og[valid] - Oi[valid]).max() <= 1e-2
        fin = np.isfinite(li)
        assert np.array_equal(np.isneginf(lg[:, valid]), ~fin[:, valid])
        assert np.abs(lg[fin] - li[fin]).max() <= LSE_TOL
        T.lse_merge(acc_o, acc_l, o, l)
    torch.cuda.synchronize()
    ao, al = f64(acc_o), f64(acc_l)
    assert np.abs(ao[valid] - O_ref[valid]).max() <= O_TOL
    fin = np.isfinite(l_ref) & valid[None, :]
    assert np.abs(al[fin] - l_ref[fin]).max() <= LSE_TOL


def test_top_left_still_rejects_unequal_lengths_on_the_device():
    c, d, cp, scale = _case(0, grad=False)
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu_q"], d["cu_kv"], d["cu_q_pad"], d["cu_kv_pad"],
                            cp_size=cp, causal=T.THD_CAUSAL_TOP_LEFT, softmax_scale=scale)
    torch.cuda.synchronize()
    assert int(st.item()) == T.THD_DEV_ERR_CAUSAL_LENGTHS
