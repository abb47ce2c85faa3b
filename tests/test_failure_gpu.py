"""Failure detection without a GPU fault: a bounded device wait that runs out.

thd_test_arm_stall makes the next launch of one attention kernel wait on a
barrier that nothing completes.  The wait is the kernels' own bounded wait
(2 s on the global timer); when it gives up, the CTA takes its abort path,
frees its tensor memory and writes THD_ERR_TIMEOUT to the call's status
word.  Checked here for the forward, dQ and dK/dV kernels: the status is
THD_ERR_TIMEOUT, the stalled kernel wrote none of its outputs (canaries
intact; a later kernel of the same call sees the status and writes nothing
either), and the next normal call on the same device succeeds and matches
the oracle."""

import time

import numpy as np
import pytest
import torch

from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T
from thd_testutil import assert_fwd_close, assert_within_bar, device_inputs, f64

pytestmark = pytest.mark.gpu
CANARY = 7.0


@pytest.fixture(scope="module", autouse=True)
def _lib(thd_lib):
    yield thd_lib
    T.thd_test_arm_stall(0)


def _tiny():
    w = inputs.make_workload("tiny")
    t = inputs.make_tensors(w, with_grad=True)
    return w, t, device_inputs(w, t)


@pytest.mark.parametrize("fwd_kernel", [T.THD_FWD_KERNEL_SINGLE, T.THD_FWD_KERNEL_DUAL], ids=["single", "dual"])
def test_forward_wait_runs_out_then_device_recovers(fwd_kernel):
    assert T.thd_test_select_fwd_kernel(fwd_kernel) == T.THD_OK
    try:
        _forward_stall_case()
    finally:
        T.thd_test_select_fwd_kernel(0)


def _forward_stall_case():
    w, t, d = _tiny()
    o = torch.full_like(d["q"], CANARY)
    assert T.thd_test_arm_stall(T.THD_KERNEL_FWD) == T.THD_OK
    t0 = time.perf_counter()
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"], cp_size=w.cp_size,
                            softmax_scale=w.softmax_scale, out=o)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 >= 1.0          # the bounded wait really ran its course
    assert int(st.item()) == T.THD_ERR_TIMEOUT
    assert torch.all(o == CANARY)                   # no output written
    o2, lse2, st2 = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"],
                               cp_size=w.cp_size, softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    assert_fwd_close(w, t, o2, lse2)


@pytest.mark.parametrize("kernel", ["dq", "dkdv"])
def test_backward_wait_runs_out_then_device_recovers(kernel):
    w, t, d = _tiny()
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"], cp_size=w.cp_size,
                            softmax_scale=w.softmax_scale)
    grads = [torch.full((w.T, H, w.D), CANARY, dtype=torch.bfloat16, device="cuda") for H in (w.Hq, w.Hkv, w.Hkv)]
    kid = T.THD_KERNEL_BWD_DQ if kernel == "dq" else T.THD_KERNEL_BWD
    assert T.thd_test_arm_stall(kid) == T.THD_OK
    dq, dk, dv, st2 = T.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], d["cu"], d["cu_pad"],
                                 d["cu_pad"], cp_size=w.cp_size, softmax_scale=w.softmax_scale, dq=grads[0],
                                 dk=grads[1], dv=grads[2])
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(st2.item()) == T.THD_ERR_TIMEOUT
    # the dQ pass runs before the dK/dV pass: when it stalls the dK/dV pass sees
    # the status and writes nothing; when the dK/dV pass stalls, dQ is complete
    assert torch.all(dk == CANARY) and torch.all(dv == CANARY)
    assert torch.all(dq == CANARY) if kernel == "dq" else not torch.any(dq == CANARY)
    dq, dk, dv, st3 = T.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], d["cu"], d["cu_pad"],
                                 d["cu_pad"], cp_size=w.cp_size, softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert int(st3.item()) == 0
    ref = orc.attn_bwd(*(t[x].float().numpy() for x in ("q", "k", "v", "do")), w.cu_seqlens, w.cu_seqlens,
                       softmax_scale=w.softmax_scale)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_within_bar(name, f64(g), r)


def test_stall_hook_is_one_shot_and_checks_its_argument():
    assert T.thd_test_select_fwd_kernel(3) == T.THD_ERR_INVALID_ARG
    assert T.thd_test_arm_stall(T.THD_KERNEL_LSE_MERGE) == T.THD_ERR_INVALID_ARG
    assert T.thd_test_arm_stall(T.THD_KERNEL_FWD) == T.THD_OK
    assert T.thd_test_arm_stall(0) == T.THD_OK      # disarmed: the next forward runs normally
    w, t, d = _tiny()
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"], cp_size=w.cp_size,
                            softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.isfinite(lse.cpu().numpy()).all()
