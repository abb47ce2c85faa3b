"""The allocation-free forward entry point (thd_attn_fwd_noalloc).

It serves callers that cannot allocate device memory at the call site (a
plug-in handed only input/output pointers by a framework that owns the
device memory, a serving loop with a fixed memory plan, code that must not
call cudaMalloc).  Its scratch is a static array inside the library.  Checked
here through the C ABI against thd_attn_fwd, on two calls in a row (the
second reuses the array the first left behind), plus the size limit.  This
file is collected last so that a failure here never hides another test."""

import pytest
import torch

from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T
from thd_testutil import device_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(thd_lib):
    return thd_lib


def _noalloc(w, d):
    o = torch.empty_like(d["q"])
    lse = torch.empty((w.Hq, w.T), dtype=torch.float32, device="cuda")
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    rc = T.thd_attn_fwd_noalloc(d["q"], d["k"], d["v"], o, lse, d["cu"], d["cu"], d["cu_pad"], d["cu_pad"], w.B,
                                w.T, w.T, w.Hq, w.Hkv, w.D, 1, w.softmax_scale, w.cp_size, -1, st)
    assert rc == T.THD_OK, T.thd_status_string(rc)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o, lse


def _with_workspace(w, d):
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"],
                            cp_size=w.cp_size, softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o, lse


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    cases = [
        inputs.make_workload("custom", 3, lengths=[600, 16, 1000], pad_to=64, Hq=4, Hkv=2, D=128, cp_size=4),
        inputs.make_workload("tiny"),
    ]
    for w in cases:   # two calls in a row on different problems share the one static array
        d = device_inputs(w, inputs.make_tensors(w))
        o1, l1 = _noalloc(w, d)
        o2, l2 = _with_workspace(w, d)
        # the same planner and kernels with the same grid: the results agree
        # bit for bit (a tolerance could hide stale scratch from the call before)
        assert torch.equal(o1, o2)
        assert torch.equal(l1, l2)


def test_noalloc_rejects_problems_beyond_its_static_scratch():
    # far more schedule entries than 1 MiB holds: refused before any launch
    n0 = T.thd_launch_count()
    rc = T.thd_attn_fwd_noalloc(16, 16, 16, 16, 16, 16, 16, None, None, 1, 1 << 30, 1 << 30, 1, 1, 128, 1, 0.1,
                                1, -1, 16, stream=0)
    assert rc == T.THD_ERR_WORKSPACE
    assert T.thd_launch_count() == n0


def test_noalloc_reports_the_same_errors_as_the_workspace_entry_point():
    # an unsupported head dim is UNSUPPORTED through both entry points, and nothing is launched
    n0 = T.thd_launch_count()
    args = (16, 16, 16, 16, 16, 16, 16, None, None, 1, 128, 128, 2, 2, 96, 1, 0.1, 1, -1)
    rc = T.thd_attn_fwd_noalloc(*args, 16, stream=0)
    assert rc == T.THD_ERR_UNSUPPORTED
    assert T.thd_attn_fwd(*args, None, 0, 16, stream=0) == rc
    assert T.thd_launch_count() == n0
