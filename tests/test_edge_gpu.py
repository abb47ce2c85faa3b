"""GPU parity on the edges of the metadata the entry points accept, against
the CPU fp64 oracle, forward (both forward kernels) and backward:

* hundreds of short sequences (0-64 tokens), so that most CP chunks hold a
  handful of rows or none;
* a large CP size (32: 64 chunks of 32 and 64 rows);
* multi-query attention (one kv head for eight query heads).

Bars as everywhere: the bf16 bar on O, dQ, dK, dV (error beyond the result's
own bf16 rounding within 2e-2), lse within 1e-3; rows without a valid token
exactly 0 (and -inf for lse).  Head dimension 128, that of every benchmark
workload: with 64 the short-sequence backward case reaches a raw dQ error of
0.022 at |dQ| = 1.2 (up to 0.014 of it from Delta = rowsum(dO * O) taken on
the bf16 O the backward receives, which the fp64 oracle does not round)."""

import numpy as np
import pytest
import torch

from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T
from thd_testutil import assert_fwd_close, assert_within_bar, device_inputs, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(thd_lib):
    yield thd_lib
    T.thd_test_select_fwd_kernel(0)


def _many_short():
    rng = np.random.default_rng(71)
    return rng.integers(0, 65, size=400).tolist()


CASES = {
    # name: (lengths, cp, Hq, Hkv, D, pad_to)
    "many_short": (_many_short(), 4, 4, 2, 128, 8),
    "cp32": ([2048, 4096], 32, 2, 1, 128, 0),
    "mqa": ([1000, 3000], 4, 8, 1, 128, 0),
}


def _workload(name):
    lengths, cp, Hq, Hkv, D, pad_to = CASES[name]
    return inputs.make_workload("custom", 90, lengths=lengths, pad_to=pad_to, Hq=Hq, Hkv=Hkv, D=D, cp_size=cp,
                                grad_slack=0.05)


@pytest.mark.parametrize("kernel", [T.THD_FWD_KERNEL_SINGLE, T.THD_FWD_KERNEL_DUAL], ids=["single", "dual"])
@pytest.mark.parametrize("name", list(CASES))
def test_forward_on_metadata_edges(name, kernel):
    w = _workload(name)
    t = inputs.make_tensors(w)
    d = device_inputs(w, t)
    assert T.thd_test_select_fwd_kernel(kernel) == T.THD_OK
    try:
        o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"],
                                cp_size=w.cp_size, softmax_scale=w.softmax_scale)
        torch.cuda.synchronize()
    finally:
        T.thd_test_select_fwd_kernel(0)
    assert int(st.item()) == 0
    assert_fwd_close(w, t, o, lse)


@pytest.mark.parametrize("name", list(CASES))
def test_backward_on_metadata_edges(name):
    w = _workload(name)
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"], cp_size=w.cp_size,
                            softmax_scale=w.softmax_scale)
    canary = 7.0
    dq = torch.full((w.dq_rows, w.Hq, w.D), canary, dtype=torch.bfloat16, device="cuda")
    dk = torch.full((w.dkv_rows, w.Hkv, w.D), canary, dtype=torch.bfloat16, device="cuda")
    dv = torch.full_like(dk, canary)
    dq, dk, dv, st2 = T.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], d["cu"], d["cu_pad"],
                                 d["cu_pad"], cp_size=w.cp_size, softmax_scale=w.softmax_scale, dq_rows=w.dq_rows,
                                 dkv_rows=w.dkv_rows, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and int(st2.item()) == 0
    ref = orc.attn_bwd(*(t[x].float().numpy() for x in ("q", "k", "v", "do")), w.cu_seqlens, w.cu_seqlens,
                       w.cu_seqlens_padded, w.cu_seqlens_padded, softmax_scale=w.softmax_scale, dq_rows=w.dq_rows,
                       dkv_rows=w.dkv_rows)
    valid = np.zeros(w.dq_rows, bool)
    valid[:w.T] = inputs.valid_row_mask(w)
    for gname, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = f64(got)
        assert_within_bar(gname, g[valid], r[valid])
        assert np.all(g[~valid] == 0), f"{gname}: rows without a valid token (pad, slack) must be 0"


def _offset_buffer(shape, dtype, offset):
    """A [shape] view that starts `offset` elements past a 256-byte aligned allocation."""
    n = int(np.prod(shape))
    big = torch.full((n + offset,), 7.0, dtype=dtype, device="cuda")
    return big[offset:].view(*shape)


@pytest.mark.parametrize("kernel", [T.THD_FWD_KERNEL_SINGLE, T.THD_FWD_KERNEL_DUAL], ids=["single", "dual"])
def test_forward_into_16_byte_aligned_buffers_is_bit_identical(kernel):
    """O buffers aligned to 16 bytes but not 32 (bf16 O and bf16 / fp32 step
    partials): the forward kernels then write rows with 16-byte stores instead
    of 32-byte ones; the results must be the same bits."""
    w = _workload("mqa")
    t = inputs.make_tensors(w)
    d = device_inputs(w, t)
    shape = (w.T, w.Hq, w.D)
    assert T.thd_test_select_fwd_kernel(kernel) == T.THD_OK
    try:
        def run(offset_bf16, offset_f32):
            o, _, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"],
                                  cp_size=w.cp_size, softmax_scale=w.softmax_scale,
                                  out=_offset_buffer(shape, torch.bfloat16, offset_bf16))
            ob, _, stb = T.attn_fwd_step_bf16(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"],
                                              step=1, cp_size=w.cp_size, softmax_scale=w.softmax_scale,
                                              out=_offset_buffer(shape, torch.bfloat16, offset_bf16))
            of, _, stf = T.attn_fwd_step(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"],
                                         step=1, cp_size=w.cp_size, softmax_scale=w.softmax_scale,
                                         out=_offset_buffer(shape, torch.float32, offset_f32))
            torch.cuda.synchronize()
            assert int(st.item()) == 0 and int(stb.item()) == 0 and int(stf.item()) == 0
            return o, ob, of

        a = run(0, 0)
        b = run(8, 4)  # 16 bytes past a 256-byte aligned allocation
        assert b[0].data_ptr() % 32 == 16 and b[2].data_ptr() % 32 == 16
        for x, y in zip(a, b):
            assert torch.equal(x, y)
    finally:
        T.thd_test_select_fwd_kernel(0)


def test_backward_into_16_byte_aligned_buffers_is_bit_identical():
    """dQ/dK/dV buffers aligned to 16 bytes but not 32 (the API's minimum):
    the kernels then write rows with 16-byte stores instead of 32-byte ones;
    the results must be the same bits."""
    w = _workload("mqa")
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"], cp_size=w.cp_size,
                            softmax_scale=w.softmax_scale)

    def run(offset):
        out = [_offset_buffer((rows, H, w.D), torch.bfloat16, offset)
               for rows, H in ((w.dq_rows, w.Hq), (w.dkv_rows, w.Hkv), (w.dkv_rows, w.Hkv))]
        dq, dk, dv, st2 = T.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], d["cu"], d["cu_pad"],
                                     d["cu_pad"], cp_size=w.cp_size, softmax_scale=w.softmax_scale,
                                     dq_rows=w.dq_rows, dkv_rows=w.dkv_rows, dq=out[0], dk=out[1], dv=out[2])
        torch.cuda.synchronize()
        assert int(st2.item()) == 0
        return dq, dk, dv

    a = run(0)
    b = run(8)  # 8 bf16 = 16 bytes past a 256-byte aligned allocation
    assert b[0].data_ptr() % 32 == 16 and b[1].data_ptr() % 32 == 16
    for x, y in zip(a, b):
        assert torch.equal(x, y)
