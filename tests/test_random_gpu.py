"""GPU parity on seeded random metadata, against the CPU fp64 oracle: batch
size, sequence lengths (empty ones included), cp size, the GQA ratio, head
dimension, padding between sequences, causal or not, and gradient-buffer
slack are all drawn per case, so that chunk boundaries land at every offset
inside the 128-row tiles.  Each case runs the forward on both forward
kernels and the backward, through the C-ABI binding.

Bars as everywhere: the bf16 bar on O, dQ, dK, dV (error beyond the result's
own bf16 rounding within 2e-2, raw error within 2e-2 where |ref| < 2), lse
within 1e-3; rows without a valid token exactly 0 (-inf for lse)."""

import numpy as np
import pytest
import torch

from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T
from thd_testutil import assert_fwd_close, assert_within_bar, device_inputs, f64

N_CASES = 40


@pytest.fixture(scope="module")
def _lib(thd_lib):
    yield thd_lib
    T.thd_test_select_fwd_kernel(0)


def _draw(seed):
    """One random configuration.  Padded lengths must be multiples of 2 cp:
    without padding the lengths are drawn as such multiples, with padding
    the pad unit is one."""
    rng = np.random.default_rng(5000 + seed)
    cp = int(rng.choice([1, 2, 3, 4, 6, 8]))
    D = int(rng.choice([64, 128]))
    Hkv = int(rng.choice([1, 2, 4]))
    G = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 7))
    unit = 2 * cp
    padded = bool(rng.integers(0, 2))
    if padded:
        pad_to = unit * int(rng.choice([1, 2, 4, 8]))
        lengths = rng.integers(0, 1600, size=B)
    else:
        pad_to = 0
        lengths = unit * rng.integers(0, 1600 // unit + 1, size=B)
    lengths[rng.random(B) < 0.15] = 0          # some empty sequences
    if not lengths.any():
        lengths[0] = unit                      # but never an empty batch
    causal = bool(rng.random() < 0.75)
    slack = float(rng.choice([0.0, 0.05, 0.3]))
    w = inputs.make_workload("custom", 6000 + seed, lengths=[int(x) for x in lengths], pad_to=pad_to,
                             Hq=Hkv * G, Hkv=Hkv, D=D, cp_size=cp, grad_slack=slack)
    return w, causal


@pytest.mark.gpu
@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_metadata_matches_oracle(seed, _lib):
    w, causal = _draw(seed)
    t = inputs.make_tensors(w, with_grad=True)
    d = device_inputs(w, t)
    outs = []
    for kernel in (T.THD_FWD_KERNEL_SINGLE, T.THD_FWD_KERNEL_DUAL):
        assert T.thd_test_select_fwd_kernel(kernel) == T.THD_OK
        try:
            o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"],
                                    cp_size=w.cp_size, causal=causal, softmax_scale=w.softmax_scale)
            torch.cuda.synchronize()
        finally:
            T.thd_test_select_fwd_kernel(0)
        assert int(st.item()) == 0
        assert_fwd_close(w, t, o, lse, causal=causal)
        outs.append((o, lse))
    o, lse = outs[1]
    canary = 7.0
    dq = torch.full((w.dq_rows, w.Hq, w.D), canary, dtype=torch.bfloat16, device="cuda")
    dk = torch.full((w.dkv_rows, w.Hkv, w.D), canary, dtype=torch.bfloat16, device="cuda")
    dv = torch.full_like(dk, canary)
    dq, dk, dv, st2 = T.attn_bwd(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], d["cu"], d["cu_pad"],
                                 d["cu_pad"], cp_size=w.cp_size, causal=causal, softmax_scale=w.softmax_scale,
                                 dq_rows=w.dq_rows, dkv_rows=w.dkv_rows, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    ref = orc.attn_bwd(*(t[x].float().numpy() for x in ("q", "k", "v", "do")), w.cu_seqlens, w.cu_seqlens,
                       w.cu_seqlens_padded, w.cu_seqlens_padded, causal=causal, softmax_scale=w.softmax_scale,
                       dq_rows=w.dq_rows, dkv_rows=w.dkv_rows)
    valid = np.zeros(w.dq_rows, bool)
    valid[:w.T] = inputs.valid_row_mask(w)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        g = f64(got)
        if valid.any():
            assert_within_bar(name, g[valid], r[valid])
        assert np.all(g[~valid] == 0), f"{name}: rows without a valid token must be 0"


def test_random_draws_cover_the_space():
    """The drawn cases span what they are meant to: several cp sizes, both
    head dimensions, GQA and MHA, padded and unpadded, an empty sequence,
    non-causal and slack (the metadata alone: no GPU needed)."""
    ws = [_draw(s) for s in range(N_CASES)]
    assert len({w.cp_size for w, _ in ws}) >= 4
    assert {w.D for w, _ in ws} == {64, 128}
    assert any(w.Hq > w.Hkv for w, _ in ws) and any(w.Hq == w.Hkv for w, _ in ws)
    assert any(not np.array_equal(w.cu_seqlens, w.cu_seqlens_padded) for w, _ in ws)
    assert any(np.array_equal(w.cu_seqlens, w.cu_seqlens_padded) for w, _ in ws)
    assert any(0 in w.lengths for w, _ in ws)
    assert any(not c for _, c in ws) and any(c for _, c in ws)
    assert any(w.grad_slack > 0 for w, _ in ws)
