"""GPU parity of the forward path (thd_attn_fwd / thd_attn_fwd_step /
thd_lse_merge) against the CPU fp64 oracle, through the C-ABI binding.

Bars: max-abs <= 2e-2 on O and <= 1e-3 on lse over valid rows; rows without a
valid token exactly 0 / -inf; value-equal padded metadata bit-identical."""

import numpy as np
import pytest
import torch

from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T
from thd_testutil import LSE_TOL, O_TOL, assert_fwd_close, device_inputs, f64, run_fwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True, params=[T.THD_FWD_KERNEL_SINGLE, T.THD_FWD_KERNEL_DUAL],
                ids=["single", "dual"])
def _lib(thd_lib, request):
    """Every test of this module runs once per forward kernel (the
    single-item kernel the library picks for long sequences, and the
    two-item one it picks for shorter ones)."""
    assert T.thd_test_select_fwd_kernel(request.param) == T.THD_OK
    yield thd_lib
    T.thd_test_select_fwd_kernel(0)


def _custom(lengths, cp, Hq=2, Hkv=2, D=64, pad_to=0, seed=0):
    return inputs.make_workload("custom", seed, lengths=lengths, pad_to=pad_to, Hq=Hq, Hkv=Hkv, D=D, cp_size=cp)


def test_tiny_workload_matches_oracle():
    w = inputs.make_workload("tiny")
    t = inputs.make_tensors(w)
    d = device_inputs(w, t)
    o, lse, st = run_fwd(w, d)
    assert st == 0
    assert_fwd_close(w, t, o, lse)


def test_value_equal_padded_metadata_is_bit_identical():
    """[P2]: a separately allocated, value-equal padded cu_seqlens must take
    the no-padding path; every way of saying 'no padding' gives the same bits."""
    w = inputs.make_workload("tiny")
    t = inputs.make_tensors(w)
    d = device_inputs(w, t)
    assert d["cu_pad"].data_ptr() != d["cu"].data_ptr()
    ref_o, ref_l, st = run_fwd(w, d, cu_pad=None)
    assert st == 0
    variants = [
        dict(pad_flag=-1, cu_pad=d["cu"]),        # same pointer
        dict(pad_flag=-1, cu_pad=d["cu_pad"]),    # value-equal clone, auto
        dict(pad_flag=0, cu_pad=d["cu_pad"]),
        dict(pad_flag=1, cu_pad=d["cu_pad"]),     # forced padding with equal values
    ]
    for kw in variants:
        o, l, st = run_fwd(w, d, **kw)
        assert st == 0
        assert torch.equal(o, ref_o), kw
        assert torch.equal(l, ref_l), kw


CASES = [
    # lengths, cp, Hq, Hkv, D, pad_to
    ([8, 16, 24], 1, 2, 1, 64, 0),
    ([4, 252, 8, 132], 2, 2, 2, 64, 0),
    ([512, 1024, 264], 4, 4, 2, 128, 0),
    ([600, 16, 1000], 4, 4, 4, 128, 64),          # inter-sequence padding
    ([130, 3, 257, 0, 61], 2, 6, 2, 64, 16),      # ragged, an empty sequence, GQA
    ([1536, 24], 3, 2, 1, 128, 0),                # cp = 3
    ([2048], 8, 2, 2, 128, 0),                    # cb = 128 exactly
    ([96, 160, 2000], 8, 4, 1, 64, 0),            # tiny chunks (6, 10 rows)
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_custom_cases_match_oracle(case):
    lengths, cp, Hq, Hkv, D, pad_to = CASES[case]
    w = _custom(lengths, cp, Hq, Hkv, D, pad_to, seed=case)
    t = inputs.make_tensors(w)
    d = device_inputs(w, t)
    o, lse, st = run_fwd(w, d)
    assert st == 0
    assert_fwd_close(w, t, o, lse)


@pytest.mark.parametrize("case", [1, 3, 4])
def test_non_causal_matches_oracle(case):
    lengths, cp, Hq, Hkv, D, pad_to = CASES[case]
    w = _custom(lengths, cp, Hq, Hkv, D, pad_to, seed=10 + case)
    t = inputs.make_tensors(w)
    d = device_inputs(w, t)
    o, lse, st = run_fwd(w, d, causal=False)
    assert st == 0
    assert_fwd_close(w, t, o, lse, causal=False)


def test_buffer_tail_rows_are_zero():
    w = _custom([256, 64], 2, 2, 2, 64)
    t = inputs.make_tensors(w)
    d = device_inputs(w, t)
    o, lse, st = run_fwd(w, d, T_q=w.T + 77)
    assert st == 0
    og, lg = f64(o), f64(lse)
    assert np.all(og[w.T:] == 0) and np.all(np.isneginf(lg[:, w.T:]))


def test_invalid_metadata_sets_status_and_leaves_output_untouched():
    w = _custom([64, 128], 2, 2, 2, 64)
    t = inputs.make_tensors(w)
    d = device_inputs(w, t)
    d["cu"] = torch.tensor([0, 62, 190], dtype=torch.int32, device="cuda")   # 62 % 4 != 0
    canary = 3.0
    o, lse, st = run_fwd(w, d, cu_pad=None, out_canary=canary)
    assert st == T.THD_DEV_ERR_NOT_DIVISIBLE
    assert torch.all(o == canary)


def test_step_partials_match_oracle_ring_and_merge_to_fused():
    """Materialised ring: each step's partial against the oracle's emulated
    ring, and thd_lse_merge over the steps equals the fused result."""
    w = _custom([320, 96, 640], 4, 4, 2, 128, seed=7)
    t = inputs.make_tensors(w)
    d = device_inputs(w, t)
    qn, kn, vn = (t[x].float().numpy() for x in ("q", "k", "v"))
    _, _, parts = orc.cp_ring_fwd(qn, kn, vn, w.cu_seqlens, w.cu_seqlens_padded, w.cp_size,
                                  softmax_scale=w.softmax_scale, return_partials=True)
    valid = inputs.valid_row_mask(w)
    acc_o = torch.zeros((w.T, w.Hq, w.D), dtype=torch.float32, device="cuda")
    acc_l = torch.full((w.Hq, w.T), float("-inf"), dtype=torch.float32, device="cuda")
    for i in range(w.cp_size):
        o_i, l_i, st = T.attn_fwd_step(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"],
                                       step=i, cp_size=w.cp_size, softmax_scale=w.softmax_scale)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        O_ref, l_ref = parts[i]
        og, lg = f64(o_i), f64(l_i)
        fin = np.isfinite(l_ref)
        assert np.array_equal(fin, np.isfinite(lg)), f"step {i}: rows with a contribution differ"
        assert np.abs(og[valid] - O_ref[valid]).max() <= 5e-3
        assert np.abs(lg[fin] - l_ref[fin]).max() <= LSE_TOL
        T.lse_merge(acc_o, acc_l, o_i, l_i)
    torch.cuda.synchronize()
    o, lse, st = run_fwd(w, d)
    assert st == 0
    assert (acc_o[valid] - o.float()[valid]).abs().max().item() <= O_TOL
    assert (acc_l[:, valid] - lse[:, valid]).abs().max().item() <= LSE_TOL
    assert_fwd_close(w, t, acc_o, acc_l)


@pytest.mark.parametrize("name", ["packed", "padded"])
def test_forward_is_bit_reproducible_over_repeats(name):
    """Every output element is produced by one work item in a fixed order, so
    repeated calls must agree bit for bit; a pipeline race between the MMA,
    producer and softmax roles shows up here as run-to-run differences."""
    w = inputs.make_workload(name)
    t = inputs.make_tensors(w, with_grad=False)
    d = device_inputs(w, t)
    o0, l0, st = run_fwd(w, d)
    assert st == 0
    for _ in range(25):
        o, lse, st = T.attn_fwd(d["q"], d["k"], d["v"], d["cu"], d["cu"], d["cu_pad"], d["cu_pad"],
                                cp_size=w.cp_size, softmax_scale=w.softmax_scale)
        assert torch.equal(o, o0) and torch.equal(lse, l0)
    torch.cuda.synchronize()
