"""GPU checks of the integer and HBM-bound entry points: thd_cp_partition
(bit-exact), thd_lse_merge and thd_grad_tail_zero."""

import os

import numpy as np
import pytest
import torch

from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import thd_attn as T

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib(thd_lib):
    return thd_lib


def _gpu_partition(cu, cu_pad, cp, pad_flag=-1):
    cu_t = torch.tensor(cu, dtype=torch.int32, device="cuda")
    pad_t = None if cu_pad is None else torch.tensor(cu_pad, dtype=torch.int32, device="cuda")
    T_ = int((cu if cu_pad is None else cu_pad)[-1])
    out, st = T.cp_partition(cu_t, pad_t, cp_size=cp, pad_between_seqs=pad_flag, token_map_capacity=max(T_, 1))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}, int(st.item()), T_


@pytest.mark.parametrize("fixture,cu,cu_pad", [
    ("tiny_partition.txt", [0, 64, 192], [0, 64, 192]),
    ("tiny_padded_partition.txt", [0, 50, 150], [0, 64, 192]),
])
def test_partition_matches_hand_derived_fixture(fixture, cu, cu_pad):
    from test_oracle_pins import _parse_golden
    g = _parse_golden(os.path.join(GOLDEN, fixture))
    cp = g["cp_size"]
    out, st, T_ = _gpu_partition(cu, cu_pad, cp)
    assert st == 0
    per = T_ // cp
    for r in range(cp):
        assert out["cu_rank"][r].tolist() == g["cu_rank"][r]
        assert out["cu_rank_padded"][r].tolist() == g["cu_rank_padded"][r]
        assert out["cu_rank_half"][r, 0].tolist() == g["cu_rank_half_first"][r]
        assert out["cu_rank_half"][r, 1].tolist() == g["cu_rank_half_second"][r]
        assert out["token_map"][r * per:(r + 1) * per].tolist() == g["token_map"][r]


@pytest.mark.parametrize("seed", range(10))
def test_partition_bit_exact_random(seed):
    rng = np.random.default_rng(seed)
    cp = int(rng.integers(1, 9))
    B = int(rng.integers(1, 40))
    unit = 2 * cp
    P = unit * rng.integers(0, 200, size=B)
    L = np.array([int(rng.integers(0, p + 1)) for p in P]) if seed % 2 else P.copy()
    cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    cu_pad = np.concatenate([[0], np.cumsum(P)]).astype(np.int32)
    out, st, T_ = _gpu_partition(cu, cu_pad, cp)
    assert st == 0
    ref = orc.cp_partition(cu, cu_pad, cp)
    assert np.array_equal(out["cu_rank"], ref["cu_rank"])
    assert np.array_equal(out["cu_rank_padded"], ref["cu_rank_padded"])
    assert np.array_equal(out["cu_rank_half"], ref["cu_rank_half"])
    if T_:
        assert np.array_equal(out["token_map"][:T_], ref["token_map"].reshape(-1))


def test_partition_pad_flag_and_errors():
    cu = [0, 50, 150]
    cu_pad = [0, 64, 192]
    out, st, _ = _gpu_partition(cu, cu_pad, 2, pad_flag=1)
    assert st == 0
    ref = orc.cp_partition(np.array(cu), np.array(cu_pad), 2)
    assert np.array_equal(out["cu_rank"], ref["cu_rank"])
    # pad flag 0: the padded array is ignored, so 50 % 4 != 0 is an error
    _, st, _ = _gpu_partition(cu, cu_pad, 2, pad_flag=0)
    assert st == T.THD_DEV_ERR_NOT_DIVISIBLE
    _, st, _ = _gpu_partition([0, 70], [0, 64], 2, pad_flag=1)
    assert st == T.THD_DEV_ERR_VALID_GT_PAD
    _, st, _ = _gpu_partition([0, 64, 32], None, 2)
    assert st == T.THD_DEV_ERR_NOT_MONOTONE
    _, st, _ = _gpu_partition([4, 64], None, 2)
    assert st == T.THD_DEV_ERR_NONZERO_START


@pytest.mark.parametrize("D", [64, 128, 12, 160, 4])
def test_lse_merge_matches_oracle(D):
    """D = 12 puts several rows in one warp (3 float4 each), D = 160 spreads a
    row over more float4s than a warp has lanes: the merged lse must come from
    the two inputs, never from a row's already-merged value."""
    rng = np.random.default_rng(D)
    Tn, H = 333, 3
    oa = rng.standard_normal((Tn, H, D)).astype(np.float32)
    ob = rng.standard_normal((Tn, H, D)).astype(np.float32)
    a = (rng.standard_normal((H, Tn)) * 4).astype(np.float32)
    b = (rng.standard_normal((H, Tn)) * 4).astype(np.float32)
    a[:, ::7] = -np.inf
    b[:, ::5] = -np.inf
    b[0, :10] = a[0, :10]
    oa[~np.isfinite(a).T] = 0
    ob[~np.isfinite(b).T] = 0
    O_ref, l_ref = orc.lse_merge(oa, a, ob, b)
    acc_o, acc_l = torch.tensor(oa, device="cuda"), torch.tensor(a, device="cuda")
    T.lse_merge(acc_o, acc_l, torch.tensor(ob, device="cuda"), torch.tensor(b, device="cuda"))
    torch.cuda.synchronize()
    go, gl = acc_o.cpu().numpy(), acc_l.cpu().numpy()
    assert np.array_equal(np.isneginf(gl), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.abs(gl[fin] - l_ref[fin]).max() <= 1e-5
    assert np.abs(go - O_ref).max() <= 1e-5
    assert np.all(go[np.isneginf(l_ref).T] == 0)


@pytest.mark.parametrize("D", [128, 12])
def test_lse_merge_bf16_partial_matches_oracle(D):
    """The bf16-partial merge equals the oracle's merge of the same (bf16-
    rounded) partial into the fp32 accumulator."""
    rng = np.random.default_rng(100 + D)
    Tn, H = 257, 4
    oa = rng.standard_normal((Tn, H, D)).astype(np.float32)
    ob16 = torch.tensor(rng.standard_normal((Tn, H, D)).astype(np.float32)).to(torch.bfloat16)
    ob = ob16.float().numpy()
    a = (rng.standard_normal((H, Tn)) * 4).astype(np.float32)
    b = (rng.standard_normal((H, Tn)) * 4).astype(np.float32)
    a[:, ::7] = -np.inf
    b[:, ::5] = -np.inf
    oa[~np.isfinite(a).T] = 0
    ob16[torch.from_numpy(~np.isfinite(b).T)] = 0
    ob = ob16.float().numpy()
    O_ref, l_ref = orc.lse_merge(oa, a, ob, b)
    acc_o, acc_l = torch.tensor(oa, device="cuda"), torch.tensor(a, device="cuda")
    T.lse_merge_bf16(acc_o, acc_l, ob16.cuda(), torch.tensor(b, device="cuda"))
    torch.cuda.synchronize()
    go, gl = acc_o.cpu().numpy(), acc_l.cpu().numpy()
    assert np.array_equal(np.isneginf(gl), np.isneginf(l_ref))
    fin = np.isfinite(l_ref)
    assert np.abs(gl[fin] - l_ref[fin]).max() <= 1e-5
    assert np.abs(go - O_ref).max() <= 1e-5


@pytest.mark.parametrize("end", [-16, 200])
def test_grad_tail_zero_ignores_an_endpoint_outside_the_buffer(end):
    """A corrupt endpoint (negative, or past the buffer's rows) writes nothing:
    the rows before the buffer (a canary) and the buffer itself stay as they were."""
    Hq, Hkv, D = 2, 2, 64
    pad = torch.tensor([0, 32, end], dtype=torch.int32, device="cuda")
    big = [torch.full((160, H, D), 3.0, dtype=torch.bfloat16, device="cuda") for H in (Hq, Hkv, Hkv)]
    dq, dk, dv = (x[32:128] for x in big)     # 96-row buffers with 32 canary rows on each side
    T.grad_tail_zero(dq, dk, dv, pad, pad)
    torch.cuda.synchronize()
    for x in big:
        assert torch.all(x == 3)


def test_grad_tail_zero_clears_slack_and_keeps_canary():
    Hq, Hkv, D = 4, 2, 64
    cuq = torch.tensor([0, 40, 100], dtype=torch.int32, device="cuda")
    cukv = torch.tensor([0, 40, 100], dtype=torch.int32, device="cuda")
    big_q = torch.full((140, Hq, D), 3.0, dtype=torch.bfloat16, device="cuda")
    big_k = torch.full((130, Hkv, D), 3.0, dtype=torch.bfloat16, device="cuda")
    big_v = torch.full((130, Hkv, D), 3.0, dtype=torch.bfloat16, device="cuda")
    dq, dk, dv = big_q[:120], big_k[:110], big_v[:110]     # buffers; rows past them are canaries
    T.grad_tail_zero(dq, dk, dv, cuq, cukv)
    torch.cuda.synchronize()
    assert torch.all(big_q[:100] == 3) and torch.all(big_q[100:120] == 0) and torch.all(big_q[120:] == 3)
    assert torch.all(big_k[:100] == 3) and torch.all(big_k[100:110] == 0) and torch.all(big_k[110:] == 3)
    assert torch.all(big_v[100:110] == 0) and torch.all(big_v[110:] == 3)


def test_grad_tail_zero_is_a_no_op_without_tail():
    Hq, Hkv, D = 2, 2, 64
    cu = torch.tensor([0, 64, 128], dtype=torch.int32, device="cuda")
    g = [torch.randn((128, Hq, D), device="cuda").to(torch.bfloat16) for _ in range(3)]
    before = [x.clone() for x in g]
    T.grad_tail_zero(g[0], g[1], g[2], cu, cu)          # end == rows: device reads it, writes nothing
    n0 = T.thd_launch_count()
    T.grad_tail_zero(g[0], g[1], g[2], cu, cu, host_knows_no_tail=True)   # no launch at all
    torch.cuda.synchronize()
    assert T.thd_launch_count() == n0
    for a, b in zip(g, before):
        assert torch.equal(a, b)
