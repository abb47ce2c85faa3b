"""GPU parity of the emulated Ulysses (A2A) and hierarchical a2a+p2p path
(thd_cp_a2a, thd_attn_fwd_a2a, thd_attn_bwd_a2a) against the CPU fp64
oracle, through the C-ABI binding.  Layout moves are bit-exact (random bit
patterns, rows past the last sequence untouched); attention and gradients
are held to the ring path's bar (max-abs <= 2e-2, lse <= 1e-3 on valid rows,
pad rows exactly 0)."""

import numpy as np
import pytest
import torch

from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T
from thd_testutil import LSE_TOL, O_TOL, assert_within_bar, f64

pytestmark = pytest.mark.gpu

CANARY = 0x7F7F  # a bf16 bit pattern no move writes in these tests


@pytest.fixture(scope="module", autouse=True)
def _lib(thd_lib):
    return thd_lib


def _bits(x: torch.Tensor) -> np.ndarray:
    return x.view(torch.int16).cpu().numpy().view(np.uint16)


def _canary(shape) -> torch.Tensor:
    return torch.full(shape, CANARY, dtype=torch.int16, device="cuda").view(torch.bfloat16)


# ---------------------------------------------------------------- layout moves

# padded lengths (each a multiple of 2 cp), cp, a2a, H, D
LAYOUT = [
    ([16, 48, 8], 2, 2, 4, 64),
    ([64, 0, 128, 32], 4, 2, 6, 128),
    ([96, 24], 4, 4, 8, 128),
    ([48, 144], 6, 3, 3, 64),
    ([256], 8, 1, 2, 128),
    ([40, 80, 120], 4, 4, 4, 8),
    ([2048, 512, 1024], 4, 2, 16, 128),
]


@pytest.mark.parametrize("case", range(len(LAYOUT)))
def test_a2a_layout_bit_exact(case):
    lens, cp, a, H, D = LAYOUT[case]
    rng = np.random.default_rng(60 + case)
    pad = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    Tend = int(pad[-1])
    T_ = Tend + cp * 2 * (case % 2)            # odd cases: two slack rows per shard
    x = rng.integers(0, 1 << 16, size=(cp, T_ // cp, H, D), dtype=np.uint16)
    pad_d = torch.from_numpy(pad).cuda()
    xs = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    y = _canary((a, T_, H // a, D))
    _, st = T.cp_a2a(xs, pad_d, cp_size=cp, a2a_size=a, direction=T.THD_A2A_TO_GROUPS, out=y)
    assert T.check_status(st) == 0
    got = _bits(y)
    ref = orc.a2a_seq_to_head(x[:, :Tend // cp], pad, cp, a)
    assert np.array_equal(got[:, :Tend], ref)
    assert np.all(got[:, Tend:] == CANARY)
    back = _canary(tuple(xs.shape))
    _, st = T.cp_a2a(y, pad_d, cp_size=cp, a2a_size=a, direction=T.THD_A2A_TO_SHARDS, out=back)
    assert T.check_status(st) == 0
    gb = _bits(back)
    assert np.array_equal(gb[:, :Tend // cp], x[:, :Tend // cp])
    assert np.all(gb[:, Tend // cp:] == CANARY)


@pytest.mark.parametrize("lens,T_,code", [([10, 16], 28, T.THD_DEV_ERR_NOT_DIVISIBLE),
                                          ([16, 16], 28, T.THD_DEV_ERR_EXCEEDS_BUF)])
def test_a2a_bad_metadata_leaves_outputs_untouched(lens, T_, code):
    cp, a, H, D = 2, 2, 2, 64
    pad = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).cuda()
    xs = torch.zeros((cp, T_ // cp, H, D), dtype=torch.bfloat16, device="cuda")
    y = _canary((a, T_, H // a, D))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert T.thd_cp_a2a(xs, y, pad, len(lens), T_, H, D, cp, a, T.THD_A2A_TO_GROUPS, st) == T.THD_OK
    torch.cuda.synchronize()
    assert int(st.item()) == code
    assert np.all(_bits(y) == CANARY)


# ---------------------------------------------------------------- attention through the layer

def _shards(w, t):
    """Global [T, H, D] tensors -> per-rank shards [cp, T/cp, H, D] (oracle move)."""
    pad = w.cu_seqlens_padded
    return {x: torch.from_numpy(orc.a2a_head_to_seq(t[x].view(torch.int16).numpy()[None], pad, w.cp_size, 1))
            .view(torch.bfloat16) for x in t}


def _valid_shards(w):
    m = inputs.valid_row_mask(w)[None, :, None]
    return orc.a2a_head_to_seq(m, w.cu_seqlens_padded, w.cp_size, 1)[:, :, 0]


# lengths, pad_to, cp, a2a, Hq, Hkv, D
ATTN = [
    ([64, 128], 0, 2, 2, 2, 2, 64),
    ([96, 200, 24], 16, 4, 2, 4, 2, 128),
    ([512, 256], 0, 4, 4, 8, 4, 128),
    ([300, 40], 8, 2, 1, 2, 1, 64),
    ([130, 3, 257], 16, 4, 2, 4, 4, 64),
]


def _attn_case(case, with_grad):
    lens, pad_to, cp, a, Hq, Hkv, D = ATTN[case]
    w = inputs.make_workload("custom", 90 + case, lengths=lens, pad_to=pad_to, Hq=Hq, Hkv=Hkv, D=D, cp_size=cp)
    t = inputs.make_tensors(w, with_grad=with_grad)
    sh = _shards(w, t)
    d = {x: sh[x].cuda() for x in sh}
    d["cu"] = torch.from_numpy(w.cu_seqlens).cuda()
    d["cu_pad"] = torch.from_numpy(w.cu_seqlens_padded).cuda()
    return w, sh, d, cp, a


@pytest.mark.parametrize("case", range(len(ATTN)))
def test_attn_fwd_a2a_matches_oracle(case):
    w, sh, d, cp, a = _attn_case(case, False)
    o, lse, st = T.attn_fwd_a2a(d["q"], d["k"], d["v"], d["cu"], d["cu_pad"], cp_size=cp, a2a_size=a,
                                softmax_scale=w.softmax_scale)
    assert T.check_status(st) == 0
    O_ref, lse_ref = orc.cp_a2a_attn_fwd(sh["q"].float().numpy(), sh["k"].float().numpy(), sh["v"].float().numpy(),
                                         w.cu_seqlens, w.cu_seqlens_padded, cp, a, softmax_scale=w.softmax_scale)
    vs = _valid_shards(w)
    og = f64(o)
    assert np.abs(og[vs] - O_ref[vs]).max() <= O_TOL
    assert np.all(og[~vs] == 0)
    valid = inputs.valid_row_mask(w)
    lg = f64(lse)
    assert np.abs(lg[:, valid] - lse_ref[:, valid]).max() <= LSE_TOL
    assert np.all(np.isneginf(lg[:, ~valid]))


@pytest.mark.parametrize("case", [0, 1, 2, 4])
def test_attn_bwd_a2a_matches_oracle(case):
    w, sh, d, cp, a = _attn_case(case, True)
    o, lse, st = T.attn_fwd_a2a(d["q"], d["k"], d["v"], d["cu"], d["cu_pad"], cp_size=cp, a2a_size=a,
                                softmax_scale=w.softmax_scale)
    dq, dk, dv, st2 = T.attn_bwd_a2a(d["q"], d["k"], d["v"], o, lse, d["do"], d["cu"], d["cu_pad"], cp_size=cp,
                                     a2a_size=a, softmax_scale=w.softmax_scale)
    assert T.check_status(st) == 0 and T.check_status(st2) == 0
    ref = orc.cp_a2a_attn_bwd(*(sh[x].float().numpy() for x in ("q", "k", "v", "do")), w.cu_seqlens,
                              w.cu_seqlens_padded, cp, a, softmax_scale=w.softmax_scale)
    vs = _valid_shards(w)
    for name, g, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        gg = f64(g)
        assert_within_bar(name, gg[vs], r[vs])
        assert np.all(gg[~vs] == 0), f"{name}: pad rows must be 0"


@pytest.mark.parametrize("a", [4, 2])
def test_attn_a2a_full_size_every_row(a):
    """The packed workload (8 sequences, 14,632 tokens, 16 heads, cp 4)
    through Ulysses (a2a 4) and hierarchical [2, 2]: the shards are
    un-sharded by the oracle's move, and O, lse, dQ, dK and dV are compared
    with the oracle's unsplit attention on every valid row of every head (the
    oracle in a process pool, the bars of oracle_pool)."""
    import os
    import oracle_pool as op
    w = inputs.make_workload("packed")
    t = inputs.make_tensors(w, with_grad=True)
    sh = _shards(w, t)
    d = {x: sh[x].cuda() for x in sh}
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    cup = torch.from_numpy(w.cu_seqlens_padded).cuda()
    o, lse, st = T.attn_fwd_a2a(d["q"], d["k"], d["v"], cu, cup, cp_size=w.cp_size, a2a_size=a,
                                softmax_scale=w.softmax_scale)
    dq, dk, dv, st2 = T.attn_bwd_a2a(d["q"], d["k"], d["v"], o, lse, d["do"], cu, cup, cp_size=w.cp_size,
                                     a2a_size=a, softmax_scale=w.softmax_scale)
    assert T.check_status(st) == 0 and T.check_status(st2) == 0
    pad = w.cu_seqlens_padded

    def unshard(x):
        return torch.from_numpy(orc.a2a_seq_to_head(x.view(torch.int16).cpu().numpy(), pad, w.cp_size, 1)[0]) \
            .view(torch.bfloat16).float().numpy()

    store = op.Store()
    try:
        for k_ in ("q", "k", "v", "do"):
            store.put(k_, t[k_].float().numpy())
        for k_, x in (("o", o), ("dq", dq), ("dk", dk), ("dv", dv)):
            store.put(k_, unshard(x))
        store.put("lse", lse.cpu().numpy())
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        specs = [{"root": root, "dir": store.dir, "off": int(pad[b]), "L": int(w.lengths[b]), "kv_heads": [hk],
                  "G": w.Hq // w.Hkv, "scale": w.softmax_scale, "bwd": True}
                 for b in range(w.B) if w.lengths[b] > 0 for hk in range(w.Hkv)]
        specs.sort(key=lambda s_: -s_["L"])
        res = op.run(op._worker_seq, specs)
    finally:
        store.close()
    for k_ in ("o", "dq", "dk", "dv"):
        st_ = None
        for r in res:
            st_ = op.merge_stats(st_, r[k_])
        assert st_["excess"] <= op.TOL and st_["raw_small"] <= op.TOL, (k_, st_)
    assert max(r["lse"] for r in res) <= op.LSE_TOL
    for g in (o, dq, dk, dv):
        assert torch.isfinite(g.float()).all()


def test_a2a_matches_fused_ring_bitwise_when_a2a_is_one():
    """a2a 1 runs the fused ring on the un-sharded tensor with the same
    launch configuration as thd_attn_fwd: the outputs agree bit for bit."""
    w = inputs.make_workload("tiny")
    t = inputs.make_tensors(w)
    sh = _shards(w, t)
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    cup = torch.from_numpy(w.cu_seqlens_padded).cuda()
    o, lse, st = T.attn_fwd_a2a(sh["q"].cuda(), sh["k"].cuda(), sh["v"].cuda(), cu, cup, cp_size=w.cp_size,
                                a2a_size=1, softmax_scale=w.softmax_scale)
    o2, lse2, st2 = T.attn_fwd(t["q"].cuda(), t["k"].cuda(), t["v"].cuda(), cu, cu, cup, cup, cp_size=w.cp_size,
                               softmax_scale=w.softmax_scale)
    assert T.check_status(st) == 0 and T.check_status(st2) == 0
    ref_sh = orc.a2a_head_to_seq(o2.view(torch.int16).cpu().numpy()[None], w.cu_seqlens_padded, w.cp_size, 1)
    assert np.array_equal(_bits(o), ref_sh.view(np.uint16))
    assert torch.equal(lse, lse2)


def test_ulysses_matches_unchunked_attention_bitwise():
    """a2a = cp leaves a ring of one rank: every member attends its heads over
    whole sequences, the thd_attn_fwd launch with cp_size 1, bit for bit."""
    w = inputs.make_workload("custom", 7, lengths=[96, 200, 24], pad_to=16, Hq=8, Hkv=4, D=128, cp_size=4)
    t = inputs.make_tensors(w)
    sh = _shards(w, t)
    cu = torch.from_numpy(w.cu_seqlens).cuda()
    cup = torch.from_numpy(w.cu_seqlens_padded).cuda()
    o, lse, st = T.attn_fwd_a2a(sh["q"].cuda(), sh["k"].cuda(), sh["v"].cuda(), cu, cup, cp_size=4, a2a_size=4,
                                softmax_scale=w.softmax_scale)
    o2, lse2, st2 = T.attn_fwd(t["q"].cuda(), t["k"].cuda(), t["v"].cuda(), cu, cu, cup, cup, cp_size=1,
                               softmax_scale=w.softmax_scale)
    assert T.check_status(st) == 0 and T.check_status(st2) == 0
    ref_sh = orc.a2a_head_to_seq(o2.view(torch.int16).cpu().numpy()[None], w.cu_seqlens_padded, 4, 1)
    assert np.array_equal(_bits(o), ref_sh.view(np.uint16))
    assert torch.equal(lse, lse2)
