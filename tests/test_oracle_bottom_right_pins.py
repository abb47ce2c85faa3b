"""Pins for the oracle's bottom-right causal mode (T_q != T_kv per sequence):
scalar brute force, torch's lower-right causal bias in fp64, the equal-length
special case, gradients against torch autograd, and a planted offset sign
mistake; and for the ring written with positional masks (every mask mode):
its merge equals unsplit attention and, for equal-length causal
self-attention, each step equals the hand-ruled ring's step.  CPU only."""

import math

import numpy as np
import pytest
import torch

from oracle import thd_oracle as orc

BR = orc.BOTTOM_RIGHT


def _case(rng, lq, lkv, pad=0, Hq=2, Hkv=1, D=8):
    """Separate q and kv metadata; q/kv padded to multiples of `pad` (if any)."""
    def cu(lengths, mult):
        P = [((L + mult - 1) // mult) * mult if mult else L for L in lengths]
        return (np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32),
                np.concatenate([[0], np.cumsum(P)]).astype(np.int32))
    cq, pq = cu(lq, pad)
    ck, pk = cu(lkv, pad)
    q = rng.standard_normal((int(pq[-1]), Hq, D))
    k = rng.standard_normal((int(pk[-1]), Hkv, D))
    v = rng.standard_normal((int(pk[-1]), Hkv, D))
    do = rng.standard_normal((int(pq[-1]), Hq, D))
    return cq, ck, pq, pk, q, k, v, do


def _brute(q, k, v, cq, ck, pq, pk, scale):
    """Scalar loops: query i of sequence b sees key j iff j <= i + Lkv - Lq."""
    Tq, Hq, D = q.shape
    G = Hq // k.shape[1]
    O = np.zeros((Tq, Hq, D))
    lse = np.full((Hq, Tq), -np.inf)
    for b in range(len(cq) - 1):
        Lq, Lkv = int(cq[b + 1] - cq[b]), int(ck[b + 1] - ck[b])
        for h in range(Hq):
            for i in range(Lq):
                s = [scale * float(np.dot(q[pq[b] + i, h], k[pk[b] + j, h // G]))
                     for j in range(Lkv) if j <= i + Lkv - Lq]
                if not s:
                    continue
                m = max(s)
                z = sum(math.exp(x - m) for x in s)
                lse[h, pq[b] + i] = m + math.log(z)
                for j, x in enumerate(s):
                    O[pq[b] + i, h] += math.exp(x - m) / z * v[pk[b] + j, h // G]
    return O, lse


@pytest.mark.parametrize("lq,lkv,pad", [([5, 9], [12, 9], 0), ([7, 3], [4, 6], 0), ([16, 1, 6], [30, 5, 6], 8),
                                        ([4], [4], 0)])
def test_bottom_right_matches_scalar_brute_force(lq, lkv, pad):
    rng = np.random.default_rng(sum(lq) * 31 + sum(lkv))
    cq, ck, pq, pk, q, k, v, _ = _case(rng, lq, lkv, pad)
    O, lse = orc.attn_fwd(q, k, v, cq, ck, pq, pk, causal=BR, softmax_scale=0.37)
    Ob, lb = _brute(q, k, v, cq, ck, pq, pk, 0.37)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    assert np.array_equal(np.isfinite(lse), np.isfinite(lb))
    np.testing.assert_allclose(lse[np.isfinite(lse)], lb[np.isfinite(lb)], rtol=0, atol=1e-12)


def _torch_lower_right(q, k, v, cq, ck, pq, pk, scale, need_grad=False, do=None):
    """Per sequence, torch's scaled_dot_product_attention with the lower-right
    causal bias, fp64 on the CPU.  Rows without any visible key come out NaN
    from torch; they are returned as NaN for the caller to mask."""
    from torch.nn.attention.bias import causal_lower_right
    Hq, Hkv = q.shape[1], k.shape[1]
    G = Hq // Hkv
    qt = torch.tensor(q, dtype=torch.float64, requires_grad=need_grad)
    kt = torch.tensor(k, dtype=torch.float64, requires_grad=need_grad)
    vt = torch.tensor(v, dtype=torch.float64, requires_grad=need_grad)
    outs = torch.zeros_like(qt)
    pieces = []
    for b in range(len(cq) - 1):
        Lq, Lkv = int(cq[b + 1] - cq[b]), int(ck[b + 1] - ck[b])
        Q = qt[pq[b]:pq[b] + Lq].transpose(0, 1)                                # [Hq, Lq, D]
        K = kt[pk[b]:pk[b] + Lkv].repeat_interleave(G, dim=1).transpose(0, 1)   # [Hq, Lkv, D]
        V = vt[pk[b]:pk[b] + Lkv].repeat_interleave(G, dim=1).transpose(0, 1)
        bias = causal_lower_right(Lq, Lkv)
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=bias, scale=scale)
        pieces.append((b, Lq, o.transpose(0, 1)))
    out = outs.clone()
    for b, Lq, o in pieces:
        out = torch.cat([out[:pq[b]], o, out[pq[b] + Lq:]])
    if need_grad:
        d = torch.tensor(do, dtype=torch.float64)
        vis = ~torch.isnan(out)
        (torch.where(vis, out, torch.zeros_like(out)) * d).sum().backward()
        return out.detach().numpy(), qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()
    return out.detach().numpy()


@pytest.mark.parametrize("seed", range(4))
def test_bottom_right_matches_torch_lower_right(seed):
    rng = np.random.default_rng(40 + seed)
    lq = [int(x) for x in rng.integers(1, 20, size=3)]
    lkv = [int(x) + int(y) for x, y in zip(lq, rng.integers(0, 12, size=3))]   # Lq <= Lkv
    cq, ck, pq, pk, q, k, v, _ = _case(rng, lq, lkv, pad=8 * (seed % 2), Hq=4, Hkv=2)
    O, _ = orc.attn_fwd(q, k, v, cq, ck, pq, pk, causal=BR, softmax_scale=0.3)
    ref = _torch_lower_right(q, k, v, cq, ck, pq, pk, 0.3)
    for b in range(len(cq) - 1):
        sl = slice(int(pq[b]), int(pq[b]) + lq[b])
        np.testing.assert_allclose(O[sl], ref[sl], rtol=0, atol=1e-12)


def test_bottom_right_with_more_queries_than_keys():
    """Lq > Lkv: the first Lq - Lkv queries see nothing (0 / -inf); the rest
    match torch's lower-right bias."""
    rng = np.random.default_rng(5)
    cq, ck, pq, pk, q, k, v, _ = _case(rng, [9, 4], [5, 4], Hq=2, Hkv=2)
    O, lse = orc.attn_fwd(q, k, v, cq, ck, pq, pk, causal=BR, softmax_scale=0.5)
    ref = _torch_lower_right(q, k, v, cq, ck, pq, pk, 0.5)
    assert np.all(O[:4] == 0) and np.all(np.isneginf(lse[:, :4]))
    np.testing.assert_allclose(O[4:], ref[4:], rtol=0, atol=1e-12)


def test_bottom_right_equals_top_left_on_equal_lengths():
    rng = np.random.default_rng(6)
    cq, ck, pq, pk, q, k, v, do = _case(rng, [12, 7], [12, 7], pad=4)
    a = orc.attn_fwd(q, k, v, cq, ck, pq, pk, causal=BR)
    b = orc.attn_fwd(q, k, v, cq, ck, pq, pk, causal=True)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    ga = orc.attn_bwd(q, k, v, do, cq, ck, pq, pk, causal=BR)
    gb = orc.attn_bwd(q, k, v, do, cq, ck, pq, pk, causal=True)
    assert all(np.array_equal(x, y) for x, y in zip(ga, gb))


def test_top_left_still_rejects_unequal_lengths():
    rng = np.random.default_rng(7)
    cq, ck, pq, pk, q, k, v, _ = _case(rng, [4], [6])
    with pytest.raises(ValueError):
        orc.attn_fwd(q, k, v, cq, ck, pq, pk, causal=True)
    with pytest.raises(ValueError):
        orc.attn_fwd(q, k, v, cq, ck, pq, pk, causal="top_right")


def test_bottom_right_gradients_match_torch_autograd():
    rng = np.random.default_rng(8)
    cq, ck, pq, pk, q, k, v, do = _case(rng, [6, 10], [9, 13], Hq=4, Hkv=2)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, cq, ck, pq, pk, causal=BR, softmax_scale=0.4)
    _, rq, rk, rv = _torch_lower_right(q, k, v, cq, ck, pq, pk, 0.4, need_grad=True, do=do)
    for g, r in ((dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(g, r, rtol=0, atol=1e-11)


def test_bottom_right_rows_helper_agrees():
    rng = np.random.default_rng(9)
    cq, ck, pq, pk, q, k, v, _ = _case(rng, [11, 8], [15, 8])
    O, lse = orc.attn_fwd(q, k, v, cq, ck, pq, pk, causal=BR)
    for b in range(2):
        L = int(cq[b + 1] - cq[b])
        Or, lr = orc.attn_fwd_rows(q, k, v, cq, ck, pq, pk, b, 1, range(L), causal=BR)
        np.testing.assert_allclose(Or, O[pq[b]:pq[b] + L, 1], rtol=0, atol=1e-12)
        np.testing.assert_allclose(lr, lse[1, pq[b]:pq[b] + L], rtol=0, atol=1e-12)


def test_planted_offset_sign_mistake_is_caught(monkeypatch):
    real = orc._key_offset

    def wrong(causal, Lq, Lkv):   # aligned the wrong way round
        o = real(causal, Lq, Lkv)
        return -o if causal == BR else o
    monkeypatch.setattr(orc, "_key_offset", wrong)
    with pytest.raises(AssertionError):
        test_bottom_right_matches_torch_lower_right(0)


# ---------------------------------------------------------------- the ring with positional masks

def _padded_case(rng, cp, lq, lkv, Hq=4, Hkv=2, D=8):
    unit = 2 * cp
    Pq = [unit * -(-max(L, 1) // unit) for L in lq]
    Pkv = [unit * -(-max(L, 1) // unit) for L in lkv]
    cq = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    ck = np.concatenate([[0], np.cumsum(lkv)]).astype(np.int32)
    pq = np.concatenate([[0], np.cumsum(Pq)]).astype(np.int32)
    pk = np.concatenate([[0], np.cumsum(Pkv)]).astype(np.int32)
    q = rng.standard_normal((int(pq[-1]), Hq, D))
    k = rng.standard_normal((int(pk[-1]), Hkv, D))
    v = rng.standard_normal((int(pk[-1]), Hkv, D))
    return cq, ck, pq, pk, q, k, v


@pytest.mark.parametrize("cp", [1, 2, 3, 4])
@pytest.mark.parametrize("mode", [True, False, BR])
def test_masked_ring_merges_to_unsplit(cp, mode):
    rng = np.random.default_rng(100 + 10 * cp + (0 if mode is True else 1 if mode is False else 2))
    lq = [int(x) for x in rng.integers(1, 40, size=3)]
    lkv = lq if mode is True else [int(x) for x in rng.integers(1, 50, size=3)]
    cq, ck, pq, pk, q, k, v = _padded_case(rng, cp, lq, lkv)
    O, lse = orc.attn_fwd(q, k, v, cq, ck, pq, pk, causal=mode, softmax_scale=0.3)
    Or, lr = orc.cp_ring_fwd_masked(q, k, v, cq, ck, pq, pk, cp, causal=mode, softmax_scale=0.3)
    np.testing.assert_allclose(Or, O, rtol=0, atol=1e-12)
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(lr))
    np.testing.assert_allclose(lr[fin], lse[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("cp", [2, 3, 4])
def test_masked_ring_steps_equal_the_causal_ring_rules(cp):
    """Equal-length causal self-attention: step i's partial from positions alone
    equals the partial of the ring's three hand rules (local causal step;
    s < r: all rows against chunk s; s > r: second-half rows only)."""
    rng = np.random.default_rng(200 + cp)
    lens = [int(x) for x in rng.integers(1, 40, size=3)]
    cq, ck, pq, pk, q, k, v = _padded_case(rng, cp, lens, lens)
    _, _, pa = orc.cp_ring_fwd_masked(q, k, v, cq, ck, pq, pk, cp, causal=True, softmax_scale=0.3,
                                      return_partials=True)
    _, _, pb = orc.cp_ring_fwd(q, k, v, cq, pq, cp, softmax_scale=0.3, return_partials=True)
    for (oa, la), (ob, lb) in zip(pa, pb):
        np.testing.assert_allclose(oa, ob, rtol=0, atol=1e-12)
        assert np.array_equal(np.isfinite(la), np.isfinite(lb))
        np.testing.assert_allclose(la[np.isfinite(la)], lb[np.isfinite(lb)], rtol=0, atol=1e-12)
