"""Pins for the oracle's Ulysses (A2A) and hierarchical a2a+p2p emulation
(CPU, no GPU): hand-derived layouts, a row-by-row ownership scan, the
round trip, the grouping reading, and attention through the decomposition
against unsplit attention."""

import os

import numpy as np
import pytest

from oracle import thd_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _parse(path):
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            if key in ("cp_size", "a2a_size"):
                out[key] = int(rest[0])
            else:
                out.setdefault(key, {})[int(rest[0])] = [int(x) for x in rest[1:]]
    return out


def _owner_scan(cu_pad, cp):
    """(owner rank, rank-local row) of every global padded row, by walking each
    sequence's rows and asking which of its 2*cp chunks the row falls in."""
    out = []
    for b in range(len(cu_pad) - 1):
        P = int(cu_pad[b + 1] - cu_pad[b])
        cb = P // (2 * cp)
        for pos in range(P):
            chunk = pos // cb
            owner = chunk if chunk < cp else 2 * cp - 1 - chunk
            local = pos - chunk * cb + (0 if chunk == owner else cb)
            out.append((owner, int(cu_pad[b]) // cp + local))
    return out


def _shard(x, cu_pad, cp):
    """Global rows -> per-rank shards [cp, T/cp, ...] by the ownership scan."""
    T = int(cu_pad[-1])
    s = np.zeros((cp, T // cp) + x.shape[1:], x.dtype)
    for g, (r, l) in enumerate(_owner_scan(cu_pad, cp)):
        s[r, l] = x[g]
    return s


def _case(rng, B, cp, max_units=4, pad=True, Hq=4, Hkv=2, D=8):
    unit = 2 * cp
    lens, pads = [], []
    for _ in range(B):
        P = unit * int(rng.integers(1, max_units + 1))
        L = int(rng.integers(1, P + 1)) if pad else P
        lens.append(L)
        pads.append(P)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cu_pad = np.concatenate([[0], np.cumsum(pads)]).astype(np.int32)
    T = int(cu_pad[-1])
    valid = np.zeros(T, bool)
    for b in range(B):
        valid[cu_pad[b]:cu_pad[b] + lens[b]] = True
    q, k, v, do = (rng.standard_normal((T, H, D)) for H in (Hq, Hkv, Hkv, Hq))
    for t in (q, k, v, do):
        t[~valid] = 0
    return cu, cu_pad, q, k, v, do


# ---------------------------------------------------------------- layout

@pytest.mark.parametrize("fixture,cu_pad", [("tiny_a2a.txt", [0, 8, 16]), ("tiny_hier_a2a.txt", [0, 16])])
def test_a2a_matches_hand_derived_fixture(fixture, cu_pad):
    g = _parse(os.path.join(GOLDEN, fixture))
    cp, a = g["cp_size"], g["a2a_size"]
    T = cu_pad[-1]
    x = np.zeros((cp, T // cp, 2, 1), np.int64)
    for r in range(cp):
        for l in range(T // cp):
            for h in range(2):
                x[r, l, h, 0] = 100 * r + 10 * l + h
    y = orc.a2a_seq_to_head(x, np.array(cu_pad, np.int32), cp, a)
    assert y.shape == (a, T, 2 // a, 1)
    for i in range(a):
        assert y[i, :, 0, 0].tolist() == g["y"][i]
    assert np.array_equal(orc.a2a_head_to_seq(y, np.array(cu_pad, np.int32), cp, a), x)


@pytest.mark.parametrize("seed", range(8))
def test_a2a_is_a_head_split_of_the_unsharded_tensor(seed):
    rng = np.random.default_rng(700 + seed)
    cp = int(rng.integers(1, 5))
    divs = [d for d in range(1, cp + 1) if cp % d == 0]
    a = divs[int(rng.integers(len(divs)))]
    H = a * int(rng.integers(1, 4))
    cu, cu_pad, *_ = _case(rng, int(rng.integers(1, 5)), cp)
    T = int(cu_pad[-1])
    glob = rng.standard_normal((T, H, 3))
    x = _shard(glob, cu_pad, cp)
    y = orc.a2a_seq_to_head(x, cu_pad, cp, a)
    Hg = H // a
    for i in range(a):
        assert np.array_equal(y[i], glob[:, i * Hg:(i + 1) * Hg])
    assert np.array_equal(orc.a2a_head_to_seq(y, cu_pad, cp, a), x)


@pytest.mark.parametrize("sizes", [(1, 4), (2, 2), (4, 1), (2, 3), (3, 2)])
def test_hierarchical_groups_hold_the_p2p_shards(sizes):
    """Reading of the hierarchical layout: with groups of consecutive ranks,
    the rows group j holds are exactly the rows p2p rank j owns under the
    2*p2p split, so the ring across groups is the load-balanced P2P ring."""
    a, p = sizes
    cp = a * p
    rng = np.random.default_rng(sum(sizes))
    _, cu_pad, *_ = _case(rng, 4, cp)
    own_cp = _owner_scan(cu_pad, cp)
    own_p = _owner_scan(cu_pad, p)
    assert [r // a for r, _ in own_cp] == [r for r, _ in own_p]


def test_hierarchical_sizes_validation():
    assert orc.hierarchical_cp_sizes([2, 2], 4) == (2, 2)
    assert orc.hierarchical_cp_sizes((4, 2), 8) == (4, 2)
    for bad, cp in (([2, 2], 8), ([3], 3), ([0, 4], 4), ([2, 2, 1], 4)):
        with pytest.raises(ValueError):
            orc.hierarchical_cp_sizes(bad, cp)
    with pytest.raises(ValueError):
        orc.a2a_seq_to_head(np.zeros((4, 4, 3, 1)), [0, 16], 4, 2)   # 3 heads over 2 members
    with pytest.raises(ValueError):
        orc.a2a_seq_to_head(np.zeros((4, 4, 4, 1)), [0, 16], 4, 3)   # 3 does not divide cp


# ---------------------------------------------------------------- attention through the decomposition

@pytest.mark.parametrize("cp,a", [(2, 2), (4, 4), (4, 2), (4, 1), (3, 3), (6, 2)])
def test_a2a_attention_equals_unsplit(cp, a):
    rng = np.random.default_rng(800 + 10 * cp + a)
    Hq, Hkv = 2 * max(a, 1), max(a, 1)
    cu, cu_pad, q, k, v, _ = _case(rng, 3, cp, Hq=Hq, Hkv=Hkv)
    O, lse = orc.attn_fwd(q, k, v, cu, cu, cu_pad, cu_pad, causal=True, softmax_scale=0.4)
    Os, lses = orc.cp_a2a_attn_fwd(_shard(q, cu_pad, cp), _shard(k, cu_pad, cp), _shard(v, cu_pad, cp), cu, cu_pad,
                                   cp, a, softmax_scale=0.4)
    np.testing.assert_allclose(Os, _shard(O, cu_pad, cp), rtol=0, atol=1e-12)
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(lses))
    np.testing.assert_allclose(lses[fin], lse[fin], rtol=0, atol=1e-12)


@pytest.mark.parametrize("cp,a", [(2, 2), (4, 2)])
def test_a2a_backward_equals_unsplit(cp, a):
    rng = np.random.default_rng(900 + cp + a)
    cu, cu_pad, q, k, v, do = _case(rng, 2, cp, Hq=2 * a, Hkv=a)
    ref = orc.attn_bwd(q, k, v, do, cu, cu, cu_pad, cu_pad, softmax_scale=0.4)
    got = orc.cp_a2a_attn_bwd(*(_shard(t, cu_pad, cp) for t in (q, k, v, do)), cu, cu_pad, cp, a,
                              softmax_scale=0.4)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, _shard(r, cu_pad, cp), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- planted mistakes

def test_planted_member_order_mistake_is_caught(monkeypatch):
    """Members receiving each other's heads, consistently in both directions,
    still round-trip; the hand-derived layouts catch it."""
    real_fwd, real_inv = orc.a2a_seq_to_head, orc.a2a_head_to_seq

    def wrong_fwd(x, pad, cp, a):
        return real_fwd(x, pad, cp, a)[::-1].copy()

    def wrong_inv(y, pad, cp, a):
        return real_inv(np.asarray(y)[::-1].copy(), pad, cp, a)
    monkeypatch.setattr(orc, "a2a_seq_to_head", wrong_fwd)
    monkeypatch.setattr(orc, "a2a_head_to_seq", wrong_inv)
    x = np.arange(4 * 4 * 2, dtype=np.int64).reshape(4, 4, 2, 1)
    assert np.array_equal(orc.a2a_head_to_seq(orc.a2a_seq_to_head(x, [0, 16], 4, 2), [0, 16], 4, 2), x)
    with pytest.raises(AssertionError):
        test_a2a_matches_hand_derived_fixture("tiny_a2a.txt", [0, 8, 16])


def test_planted_ring_size_mistake_is_caught(monkeypatch):
    """Running each member's ring over cp ranks instead of cp / a2a would still
    cover every causal pair here (the ring emulation reads global rows), so
    the mistake planted is the other plausible one: a member attending only
    its own group's rows (no ring across groups)."""
    real = orc.cp_ring_fwd

    def wrong(q, k, v, cu, pad, cp_size, **kw):
        return real(q, k, v, cu, pad, cp_size, steps=1, **kw)
    monkeypatch.setattr(orc, "cp_ring_fwd", wrong)
    with pytest.raises(AssertionError):
        test_a2a_attention_equals_unsplit(4, 2)
