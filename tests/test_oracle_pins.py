"""Pins for the CPU oracle: each function is checked against something other
than itself -- hand-derived fixtures, brute force, closed forms, a library
special case (torch SDPA in fp64 on the CPU) and invariants -- chosen so
that a dropped term, a wrong sign or index, or a transposed operand fails
at least one of them.  The last tests plant such mistakes in the oracle (on
the CPU) and check that the pins catch them.
"""

import math
import os

import numpy as np
import pytest

from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers

def _parse_golden(path):
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            if key == "cp_size":
                out[key] = int(rest[0])
                continue
            r = int(rest[0])
            vals = []
            for tok in rest[1:]:
                if "-" in tok:
                    a, b = tok.split("-")
                    vals.extend(range(int(a), int(b) + 1))
                else:
                    vals.append(int(tok))
            out.setdefault(key, {})[r] = vals
    return out


def _rand_case(rng, B, max_len, cp, pad_mult=0, Hq=2, Hkv=1, D=4, zero_len_ok=True):
    unit = 2 * cp
    lens, pads = [], []
    for _ in range(B):
        if pad_mult:
            P = unit * int(rng.integers(1, max_len // unit + 1))
            L = int(rng.integers(0 if zero_len_ok else 1, P + 1))
        else:
            L = unit * int(rng.integers(0 if zero_len_ok else 1, max_len // unit + 1))
            P = L
        lens.append(L)
        pads.append(P)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cu_pad = np.concatenate([[0], np.cumsum(pads)]).astype(np.int32)
    T = int(cu_pad[-1])
    q = rng.standard_normal((T, Hq, D))
    k = rng.standard_normal((T, Hkv, D))
    v = rng.standard_normal((T, Hkv, D))
    valid = np.zeros(T, bool)
    for b in range(B):
        valid[cu_pad[b]:cu_pad[b] + lens[b]] = True
    q[~valid] = 0
    k[~valid] = 0
    v[~valid] = 0
    return cu, cu_pad, q, k, v, lens, valid


def _brute_fwd(q, k, v, cu, cu_pad, causal, scale):
    """Pure-Python loops, no vectorisation: the definition element by element."""
    T, Hq, D = q.shape
    G = Hq // k.shape[1]
    O = [[[0.0] * D for _ in range(Hq)] for _ in range(T)]
    lse = [[float("-inf")] * T for _ in range(Hq)]
    for b in range(len(cu) - 1):
        L = int(cu[b + 1] - cu[b])
        off = int(cu_pad[b])
        for h in range(Hq):
            for i in range(L):
                scores = []
                for j in range(L):
                    if causal and j > i:
                        continue
                    s = 0.0
                    for d in range(D):
                        s += q[off + i][h][d] * k[off + j][h // G][d]
                    scores.append((j, scale * s))
                m = max(s for _, s in scores)
                z = sum(math.exp(s - m) for _, s in scores)
                l = m + math.log(z)
                lse[h][off + i] = l
                for d in range(D):
                    O[off + i][h][d] = sum(math.exp(s - l) * v[off + j][h // G][d] for j, s in scores)
    return np.array(O), np.array(lse)


# ---------------------------------------------------------------- partition

@pytest.mark.parametrize("fixture,cu,cu_pad", [
    ("tiny_partition.txt", [0, 64, 192], [0, 64, 192]),
    ("tiny_padded_partition.txt", [0, 50, 150], [0, 64, 192]),
])
def test_partition_matches_hand_derived_fixture(fixture, cu, cu_pad):
    g = _parse_golden(os.path.join(GOLDEN, fixture))
    cp = g["cp_size"]
    part = orc.cp_partition(np.array(cu, np.int32), np.array(cu_pad, np.int32), cp)
    for r in range(cp):
        assert part["cu_rank"][r].tolist() == g["cu_rank"][r]
        assert part["cu_rank_padded"][r].tolist() == g["cu_rank_padded"][r]
        assert part["cu_rank_half"][r, 0].tolist() == g["cu_rank_half_first"][r]
        assert part["cu_rank_half"][r, 1].tolist() == g["cu_rank_half_second"][r]
        assert part["token_map"][r].tolist() == g["token_map"][r]


def _brute_owner_table(cu, cu_pad, cp):
    """For every global padded row: (owner rank, rank-local row, valid?), by
    scanning rows one at a time and asking which chunk each falls in."""
    out = {}
    B = len(cu) - 1
    for b in range(B):
        P = int(cu_pad[b + 1] - cu_pad[b])
        L = int(cu[b + 1] - cu[b])
        cb = P // (2 * cp)
        for pos in range(P):
            chunk = pos // cb
            owner = chunk if chunk < cp else 2 * cp - 1 - chunk
            local = (pos - owner * cb) if chunk == owner else cb + (pos - (2 * cp - 1 - owner) * cb)
            out[int(cu_pad[b]) + pos] = (owner, int(cu_pad[b]) // cp + local, pos < L, b)
    return out


@pytest.mark.parametrize("seed", range(12))
def test_partition_brute_force(seed):
    rng = np.random.default_rng(seed)
    cp = int(rng.integers(1, 6))
    B = int(rng.integers(1, 6))
    cu, cu_pad, *_ = _rand_case(rng, B, 64, cp, pad_mult=seed % 2)
    part = orc.cp_partition(cu, cu_pad, cp)
    table = _brute_owner_table(cu, cu_pad, cp)
    T = int(cu_pad[-1])
    # token map agrees with the row-by-row ownership and is a permutation of [0, T)
    seen = []
    for r in range(cp):
        for p, g in enumerate(part["token_map"][r].tolist()):
            owner, local, _, _ = table[g]
            assert owner == r and local == p
            seen.append(g)
    assert sorted(seen) == list(range(T))
    # valid counts per (rank, sequence) match the count of valid owned rows
    for r in range(cp):
        for b in range(B):
            n = sum(1 for g, (o, _, val, bb) in table.items() if o == r and bb == b and val)
            assert part["cu_rank"][r, b + 1] - part["cu_rank"][r, b] == n
            n1 = sum(1 for g, (o, loc, val, bb) in table.items()
                     if o == r and bb == b and val and loc - int(cu_pad[b]) // cp < (int(cu_pad[b + 1] - cu_pad[b]) // (2 * cp)))
            assert part["cu_rank_half"][r, 0, b + 1] - part["cu_rank_half"][r, 0, b] == n1
        assert part["cu_rank_padded"][r].tolist() == [int(x) // cp for x in cu_pad]
    # the ranks' valid counts add up to each sequence's length
    for b in range(B):
        assert sum(int(part["cu_rank"][r, b + 1] - part["cu_rank"][r, b]) for r in range(cp)) == int(cu[b + 1] - cu[b])


def test_detect_pad_by_value_not_identity():
    cu = np.array([0, 64, 192], np.int32)
    clone = cu.copy()
    assert clone is not cu
    assert orc.detect_pad_between_seqs(cu, clone) is False
    assert orc.detect_pad_between_seqs(cu, None) is False
    assert orc.detect_pad_between_seqs(cu, np.array([0, 64, 200], np.int32)) is True
    assert orc.effective_padded(cu, np.array([0, 64, 200], np.int32), 0) == [0, 64, 192]
    assert orc.effective_padded(cu, np.array([0, 64, 200], np.int32), 1) == [0, 64, 200]


def test_validate_rejects_bad_metadata():
    with pytest.raises(ValueError):
        orc.validate([0, 60], [0, 60], 4, 60)           # 60 % 8 != 0
    with pytest.raises(ValueError):
        orc.validate([0, 70], [0, 64], 2, 64)           # valid > padded
    with pytest.raises(ValueError):
        orc.validate([0, 64], [0, 64], 2, 32)           # exceeds the buffer
    with pytest.raises(ValueError):
        orc.validate([0, 64, 32], [0, 64, 32], 2, 64)   # not monotone
    orc.validate([0, 50, 150], [0, 64, 192], 2, 192)


# ---------------------------------------------------------------- forward

@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("causal", [True, False])
def test_fwd_matches_brute_force_loops(seed, causal):
    rng = np.random.default_rng(100 + seed)
    Hkv = int(rng.integers(1, 3))
    G = int(rng.integers(1, 3))
    D = int(rng.integers(1, 9))
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, int(rng.integers(1, 4)), 16, 2,
                                                  pad_mult=seed % 2, Hq=Hkv * G, Hkv=Hkv, D=D)
    scale = float(rng.uniform(0.2, 1.0))
    O, lse = orc.attn_fwd(q, k, v, cu, cu, cu_pad, cu_pad, causal=causal, softmax_scale=scale)
    Ob, lseb = _brute_fwd(q, k, v, cu, cu_pad, causal, scale)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    fin = np.isfinite(lseb)
    assert np.array_equal(fin, np.isfinite(lse))
    np.testing.assert_allclose(lse[fin], lseb[fin], rtol=0, atol=1e-12)


def _sdpa_reference(q, k, v, cu, cu_pad, causal, scale, need_grad=False, do=None):
    import torch
    import torch.nn.functional as F
    T, Hq, D = q.shape
    G = Hq // k.shape[1]
    O = np.zeros_like(q)
    grads = [np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)]
    for b in range(len(cu) - 1):
        L = int(cu[b + 1] - cu[b])
        o = int(cu_pad[b])
        if L == 0:
            continue
        tq = torch.tensor(q[o:o + L]).permute(1, 0, 2)[None].requires_grad_(need_grad)
        tk = torch.tensor(k[o:o + L]).permute(1, 0, 2)[None].requires_grad_(need_grad)
        tv = torch.tensor(v[o:o + L]).permute(1, 0, 2)[None].requires_grad_(need_grad)
        ke = tk.repeat_interleave(G, dim=1)
        ve = tv.repeat_interleave(G, dim=1)
        out = F.scaled_dot_product_attention(tq, ke, ve, is_causal=causal, scale=scale)
        O[o:o + L] = out[0].permute(1, 0, 2).detach().numpy()
        if need_grad:
            g = torch.tensor(do[o:o + L]).permute(1, 0, 2)[None]
            out.backward(g)
            grads[0][o:o + L] = tq.grad[0].permute(1, 0, 2).numpy()
            grads[1][o:o + L] = tk.grad[0].permute(1, 0, 2).numpy()
            grads[2][o:o + L] = tv.grad[0].permute(1, 0, 2).numpy()
    return O, grads


@pytest.mark.parametrize("seed", range(4))
def test_fwd_matches_torch_sdpa_fp64(seed):
    rng = np.random.default_rng(200 + seed)
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, 3, 96, 2, pad_mult=seed % 2, Hq=4, Hkv=2, D=16)
    scale = 1 / math.sqrt(16)
    O, _ = orc.attn_fwd(q, k, v, cu, cu, cu_pad, cu_pad, causal=True, softmax_scale=scale)
    Oref, _ = _sdpa_reference(q, k, v, cu, cu_pad, True, scale)
    np.testing.assert_allclose(O, Oref, rtol=0, atol=1e-12)


def test_fwd_blocks_rows_consistently():
    # a sequence longer than the oracle's query block: blocking must not change the result
    rng = np.random.default_rng(7)
    L = orc.Q_BLOCK + 40
    q = rng.standard_normal((L, 1, 8)); k = rng.standard_normal((L, 1, 8)); v = rng.standard_normal((L, 1, 8))
    cu = np.array([0, L], np.int32)
    O, lse = orc.attn_fwd(q, k, v, cu, cu, causal=True, softmax_scale=0.3)
    Oref, _ = _sdpa_reference(q, k, v, cu, cu, True, 0.3)
    np.testing.assert_allclose(O, Oref, rtol=0, atol=1e-12)


def test_fwd_constant_v_gives_v():
    rng = np.random.default_rng(3)
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, 3, 32, 2, Hq=2, Hkv=1, D=4, zero_len_ok=False)
    const = rng.standard_normal(4)
    v[:] = const
    O, _ = orc.attn_fwd(q, k, v, cu, cu, causal=True, softmax_scale=0.5)
    np.testing.assert_allclose(O[valid], np.broadcast_to(const, O[valid].shape), rtol=0, atol=1e-13)


def test_fwd_single_token_closed_form():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((1, 2, 8)); k = rng.standard_normal((1, 1, 8)); v = rng.standard_normal((1, 1, 8))
    cu = np.array([0, 1], np.int32)
    O, lse = orc.attn_fwd(q, k, v, cu, cu, causal=True, softmax_scale=0.25)
    for h in range(2):
        np.testing.assert_allclose(O[0, h], v[0, 0], atol=1e-15)
        assert abs(lse[h, 0] - 0.25 * float(q[0, h] @ k[0, 0])) < 1e-14


def test_fwd_first_row_attends_only_itself():
    # causal: row 0 sees key 0 only, so O[0] = v[0] and lse[0] = scale q0.k0
    rng = np.random.default_rng(5)
    q = rng.standard_normal((24, 1, 4)); k = rng.standard_normal((24, 1, 4)); v = rng.standard_normal((24, 1, 4))
    cu = np.array([0, 8, 24], np.int32)
    O, lse = orc.attn_fwd(q, k, v, cu, cu, causal=True, softmax_scale=0.7)
    for start in (0, 8):
        np.testing.assert_allclose(O[start, 0], v[start, 0], atol=1e-15)
        assert abs(lse[0, start] - 0.7 * float(q[start, 0] @ k[start, 0])) < 1e-14
    # two equal keys at row 1 with k0 == k1: uniform weights
    k[9] = k[8]
    O, lse = orc.attn_fwd(q, k, v, cu, cu, causal=True, softmax_scale=0.7)
    np.testing.assert_allclose(O[9, 0], 0.5 * (v[8, 0] + v[9, 0]), atol=1e-14)


@pytest.mark.parametrize("seed", range(3))
def test_fwd_rows_equals_full_definition(seed):
    rng = np.random.default_rng(600 + seed)
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, 3, 40, 2, pad_mult=seed % 2, Hq=4, Hkv=2, D=8,
                                                  zero_len_ok=False)
    O, lse = orc.attn_fwd(q, k, v, cu, cu, cu_pad, cu_pad, causal=bool(seed % 2 == 0), softmax_scale=0.4)
    for b in range(len(lens)):
        for h in (0, 3):
            pos = list(range(int(cu_pad[b + 1] - cu_pad[b])))
            Or, lr = orc.attn_fwd_rows(q, k, v, cu, cu, cu_pad, cu_pad, b, h, pos,
                                       causal=bool(seed % 2 == 0), softmax_scale=0.4)
            rows = int(cu_pad[b]) + np.arange(len(pos))
            np.testing.assert_allclose(Or, O[rows, h], rtol=0, atol=1e-13)
            assert np.array_equal(np.isfinite(lr), np.isfinite(lse[h, rows]))
            fin = np.isfinite(lr)
            np.testing.assert_allclose(lr[fin], lse[h, rows][fin], rtol=0, atol=1e-13)


# ---------------------------------------------------------------- padding

def test_value_equal_padded_metadata_is_bit_identical():
    rng = np.random.default_rng(11)
    cu, _, q, k, v, lens, valid = _rand_case(rng, 3, 48, 2, Hq=2, Hkv=2, D=8)
    clone = cu.copy()
    ref = orc.attn_fwd(q, k, v, cu, cu, None, None, causal=True)
    for pad_flag in (-1, 0, 1):
        got = orc.attn_fwd(q, k, v, cu, cu, clone, clone.copy(), causal=True, pad_between_seqs=pad_flag)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    do = rng.standard_normal(q.shape)
    gref = orc.attn_bwd(q, k, v, do, cu, cu, None, None)
    gclone = orc.attn_bwd(q, k, v, do, cu, cu, clone, clone.copy(), pad_between_seqs=1)
    for a, b in zip(gref, gclone):
        assert np.array_equal(a, b)


def test_pad_rows_are_zero_and_lse_neg_inf():
    rng = np.random.default_rng(12)
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, 4, 64, 2, pad_mult=1, Hq=2, Hkv=1, D=8)
    assert (~valid).any()
    q[~valid] = 5.0  # pad content must not leak into results
    O, lse = orc.attn_fwd(q, k, v, cu, cu, cu_pad, cu_pad, causal=True)
    assert np.all(O[~valid] == 0)
    assert np.all(np.isneginf(lse[:, ~valid]))
    assert np.all(np.isfinite(lse[:, valid]))
    do = rng.standard_normal(q.shape)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, cu, cu, cu_pad, cu_pad)
    assert np.all(dq[~valid] == 0) and np.all(dk[~valid] == 0) and np.all(dv[~valid] == 0)


# ---------------------------------------------------------------- LSE merge

def test_lse_merge_closed_forms():
    rng = np.random.default_rng(13)
    oa = rng.standard_normal((5, 2, 3)); ob = rng.standard_normal((5, 2, 3))
    a = rng.standard_normal((2, 5)); b = a.copy()
    O, lse = orc.lse_merge(oa, a, ob, b)
    np.testing.assert_allclose(lse, a + math.log(2.0), atol=1e-15)
    np.testing.assert_allclose(O, 0.5 * (oa + ob), atol=1e-15)
    # one side -inf: the other passes through unchanged
    ninf = np.full((2, 5), -np.inf)
    O, lse = orc.lse_merge(oa, a, ob, ninf)
    assert np.array_equal(lse, a) and np.allclose(O, oa, atol=0)
    O, lse = orc.lse_merge(oa, ninf, ob, b)
    assert np.array_equal(lse, b) and np.allclose(O, ob, atol=0)
    # both -inf: (0, -inf), no NaN
    O, lse = orc.lse_merge(oa, ninf, ob, ninf)
    assert np.all(O == 0) and np.all(np.isneginf(lse))
    # unequal: weights e^(a-lse) and e^(b-lse) sum to 1 and lse = log(e^a + e^b)
    b2 = a + rng.uniform(-3, 3, a.shape)
    O, lse = orc.lse_merge(oa, a, ob, b2)
    np.testing.assert_allclose(lse, np.log(np.exp(a) + np.exp(b2)), atol=1e-13)
    wa = np.exp(a - lse).T[:, :, None]
    np.testing.assert_allclose(O, wa * oa + (1 - wa) * ob, atol=1e-13)


def test_lse_merge_splits_keys_exactly():
    # attention over keys K split into two disjoint sets, merged == unsplit
    rng = np.random.default_rng(14)
    L, D = 12, 4
    q = rng.standard_normal((L, 1, D)); k = rng.standard_normal((L, 1, D)); v = rng.standard_normal((L, 1, D))
    cu = np.array([0, L], np.int32)
    O, lse = orc.attn_fwd(q, k, v, cu, cu, causal=False, softmax_scale=0.4)
    S = 0.4 * q[:, 0] @ k[:, 0].T
    parts = []
    for sel in (slice(0, 5), slice(5, L)):
        Ss = S[:, sel]
        l = np.log(np.exp(Ss).sum(1))
        parts.append(((np.exp(Ss - l[:, None]) @ v[sel, 0])[:, None, :], l[None, :]))
    Om, lm = orc.lse_merge(parts[0][0], parts[0][1], parts[1][0], parts[1][1])
    np.testing.assert_allclose(Om, O, atol=1e-13)
    np.testing.assert_allclose(lm, lse, atol=1e-13)


# ---------------------------------------------------------------- the ring

@pytest.mark.parametrize("cp", [1, 2, 3, 4])
@pytest.mark.parametrize("pad_mult", [0, 1])
def test_ring_partials_merge_to_unsplit(cp, pad_mult):
    rng = np.random.default_rng(300 + cp * 10 + pad_mult)
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, 3, 48, cp, pad_mult=pad_mult, Hq=4, Hkv=2, D=8)
    O, lse = orc.attn_fwd(q, k, v, cu, cu, cu_pad, cu_pad, causal=True, softmax_scale=0.3)
    Or, lser = orc.cp_ring_fwd(q, k, v, cu, cu_pad, cp, softmax_scale=0.3)
    np.testing.assert_allclose(Or, O, rtol=0, atol=1e-12)
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(lser))
    np.testing.assert_allclose(lser[fin], lse[fin], rtol=0, atol=1e-12)


def test_ring_local_chunk_only_is_wrong():
    # "Pitfalls" item 5 of the HCP skill page: attending only the local chunk
    # runs but gives wrong results; the merge invariant exposes it.
    rng = np.random.default_rng(15)
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, 2, 64, 4, Hq=2, Hkv=2, D=8, zero_len_ok=False)
    O, _ = orc.attn_fwd(q, k, v, cu, cu, causal=True)
    Ol, _ = orc.cp_ring_fwd(q, k, v, cu, cu_pad, 4, steps=1)
    assert np.abs(Ol - O).max() > 1e-2


def test_ring_step_rules():
    # at step i > 0 with s > r the first-half rows of rank r get nothing
    rng = np.random.default_rng(16)
    cp = 3
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, 1, 48, cp, Hq=1, Hkv=1, D=4, zero_len_ok=False)
    L = lens[0]
    cb = L // (2 * cp)
    _, _, parts = orc.cp_ring_fwd(q, k, v, cu, cu_pad, cp, return_partials=True)
    for i in range(1, cp):
        lse_i = parts[i][1][0]
        for r in range(cp):
            s = (r - i) % cp
            first = slice(r * cb, (r + 1) * cb)
            second = slice((2 * cp - 1 - r) * cb, (2 * cp - r) * cb)
            if s > r:
                assert np.all(np.isneginf(lse_i[first]))
            else:
                assert np.all(np.isfinite(lse_i[first]))
            assert np.all(np.isfinite(lse_i[second]))


# ---------------------------------------------------------------- backward

def _loss(q, k, v, do, cu, cu_pad, scale):
    O, _ = orc.attn_fwd(q, k, v, cu, cu, cu_pad, cu_pad, causal=True, softmax_scale=scale)
    return float((O * do).sum())


@pytest.mark.parametrize("seed", range(3))
def test_bwd_matches_central_finite_differences(seed):
    rng = np.random.default_rng(400 + seed)
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, 2, 8, 2, pad_mult=seed % 2, Hq=2, Hkv=1, D=3,
                                                  zero_len_ok=False)
    do = rng.standard_normal(q.shape)
    do[~valid] = 0
    scale = 0.6
    dq, dk, dv = orc.attn_bwd(q, k, v, do, cu, cu, cu_pad, cu_pad, softmax_scale=scale)
    eps = 1e-6
    for arr, grad in ((q, dq), (k, dk), (v, dv)):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            old = arr[idx]
            arr[idx] = old + eps
            lp = _loss(q, k, v, do, cu, cu_pad, scale)
            arr[idx] = old - eps
            lm = _loss(q, k, v, do, cu, cu_pad, scale)
            arr[idx] = old
            fd[idx] = (lp - lm) / (2 * eps)
        fd[~valid] = 0  # pad rows are not inputs of the function
        np.testing.assert_allclose(grad, fd, rtol=0, atol=1e-7)


@pytest.mark.parametrize("seed", range(3))
def test_bwd_matches_torch_autograd_fp64(seed):
    rng = np.random.default_rng(500 + seed)
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, 3, 64, 2, pad_mult=seed % 2, Hq=4, Hkv=2, D=8)
    do = rng.standard_normal(q.shape)
    do[~valid] = 0
    scale = 1 / math.sqrt(8)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, cu, cu, cu_pad, cu_pad, softmax_scale=scale)
    _, (gq, gk, gv) = _sdpa_reference(q, k, v, cu, cu_pad, True, scale, need_grad=True, do=do)
    np.testing.assert_allclose(dq, gq, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, gk, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, gv, rtol=0, atol=1e-11)


def test_bwd_slack_rows_zero():
    rng = np.random.default_rng(17)
    cu, cu_pad, q, k, v, lens, valid = _rand_case(rng, 2, 32, 2, Hq=2, Hkv=2, D=4)
    do = rng.standard_normal(q.shape)
    T = q.shape[0]
    dq, dk, dv = orc.attn_bwd(q, k, v, do, cu, cu, dq_rows=T + 7, dkv_rows=T + 5)
    assert dq.shape[0] == T + 7 and dk.shape[0] == T + 5
    assert np.all(dq[T:] == 0) and np.all(dk[T:] == 0) and np.all(dv[T:] == 0)


# ---------------------------------------------------------------- tail-zero

def test_grad_tail_zero():
    rng = np.random.default_rng(18)
    dq = rng.standard_normal((20, 2, 4)); dk = rng.standard_normal((22, 1, 4)); dv = rng.standard_normal((22, 1, 4))
    cuq = np.array([0, 8, 16], np.int32)
    cukv = np.array([0, 8, 22], np.int32)
    zq, zk, zv = orc.grad_tail_zero(dq, dk, dv, cuq, cukv)
    assert np.all(zq[16:] == 0) and np.array_equal(zq[:16], dq[:16])
    assert np.array_equal(zk, dk) and np.array_equal(zv, dv)   # no tail: untouched


# ---------------------------------------------------------------- input recipes

def test_workload_recipes():
    w = inputs.make_workload("packed")
    assert w.lengths == [3472, 1256, 672, 1400, 1848, 3384, 1992, 608] and w.T == 14632
    w = inputs.make_workload("padded")
    assert int(w.cu_seqlens[-1]) == 38992 and w.T == 39232 and w.padded
    assert all(int(x) % 64 == 0 for x in w.cu_seqlens_padded)
    w = inputs.make_workload("fwdbwd")
    assert w.T == 41888 and w.dq_rows == 46077
    w = inputs.make_workload("tiny")
    assert w.cu_seqlens.tolist() == [0, 64, 192]
    assert w.cu_seqlens_padded is not w.cu_seqlens and not w.padded
    for name in inputs.CONFIG_NAMES:
        w = inputs.make_workload(name)
        for b in range(w.B):
            assert (int(w.cu_seqlens_padded[b + 1] - w.cu_seqlens_padded[b])) % (2 * w.cp_size) == 0


def test_algorithmic_flops():
    fwd, both = inputs.algorithmic_flops([1, 2], 2, 64, causal=True)
    assert fwd == 4 * 64 * 2 * (1 + 3) and both == 3.5 * fwd


# ---------------------------------------------------------------- planted mistakes

def test_planted_partition_mistake_is_caught(monkeypatch):
    real = orc.cp_partition

    def wrong(cu, cu_pad, cp):   # owner of the second chunk off by one
        out = real(cu, cu_pad, cp)
        out["token_map"] = np.roll(out["token_map"], 1, axis=0)
        return out
    monkeypatch.setattr(orc, "cp_partition", wrong)
    with pytest.raises(AssertionError):
        test_partition_matches_hand_derived_fixture("tiny_partition.txt", [0, 64, 192], [0, 64, 192])


def test_planted_merge_mistake_is_caught(monkeypatch):
    def wrong(o_a, lse_a, o_b, lse_b):   # forgets the log1p correction term
        a, b = np.asarray(lse_a, float), np.asarray(lse_b, float)
        lse = np.maximum(a, b)
        with np.errstate(invalid="ignore"):
            wa = np.nan_to_num(np.exp(a - lse)); wb = np.nan_to_num(np.exp(b - lse))
        return wa.T[:, :, None] * o_a + wb.T[:, :, None] * o_b, lse
    monkeypatch.setattr(orc, "lse_merge", wrong)
    with pytest.raises(AssertionError):
        test_lse_merge_closed_forms()
    with pytest.raises(AssertionError):
        test_ring_partials_merge_to_unsplit(2, 0)


def test_planted_ring_rule_mistake_is_caught(monkeypatch):
    real = orc._ring_step_partial

    def wrong(Ql, Kl, Vl, nQ, nK, vq, vk, r, s, i, scale):   # s > r step also feeds first-half rows
        if i > 0 and s > r:
            return real(Ql, Kl, Vl, nQ, nK, vq, vk, r, s, 0, scale)
        return real(Ql, Kl, Vl, nQ, nK, vq, vk, r, s, i, scale)
    monkeypatch.setattr(orc, "_ring_step_partial", wrong)
    with pytest.raises(AssertionError):
        test_ring_partials_merge_to_unsplit(3, 0)


def test_planted_backward_mistake_is_caught(monkeypatch):
    real = orc.attn_bwd

    def wrong(*a, **kw):   # transposed dK contribution (uses Q of the wrong head group)
        dq, dk, dv = real(*a, **kw)
        return dq, dk[:, ::-1].copy(), dv
    monkeypatch.setattr(orc, "attn_bwd", wrong)
    with pytest.raises(AssertionError):
        test_bwd_matches_torch_autograd_fp64(0)
