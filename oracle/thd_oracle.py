"""CPU fp64 oracle for causal attention over packed THD tensors with an emulated
P2P (ring) context-parallel decomposition.

TEST INFRASTRUCTURE ONLY.  This module is the slow, obviously-correct
definition that the CUDA path is checked against.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline / reference leg of
``bench.py`` may import it.  The library under ``packed_sequence_context_gb300``
never imports it, and this module imports nothing from there: the two share
no code, tables or helpers.

Sources (web pages; cited as [P1], [P2], [P3] with the section on the page):

* [P1] TransformerEngine issue #2208, "thd format is not supported with
  hierarchical CP implementation yet" -- the traceback through
  ``AttnFuncWithCPAndKVP2P`` (the P2P ring) and the maintainer's reply on P2P
  versus A2A.
* [P2] TransformerEngine issue #3487, "THD P2P context-parallel regression
  when padded cu_seqlens are value-equal but not object-identical" --
  sections "Describe the bug", "Steps/Code to reproduce bug",
  "Expected behavior".
* [P3] "Hybrid / Hierarchical Context Parallel Skill" -- section
  "Contraintes requises" (``seq_length % (2 * context_parallel_size) == 0``)
  and "Pitfalls" item 5 (local-chunk-only attention is fast but wrong).

The pages name the operations but print no formula.  Where they are silent
this module takes the plainest reading that the rest supports:

* THD layout: tokens of all sequences concatenated, ``[T, H, D]``; sequence b
  occupies buffer rows ``[cu_pad[b], cu_pad[b] + L_b)`` with
  ``L_b = cu[b+1] - cu[b]``; rows ``[cu_pad[b] + L_b, cu_pad[b+1])`` are pad.
* Attention: ``S = scale * q k^T`` per sequence and head, causal mask
  ``j <= i`` (top-left), ``lse = logsumexp_j S`` (natural log),
  ``O = softmax(S) V``.  GQA: query head h reads key/value head
  ``h // (Hq // Hkv)``.  Pad rows: ``O = 0``, ``lse = -inf``.
* CP chunking: each sequence's padded length is cut into ``2*CP`` equal
  chunks (length ``cb = P_b / (2 CP)``); rank r owns chunks r and
  ``2CP-1-r``; at ring step i rank r holds the KV of rank
  ``s = (r - i) mod CP``.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
(the Ulysses/A2A and hierarchical functions in ``tests/test_oracle_a2a_pins.py``,
the bottom-right causal mode in ``tests/test_oracle_bottom_right_pins.py``)
against brute force, closed forms, library special cases (torch SDPA in
fp64 on the CPU) and invariants.  No function is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

NEG_INF = float("-inf")
Q_BLOCK = 1024  # query rows per block, so a 131072-token sequence never builds its full S


# ---------------------------------------------------------------------------
# metadata
# ---------------------------------------------------------------------------

def _as_int_list(a) -> list[int]:
    return [int(x) for x in np.asarray(a).reshape(-1)]


def detect_pad_between_seqs(cu_seqlens, cu_seqlens_padded) -> bool:
    """Padding between sequences, decided from VALUES.

    [P2 "Describe the bug"] shows the detector deciding by object identity,
    so a value-equal clone is classified as padded; [P2 "Expected behavior"]
    asks that value-equal metadata not select the padding path.  Here the
    decision is: padded iff some entry differs.
    """
    if cu_seqlens_padded is None:
        return False
    a = _as_int_list(cu_seqlens)
    b = _as_int_list(cu_seqlens_padded)
    if len(a) != len(b):
        raise ValueError("cu_seqlens and cu_seqlens_padded differ in length")
    return any(x != y for x, y in zip(a, b))


def effective_padded(cu_seqlens, cu_seqlens_padded, pad_between_seqs: int = -1) -> list[int]:
    """Padded offsets that the computation uses.

    pad_between_seqs: -1 decide from values, 0 no padding (the padded array is
    ignored and offsets come from cu_seqlens), 1 padding (offsets from the
    padded array).  [P2 "Describe the bug"]: the tri-state None/False/True.
    """
    if pad_between_seqs == -1:
        pad = detect_pad_between_seqs(cu_seqlens, cu_seqlens_padded)
    elif pad_between_seqs in (0, 1):
        pad = bool(pad_between_seqs)
        if pad and cu_seqlens_padded is None:
            raise ValueError("pad_between_seqs=1 needs cu_seqlens_padded")
    else:
        raise ValueError("pad_between_seqs must be -1, 0 or 1")
    return _as_int_list(cu_seqlens_padded if pad else cu_seqlens)


def validate(cu_seqlens, cu_pad, cp_size: int, rows: int) -> None:
    """The constraints the decomposition needs.

    [P3 "Contraintes requises"]: ``seq_length % (2 * context_parallel_size) == 0``,
    read per sequence on the padded length for THD.  The other checks
    (monotone offsets, valid <= padded, fits the buffer) are what the layout
    itself requires.
    """
    cu = _as_int_list(cu_seqlens)
    pad = _as_int_list(cu_pad)
    if len(cu) != len(pad) or len(cu) < 2:
        raise ValueError("bad cu_seqlens length")
    if cu[0] != 0 or pad[0] != 0:
        raise ValueError("cu_seqlens must start at 0")
    for b in range(len(cu) - 1):
        L = cu[b + 1] - cu[b]
        P = pad[b + 1] - pad[b]
        if L < 0 or P < 0:
            raise ValueError("cu_seqlens not monotone")
        if L > P:
            raise ValueError("valid length exceeds padded length")
        if P % (2 * cp_size) != 0:
            raise ValueError("padded length not divisible by 2*cp_size")
    if pad[-1] > rows:
        raise ValueError("sequences exceed the buffer")


# ---------------------------------------------------------------------------
# a2: per-rank partition (get_cu_seqlens_on_cp_rank, one call for all ranks)
# ---------------------------------------------------------------------------

def cp_partition(cu_seqlens, cu_seqlens_padded, cp_size: int):
    """Per-rank cu_seqlens for THD + P2P context parallelism.

    [P2 "Describe the bug" / "Hướng nghiên cứu"] name the helper
    ``get_cu_seqlens_on_cp_rank``; [P3 "Contraintes requises"] fixes the
    2*CP split.  Reading: rank r's share of sequence b is chunk r followed by
    chunk 2CP-1-r, each ``cb = P_b/(2CP)`` padded rows; the valid counts are

        v1 = clamp(L_b - r*cb, 0, cb)            (first half, chunk r)
        v2 = clamp(L_b - (2CP-1-r)*cb, 0, cb)    (second half, chunk 2CP-1-r)

    Returns a dict of int32 arrays:
      cu_rank        [cp][B+1]  exclusive prefix sums of v1+v2
      cu_rank_padded [cp][B+1]  cu_pad[b] / cp   (each rank holds P_b/cp rows)
      cu_rank_half   [cp][2][B+1]  prefix sums of v1 and of v2 separately
      token_map      [cp][T/cp] global padded row of each rank-local row,
                     built by enumerating the chunks one row at a time.
    """
    cu = _as_int_list(cu_seqlens)
    pad = _as_int_list(cu_seqlens if cu_seqlens_padded is None else cu_seqlens_padded)
    B = len(cu) - 1
    T = pad[-1]
    cp = int(cp_size)
    cu_rank = np.zeros((cp, B + 1), np.int32)
    cu_rank_padded = np.zeros((cp, B + 1), np.int32)
    cu_rank_half = np.zeros((cp, 2, B + 1), np.int32)
    for r in range(cp):
        acc = acc1 = acc2 = 0
        for b in range(B):
            L = cu[b + 1] - cu[b]
            P = pad[b + 1] - pad[b]
            cb = P // (2 * cp)
            v1 = min(max(L - r * cb, 0), cb)
            v2 = min(max(L - (2 * cp - 1 - r) * cb, 0), cb)
            acc += v1 + v2
            acc1 += v1
            acc2 += v2
            cu_rank[r, b + 1] = acc
            cu_rank_half[r, 0, b + 1] = acc1
            cu_rank_half[r, 1, b + 1] = acc2
        for b in range(B + 1):
            cu_rank_padded[r, b] = pad[b] // cp
    token_map = np.zeros((cp, T // cp), np.int32)
    for r in range(cp):
        p = 0
        for b in range(B):
            cb = (pad[b + 1] - pad[b]) // (2 * cp)
            for chunk in (r, 2 * cp - 1 - r):
                for j in range(cb):
                    token_map[r, p] = pad[b] + chunk * cb + j
                    p += 1
    return {
        "cu_rank": cu_rank,
        "cu_rank_padded": cu_rank_padded,
        "cu_rank_half": cu_rank_half,
        "token_map": token_map,
    }


# ---------------------------------------------------------------------------
# attention (the plain definition)
# ---------------------------------------------------------------------------

def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


def _seq_table(cu_q, cu_kv, pad_q, pad_kv):
    B = len(cu_q) - 1
    out = []
    for b in range(B):
        out.append((pad_q[b], cu_q[b + 1] - cu_q[b], pad_kv[b], cu_kv[b + 1] - cu_kv[b]))
    return out


def _logsumexp_rows(S: np.ndarray) -> np.ndarray:
    if S.shape[1] == 0:
        return np.full(S.shape[0], NEG_INF)
    m = S.max(axis=1)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    with np.errstate(under="ignore"):
        s = np.exp(S - m_safe[:, None]).sum(axis=1)
    with np.errstate(divide="ignore"):
        return np.where(finite, m_safe + np.log(s), NEG_INF)


BOTTOM_RIGHT = "bottom_right"


def _key_offset(causal, Lq: int, Lkv: int):
    """None for no mask, else the offset o of the causal mask j <= i + o.

    ``causal`` True is the top-left mask (o = 0), which the pages' training
    setting uses and which needs equal query and key lengths per sequence.
    ``BOTTOM_RIGHT`` aligns the last query with the last key, o = Lkv - Lq
    (the T_q != T_kv case; not on the pages, the usual convention for a
    query block at the end of its keys): with Lq > Lkv the first Lq - Lkv
    queries see no key and get O = 0, lse = -inf like pad rows.
    """
    if causal == BOTTOM_RIGHT:
        return Lkv - Lq
    if causal is True or causal == 1:
        if Lq != Lkv:
            raise ValueError("causal attention needs equal q/kv lengths per sequence")
        return 0
    if causal is False or causal == 0:
        return None
    raise ValueError(f"unknown causal mode {causal!r}")


def _mask(i0: int, nq: int, Lkv: int, offset) -> np.ndarray:
    """Allowed (i, j) for query rows i0..i0+nq-1: j < Lkv, and j <= i + offset
    unless offset is None (no causal mask)."""
    i = np.arange(i0, i0 + nq)[:, None]
    j = np.arange(Lkv)[None, :]
    return (j <= i + offset) if offset is not None else np.ones((nq, Lkv), bool)


def attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded=None,
             cu_seqlens_kv_padded=None, causal: bool = True, softmax_scale: float | None = None,
             pad_between_seqs: int = -1, heads=None):
    """Causal softmax attention within each packed sequence, fp64.

    q [Tq, Hq, D], k/v [Tkv, Hkv, D] (any float dtype; upcast to fp64).
    Returns O [Tq, Hq, D] fp64 and lse [Hq, Tq] fp64 (natural log).  Every
    row that holds no valid query token (pad rows, the buffer tail) has
    O = 0 and lse = -inf.  ``heads`` restricts the query heads computed
    (others stay 0 / -inf), for bounded timing samples.

    Causal is the top-left mask j <= i, which needs equal query and key
    lengths per sequence; ``causal=BOTTOM_RIGHT`` is j <= i + Lkv - Lq.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, Hq, D = q.shape
    Tkv, Hkv, _ = k.shape
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    cu_q, cu_kv = _as_int_list(cu_seqlens_q), _as_int_list(cu_seqlens_kv)
    pq = effective_padded(cu_q, cu_seqlens_q_padded, pad_between_seqs)
    pkv = effective_padded(cu_kv, cu_seqlens_kv_padded, pad_between_seqs)
    O = np.zeros((Tq, Hq, D))
    lse = np.full((Hq, Tq), NEG_INF)
    hs = range(Hq) if heads is None else heads
    for (oq, Lq, ok, Lkv) in _seq_table(cu_q, cu_kv, pq, pkv):
        off = _key_offset(causal, Lq, Lkv)
        for h in hs:
            K = k[ok:ok + Lkv, h // G]
            V = v[ok:ok + Lkv, h // G]
            for i0 in range(0, Lq, Q_BLOCK):
                nq = min(Q_BLOCK, Lq - i0)
                Qb = q[oq + i0:oq + i0 + nq, h]
                S = scale * (Qb @ K.T)
                S = np.where(_mask(i0, nq, Lkv, off), S, NEG_INF)
                l = _logsumexp_rows(S)
                with np.errstate(invalid="ignore", under="ignore"):
                    P = np.where(np.isfinite(l)[:, None], np.exp(S - l[:, None]), 0.0)
                O[oq + i0:oq + i0 + nq, h] = P @ V
                lse[h, oq + i0:oq + i0 + nq] = l
    return O, lse


def attn_bwd(q, k, v, do, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded=None,
             cu_seqlens_kv_padded=None, causal: bool = True, softmax_scale: float | None = None,
             pad_between_seqs: int = -1, dq_rows: int | None = None, dkv_rows: int | None = None,
             heads=None):
    """Gradients of ``attn_fwd`` w.r.t. q, k, v for upstream dO, fp64.

    Textbook softmax-attention backward (recomputes P from q, k in fp64):
        P  = exp(S - lse),  dV = P^T dO,  dP = dO V^T,
        Delta = rowsum(dO * O),  dS = P * (dP - Delta),
        dQ = scale dS K,  dK = scale dS^T Q,
    with dK/dV summed over the query heads of each GQA group.  [P2 "Steps/Code
    to reproduce bug"] runs forward and backward on this layout; [P2
    "Describe the bug"] has THD dQ/dK/dV rows past the valid endpoint
    zeroed: here every row without a valid token is 0, including the slack
    rows ``[cu_pad[B], rows)`` of buffers longer than the data.  ``causal``
    takes the same modes as ``attn_fwd`` (``BOTTOM_RIGHT`` included).
    """
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    Tq, Hq, D = q.shape
    Tkv, Hkv, _ = k.shape
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    cu_q, cu_kv = _as_int_list(cu_seqlens_q), _as_int_list(cu_seqlens_kv)
    pq = effective_padded(cu_q, cu_seqlens_q_padded, pad_between_seqs)
    pkv = effective_padded(cu_kv, cu_seqlens_kv_padded, pad_between_seqs)
    dq = np.zeros((Tq if dq_rows is None else dq_rows, Hq, D))
    dk = np.zeros((Tkv if dkv_rows is None else dkv_rows, Hkv, D))
    dv = np.zeros_like(dk)
    hs = range(Hq) if heads is None else heads
    for (oq, Lq, ok, Lkv) in _seq_table(cu_q, cu_kv, pq, pkv):
        off = _key_offset(causal, Lq, Lkv)
        for h in hs:
            K = k[ok:ok + Lkv, h // G]
            V = v[ok:ok + Lkv, h // G]
            dK = np.zeros_like(K)
            dV = np.zeros_like(V)
            for i0 in range(0, Lq, Q_BLOCK):
                nq = min(Q_BLOCK, Lq - i0)
                Qb = q[oq + i0:oq + i0 + nq, h]
                dOb = do[oq + i0:oq + i0 + nq, h]
                S = scale * (Qb @ K.T)
                S = np.where(_mask(i0, nq, Lkv, off), S, NEG_INF)
                l = _logsumexp_rows(S)
                with np.errstate(invalid="ignore", under="ignore"):
                    P = np.where(np.isfinite(l)[:, None], np.exp(S - l[:, None]), 0.0)
                Ob = P @ V
                dV += P.T @ dOb
                dP = dOb @ V.T
                delta = (dOb * Ob).sum(axis=1)
                dS = P * (dP - delta[:, None])
                dq[oq + i0:oq + i0 + nq, h] = scale * (dS @ K)
                dK += scale * (dS.T @ Qb)
            dk[ok:ok + Lkv, h // G] += dK
            dv[ok:ok + Lkv, h // G] += dV
    return dq, dk, dv


def attn_fwd_rows(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, b: int,
                  h: int, positions, causal: bool = True, softmax_scale: float | None = None,
                  pad_between_seqs: int = -1):
    """The same definition as ``attn_fwd`` for a few query positions of one
    sequence b and query head h only (so that full-size workloads can be
    checked on samples).  Returns (O [n, D], lse [n]); positions at or past
    the valid length give (0, -inf)."""
    q, k, v = np.asarray(q), np.asarray(k), np.asarray(v)
    Hq, D = q.shape[1], q.shape[2]
    G = Hq // k.shape[1]
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    cu_q, cu_kv = _as_int_list(cu_seqlens_q), _as_int_list(cu_seqlens_kv)
    pq = effective_padded(cu_q, cu_seqlens_q_padded, pad_between_seqs)
    pkv = effective_padded(cu_kv, cu_seqlens_kv_padded, pad_between_seqs)
    Lq, Lkv = cu_q[b + 1] - cu_q[b], cu_kv[b + 1] - cu_kv[b]
    off = _key_offset(causal, Lq, Lkv)
    K = _f64(k[pkv[b]:pkv[b] + Lkv, h // G])
    V = _f64(v[pkv[b]:pkv[b] + Lkv, h // G])
    pos = [int(x) for x in positions]
    O = np.zeros((len(pos), D))
    lse = np.full(len(pos), NEG_INF)
    for n, i in enumerate(pos):
        if i >= Lq:
            continue
        S = scale * (K @ _f64(q[pq[b] + i, h]))
        if off is not None:
            S[max(i + off + 1, 0):] = NEG_INF
        l = _logsumexp_rows(S[None, :])[0]
        lse[n] = l
        if np.isfinite(l):
            O[n] = np.exp(S - l) @ V
    return O, lse


# ---------------------------------------------------------------------------
# a5: LSE merge
# ---------------------------------------------------------------------------

def lse_merge(o_a, lse_a, o_b, lse_b):
    """Merge two partial softmax results over disjoint key sets.

    The pages give no formula (the ring's per-step correction is only named
    in [P1]'s traceback); this is the log-sum-exp identity:
        lse = max(a, b) + log1p(exp(-|a - b|))
        O   = exp(a - lse) O_a + exp(b - lse) O_b
    A side with lse = -inf contributes nothing; both -inf give (0, -inf).
    Layout: o [T, H, D], lse [H, T].
    """
    o_a, o_b = _f64(o_a), _f64(o_b)
    a, b = _f64(lse_a), _f64(lse_b)
    hi = np.maximum(a, b)
    lo = np.minimum(a, b)
    both_inf = ~np.isfinite(hi)
    with np.errstate(invalid="ignore", over="ignore", under="ignore"):
        gap = np.where(np.isfinite(lo), lo - hi, NEG_INF)
        lse = np.where(both_inf, NEG_INF, hi + np.log1p(np.exp(gap)))
        wa = np.where(both_inf | ~np.isfinite(a), 0.0, np.exp(a - lse))
        wb = np.where(both_inf | ~np.isfinite(b), 0.0, np.exp(b - lse))
    O = wa.T[:, :, None] * o_a + wb.T[:, :, None] * o_b
    return O, lse


# ---------------------------------------------------------------------------
# the emulated P2P ring, written in rank-local terms (used to check the
# decomposition invariant, never as the reference result)
# ---------------------------------------------------------------------------

def _ring_step_partial(Ql, Kl, Vl, nQ, nK, cb_valid_q, cb_valid_k, r: int, s: int, i: int,
                       scale: float):
    """Partial attention of rank r at ring step i (KV of rank s) for one
    sequence and head, in rank-local rows.

    Rank-local rows are [chunk r ; chunk 2CP-1-r] (cb rows each); the valid
    rows of each half are a prefix of it: ``cb_valid_q = (v1, v2)``.

      i == 0 : local Q against local KV, causal on local positions;
      s <  r : all local Q rows against the first half of s's KV (chunk s),
               no mask (chunk 2CP-1-s lies after every local query);
      s >  r : only the second-half rows (chunk 2CP-1-r) against both halves
               of s's KV, no mask; first-half rows get nothing (lse = -inf).

    Returns O_i [2cb, D] and lse_i [2cb].
    """
    cb = nQ // 2
    v1, v2 = cb_valid_q
    k1, k2 = cb_valid_k
    qvalid = np.zeros(nQ, bool)
    qvalid[:v1] = True
    qvalid[cb:cb + v2] = True
    kvalid = np.zeros(nK, bool)
    kvalid[:k1] = True
    kvalid[cb:cb + k2] = True
    allowed = np.zeros((nQ, nK), bool)
    if i == 0:
        allowed = np.tril(np.ones((nQ, nK), bool))
    elif s < r:
        allowed[:, :cb] = True
    else:
        allowed[cb:, :] = True
    allowed &= qvalid[:, None] & kvalid[None, :]
    S = np.where(allowed, scale * (Ql @ Kl.T), NEG_INF)
    l = _logsumexp_rows(S)
    with np.errstate(invalid="ignore", under="ignore"):
        P = np.where(np.isfinite(l)[:, None], np.exp(S - l[:, None]), 0.0)
    return P @ Vl, l


def cp_ring_fwd(q, k, v, cu_seqlens, cu_seqlens_padded, cp_size: int, causal: bool = True,
                softmax_scale: float | None = None, pad_between_seqs: int = -1,
                steps: int | None = None, return_partials: bool = False):
    """Forward attention through the emulated P2P ring, merged by ``lse_merge``.

    [P1 traceback]: ``AttnFuncWithCPAndKVP2P`` rotates KV among CP ranks and
    corrects the running output per step; [P3 "Contraintes requises"]: the
    2*CP split.  Every rank and step runs here on one host, with the KV
    "received" at step i read from rank (r - i) mod CP's rows.

    ``steps`` < cp_size truncates the ring (only the first ``steps`` steps);
    with steps=1 every rank sees only its local chunks -- the silent failure
    of [P3 "Pitfalls" item 5].  ``return_partials`` also returns the per-step
    partials scattered back to global rows: lists of (O_i [T,Hq,D],
    lse_i [Hq,T]).
    Only causal self-attention (same metadata for q and kv) is emulated here.
    """
    if not causal:
        raise ValueError("the ring emulation here covers causal self-attention")
    q, k, v = _f64(q), _f64(k), _f64(v)
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    cp = int(cp_size)
    cu = _as_int_list(cu_seqlens)
    pad = effective_padded(cu, cu_seqlens_padded, pad_between_seqs)
    part = cp_partition(cu, pad, cp)
    tmap = part["token_map"]
    half = part["cu_rank_half"]
    B = len(cu) - 1
    nsteps = cp if steps is None else int(steps)
    O = np.zeros((T, Hq, D))
    lse = np.full((Hq, T), NEG_INF)
    partials = [(np.zeros((T, Hq, D)), np.full((Hq, T), NEG_INF)) for _ in range(nsteps)]
    for b in range(B):
        P_b = pad[b + 1] - pad[b]
        cb = P_b // (2 * cp)
        base = pad[b] // cp
        rows = {r: tmap[r, base:base + 2 * cb] for r in range(cp)}
        valid = {r: (int(half[r, 0, b + 1] - half[r, 0, b]), int(half[r, 1, b + 1] - half[r, 1, b]))
                 for r in range(cp)}
        for h in range(Hq):
            for r in range(cp):
                Ql = q[rows[r], h]
                acc_o = np.zeros((2 * cb, D))
                acc_l = np.full(2 * cb, NEG_INF)
                for i in range(nsteps):
                    s = (r - i) % cp
                    Kl = k[rows[s], h // G]
                    Vl = v[rows[s], h // G]
                    Oi, li = _ring_step_partial(Ql, Kl, Vl, 2 * cb, 2 * cb, valid[r], valid[s],
                                                r, s, i, scale)
                    partials[i][0][rows[r], h] = Oi
                    partials[i][1][h, rows[r]] = li
                    m_o, m_l = lse_merge(acc_o[:, None, :], acc_l[None, :],
                                         Oi[:, None, :], li[None, :])
                    acc_o, acc_l = m_o[:, 0, :], m_l[0]
                O[rows[r], h] = acc_o
                lse[h, rows[r]] = acc_l
    if return_partials:
        return O, lse, partials
    return O, lse


# ---------------------------------------------------------------------------
# next: Ulysses (A2A) and hierarchical a2a+p2p decompositions, emulated
# ---------------------------------------------------------------------------

def hierarchical_cp_sizes(sizes, cp_size: int) -> tuple[int, int]:
    """The two levels of a hierarchical CP layer, (a2a group size, p2p group size).

    [P3, the ``hierarchical_context_parallel_sizes`` docstring: the first value
    is the a2a group size, the second the p2p group size] and [P3
    "Contraintes requises" / "Pitfalls" item 6: their product must equal the
    CP size, else an assertion].
    """
    s = [int(x) for x in sizes]
    if len(s) != 2 or min(s) < 1:
        raise ValueError("hierarchical CP takes two sizes, a2a then p2p")
    if s[0] * s[1] != int(cp_size):
        raise ValueError("prod(hierarchical sizes) != cp_size")
    return s[0], s[1]


def _a2a_shape_check(H: int, cp: int, a2a: int) -> int:
    if cp < 1 or a2a < 1 or cp % a2a != 0:
        raise ValueError("the a2a group size must divide cp_size")
    if H % a2a != 0:
        raise ValueError("heads must divide evenly over the a2a group")
    return H // a2a


def a2a_seq_to_head(x_shards, cu_seqlens_padded, cp_size: int, a2a_size: int) -> np.ndarray:
    """The all-to-all in front of attention: scatter heads, gather the sequence.

    [P1, the maintainer's reply]: A2A (Ulysses) context parallelism, which
    THD lacked; [P3]: hierarchical CP runs that A2A inside groups of
    ``a2a_size`` ranks and the P2P ring across the groups.  Readings (the
    pages print no layout):

    * Before the A2A, CP rank r holds its THD shard ``x_shards[r]``
      (``[T/cp, H, ...]``): rank-local rows in ``cp_partition``'s token_map
      order, chunk r then chunk ``2cp-1-r`` of every sequence.
    * Groups are runs of consecutive ranks: rank ``j*a2a + i`` is member i of
      group j.  Member i receives query/key/value heads
      ``[i*H/a2a, (i+1)*H/a2a)`` of every token its group holds, placed at the
      token's global padded row.  With ``a2a_size == cp_size`` (pure Ulysses)
      there is one group that holds every token.
    * Emulated on one host, member i's buffers of all groups form one tensor in
      global order, so the result is ``y[i, g] = x[r, l, i*Hg:(i+1)*Hg]`` for
      every (r, l) with ``token_map[r, l] == g``; ``y`` is
      ``[a2a, T, H/a2a, ...]``.
    """
    x = np.asarray(x_shards)
    cp, rows_r, H = x.shape[0], x.shape[1], x.shape[2]
    a = int(a2a_size)
    if cp != int(cp_size):
        raise ValueError("x_shards must hold cp_size shards")
    Hg = _a2a_shape_check(H, cp, a)
    pad = _as_int_list(cu_seqlens_padded)
    T = pad[-1]
    if rows_r * cp != T:
        raise ValueError("each shard holds T/cp rows")
    tmap = cp_partition(pad, pad, cp)["token_map"]
    y = np.zeros((a, T, Hg) + x.shape[3:], x.dtype)
    for r in range(cp):
        for l in range(rows_r):
            g = int(tmap[r, l])
            for i in range(a):
                y[i, g] = x[r, l, i * Hg:(i + 1) * Hg]
    return y


def a2a_head_to_seq(y, cu_seqlens_padded, cp_size: int, a2a_size: int) -> np.ndarray:
    """The all-to-all behind attention, the inverse of ``a2a_seq_to_head``:
    ``x[r, l, i*Hg:(i+1)*Hg] = y[i, token_map[r, l]]``; ``x`` is
    ``[cp, T/cp, H, ...]``."""
    y = np.asarray(y)
    a, T, Hg = y.shape[0], y.shape[1], y.shape[2]
    cp = int(cp_size)
    if a != int(a2a_size):
        raise ValueError("y must hold a2a_size head groups")
    _a2a_shape_check(a * Hg, cp, a)
    pad = _as_int_list(cu_seqlens_padded)
    if pad[-1] != T or T % cp != 0:
        raise ValueError("y must hold the T padded rows")
    tmap = cp_partition(pad, pad, cp)["token_map"]
    x = np.zeros((cp, T // cp, a * Hg) + y.shape[3:], y.dtype)
    for r in range(cp):
        for l in range(T // cp):
            g = int(tmap[r, l])
            for i in range(a):
                x[r, l, i * Hg:(i + 1) * Hg] = y[i, g]
    return x


def cp_a2a_attn_fwd(q_shards, k_shards, v_shards, cu_seqlens, cu_seqlens_padded, cp_size: int, a2a_size: int,
                    softmax_scale: float | None = None):
    """Causal attention through the emulated A2A (``a2a_size == cp_size``) or
    hierarchical a2a+p2p (``p2p = cp_size / a2a_size``) decomposition.

    1. ``a2a_seq_to_head`` of q, k and v (GQA: the KV heads split the same way);
    2. member i of every group runs the P2P ring of ``p2p`` ranks over its
       heads (``cp_ring_fwd``, which for ``p2p == 1`` is plain causal
       attention on the whole sequence);
    3. ``a2a_head_to_seq`` of the output.

    Returns the output shards ``[cp, T/cp, Hq, D]`` and lse ``[Hq, T]`` in
    global row order (the members' heads stacked are the global heads).
    """
    cp, a = int(cp_size), int(a2a_size)
    p2p = cp // a
    qh = a2a_seq_to_head(_f64(q_shards), cu_seqlens_padded, cp, a)
    kh = a2a_seq_to_head(_f64(k_shards), cu_seqlens_padded, cp, a)
    vh = a2a_seq_to_head(_f64(v_shards), cu_seqlens_padded, cp, a)
    Hg, T = qh.shape[2], qh.shape[1]
    oh = np.zeros_like(qh)
    lse = np.full((a * Hg, T), NEG_INF)
    for i in range(a):
        oh[i], lse[i * Hg:(i + 1) * Hg] = cp_ring_fwd(qh[i], kh[i], vh[i], cu_seqlens, cu_seqlens_padded, p2p,
                                                      softmax_scale=softmax_scale)
    return a2a_head_to_seq(oh, cu_seqlens_padded, cp, a), lse


def cp_a2a_attn_bwd(q_shards, k_shards, v_shards, do_shards, cu_seqlens, cu_seqlens_padded, cp_size: int,
                    a2a_size: int, causal: bool = True, softmax_scale: float | None = None):
    """Gradients through the same decomposition: dO goes through
    ``a2a_seq_to_head`` with q, k, v; member i's gradients are those of its
    heads' attention (``attn_bwd``); dQ, dK, dV come back through
    ``a2a_head_to_seq``.  Returns the three gradient shard arrays."""
    cp, a = int(cp_size), int(a2a_size)
    pad = cu_seqlens_padded
    qh, kh, vh, doh = (a2a_seq_to_head(_f64(x), pad, cp, a) for x in (q_shards, k_shards, v_shards, do_shards))
    dqh, dkh, dvh = np.zeros_like(qh), np.zeros_like(kh), np.zeros_like(vh)
    T = qh.shape[1]
    for i in range(a):
        dqh[i], dkh[i], dvh[i] = attn_bwd(qh[i], kh[i], vh[i], doh[i], cu_seqlens, cu_seqlens, pad, pad,
                                          causal=causal, softmax_scale=softmax_scale, dq_rows=T, dkv_rows=T)
    return tuple(a2a_head_to_seq(g, pad, cp, a) for g in (dqh, dkh, dvh))


def _rank_rows(off: int, P: int, cp: int, r: int) -> np.ndarray:
    """Buffer rows of rank r's share of one sequence (padded length P at row
    off): chunk r then chunk 2cp-1-r, chunk = P / (2cp) rows."""
    cb = P // (2 * cp)
    return np.concatenate([off + r * cb + np.arange(cb), off + (2 * cp - 1 - r) * cb + np.arange(cb)]).astype(int)


def cp_ring_fwd_masked(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
                       cp_size: int, causal=True, softmax_scale: float | None = None, pad_between_seqs: int = -1,
                       return_partials: bool = False):
    """The P2P ring written with positional masks, for any mask mode.

    At step i rank r attends its query rows (its two q chunks) to the KV rows
    of rank s = (r - i) mod cp (s's two kv chunks), the mask taken from the
    rows' positions in the sequence (``_key_offset``: top-left causal,
    bottom-right causal or none), and the partials are merged with
    ``lse_merge``.  q and kv are chunked separately (``P_q / 2cp`` and
    ``P_kv / 2cp`` rows).  For equal-length causal self-attention the
    step-by-step partials are those of ``cp_ring_fwd``'s three rules; here
    they follow from positions alone, which also covers non-causal and
    bottom-right causal attention.  Returns (O, lse) like ``attn_fwd`` and,
    with ``return_partials``, the per-step partials scattered to global rows.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, Hq, D = q.shape
    G = Hq // k.shape[1]
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    cp = int(cp_size)
    cu_q, cu_kv = _as_int_list(cu_seqlens_q), _as_int_list(cu_seqlens_kv)
    pq = effective_padded(cu_q, cu_seqlens_q_padded, pad_between_seqs)
    pkv = effective_padded(cu_kv, cu_seqlens_kv_padded, pad_between_seqs)
    O = np.zeros((Tq, Hq, D))
    lse = np.full((Hq, Tq), NEG_INF)
    partials = [(np.zeros((Tq, Hq, D)), np.full((Hq, Tq), NEG_INF)) for _ in range(cp)]
    for b in range(len(cu_q) - 1):
        Lq, Lkv = cu_q[b + 1] - cu_q[b], cu_kv[b + 1] - cu_kv[b]
        Pq, Pkv = pq[b + 1] - pq[b], pkv[b + 1] - pkv[b]
        if Pq % (2 * cp) or Pkv % (2 * cp):
            raise ValueError("padded length not divisible by 2*cp_size")
        off = _key_offset(causal, Lq, Lkv)
        for r in range(cp):
            qrows = _rank_rows(pq[b], Pq, cp, r)
            qpos = qrows - pq[b]
            for h in range(Hq):
                acc_o = np.zeros((len(qrows), D))
                acc_l = np.full(len(qrows), NEG_INF)
                for i in range(cp):
                    s = (r - i) % cp
                    krows = _rank_rows(pkv[b], Pkv, cp, s)
                    kpos = krows - pkv[b]
                    allowed = (qpos[:, None] < Lq) & (kpos[None, :] < Lkv)
                    if off is not None:
                        allowed &= kpos[None, :] <= qpos[:, None] + off
                    S = np.where(allowed, scale * (q[qrows, h] @ k[krows, h // G].T), NEG_INF)
                    l = _logsumexp_rows(S)
                    with np.errstate(invalid="ignore", under="ignore"):
                        P = np.where(np.isfinite(l)[:, None], np.exp(S - l[:, None]), 0.0)
                    Oi = P @ v[krows, h // G]
                    partials[i][0][qrows, h] = Oi
                    partials[i][1][h, qrows] = l
                    m_o, m_l = lse_merge(acc_o[:, None, :], acc_l[None, :], Oi[:, None, :], l[None, :])
                    acc_o, acc_l = m_o[:, 0, :], m_l[0]
                O[qrows, h] = acc_o
                lse[h, qrows] = acc_l
    if return_partials:
        return O, lse, partials
    return O, lse


# ---------------------------------------------------------------------------
# a9: gradient tail-zero
# ---------------------------------------------------------------------------

def grad_tail_zero(dq, dk, dv, cu_seqlens_q_padded, cu_seqlens_kv_padded):
    """Zero gradient rows past the last padded endpoint.

    [P2 "Describe the bug"]: THD dQ/dK/dV tail-zeroing; [P2 "Expected
    behavior"]: nothing to do when the valid endpoint equals the buffer end.
    Returns copies with rows ``[cu_pad[B], rows)`` set to 0.
    """
    out = []
    for g, cu in ((dq, cu_seqlens_q_padded), (dk, cu_seqlens_kv_padded), (dv, cu_seqlens_kv_padded)):
        g = np.array(g, copy=True)
        end = _as_int_list(cu)[-1]
        g[end:] = 0
        out.append(g)
    return tuple(out)

