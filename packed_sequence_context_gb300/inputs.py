"""Seeded synthetic workloads for THD attention.

This module only draws inputs: sequence lengths, cu_seqlens metadata and
N(0, 1) tensors.  It holds none of the attention arithmetic, so both the CUDA
path and the CPU oracle can be fed from it.

Recipes (the pages use no dataset; the shapes follow the five workloads the
library is measured on):

* ``tiny``     : 2 sequences of 64 and 128 tokens, cu_seqlens = [0, 64, 192]
                 with a separately allocated padded copy holding equal
                 values; Hq = Hkv = 2, D = 64, CP = 2, forward.
* ``packed``   : 8 lengths ``8 * integers(32, 513)`` (256..4096 tokens,
                 about 16K in total); Hq = Hkv = 16, D = 128, CP = 4.
* ``padded``   : 12 lengths ``8 * integers(16, 1025)``, each padded up to a
                 multiple of 64 in cu_seqlens_padded, pad tokens zero-filled;
                 Hq = 32, Hkv = 8 (GQA), D = 128, CP = 4.
* ``long``     : one sequence of 131072 tokens; Hq = 32, Hkv = 8, D = 128,
                 CP = 4 (8 chunks of 16384).
* ``fwdbwd``   : 16 lognormal lengths,
                 ``clip(16 * rint(exp(ln 2048 + 0.8 z) / 16), 128, 16384)``;
                 Hq = Hkv = 32, D = 128, CP = 8; gradient buffers have
                 ``ceil(0.1 T)`` slack rows past the last sequence.

Lengths come from ``numpy.random.default_rng(seed)``; tensors are drawn in
fp32 ``standard_normal`` from a second generator seeded ``seed + 1000`` and
rounded to bf16 with a round-to-nearest-even cast.  Pad tokens (rows between
a sequence's valid end and the next padded offset) are zero.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

CONFIG_NAMES = ("tiny", "packed", "padded", "long", "fwdbwd")
CONFIG_ALIASES = {"C1": "tiny", "C2": "packed", "C3": "padded", "C4": "long", "C5": "fwdbwd"}
DEFAULT_SEEDS = {"tiny": 1, "packed": 2, "padded": 3, "long": 4, "fwdbwd": 5}


@dataclass
class Workload:
    name: str
    seed: int
    lengths: list
    cu_seqlens: np.ndarray            # int32 [B+1]
    cu_seqlens_padded: np.ndarray     # int32 [B+1], a separate array (equal values when unpadded)
    Hq: int
    Hkv: int
    D: int
    cp_size: int
    causal: bool = True
    backward: bool = False
    grad_slack: float = 0.0
    extra: dict = field(default_factory=dict)

    @property
    def B(self) -> int:
        return len(self.lengths)

    @property
    def T(self) -> int:
        return int(self.cu_seqlens_padded[-1])

    @property
    def dq_rows(self) -> int:
        return self.T + int(math.ceil(self.grad_slack * self.T))

    @property
    def dkv_rows(self) -> int:
        return self.dq_rows

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def padded(self) -> bool:
        return bool(np.any(self.cu_seqlens != self.cu_seqlens_padded))


def _cumsum0(x) -> np.ndarray:
    out = np.zeros(len(x) + 1, np.int64)
    out[1:] = np.cumsum(np.asarray(x, np.int64))
    return out.astype(np.int32)


def make_workload(name: str, seed: int | None = None, *, lengths=None, pad_to: int = 0,
                  Hq=None, Hkv=None, D=None, cp_size=None, grad_slack=None) -> Workload:
    """Build one named workload's metadata.  Keyword overrides build custom
    small cases for tests (``name='custom'`` requires ``lengths``)."""
    name = CONFIG_ALIASES.get(name, name)
    if seed is None:
        seed = DEFAULT_SEEDS.get(name, 0)
    rng = np.random.default_rng(seed)
    backward = False
    slack = 0.0
    if name == "tiny":
        L = [64, 128]
        hq, hkv, d, cp = 2, 2, 64, 2
        pad_mult = 0
    elif name == "packed":
        L = (8 * rng.integers(32, 513, size=8)).tolist()
        hq, hkv, d, cp = 16, 16, 128, 4
        pad_mult = 0
    elif name == "padded":
        L = (8 * rng.integers(16, 1025, size=12)).tolist()
        hq, hkv, d, cp = 32, 8, 128, 4
        pad_mult = 64
    elif name == "long":
        L = [131072]
        hq, hkv, d, cp = 32, 8, 128, 4
        pad_mult = 0
    elif name == "fwdbwd":
        z = rng.standard_normal(16)
        L = np.clip(16 * np.rint(np.exp(np.log(2048.0) + 0.8 * z) / 16), 128, 16384).astype(int).tolist()
        hq, hkv, d, cp = 32, 32, 128, 8
        pad_mult = 0
        backward = True
        slack = 0.1
    elif name == "custom":
        if lengths is None:
            raise ValueError("custom workload needs lengths")
        L = [int(x) for x in lengths]
        hq, hkv, d, cp = 2, 2, 64, 2
        pad_mult = pad_to
    else:
        raise KeyError(name)
    if lengths is not None:
        L = [int(x) for x in lengths]
    if pad_to:
        pad_mult = pad_to
    hq = hq if Hq is None else Hq
    hkv = hkv if Hkv is None else Hkv
    d = d if D is None else D
    cp = cp if cp_size is None else cp_size
    slack = slack if grad_slack is None else grad_slack
    P = [((x + pad_mult - 1) // pad_mult) * pad_mult if pad_mult else x for x in L]
    cu = _cumsum0(L)
    cu_pad = _cumsum0(P) if pad_mult else cu.copy()   # separately allocated even when equal
    return Workload(name=name, seed=seed, lengths=L, cu_seqlens=cu, cu_seqlens_padded=cu_pad,
                    Hq=hq, Hkv=hkv, D=d, cp_size=cp, causal=True, backward=backward,
                    grad_slack=slack)


def _bf16_normal(rng, shape):
    """fp32 standard normal rounded to bf16 (torch's RNE cast), as a CPU tensor."""
    import torch
    x = rng.standard_normal(size=shape, dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def make_tensors(w: Workload, *, with_grad: bool | None = None):
    """q, k, v (and dO when ``with_grad``) as bf16 CPU tensors of shape [T, H, D].

    Pad rows are zero-filled.  Returns a dict of torch tensors.
    """
    import torch
    rng = np.random.default_rng(w.seed + 1000)
    T = w.T
    q = _bf16_normal(rng, (T, w.Hq, w.D))
    k = _bf16_normal(rng, (T, w.Hkv, w.D))
    v = _bf16_normal(rng, (T, w.Hkv, w.D))
    out = {"q": q, "k": k, "v": v}
    if with_grad if with_grad is not None else w.backward:
        out["do"] = _bf16_normal(rng, (T, w.Hq, w.D))
    mask = valid_row_mask(w)
    if not mask.all():
        m = torch.from_numpy(~mask)
        for t in out.values():
            t[m] = 0
    return out


def valid_row_mask(w: Workload) -> np.ndarray:
    """Boolean [T]: True on rows that hold a valid token."""
    m = np.zeros(w.T, bool)
    for b in range(w.B):
        o = int(w.cu_seqlens_padded[b])
        m[o:o + w.lengths[b]] = True
    return m


def algorithmic_flops(lengths, Hq: int, D: int, causal: bool = True) -> tuple[float, float]:
    """FLOPs credited for (forward, forward+backward), valid pairs only.

    pairs = sum_b L_b (L_b + 1) / 2 (causal) or L_b^2; forward = 4 D Hq pairs
    (QK^T and PV), backward = 2.5 x forward (five GEMMs), so fwd+bwd = 3.5 x.
    Masked halves of diagonal tiles, skipped tiles and pad tokens are not
    credited.
    """
    pairs = 0
    for L in lengths:
        L = int(L)
        pairs += L * (L + 1) // 2 if causal else L * L
    fwd = 4.0 * D * Hq * pairs
    return fwd, 3.5 * fwd


def make_cross(lengths_q, lengths_kv, *, pad_to: int, Hq: int, Hkv: int, D: int, cp_size: int, seed: int,
               with_grad: bool = True):
    """A packed batch whose query and key sequences differ in length (the
    bottom-right causal case): per sequence b, L_q[b] queries and L_kv[b]
    keys, each padded up to a multiple of ``pad_to`` (which must itself be a
    multiple of 2 * cp_size).  Returns a dict of the metadata (int32 numpy:
    cu_q, cu_kv, cu_q_pad, cu_kv_pad) and bf16 CPU tensors q [T_q, Hq, D],
    k, v [T_kv, Hkv, D] and, with ``with_grad``, dO [T_q, Hq, D]; pad rows zero.
    Drawn like make_tensors (fp32 standard normal, RNE to bf16) from
    ``numpy.random.default_rng(seed + 1000)``."""
    import torch
    if pad_to % (2 * cp_size):
        raise ValueError("pad_to must be a multiple of 2 * cp_size")
    Lq = [int(x) for x in lengths_q]
    Lk = [int(x) for x in lengths_kv]
    Pq = [-(-x // pad_to) * pad_to for x in Lq]
    Pk = [-(-x // pad_to) * pad_to for x in Lk]
    meta = {"cu_q": _cumsum0(Lq), "cu_kv": _cumsum0(Lk), "cu_q_pad": _cumsum0(Pq), "cu_kv_pad": _cumsum0(Pk),
            "L_q": Lq, "L_kv": Lk}
    rng = np.random.default_rng(seed + 1000)
    Tq, Tk = int(meta["cu_q_pad"][-1]), int(meta["cu_kv_pad"][-1])
    t = {"q": _bf16_normal(rng, (Tq, Hq, D)), "k": _bf16_normal(rng, (Tk, Hkv, D)),
         "v": _bf16_normal(rng, (Tk, Hkv, D))}
    if with_grad:
        t["do"] = _bf16_normal(rng, (Tq, Hq, D))
    for names, L, pad in ((("q", "do"), Lq, meta["cu_q_pad"]), (("k", "v"), Lk, meta["cu_kv_pad"])):
        m = np.ones(int(pad[-1]), bool)
        for b, n in enumerate(L):
            m[int(pad[b]):int(pad[b]) + n] = False
        for x in names:
            if x in t:
                t[x][torch.from_numpy(m)] = 0
    meta.update(t)
    return meta
