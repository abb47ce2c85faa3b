"""Helpers shared by the GPU parity tests: move a seeded workload to the GPU,
run the library through its C ABI binding, and compare with the oracle."""

from __future__ import annotations

import numpy as np
import torch

from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T

O_TOL = 2e-2     # max-abs on valid rows, outputs and gradients (bf16 results)
LSE_TOL = 1e-3   # max-abs on valid rows


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the bf16 spacing at |x|: the rounding error a correctly rounded
    bf16 result may carry (0.0156 for |x| in [4, 8), 0.031 in [8, 16))."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return 0.5 * np.exp2(np.floor(np.log2(ax)) - 7)


def rounding_aware_excess(got: np.ndarray, ref: np.ndarray) -> float:
    """max(|got - ref| - half_ulp_bf16(ref)): the error left after the bf16
    rounding of the result itself.  Stress cases whose gradients reach |x| >= 4
    are held to O_TOL on this quantity."""
    return float((np.abs(got - ref) - bf16_half_ulp(ref)).max())


def device_inputs(w: inputs.Workload, t: dict, dev="cuda"):
    d = {k: v.to(dev) for k, v in t.items()}
    d["cu"] = torch.from_numpy(w.cu_seqlens).to(dev)
    d["cu_pad"] = torch.from_numpy(w.cu_seqlens_padded).to(dev)   # separate allocation
    return d


def f64(x: torch.Tensor) -> np.ndarray:
    return x.detach().float().cpu().numpy().astype(np.float64)


_DEFAULT = object()


def run_fwd(w, d, pad_flag=-1, cu_pad=_DEFAULT, cu_pad_kv=_DEFAULT, causal=True, T_q=None, out_canary=None):
    """cu_pad: _DEFAULT -> the workload's separately allocated padded array,
    None -> NULL (no padded array), else the tensor given."""
    q, k, v = d["q"], d["k"], d["v"]
    if T_q is not None and T_q > q.shape[0]:
        extra = T_q - q.shape[0]
        q = torch.cat([q, torch.zeros((extra,) + tuple(q.shape[1:]), dtype=q.dtype, device=q.device)])
    cp = d.get("cu_pad") if cu_pad is _DEFAULT else cu_pad
    ckv = cp if cu_pad_kv is _DEFAULT else cu_pad_kv
    o = None
    if out_canary is not None:
        o = torch.full_like(q, out_canary)
    o, lse, st = T.attn_fwd(q, k, v, d["cu"], d["cu"], cp, ckv, cp_size=w.cp_size, causal=causal,
                            softmax_scale=w.softmax_scale, pad_between_seqs=pad_flag, out=o)
    torch.cuda.synchronize()
    return o, lse, int(st.item())


def valid_rows(w, rows=None) -> np.ndarray:
    m = inputs.valid_row_mask(w)
    if rows is not None and rows > len(m):
        m = np.concatenate([m, np.zeros(rows - len(m), bool)])
    return m


def assert_fwd_close(w, t, o, lse, causal=True):
    """Full comparison against the oracle (small workloads)."""
    O_ref, lse_ref = orc.attn_fwd(t["q"].float().numpy(), t["k"].float().numpy(), t["v"].float().numpy(),
                                  w.cu_seqlens, w.cu_seqlens, w.cu_seqlens_padded, w.cu_seqlens_padded,
                                  causal=causal, softmax_scale=w.softmax_scale)
    og, lg = f64(o), f64(lse)
    T_ = O_ref.shape[0]
    valid = valid_rows(w)
    err = np.abs(og[:T_][valid] - O_ref[valid]).max() if valid.any() else 0.0
    lerr = np.abs(lg[:, :T_][:, valid] - lse_ref[:, valid]).max() if valid.any() else 0.0
    assert err <= O_TOL, f"O max-abs {err:.3e} > {O_TOL}"
    assert lerr <= LSE_TOL, f"lse max-abs {lerr:.3e} > {LSE_TOL}"
    # rows without a valid token: exactly 0 and -inf
    inv = ~valid_rows(w, og.shape[0])
    assert np.all(og[inv] == 0), "pad/tail rows of O must be 0"
    assert np.all(np.isneginf(lg[:, inv])), "pad/tail rows of lse must be -inf"
    return err, lerr


def sample_positions(L: int, cb: int, rng, n: int = 12) -> list[int]:
    """Query positions to check on a long sequence: chunk edges, tile edges,
    first/last rows and random ones."""
    cand = {0, L - 1}
    for c in range(0, L, max(cb, 1)):
        cand.update({c, c - 1, c + 127, c + 128})
    cand.update(int(x) for x in rng.integers(0, L, size=n))
    return sorted(x for x in cand if 0 <= x < L)


def assert_fwd_sampled(w, t, o, lse, heads, seed=0, causal=True):
    """Sampled comparison (full-size workloads): per sequence, a few query
    positions of the given heads are computed by the oracle one by one."""
    rng = np.random.default_rng(seed)
    og, lg = o.float().cpu().numpy(), lse.float().cpu().numpy()
    worst_o = worst_l = 0.0
    q = t["q"]
    k = t["k"]
    v = t["v"]
    for b in range(w.B):
        L = w.lengths[b]
        P = int(w.cu_seqlens_padded[b + 1] - w.cu_seqlens_padded[b])
        cb = P // (2 * w.cp_size)
        pos = sample_positions(L, cb, rng)
        off = int(w.cu_seqlens_padded[b])
        kk = k[off:off + L].float().numpy()
        vv = v[off:off + L].float().numpy()
        for h in heads:
            qq = q[off:off + L, h:h + 1].float().numpy()
            # q restricted to this head; k/v restricted to this sequence
            G = w.Hq // w.Hkv
            O_ref, l_ref = orc.attn_fwd_rows(
                np.repeat(qq, 1, axis=1), kk[:, h // G:h // G + 1], vv[:, h // G:h // G + 1],
                [0, L], [0, L], None, None, 0, 0, pos, causal=causal, softmax_scale=w.softmax_scale)
            rows = off + np.array(pos)
            worst_o = max(worst_o, float(np.abs(og[rows, h] - O_ref).max()))
            worst_l = max(worst_l, float(np.abs(lg[h, rows] - l_ref).max()))
    assert worst_o <= O_TOL, f"sampled O max-abs {worst_o:.3e}"
    assert worst_l <= LSE_TOL, f"sampled lse max-abs {worst_l:.3e}"
    return worst_o, worst_l
