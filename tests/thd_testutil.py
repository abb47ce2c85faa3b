"""Helpers shared by the GPU parity tests: move a seeded workload to the GPU,
run the library through its C ABI binding, and compare with the oracle."""

from __future__ import annotations

import numpy as np
import torch

import oracle_pool
from oracle import thd_oracle as orc
from packed_sequence_context_gb300 import inputs
from packed_sequence_context_gb300 import thd_attn as T

O_TOL = 2e-2     # max-abs on valid rows, outputs and gradients (bf16 results)
LSE_TOL = 1e-3   # max-abs on valid rows


def assert_within_bar(name: str, got: np.ndarray, ref: np.ndarray):
    """The bar for bf16 results (O, dQ, dK, dV), the same everywhere: the error
    beyond the result's own bf16 rounding within O_TOL, and the raw error
    within O_TOL wherever |ref| < 2 (see oracle_pool)."""
    s = oracle_pool.compare(got, ref)
    assert s["excess"] <= O_TOL and s["raw_small"] <= O_TOL, f"{name}: {s}"
    return s


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
