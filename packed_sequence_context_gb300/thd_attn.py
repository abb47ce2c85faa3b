"""Thin ctypes binding of ``libthdattn.so`` (see ``include/thd_attn.h``).

The ``thd_*`` functions here have the C names and argument order; they only
marshal arguments (torch tensors -> device pointers, the current torch stream
-> cudaStream_t) and return the C status code.  Every step of the
computation runs in the library's CUDA kernels; there is no Python or CPU
fallback: if the library is missing, ``lib()`` raises.

The lower-case helpers at the end (``attn_fwd``, ``attn_bwd``, ...) allocate
outputs, workspace and the device status word with torch and call the
``thd_*`` functions -- allocation and marshalling only.
"""

from __future__ import annotations

import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libthdattn.so")

THD_OK = 0
THD_ERR_INVALID_ARG = 1
THD_ERR_UNSUPPORTED = 2
THD_ERR_CUDA = 3
THD_ERR_TIMEOUT = 4
THD_ERR_WORKSPACE = 5
THD_DEV_ERR_NONZERO_START = 101
THD_DEV_ERR_NOT_MONOTONE = 102
THD_DEV_ERR_VALID_GT_PAD = 103
THD_DEV_ERR_NOT_DIVISIBLE = 104
THD_DEV_ERR_EXCEEDS_BUF = 105
THD_DEV_ERR_CAUSAL_LENGTHS = 106
THD_DEV_ERR_CAPACITY = 107

THD_KERNEL_PLAN = 1
THD_KERNEL_FWD = 2
THD_KERNEL_BWD_PREP = 3
THD_KERNEL_BWD = 4
THD_KERNEL_BWD_DQ = 5
THD_KERNEL_LSE_MERGE = 6
THD_KERNEL_TAIL_ZERO = 7
THD_KERNEL_PARTITION = 8
THD_KERNEL_A2A = 9

THD_FWD_KERNEL_SINGLE = 1
THD_FWD_KERNEL_DUAL = 2

THD_CAUSAL_NONE = 0
THD_CAUSAL_TOP_LEFT = 1
THD_CAUSAL_BOTTOM_RIGHT = 2

THD_A2A_TO_GROUPS = 0
THD_A2A_TO_SHARDS = 1

_vp = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

# name -> (restype, argtypes); mirrors include/thd_attn.h
SIGNATURES = {
    "thd_status_string": (ctypes.c_char_p, [_i32]),
    "thd_version": (_i32, []),
    "thd_workspace_size": (_sz, [_i32, _i64, _i64, _i32, _i32, _i32, _i32, _i32]),
    "thd_cp_partition": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _i64, _vp, _vp]),
    "thd_attn_fwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _i32, _i32,
                            _i32, _f32, _i32, _i32, _vp, _sz, _vp, _vp]),
    "thd_attn_fwd_step": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _i32, _i32,
                                 _i32, _f32, _i32, _i32, _i32, _vp, _sz, _vp, _vp]),
    "thd_attn_fwd_step_bf16": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _i32,
                                      _i32, _i32, _f32, _i32, _i32, _i32, _vp, _sz, _vp, _vp]),
    "thd_attn_fwd_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i64, _i32, _i32,
                                    _i32, _i32, _f32, _i32, _i32, _vp, _vp]),
    "thd_attn_bwd": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _i32,
                            _i64, _i64, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _vp, _sz, _vp, _vp]),
    "thd_lse_merge": (_i32, [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _vp]),
    "thd_lse_merge_bf16": (_i32, [_vp, _vp, _vp, _vp, _i64, _i32, _i32, _vp]),
    "thd_grad_tail_zero": (_i32, [_vp, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp, _vp, _i32, _i32, _vp]),
    "thd_cp_a2a": (_i32, [_vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32, _i32, _vp, _vp]),
    "thd_a2a_workspace_size": (_sz, [_i32, _i64, _i32, _i32, _i32, _i32, _i32, _i32]),
    "thd_attn_fwd_a2a": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32, _f32, _i32,
                                _i32, _vp, _sz, _vp, _vp]),
    "thd_attn_bwd_a2a": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32,
                                _i32, _f32, _i32, _i32, _vp, _sz, _vp, _vp]),
    "thd_profile_enable": (_i32, [_i32, _i32]),
    "thd_profile_read": (_i32, [_vp, _i32, _vp]),
    "thd_launch_count": (ctypes.c_uint64, []),
    "thd_test_arm_stall": (_i32, [_i32]),
    "thd_test_select_fwd_kernel": (_i32, [_i32]),
}

_LIB = None


def lib() -> ctypes.CDLL:
    """Load the library (once).  Raises if it has not been built."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m packed_sequence_context_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _p(x):
    """Device pointer of a tensor (or pass an int / None through)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- C names
def thd_status_string(status: int) -> str:
    return lib().thd_status_string(status).decode()


def thd_version() -> int:
    return lib().thd_version()


def thd_workspace_size(B, T_q, T_kv, Hq, Hkv, D, cp_size, for_bwd) -> int:
    return lib().thd_workspace_size(B, T_q, T_kv, Hq, Hkv, D, cp_size, for_bwd)


def thd_cp_partition(cu_seqlens, cu_seqlens_padded, B, cp_size, pad_between_seqs, cu_rank, cu_rank_padded,
                     cu_rank_half, token_map, token_map_capacity, dev_status, stream=None) -> int:
    return lib().thd_cp_partition(_p(cu_seqlens), _p(cu_seqlens_padded), B, cp_size, pad_between_seqs,
                                  _p(cu_rank), _p(cu_rank_padded), _p(cu_rank_half), _p(token_map),
                                  token_map_capacity, _p(dev_status), _s(stream))


def thd_attn_fwd(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, B, T_q,
                 T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size, pad_between_seqs, workspace, workspace_bytes,
                 dev_status, stream=None) -> int:
    return lib().thd_attn_fwd(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cu_seqlens_q), _p(cu_seqlens_kv),
                              _p(cu_seqlens_q_padded), _p(cu_seqlens_kv_padded), B, T_q, T_kv, Hq, Hkv, D, causal,
                              softmax_scale, cp_size, pad_between_seqs, _p(workspace), workspace_bytes,
                              _p(dev_status), _s(stream))


def thd_attn_fwd_step(q, k, v, o_part, lse_part, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                      cu_seqlens_kv_padded, B, T_q, T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size,
                      pad_between_seqs, step, workspace, workspace_bytes, dev_status, stream=None) -> int:
    return lib().thd_attn_fwd_step(_p(q), _p(k), _p(v), _p(o_part), _p(lse_part), _p(cu_seqlens_q),
                                   _p(cu_seqlens_kv), _p(cu_seqlens_q_padded), _p(cu_seqlens_kv_padded), B, T_q,
                                   T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size, pad_between_seqs, step,
                                   _p(workspace), workspace_bytes, _p(dev_status), _s(stream))


def thd_attn_fwd_step_bf16(q, k, v, o_part, lse_part, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                           cu_seqlens_kv_padded, B, T_q, T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size,
                           pad_between_seqs, step, workspace, workspace_bytes, dev_status, stream=None) -> int:
    return lib().thd_attn_fwd_step_bf16(_p(q), _p(k), _p(v), _p(o_part), _p(lse_part), _p(cu_seqlens_q),
                                        _p(cu_seqlens_kv), _p(cu_seqlens_q_padded), _p(cu_seqlens_kv_padded), B, T_q,
                                        T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size, pad_between_seqs, step,
                                        _p(workspace), workspace_bytes, _p(dev_status), _s(stream))


def thd_attn_fwd_noalloc(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded,
                         B, T_q, T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size, pad_between_seqs, dev_status,
                         stream=None) -> int:
    return lib().thd_attn_fwd_noalloc(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cu_seqlens_q), _p(cu_seqlens_kv),
                                      _p(cu_seqlens_q_padded), _p(cu_seqlens_kv_padded), B, T_q, T_kv, Hq, Hkv, D,
                                      causal, softmax_scale, cp_size, pad_between_seqs, _p(dev_status), _s(stream))


def thd_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, dq_rows, dkv_rows, cu_seqlens_q, cu_seqlens_kv,
                 cu_seqlens_q_padded, cu_seqlens_kv_padded, B, T_q, T_kv, Hq, Hkv, D, causal, softmax_scale,
                 cp_size, pad_between_seqs, workspace, workspace_bytes, dev_status, stream=None) -> int:
    return lib().thd_attn_bwd(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(dout), _p(dq), _p(dk), _p(dv), dq_rows,
                              dkv_rows, _p(cu_seqlens_q), _p(cu_seqlens_kv), _p(cu_seqlens_q_padded),
                              _p(cu_seqlens_kv_padded), B, T_q, T_kv, Hq, Hkv, D, causal, softmax_scale, cp_size,
                              pad_between_seqs, _p(workspace), workspace_bytes, _p(dev_status), _s(stream))


def thd_lse_merge(o_acc, lse_acc, o_part, lse_part, T, H, D, stream=None) -> int:
    return lib().thd_lse_merge(_p(o_acc), _p(lse_acc), _p(o_part), _p(lse_part), T, H, D, _s(stream))


def thd_lse_merge_bf16(o_acc, lse_acc, o_part, lse_part, T, H, D, stream=None) -> int:
    return lib().thd_lse_merge_bf16(_p(o_acc), _p(lse_acc), _p(o_part), _p(lse_part), T, H, D, _s(stream))


def thd_grad_tail_zero(dq, dk, dv, dq_rows, dkv_rows, Hq, Hkv, D, cu_seqlens_q_padded, cu_seqlens_kv_padded, B,
                       host_knows_no_tail, stream=None) -> int:
    return lib().thd_grad_tail_zero(_p(dq), _p(dk), _p(dv), dq_rows, dkv_rows, Hq, Hkv, D, _p(cu_seqlens_q_padded),
                                    _p(cu_seqlens_kv_padded), B, host_knows_no_tail, _s(stream))


def thd_cp_a2a(src, dst, cu_seqlens_padded, B, T, H, D, cp_size, a2a_size, direction, dev_status,
               stream=None) -> int:
    return lib().thd_cp_a2a(_p(src), _p(dst), _p(cu_seqlens_padded), B, T, H, D, cp_size, a2a_size, direction,
                            _p(dev_status), _s(stream))


def thd_a2a_workspace_size(B, T, Hq, Hkv, D, cp_size, a2a_size, for_bwd) -> int:
    return lib().thd_a2a_workspace_size(B, T, Hq, Hkv, D, cp_size, a2a_size, for_bwd)


def thd_attn_fwd_a2a(q, k, v, o, lse, cu_seqlens, cu_seqlens_padded, B, T, Hq, Hkv, D, causal, softmax_scale,
                     cp_size, a2a_size, workspace, workspace_bytes, dev_status, stream=None) -> int:
    return lib().thd_attn_fwd_a2a(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cu_seqlens), _p(cu_seqlens_padded), B, T,
                                  Hq, Hkv, D, causal, softmax_scale, cp_size, a2a_size, _p(workspace),
                                  workspace_bytes, _p(dev_status), _s(stream))


def thd_attn_bwd_a2a(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens, cu_seqlens_padded, B, T, Hq, Hkv, D, causal,
                     softmax_scale, cp_size, a2a_size, workspace, workspace_bytes, dev_status, stream=None) -> int:
    return lib().thd_attn_bwd_a2a(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(dout), _p(dq), _p(dk), _p(dv),
                                  _p(cu_seqlens), _p(cu_seqlens_padded), B, T, Hq, Hkv, D, causal, softmax_scale,
                                  cp_size, a2a_size, _p(workspace), workspace_bytes, _p(dev_status), _s(stream))


def thd_profile_enable(kernel_id: int, max_records: int) -> int:
    return lib().thd_profile_enable(kernel_id, max_records)


def thd_profile_read(max_out: int = 4096) -> list[float]:
    buf = (ctypes.c_float * max_out)()
    n = ctypes.c_int(0)
    rc = lib().thd_profile_read(ctypes.cast(buf, _vp), max_out, ctypes.cast(ctypes.pointer(n), _vp))
    if rc != THD_OK:
        raise RuntimeError(f"thd_profile_read: {thd_status_string(rc)}")
    return [buf[i] for i in range(n.value)]


def thd_launch_count() -> int:
    return lib().thd_launch_count()


def thd_test_arm_stall(kernel_id: int) -> int:
    return lib().thd_test_arm_stall(kernel_id)


def thd_test_select_fwd_kernel(which: int) -> int:
    return lib().thd_test_select_fwd_kernel(which)


# ----------------------------------------------------------------- helpers
class ThdError(RuntimeError):
    def __init__(self, where: str, code: int):
        super().__init__(f"{where}: {thd_status_string(code)} ({code})")
        self.code = code


def _check(where: str, rc: int):
    if rc != THD_OK:
        raise ThdError(where, rc)


def check_status(dev_status) -> int:
    """Synchronise and raise on a nonzero device status word."""
    code = int(dev_status.item())
    if code != 0:
        raise ThdError("device", code)
    return code


def _workspace(nbytes, device):
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def attn_fwd(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded=None, cu_seqlens_kv_padded=None, *,
             cp_size=1, causal=True, softmax_scale=None, pad_between_seqs=-1, out=None, lse=None,
             dev_status=None, workspace=None, stream=None):
    """Allocate O [T_q,Hq,D] bf16, lse [Hq,T_q] fp32 and call thd_attn_fwd.
    Returns (o, lse, dev_status); read dev_status after synchronising."""
    import torch
    T_q, Hq, D = q.shape
    T_kv, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((Hq, T_q), dtype=torch.float32, device=q.device) if lse is None else lse
    st = torch.zeros(1, dtype=torch.int32, device=q.device) if dev_status is None else dev_status
    nbytes = thd_workspace_size(B, T_q, T_kv, Hq, Hkv, D, cp_size, 0)
    ws = _workspace(nbytes, q.device) if workspace is None else workspace
    _check("thd_attn_fwd", thd_attn_fwd(q, k, v, o, l, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                                        cu_seqlens_kv_padded, B, T_q, T_kv, Hq, Hkv, D, int(causal), scale,
                                        cp_size, pad_between_seqs, ws, ws.numel(), st, stream))
    return o, l, st


def attn_fwd_step(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded=None, cu_seqlens_kv_padded=None, *,
                  step, cp_size=1, causal=True, softmax_scale=None, pad_between_seqs=-1, out=None, lse=None,
                  stream=None):
    """One ring step's materialised partial: (o_part fp32 [T_q,Hq,D], lse_part [Hq,T_q], dev_status)."""
    import torch
    T_q, Hq, D = q.shape
    T_kv, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    o = torch.empty((T_q, Hq, D), dtype=torch.float32, device=q.device) if out is None else out
    l = torch.empty((Hq, T_q), dtype=torch.float32, device=q.device) if lse is None else lse
    st = torch.zeros(1, dtype=torch.int32, device=q.device)
    ws = _workspace(thd_workspace_size(B, T_q, T_kv, Hq, Hkv, D, cp_size, 0), q.device)
    _check("thd_attn_fwd_step", thd_attn_fwd_step(q, k, v, o, l, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded,
                                                  cu_seqlens_kv_padded, B, T_q, T_kv, Hq, Hkv, D, int(causal),
                                                  scale, cp_size, pad_between_seqs, step, ws, ws.numel(), st,
                                                  stream))
    return o, l, st


def attn_fwd_step_bf16(q, k, v, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded=None, cu_seqlens_kv_padded=None,
                       *, step, cp_size=1, causal=True, softmax_scale=None, pad_between_seqs=-1, out=None, lse=None,
                       dev_status=None, workspace=None, stream=None):
    """One ring step's partial in bf16: (o_part bf16 [T_q,Hq,D], lse_part fp32 [Hq,T_q], dev_status)."""
    import torch
    T_q, Hq, D = q.shape
    T_kv, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    o = torch.empty((T_q, Hq, D), dtype=torch.bfloat16, device=q.device) if out is None else out
    l = torch.empty((Hq, T_q), dtype=torch.float32, device=q.device) if lse is None else lse
    st = torch.zeros(1, dtype=torch.int32, device=q.device) if dev_status is None else dev_status
    ws = _workspace(thd_workspace_size(B, T_q, T_kv, Hq, Hkv, D, cp_size, 0), q.device) if workspace is None \
        else workspace
    _check("thd_attn_fwd_step_bf16", thd_attn_fwd_step_bf16(q, k, v, o, l, cu_seqlens_q, cu_seqlens_kv,
                                                            cu_seqlens_q_padded, cu_seqlens_kv_padded, B, T_q, T_kv,
                                                            Hq, Hkv, D, int(causal), scale, cp_size,
                                                            pad_between_seqs, step, ws, ws.numel(), st, stream))
    return o, l, st


def attn_bwd(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_kv, cu_seqlens_q_padded=None,
             cu_seqlens_kv_padded=None, *, cp_size=1, causal=True, softmax_scale=None, pad_between_seqs=-1,
             dq_rows=None, dkv_rows=None, dq=None, dk=None, dv=None, dev_status=None, workspace=None, stream=None):
    """Allocate dQ/dK/dV (with optional slack rows) and call thd_attn_bwd.
    Returns (dq, dk, dv, dev_status)."""
    import torch
    T_q, Hq, D = q.shape
    T_kv, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    dq_rows = T_q if dq_rows is None else dq_rows
    dkv_rows = T_kv if dkv_rows is None else dkv_rows
    dq = torch.empty((dq_rows, Hq, D), dtype=q.dtype, device=q.device) if dq is None else dq
    dk = torch.empty((dkv_rows, Hkv, D), dtype=q.dtype, device=q.device) if dk is None else dk
    dv = torch.empty((dkv_rows, Hkv, D), dtype=q.dtype, device=q.device) if dv is None else dv
    st = torch.zeros(1, dtype=torch.int32, device=q.device) if dev_status is None else dev_status
    nbytes = thd_workspace_size(B, T_q, T_kv, Hq, Hkv, D, cp_size, 1)
    ws = _workspace(nbytes, q.device) if workspace is None else workspace
    _check("thd_attn_bwd", thd_attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, dq_rows, dkv_rows, cu_seqlens_q,
                                        cu_seqlens_kv, cu_seqlens_q_padded, cu_seqlens_kv_padded, B, T_q, T_kv, Hq,
                                        Hkv, D, int(causal), scale, cp_size, pad_between_seqs, ws, ws.numel(), st,
                                        stream))
    return dq, dk, dv, st


def cp_partition(cu_seqlens, cu_seqlens_padded=None, *, cp_size, pad_between_seqs=-1, token_map_capacity=None,
                 stream=None):
    """Per-rank partition via thd_cp_partition.  Returns a dict of device
    int32 tensors (cu_rank [cp,B+1], cu_rank_padded [cp,B+1], cu_rank_half
    [cp,2,B+1], token_map [capacity]) and the status word."""
    import torch
    B = cu_seqlens.numel() - 1
    dev = cu_seqlens.device
    cap = int(token_map_capacity) if token_map_capacity is not None else 0
    out = {
        "cu_rank": torch.empty((cp_size, B + 1), dtype=torch.int32, device=dev),
        "cu_rank_padded": torch.empty((cp_size, B + 1), dtype=torch.int32, device=dev),
        "cu_rank_half": torch.empty((cp_size, 2, B + 1), dtype=torch.int32, device=dev),
        "token_map": torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
    }
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    _check("thd_cp_partition", thd_cp_partition(cu_seqlens, cu_seqlens_padded, B, cp_size, pad_between_seqs,
                                                out["cu_rank"], out["cu_rank_padded"], out["cu_rank_half"],
                                                out["token_map"] if cap else None, cap, st, stream))
    return out, st


def lse_merge(o_acc, lse_acc, o_part, lse_part, stream=None):
    """In-place merge of (o_part, lse_part) into (o_acc, lse_acc)."""
    T, H, D = o_acc.shape
    _check("thd_lse_merge", thd_lse_merge(o_acc, lse_acc, o_part, lse_part, T, H, D, stream))


def lse_merge_bf16(o_acc, lse_acc, o_part, lse_part, stream=None):
    """In-place merge of a bf16 partial (o_part, lse_part) into the fp32 (o_acc, lse_acc)."""
    T, H, D = o_acc.shape
    _check("thd_lse_merge_bf16", thd_lse_merge_bf16(o_acc, lse_acc, o_part, lse_part, T, H, D, stream))


def grad_tail_zero(dq, dk, dv, cu_seqlens_q_padded, cu_seqlens_kv_padded, host_knows_no_tail=False, stream=None):
    Hq, D = dq.shape[1], dq.shape[2]
    Hkv = dk.shape[1]
    B = cu_seqlens_q_padded.numel() - 1
    _check("thd_grad_tail_zero", thd_grad_tail_zero(dq, dk, dv, dq.shape[0], dk.shape[0], Hq, Hkv, D,
                                                    cu_seqlens_q_padded, cu_seqlens_kv_padded, B,
                                                    int(host_knows_no_tail), stream))


def cp_a2a(src, cu_seqlens_padded, *, cp_size, a2a_size, direction, out=None, dev_status=None, stream=None):
    """Allocate the other layout and call thd_cp_a2a.  THD_A2A_TO_GROUPS:
    src shards [cp, T/cp, H, D] -> [a2a, T, H/a2a, D]; THD_A2A_TO_SHARDS: the
    reverse.  Returns (dst, dev_status)."""
    import torch
    if direction == THD_A2A_TO_GROUPS:
        cp, rows_r, H, D = src.shape
        T = cp * rows_r
        shape = (a2a_size, T, H // a2a_size, D)
    else:
        a, T, Hg, D = src.shape
        H = a * Hg
        shape = (cp_size, T // cp_size, H, D)
    B = cu_seqlens_padded.numel() - 1
    dst = torch.empty(shape, dtype=src.dtype, device=src.device) if out is None else out
    st = torch.zeros(1, dtype=torch.int32, device=src.device) if dev_status is None else dev_status
    _check("thd_cp_a2a", thd_cp_a2a(src, dst, cu_seqlens_padded, B, T, H, D, cp_size, a2a_size, direction, st,
                                    stream))
    return dst, st


def attn_fwd_a2a(q, k, v, cu_seqlens, cu_seqlens_padded, *, cp_size, a2a_size, causal=True, softmax_scale=None,
                 out=None, lse=None, dev_status=None, workspace=None, stream=None):
    """Attention through the emulated A2A / hierarchical layer on shards
    q [cp, T/cp, Hq, D], k, v [cp, T/cp, Hkv, D].  Returns (o shards,
    lse [Hq, T] in global row order, dev_status)."""
    import torch
    cp, rows_r, Hq, D = q.shape
    Hkv = k.shape[2]
    T = cp * rows_r
    B = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    o = torch.empty_like(q) if out is None else out
    l = torch.empty((Hq, T), dtype=torch.float32, device=q.device) if lse is None else lse
    st = torch.zeros(1, dtype=torch.int32, device=q.device) if dev_status is None else dev_status
    nbytes = thd_a2a_workspace_size(B, T, Hq, Hkv, D, cp_size, a2a_size, 0)
    ws = _workspace(nbytes, q.device) if workspace is None else workspace
    _check("thd_attn_fwd_a2a", thd_attn_fwd_a2a(q, k, v, o, l, cu_seqlens, cu_seqlens_padded, B, T, Hq, Hkv, D,
                                                int(causal), scale, cp_size, a2a_size, ws, ws.numel(), st, stream))
    return o, l, st


def attn_bwd_a2a(q, k, v, o, lse, dout, cu_seqlens, cu_seqlens_padded, *, cp_size, a2a_size, causal=True,
                 softmax_scale=None, dq=None, dk=None, dv=None, dev_status=None, workspace=None, stream=None):
    """Gradients through the emulated A2A / hierarchical layer; shards in and
    out.  Returns (dq, dk, dv, dev_status)."""
    import torch
    cp, rows_r, Hq, D = q.shape
    Hkv = k.shape[2]
    T = cp * rows_r
    B = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(D) if softmax_scale is None else float(softmax_scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = torch.zeros(1, dtype=torch.int32, device=q.device) if dev_status is None else dev_status
    nbytes = thd_a2a_workspace_size(B, T, Hq, Hkv, D, cp_size, a2a_size, 1)
    ws = _workspace(nbytes, q.device) if workspace is None else workspace
    _check("thd_attn_bwd_a2a", thd_attn_bwd_a2a(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens, cu_seqlens_padded, B,
                                                T, Hq, Hkv, D, int(causal), scale, cp_size, a2a_size, ws, ws.numel(),
                                                st, stream))
    return dq, dk, dv, st
