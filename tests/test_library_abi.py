"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports
every symbol include/thd_attn.h declares, and rejects bad host-side arguments
before touching the device.  No compute call runs here."""

import ctypes
import os
import re

import pytest

from packed_sequence_context_gb300 import thd_attn as T

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "thd_attn.h")


def _declared():
    src = open(HEADER).read()
    return re.findall(r"^THD_API\s+[\w\s\*]+?\b(thd_\w+)\s*\(", src, flags=re.M)


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("thd_cp_partition", "thd_attn_fwd", "thd_attn_bwd", "thd_lse_merge", "thd_grad_tail_zero",
              "thd_workspace_size", "thd_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(thd_lib):
    for name in _declared():
        assert hasattr(thd_lib, name), name
        assert name in T.SIGNATURES, f"binding lacks {name}"


def test_binding_names_match_c_names():
    for name in T.SIGNATURES:
        assert callable(getattr(T, name)), name


def test_status_strings_and_version(thd_lib):
    assert T.thd_version() >= 100
    for code in (0, 1, 2, 3, 4, 5, 101, 102, 103, 104, 105, 106, 107):
        s = T.thd_status_string(code)
        assert s and s != "unknown status"
    assert T.thd_status_string(9999) == "unknown status"


def test_workspace_size(thd_lib):
    f = T.thd_workspace_size(8, 14632, 14632, 16, 16, 128, 4, 0)
    b = T.thd_workspace_size(8, 14632, 14632, 16, 16, 128, 4, 1)
    assert 0 < f < b
    # backward: Delta (fp32 [Hq][T]) and a second schedule; dQ stays on chip
    assert b >= 14632 * 16 * 4
    assert b < 14632 * 16 * 128 * 4
    assert T.thd_workspace_size(8, 100, 100, 16, 16, 96, 4, 0) == 0   # unsupported head dim
    assert T.thd_workspace_size(0, 100, 100, 16, 16, 64, 4, 0) == 0


def test_host_side_rejections_need_no_device(thd_lib):
    # null tensors -> invalid argument, decided before any CUDA call
    rc = T.thd_attn_fwd(None, None, None, None, None, None, None, None, None, 2, 192, 192, 2, 2, 64, 1, 0.125,
                        2, -1, None, 0, None, stream=0)
    assert rc == T.THD_ERR_INVALID_ARG
    # unsupported head dim
    rc = T.thd_attn_fwd(16, 16, 16, 16, 16, 16, 16, None, None, 2, 192, 192, 2, 2, 96, 1, 0.125, 2, -1,
                        256, 1 << 20, 16, stream=0)
    assert rc == T.THD_ERR_UNSUPPORTED
    # Hq not a multiple of Hkv
    rc = T.thd_attn_fwd(16, 16, 16, 16, 16, 16, 16, None, None, 2, 192, 192, 3, 2, 64, 1, 0.125, 2, -1,
                        256, 1 << 20, 16, stream=0)
    assert rc == T.THD_ERR_INVALID_ARG
    # workspace too small
    rc = T.thd_attn_fwd(16, 16, 16, 16, 16, 16, 16, None, None, 2, 192, 192, 2, 2, 64, 1, 0.125, 2, -1,
                        256, 8, 16, stream=0)
    assert rc == T.THD_ERR_WORKSPACE
    # bad pad flag, bad scale, bad causal flag
    for args in ((2, -1.0, 1), (5, 0.125, 1), (-1, 0.125, 7)):
        pad, scale, causal = args
        rc = T.thd_attn_fwd(16, 16, 16, 16, 16, 16, 16, None, None, 2, 192, 192, 2, 2, 64, causal, scale, 2,
                            pad, 256, 1 << 20, 16, stream=0)
        assert rc == T.THD_ERR_INVALID_ARG
    # step out of range
    rc = T.thd_attn_fwd_step(16, 16, 16, 16, 16, 16, 16, None, None, 2, 192, 192, 2, 2, 64, 1, 0.125, 2, -1,
                             2, 256, 1 << 20, 16, stream=0)
    assert rc == T.THD_ERR_INVALID_ARG
    # misaligned tensor pointer
    rc = T.thd_attn_fwd(18, 16, 16, 16, 16, 16, 16, None, None, 2, 192, 192, 2, 2, 64, 1, 0.125, 2, -1,
                        256, 1 << 20, 16, stream=0)
    assert rc == T.THD_ERR_INVALID_ARG
    # backward: gradient buffers shorter than the data
    rc = T.thd_attn_bwd(16, 16, 16, 16, 16, 16, 16, 16, 16, 100, 192, 16, 16, None, None, 2, 192, 192, 2, 2, 64,
                        1, 0.125, 2, -1, 256, 1 << 30, 16, stream=0)
    assert rc == T.THD_ERR_INVALID_ARG
    # merge: D not a multiple of 4
    assert T.thd_lse_merge(16, 16, 16, 16, 10, 2, 6, stream=0) == T.THD_ERR_INVALID_ARG
    # tail-zero: the caller knows there is no tail -> OK with no launch
    before = T.thd_launch_count()
    assert T.thd_grad_tail_zero(16, 16, 16, 192, 192, 2, 2, 64, 16, 16, 2, 1, stream=0) == T.THD_OK
    assert T.thd_launch_count() == before
    # partition: bad cp
    assert T.thd_cp_partition(16, None, 2, 0, -1, None, None, None, None, 0, 16, stream=0) == T.THD_ERR_INVALID_ARG


def test_library_refuses_to_load_when_missing(monkeypatch, tmp_path):
    import importlib
    mod = importlib.reload(T)
    monkeypatch.setattr(mod, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(mod, "_LIB", None)
    with pytest.raises(RuntimeError):
        mod.lib()
    importlib.reload(T)


def test_a2a_host_side_checks(thd_lib):
    A = T.THD_A2A_TO_GROUPS
    # heads not divisible by the a2a group, a2a not dividing cp, T not divisible by cp, bad direction,
    # misaligned pointer, missing metadata: rejected before any CUDA call
    for args in ((16, 16, 16, 2, 192, 3, 64, 2, 2, A), (16, 16, 16, 2, 192, 4, 64, 4, 3, A),
                 (16, 16, 16, 2, 190, 4, 64, 4, 2, A), (16, 16, 16, 2, 192, 4, 64, 4, 2, 2),
                 (18, 16, 16, 2, 192, 4, 64, 4, 2, A), (16, 16, None, 2, 192, 4, 64, 4, 2, A),
                 (16, 16, 16, 2, 192, 4, 12, 4, 2, A)):
        assert T.thd_cp_a2a(*args, 16, stream=0) == T.THD_ERR_INVALID_ARG, args
    f = T.thd_a2a_workspace_size(8, 14632, 16, 16, 128, 4, 2, 0)
    b = T.thd_a2a_workspace_size(8, 14632, 16, 16, 128, 4, 2, 1)
    # the forward holds q, k, v, O in the group layout, the backward also dO, dQ, dK, dV
    assert f >= 4 * 14632 * 16 * 128 * 2 and b >= 8 * 14632 * 16 * 128 * 2 and b > f
    assert T.thd_a2a_workspace_size(8, 14632, 16, 16, 96, 4, 2, 0) == 0     # head dim of the attention
    assert T.thd_a2a_workspace_size(8, 14632, 16, 16, 128, 4, 3, 0) == 0    # 3 does not divide cp
    assert T.thd_a2a_workspace_size(8, 14632, 16, 6, 128, 4, 4, 0) == 0     # kv heads over 4 members
    # composites: workspace too small, bad scale
    rc = T.thd_attn_fwd_a2a(16, 16, 16, 16, 16, 16, 16, 2, 192, 4, 4, 64, 1, 0.125, 4, 2, 256, 8, 16, stream=0)
    assert rc == T.THD_ERR_WORKSPACE
    rc = T.thd_attn_fwd_a2a(16, 16, 16, 16, 16, 16, 16, 2, 192, 4, 4, 64, 1, -1.0, 4, 2, 256, 1 << 30, 16,
                            stream=0)
    assert rc == T.THD_ERR_INVALID_ARG
    rc = T.thd_attn_bwd_a2a(16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 16, 2, 192, 4, 4, 64, 1, 0.125, 4, 2, 256, 8,
                            16, stream=0)
    assert rc == T.THD_ERR_WORKSPACE
