"""Host-side checks of the C-ABI library that need no GPU: it builds for sm_103a, loads, and
exports every function include/resolvent.h declares; the host argument checks answer
before anything touches a device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def built_lib():
    from gated_causal_attention_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def declared_functions():
    text = open(os.path.join(ROOT, "include", "resolvent.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(resolvent_\w+)\s*\(", text)))


def test_header_declares_the_three_calls():
    names = declared_functions()
    for n in ("resolvent_gate_prep", "resolvent_head_forward", "resolvent_chain_scan",
              "resolvent_status_sync"):
        assert n in names


def test_library_exports_every_declared_symbol(built_lib):
    missing = [n for n in declared_functions() if not hasattr(built_lib, n)]
    assert not missing, missing


def test_host_argument_checks_without_a_gpu(built_lib):
    """Shape errors and empty calls are answered on the host, before any CUDA call."""
    import gated_causal_attention_gb300 as R
    L = R.lib()
    sw, keep = R._switches(2, 1.0, 1.0, 0.5)
    # n == 0: empty call, RS_OK, nothing launched
    assert L.resolvent_head_forward(None, None, None, None, None, sw, 1, 2, 0, 64, 64, R.RS_BF16,
                                    None, None, None, 0, None, None) == R.RS_OK
    # head_dim = 0 with n > 0: a shape error (the pages' module panics)
    assert L.resolvent_head_forward(None, None, None, None, None, sw, 1, 2, 5, 0, 64, R.RS_BF16,
                                    None, None, None, 0, None, None) == R.RS_ERR_SHAPE
    # d above 128 or not a multiple of 8
    assert L.resolvent_head_forward(None, None, None, None, None, sw, 1, 2, 5, 256, 64, R.RS_BF16,
                                    None, None, None, 0, None, None) == R.RS_ERR_UNSUPPORTED
    # a non-finite switch is refused at once
    bad, keep2 = R._switches(2, float("nan"), 1.0, 0.5)
    assert L.resolvent_head_forward(None, None, None, None, None, bad, 1, 2, 5, 64, 64, R.RS_BF16,
                                    None, None, None, 0, None, None) == R.RS_ERR_NONFINITE
    # switch count must be 1 or H
    three, keep3 = R._switches(3, [1.0, 1.0, 1.0], 1.0, 0.5)
    assert L.resolvent_chain_scan(None, None, three, None, 1, 2, 5, 4, None, None, None, 0, None,
                                  None) == R.RS_ERR_SHAPE
    assert L.resolvent_head_workspace_bytes(1, 2, 0, 64, 64, R.RS_BF16) == 0
    assert L.resolvent_head_workspace_bytes(2, 3, 300, 64, 64, R.RS_BF16) > 2 * 3 * 300 * 24
    assert L.resolvent_status_string(R.RS_ERR_NONFINITE) == b"non-finite input refused"


def test_operator_and_position_argument_checks_without_a_gpu(built_lib):
    """The operator and position-head entry points answer shape, support, switch, alignment
    and workspace errors on the host, before any CUDA call (pointer values are only
    inspected, never dereferenced)."""
    import gated_causal_attention_gb300 as R
    L = R.lib()
    A, M = 0x10000, 0x10004  # a 16-byte-aligned and a misaligned address (never dereferenced)
    sw, keep = R._switches(2, 1.0, 1.0, 0.5)
    sw0, keep0 = R._switches(2, 1.0, 1.0, 0.0)
    # operator: empty call; d = 0; d not a multiple of 8; misaligned; workspace too small
    op = lambda n, d, q, ws, wsb, s=sw: L.resolvent_operator(q, A, A, A, s, 1, 2, n, d, R.RS_BF16,
                                                              A, A, ws, wsb, A, None)
    assert op(0, 64, A, A, 0) == R.RS_OK
    assert op(5, 0, A, A, 0) == R.RS_ERR_SHAPE
    assert op(5, 60, A, A, 0) == R.RS_ERR_UNSUPPORTED
    assert op(5, 64, M, A, 1 << 30) == R.RS_ERR_ALIGN
    need = L.resolvent_operator_workspace_bytes(1, 2, 300, 64, R.RS_BF16)
    assert need > 0 and L.resolvent_operator_workspace_bytes(1, 2, 0, 64, R.RS_BF16) == 0
    assert op(300, 64, A, A, need - 1) == R.RS_ERR_WORKSPACE
    assert op(300, 64, A, None, 0) == R.RS_ERR_WORKSPACE
    # position heads: empty call; dv = 0 or above 128; a gate switch other than 0;
    # misaligned; workspace too small
    pos = lambda n, dv, v, ws, wsb, s=sw0: L.resolvent_position_head(A, v, s, 1, 2, n, dv, R.RS_BF16,
                                                                     A, ws, wsb, A, None)
    assert pos(0, 64, A, A, 0) == R.RS_OK
    assert pos(5, 0, A, A, 0) == R.RS_ERR_SHAPE
    assert pos(5, 256, A, A, 0) == R.RS_ERR_UNSUPPORTED
    assert pos(5, 64, A, A, 1 << 30, s=sw) == R.RS_ERR_UNSUPPORTED
    assert pos(5, 64, M, A, 1 << 30) == R.RS_ERR_ALIGN
    needp = L.resolvent_position_workspace_bytes(1, 2, 300, 64, R.RS_BF16)
    assert needp > 0 and L.resolvent_position_workspace_bytes(1, 2, 0, 64, R.RS_BF16) == 0
    assert pos(300, 64, A, A, needp - 1) == R.RS_ERR_WORKSPACE
    bad, keepb = R._switches(2, float("inf"), 1.0, 0.0)
    assert pos(5, 64, A, A, 1 << 30, s=bad) == R.RS_ERR_NONFINITE

