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
