"""resolvent_chain_scan_noalloc: the chain with its scratch in the library's fixed device
array, for callers that cannot allocate device memory (a framework pool that owns all of
it, a plugin host that hands out only inputs and outputs, a loop where an allocation is
not acceptable).

Called through the C ABI twice in a row (the second call must find its counters cleared
again) and compared with resolvent_chain_scan on the same inputs, within the chain
tolerance the other tests use (1e-5 of the forward-error envelope). The file name sorts
last so that a run stopping at the first failure has run every other test first.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def test_noalloc_chain_matches_the_workspace_entry_point(oracle_mod):
    import __graft_entry__
    __graft_entry__.build()
    import gated_causal_attention_gb300 as R
    assert torch.cuda.is_available()
    L = R.lib()

    B, H, n, dv = 2, 3, 1000, 64
    r = np.random.default_rng(77)
    u = r.uniform(0.9, 1.0, (B, H, n)).astype(np.float32)
    u[r.uniform(size=u.shape) < 0.01] = 0.0
    th = r.uniform(-math.pi, math.pi, (B, H, n)).astype(np.float32)
    b = r.standard_normal((B, H, n, dv)).astype(np.float32)
    gs = [1.0, 0.4, 0.0]
    du, dth, db = (torch.from_numpy(x).cuda() for x in (u, th, b))

    ref_re, ref_im = R.chain_scan(du, dth, gs, db)
    ref = ref_re.cpu().double().numpy() + 1j * ref_im.cpu().double().numpy()
    _, env, st = oracle_mod.chain_heads(u.reshape(B * H, n), th.reshape(B * H, n),
                                        np.tile(np.float32(gs).astype(np.float64), B),
                                        b.reshape(B * H, n, dv))
    assert np.all(st == 0)
    env = env.reshape(B, H, n, dv)

    sw, keep = R._switches(H, 0.0, 0.0, gs)
    status = R.new_status()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        y_re = torch.full_like(db, float("nan"))
        y_im = torch.full_like(db, float("nan"))
        rc = L.resolvent_chain_scan_noalloc(du.data_ptr(), dth.data_ptr(), sw, db.data_ptr(),
                                            B, H, n, dv, y_re.data_ptr(), y_im.data_ptr(),
                                            status.data_ptr(), stream)
        assert rc == R.RS_OK, f"call {call}: rs_status {rc}"
        R.status_sync(status)
        got = y_re.cpu().double().numpy() + 1j * y_im.cpu().double().numpy()
        assert np.all(np.isfinite(got)), f"call {call}"
        assert np.all(np.abs(got - ref) <= 1e-5 * env + 1e-30), f"call {call}"


def test_noalloc_chain_rejects_sizes_beyond_its_scratch():
    import gated_causal_attention_gb300 as R
    L = R.lib()
    sw, keep = R._switches(1, 0.0, 0.0, 1.0)
    # 128 heads x 2^20 tokens at dv = 64 need far more than the fixed 8 MiB
    assert L.resolvent_chain_workspace_bytes(1, 128, 1 << 20, 64) > 8 << 20
    rc = L.resolvent_chain_scan_noalloc(16, 16, sw, 16, 1, 1, 1 << 24, 64, 16, 16, 16, None)
    assert rc == R.RS_ERR_UNSUPPORTED
