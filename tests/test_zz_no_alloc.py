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


LIMIT = 8 << 20  # the fixed scratch array, bytes


def largest_n_within(L, B, H, dv):
    """The largest n (a multiple of the 128-token chunk) whose chain scratch fits the array."""
    n = 128
    while L.resolvent_chain_workspace_bytes(B, H, n + 128, dv) <= LIMIT:
        n += 128
    return n


def test_noalloc_chain_at_the_size_limit(oracle_mod):
    """At the largest size whose scratch still fits the array, the no-allocation entry point
    gives the workspace entry point's result (within the chain tolerance); one chunk more is
    refused with RS_ERR_UNSUPPORTED before anything is launched. The refused call gets real
    device buffers of its own size, so even a broken size check would launch in bounds."""
    import __graft_entry__
    __graft_entry__.build()
    import gated_causal_attention_gb300 as R
    L = R.lib()
    B, H, dv = 1, 8, 128
    n = largest_n_within(L, B, H, dv)
    assert L.resolvent_chain_workspace_bytes(B, H, n, dv) <= LIMIT
    n_over = n + 128
    assert L.resolvent_chain_workspace_bytes(B, H, n_over, dv) > LIMIT

    r = np.random.default_rng(78)
    u = r.uniform(0.95, 1.0, (B, H, n_over)).astype(np.float32)
    u[r.uniform(size=u.shape) < 0.01] = 0.0
    th = r.uniform(-math.pi, math.pi, (B, H, n_over)).astype(np.float32)
    du, dth = torch.from_numpy(u).cuda(), torch.from_numpy(th).cuda()
    db = torch.randn(B, H, n_over, dv, device="cuda", generator=torch.Generator("cuda").manual_seed(5))
    y_re = torch.full_like(db, float("nan"))
    y_im = torch.full_like(db, float("nan"))
    sw, keep = R._switches(H, 0.0, 0.0, 1.0)
    status = R.new_status()
    stream = torch.cuda.current_stream().cuda_stream

    # one chunk beyond the limit: refused, nothing written
    rc = L.resolvent_chain_scan_noalloc(du.data_ptr(), dth.data_ptr(), sw, db.data_ptr(), B, H,
                                        n_over, dv, y_re.data_ptr(), y_im.data_ptr(),
                                        status.data_ptr(), stream)
    assert rc == R.RS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.isnan(y_re).all()

    # at the limit: the same result as the workspace entry point
    us, ths = du[:, :, :n].contiguous(), dth[:, :, :n].contiguous()
    bs = db[:, :, :n].contiguous()
    ref_re, ref_im = R.chain_scan(us, ths, 1.0, bs)
    ys_re, ys_im = y_re[:, :, :n].contiguous(), y_im[:, :, :n].contiguous()
    rc = L.resolvent_chain_scan_noalloc(us.data_ptr(), ths.data_ptr(), sw, bs.data_ptr(), B, H, n,
                                        dv, ys_re.data_ptr(), ys_im.data_ptr(), status.data_ptr(),
                                        stream)
    assert rc == R.RS_OK
    R.status_sync(status)
    _, env, st = oracle_mod.chain_heads(u[:, :, :n].reshape(B * H, n), th[:, :, :n].reshape(B * H, n),
                                        [1.0] * (B * H), bs.cpu().numpy().reshape(B * H, n, dv))
    assert np.all(st == 0)
    env = env.reshape(B, H, n, dv)
    for got, ref in ((ys_re, ref_re), (ys_im, ref_im)):
        err = (got - ref).abs().cpu().double().numpy()
        assert np.all(np.isfinite(got.cpu().numpy()))
        assert np.all(err <= 1e-5 * env + 1e-30)
