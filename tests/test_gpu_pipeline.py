"""The overlapped host pipeline (uploads, calls and downloads on three streams with double-
buffered device memory) gives the results of the same calls made one after another: bit for
bit for the head (its kernels are deterministic), and for the chain within the chain
tolerance (1e-5 of the oracle's forward-error envelope): the single-pass scan resolves a
chunk's carry from whichever earlier chunks have published, so its rounding can differ from
run to run."""
import math

import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def R():
    import __graft_entry__
    __graft_entry__.build()
    import gated_causal_attention_gb300 as R
    assert torch.cuda.is_available()
    return R


def pinned(x, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(x)).to(dtype).pin_memory()


def test_pipelined_head_equals_serial_calls(R):
    from gated_causal_attention_gb300.pipeline import HostPipeline
    B, H, n, d, dv = 1, 4, 300, 64, 64
    shp = (B, H, n)
    batches = []
    for i in range(5):
        hi = W.head_inputs(B, H, n, d, dv, seed=60 + i, q_scale=1 / 8, u_range=(0.8, 1.0),
                           zero_frac=0.01, beta=[1.0, 0.5, 0.0, 1.0], qk=[1.0, 1.0, 1.0, 0.0],
                           g=[0.5, 0.0, 1.0, 0.3])
        batches.append([pinned(hi.q.reshape(*shp, d), torch.bfloat16),
                        pinned(hi.k.reshape(*shp, d), torch.bfloat16),
                        pinned(hi.u.reshape(shp)), pinned(hi.theta.reshape(shp)),
                        pinned(hi.v.reshape(*shp, dv), torch.bfloat16)])
    sw = dict(beta=[1.0, 0.5, 0.0, 1.0], qk=[1.0, 1.0, 1.0, 0.0], g=[0.5, 0.0, 1.0, 0.3])
    ws = torch.empty(R.head_workspace_bytes(B, H, n, d, dv, torch.bfloat16), dtype=torch.uint8,
                     device="cuda")
    status = R.new_status()

    def call(di, do, stream):
        q, k, u, th, v = di
        R.head_forward(q, k, u, th, v, sw["beta"], sw["qk"], sw["g"], out=(do[0], do[1]),
                       workspace=ws, status=status, stream=stream, sync=False)

    spec_in = [((*shp, d), torch.bfloat16), ((*shp, d), torch.bfloat16), (shp, torch.float32),
               (shp, torch.float32), ((*shp, dv), torch.bfloat16)]
    spec_out = [((*shp, dv), torch.float32)] * 2
    pipe = HostPipeline(call, spec_in, spec_out)
    outs = [[torch.empty((*shp, dv)).pin_memory() for _ in range(2)] for _ in batches]
    for hin, hout in zip(batches, outs):
        pipe.submit(hin, hout)
    pipe.synchronize()
    R.status_sync(status)
    for hin, hout in zip(batches, outs):
        q, k, u, th, v = [x.cuda() for x in hin]
        Ore, Oim = R.head_forward(q, k, u, th, v, sw["beta"], sw["qk"], sw["g"])
        assert torch.equal(Ore.cpu(), hout[0]) and torch.equal(Oim.cpu(), hout[1])


def test_pipelined_chain_equals_serial_calls(R, oracle_mod):
    from gated_causal_attention_gb300.pipeline import HostPipeline
    B, H, n, dv = 2, 3, 1000, 64
    shp = (B, H, n)
    r = np.random.default_rng(61)
    batches = [[pinned(r.uniform(0.9, 1.0, shp)), pinned(r.uniform(-math.pi, math.pi, shp)),
                pinned(r.standard_normal((*shp, dv)))] for _ in range(4)]
    ws = torch.empty(R.chain_workspace_bytes(B, H, n, dv), dtype=torch.uint8, device="cuda")
    status = R.new_status()

    def call(di, do, stream):
        u, th, b = di
        R.chain_scan(u, th, 1.0, b, out=(do[0], do[1]), workspace=ws, status=status,
                     stream=stream, sync=False)

    pipe = HostPipeline(call, [(shp, torch.float32)] * 2 + [((*shp, dv), torch.float32)],
                        [((*shp, dv), torch.float32)] * 2, depth=2)
    outs = [[torch.empty((*shp, dv)).pin_memory() for _ in range(2)] for _ in batches]
    for hin, hout in zip(batches, outs):
        pipe.submit(hin, hout)
    pipe.synchronize()
    R.status_sync(status)
    for hin, hout in zip(batches, outs):
        u, th, b = [x.cuda() for x in hin]
        yr, yi = R.chain_scan(u, th, 1.0, b)
        yref, env, st = oracle_mod.chain_heads(hin[0].numpy().reshape(B * H, n),
                                               hin[1].numpy().reshape(B * H, n), [1.0] * (B * H),
                                               hin[2].numpy().reshape(B * H, n, dv))
        assert np.all(st == 0)
        yref, env = yref.reshape(B, H, n, dv), env.reshape(B, H, n, dv)
        for re, im in ((yr.cpu(), yi.cpu()), (hout[0], hout[1])):
            y = re.double().numpy() + 1j * im.double().numpy()
            assert np.all(np.abs(y - yref) <= 1e-5 * env + 1e-30)
