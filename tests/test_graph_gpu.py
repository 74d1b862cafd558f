"""CUDA graph capture (``-m gpu``).

With caller workspaces every entry point is stream-ordered, allocates
nothing and never synchronises the host, so a step can be captured once
into a CUDA graph and replayed.  Every combine in the kernels runs in a
fixed order, so a replay reproduces the eager results bit for bit."""
import pytest
import torch

import prefix_sum_outer_gb300 as cp
from prefix_sum_outer_gb300.workloads import make_inputs, make_norm_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _ws(nbytes):
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
def test_fwd_bwd_step_replays_bitwise(dt):
    B, H, N, D, M = 2, 8, 1000, 64, 64
    q, k, v, g = (t.to(DEV) for t in make_inputs(B, H, N, D, M, dt, seed=3))
    ws_f = _ws(cp.causal_product_workspace_size(B, H, N, D, M, dt, False))
    ws_b = _ws(cp.causal_product_workspace_size(B, H, N, D, M, dt, True))
    out = torch.empty_like(v)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step(stream):
        cp.causal_product_fwd(q, k, v, out=out, workspace=ws_f, stream=stream)
        cp.causal_product_bwd(q, k, v, g, dq, dk, dv, workspace=ws_b, stream=stream)

    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    eager = [t.clone() for t in (out, dq, dk, dv)]
    for t in (out, dq, dk, dv):
        t.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(s)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    for got, ref in zip((out, dq, dk, dv), eager):
        assert torch.equal(got, ref)
    assert cp.causal_product_status(ws_f) == cp.CP_OK and cp.causal_product_status(ws_b) == cp.CP_OK


def test_normalizer_and_decode_replay_bitwise():
    B, H, N, D = 4, 8, 3000, 64
    q, k, gz = (t.to(DEV) for t in make_norm_inputs(B, H, N, D, torch.bfloat16, seed=5))
    ws = _ws(cp.load_library().causal_product_normalizer_workspace_size(B, H, N, D, 1))
    z = torch.empty((B, H, N), device=DEV)
    nq, nk = torch.empty_like(q), torch.empty_like(k)
    qt, kt, vt = (t.to(DEV) for t in make_inputs(B, H, 1, D, D, torch.bfloat16, seed=6,
                                                 backward=False)[:3])
    qt, kt, vt = qt[:, :, 0].contiguous(), kt[:, :, 0].contiguous(), vt[:, :, 0].contiguous()
    state0 = torch.randn((B, H, D, D), generator=torch.Generator().manual_seed(7)).to(DEV)
    state = state0.clone()
    ot = torch.empty_like(vt)

    def step(stream):
        cp.causal_product_normalizer(q, k, z=z, workspace=ws, stream=stream)
        cp.causal_product_normalizer_bwd(q, k, gz, nq, nk, workspace=ws, stream=stream)
        cp.causal_product_decode(qt, kt, vt, state, out=ot, stream=stream)

    step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    eager = [t.clone() for t in (z, nq, nk, ot, state)]
    state.copy_(state0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(s)
    graph.replay()   # one decoding step from state0, as in the eager call
    torch.cuda.synchronize()
    for got, ref in zip((z, nq, nk, ot, state), eager):
        assert torch.equal(got, ref)
