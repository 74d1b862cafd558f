"""Back-to-back calls on one stream with caller workspaces (``-m gpu``).

With its own workspaces a caller's launches follow one another directly:
the product kernels start as programmatic dependents of the kernel before
them and must not read their inputs before it has completed.  Each call here
consumes the previous call's output, with nothing in between: the forward's
output is the backward's grad_out, the backward's gradients are the next
forward's inputs, and a forward's final state is the next call's initial
state.  Each result is compared with the oracle on the values the GPU
actually received (the intermediates as the GPU wrote them)."""
import numpy as np
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _ws(B, H, N, D, M, dt, backward):
    n = cp.causal_product_workspace_size(B, H, N, D, M, dt, backward)
    return torch.zeros(n, dtype=torch.uint8, device=DEV)


@pytest.mark.parametrize("shape", [(8, 16, 1024, 64, 64), (2, 4, 1000, 64, 64),
                                   (1, 2, 700, 128, 128)], ids=lambda s: "x".join(map(str, s)))
def test_forward_backward_forward_chain(shape):
    B, H, N, D, M = shape
    dt = torch.bfloat16
    q, k, v, _ = (t.to(DEV) if t is not None else None
                  for t in make_inputs(B, H, N, D, M, dt, seed=N, backward=False))
    ws_f, ws_b = _ws(B, H, N, D, M, dt, False), _ws(B, H, N, D, M, dt, True)
    out = torch.empty_like(v)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    out2 = torch.empty_like(v)
    stream = torch.cuda.current_stream()
    cp.causal_product_fwd(q, k, v, out=out, workspace=ws_f, stream=stream)
    cp.causal_product_bwd(q, k, v, out, dq, dk, dv, workspace=ws_b, stream=stream)
    if D == M:
        cp.causal_product_fwd(dq, dk, dv, out=out2, workspace=ws_f, stream=stream)
    torch.cuda.synchronize()
    assert cp.causal_product_status(ws_f) == cp.CP_OK and cp.causal_product_status(ws_b) == cp.CP_OK
    qn, kn, vn, on = to_np(q), to_np(k), to_np(v), to_np(out)
    assert row_rel_err(on, oracle.fwd(qn, kn, vn)) <= TOL["bf16"]
    r = oracle.bwd(qn, kn, vn, on)
    for got, ref in zip((dq, dk, dv), r):
        assert row_rel_err(to_np(got), ref) <= TOL["bf16"]
    if D == M:
        assert row_rel_err(to_np(out2), oracle.fwd(to_np(dq), to_np(dk), to_np(dv))) <= TOL["bf16"]


def test_state_chain():
    """S_N of one forward is the next forward's S_0 and the backward's dL/dS_N,
    all launched back to back."""
    B, H, N, D, M = 4, 8, 1000, 64, 64
    dt = torch.bfloat16
    q, k, v, g = (t.to(DEV) for t in make_inputs(B, H, N, D, M, dt, seed=7))
    ws_f, ws_b = _ws(B, H, N, D, M, dt, False), _ws(B, H, N, D, M, dt, True)
    s0 = torch.randn((B, H, D, M), generator=torch.Generator().manual_seed(8)).to(DEV)
    s1, s2 = torch.empty_like(s0), torch.empty_like(s0)
    ds0 = torch.empty_like(s0)
    out1, out2 = torch.empty_like(v), torch.empty_like(v)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    cp.causal_product_fwd(q, k, v, out=out1, workspace=ws_f, state_in=s0, return_state=True,
                          state_out=s1)
    cp.causal_product_fwd(q, k, v, out=out2, workspace=ws_f, state_in=s1, return_state=True,
                          state_out=s2)
    cp.causal_product_bwd(q, k, v, g, dq, dk, dv, workspace=ws_b, state_in=s1,
                          grad_state_out=s2, return_state_grad=True, grad_state_in=ds0)
    torch.cuda.synchronize()
    qn, kn, vn, gn = to_np(q), to_np(k), to_np(v), to_np(g)
    r1, r_s1 = oracle.fwd_state(qn, kn, vn, state_in=s0.cpu().numpy())
    assert row_rel_err(to_np(out1), r1) <= TOL["bf16"]
    assert row_rel_err(to_np(s1), r_s1) <= 1e-4
    r2, r_s2 = oracle.fwd_state(qn, kn, vn, state_in=to_np(s1))
    assert row_rel_err(to_np(out2), r2) <= TOL["bf16"]
    assert row_rel_err(to_np(s2), r_s2) <= 1e-4
    rb = oracle.bwd_state(qn, kn, vn, gn, state_in=to_np(s1), grad_state_out=to_np(s2))
    for got, ref in zip((dq, dk, dv), rb[:3]):
        assert row_rel_err(to_np(got), ref) <= TOL["bf16"]
    assert row_rel_err(to_np(ds0), rb[3]) <= 1e-4


def test_feature_chain():
    """Feature-map forward, then the feature backward fed with the forward's
    own output as grad_out, back to back."""
    B, H, N, D, M = 2, 4, 800, 64, 64
    dt = torch.bfloat16
    x_q, x_k, v, _ = (t.to(DEV) if t is not None else None
                      for t in make_inputs(B, H, N, D, M, dt, seed=9, feature="normal",
                                           backward=False))
    ws_f = torch.zeros(cp.load_library().causal_product_feature_workspace_size(B, H, N, D, M, 1, 0),
                       dtype=torch.uint8, device=DEV)
    ws_b = torch.zeros(cp.load_library().causal_product_feature_workspace_size(B, H, N, D, M, 1, 1),
                       dtype=torch.uint8, device=DEV)
    out = cp.causal_product_fwd_feature(x_q, x_k, v, "elu1", workspace=ws_f)
    dq, dk, dv = cp.causal_product_bwd_feature(x_q, x_k, v, out, "elu1", workspace=ws_b)
    torch.cuda.synchronize()
    qn, kn, vn, on = to_np(x_q), to_np(x_k), to_np(v), to_np(out)
    assert row_rel_err(on, oracle.fwd_feature(qn, kn, vn)) <= TOL["bf16"]
    r = oracle.bwd_feature(qn, kn, vn, on)
    for got, ref in zip((dq, dk, dv), r):
        assert row_rel_err(to_np(got), ref) <= TOL["bf16"]
