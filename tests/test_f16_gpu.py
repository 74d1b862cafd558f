"""fp16 inputs on the GPU (``-m gpu``): every entry point with fp16 tensors
against the fp64 oracle.  fp16 values are exact in fp32, so the oracle reads
the values the GPU receives; the GPU widens them to fp32, computes in fp32
and rounds the outputs to fp16 once (bound 2e-3, parity_util)."""
import numpy as np
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import make_inputs, make_norm_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
F16 = torch.float16
T = TOL["f16"]


def _inputs(B, H, N, D, M, seed, backward=True, feature="elu"):
    return make_inputs(B, H, N, D, M, F16, seed=seed, feature=feature, backward=backward)


@pytest.mark.parametrize("shape", [(2, 3, 300, 64, 64), (1, 2, 1000, 48, 20),
                                   (8, 16, 1024, 64, 64), (1, 1, 70, 7, 5)],
                         ids=lambda s: "x".join(map(str, s)))
def test_f16_forward_and_backward(shape):
    B, H, N, D, M = shape
    q, k, v, g = _inputs(B, H, N, D, M, seed=N + D)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    out = cp.causal_product_fwd(qd, kd, vd)
    dq, dk, dv = cp.causal_product_bwd(qd, kd, vd, gd)
    torch.cuda.synchronize()
    assert out.dtype == F16 and dq.dtype == F16
    assert row_rel_err(to_np(out), oracle.fwd(to_np(q), to_np(k), to_np(v))) <= T
    ref = oracle.bwd(to_np(q), to_np(k), to_np(v), to_np(g))
    for got, r in zip((dq, dk, dv), ref):
        assert row_rel_err(to_np(got), r) <= T


def test_f16_carried_state():
    B, H, N, D, M = 1, 2, 300, 32, 24
    q, k, v, g = _inputs(B, H, N, D, M, seed=5)
    gen = torch.Generator().manual_seed(6)
    s0 = torch.randn((B, H, D, M), generator=gen)
    ds_n = torch.randn((B, H, D, M), generator=gen)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    out, s_n = cp.causal_product_fwd(qd, kd, vd, state_in=s0.to(DEV), return_state=True)
    dq, dk, dv, ds0 = cp.causal_product_bwd(qd, kd, vd, gd, state_in=s0.to(DEV),
                                            grad_state_out=ds_n.to(DEV), return_state_grad=True)
    torch.cuda.synchronize()
    r_out, r_sn = oracle.fwd_state(to_np(q), to_np(k), to_np(v), state_in=s0.numpy())
    r = oracle.bwd_state(to_np(q), to_np(k), to_np(v), to_np(g), state_in=s0.numpy(),
                         grad_state_out=ds_n.numpy())
    assert row_rel_err(to_np(out), r_out) <= T
    assert row_rel_err(to_np(s_n), r_sn) <= 1e-5
    for got, rr in zip((dq, dk, dv), r[:3]):
        assert row_rel_err(to_np(got), rr) <= T
    assert row_rel_err(to_np(ds0), r[3]) <= 1e-5


@pytest.mark.parametrize("dm", [(64, 64), (24, 20)], ids=["v4", "scalar"])
def test_f16_decode(dm):
    D, M = dm
    B, H = 4, 4
    q, k, v, _ = _inputs(B, H, 1, D, M, seed=D, backward=False)
    s0 = torch.randn((B, H, D, M), generator=torch.Generator().manual_seed(7)) * 3
    state = s0.to(DEV)
    out = cp.causal_product_decode(q[:, :, 0].to(DEV), k[:, :, 0].to(DEV), v[:, :, 0].to(DEV),
                                   state)
    torch.cuda.synchronize()
    r_out, r_state = oracle.fwd_state(to_np(q), to_np(k), to_np(v), state_in=s0.numpy())
    assert row_rel_err(to_np(out), r_out[:, :, 0]) <= T
    assert row_rel_err(to_np(state), r_state) <= 1e-5


# dq_i = g_i sum_{j<=i} k_j grows with N: with these features it passes
# fp16's largest value (65504) near N = 10^4, so the long case stays below
@pytest.mark.parametrize("shape", [(2, 3, 1000, 64), (1, 1, 4000, 128)],
                         ids=lambda s: "x".join(map(str, s)))
def test_f16_normalizer(shape):
    B, H, N, D = shape
    q, k, gz = make_norm_inputs(B, H, N, D, F16, seed=N)
    z = cp.causal_product_normalizer(q.to(DEV), k.to(DEV))
    dq, dk = cp.causal_product_normalizer_bwd(q.to(DEV), k.to(DEV), gz.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.norm(to_np(q), to_np(k))
    scale = oracle.norm(np.abs(to_np(q)), np.abs(to_np(k)))
    assert float(np.max(np.abs(to_np(z) - ref) / scale)) <= 1e-4
    r_dq, r_dk = oracle.norm_bwd(to_np(q), to_np(k), gz.numpy())
    assert row_rel_err(to_np(dq), r_dq) <= T
    assert row_rel_err(to_np(dk), r_dk) <= T


def test_f16_feature_map():
    B, H, N, D, M = 2, 3, 300, 64, 64
    q, k, v, g = _inputs(B, H, N, D, M, seed=17, feature="normal")
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    out = cp.causal_product_fwd_feature(qd, kd, vd, "elu1")
    dq, dk, dv = cp.causal_product_bwd_feature(qd, kd, vd, gd, "elu1")
    torch.cuda.synchronize()
    assert row_rel_err(to_np(out), oracle.fwd_feature(to_np(q), to_np(k), to_np(v))) <= T
    ref = oracle.bwd_feature(to_np(q), to_np(k), to_np(v), to_np(g))
    for got, r in zip((dq, dk, dv), ref):
        assert row_rel_err(to_np(got), r) <= T


def test_f16_autograd():
    B, H, N, D, M = 2, 2, 200, 32, 32
    q, k, v, g = _inputs(B, H, N, D, M, seed=23)
    qd, kd, vd = (t.to(DEV).requires_grad_() for t in (q, k, v))
    out = cp.causal_product(qd, kd, vd)
    out.backward(g.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.bwd(to_np(q), to_np(k), to_np(v), to_np(g))
    for t, r in zip((qd, kd, vd), ref):
        assert row_rel_err(to_np(t.grad), r) <= T
