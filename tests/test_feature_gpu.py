"""Feature map fused into the product on the GPU (``-m gpu``): the causal
product of phi(q), phi(k) and v with phi(x) = elu(x) + 1 applied inside the
kernels, and its backward with respect to the raw q, k, v, against the fp64
oracle (which maps the raw inputs in double)."""
import numpy as np
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DT = {"f32": torch.float32, "bf16": torch.bfloat16}

# (B, H, N, D, M, dtype): unsplit and segmented scans (the aggregate pass
# maps K too), every tile geometry of the tensor-core path, ragged tails
FWD_SHAPES = [
    (8, 16, 4096, 64, 64, "bf16"),
    (2, 4, 1000, 64, 64, "bf16"),
    (1, 2, 8229, 128, 128, "bf16"),
    (1, 2, 700, 256, 64, "bf16"),
    (2, 2, 300, 192, 64, "bf16"),
    (3, 5, 129, 64, 128, "bf16"),
    (2, 3, 500, 48, 64, "bf16"),      # D below the 64-column box: padded columns
    (1, 2, 333, 96, 64, "bf16"),
    (2, 3, 200, 16, 16, "f32"),
    (1, 2, 513, 36, 20, "f32"),
]
BWD_SHAPES = [
    (2, 4, 1000, 64, 64, "bf16"),
    (8, 16, 1024, 64, 64, "bf16"),
    (1, 2, 777, 128, 128, "bf16"),
    (2, 2, 400, 40, 64, "bf16"),
    (2, 3, 200, 16, 16, "f32"),
]


def _raw(shape, seed, backward):
    B, H, N, D, M, dt = shape
    # raw (pre-feature) inputs: standard normal, both signs, so both branches
    # of phi are taken
    return make_inputs(B, H, N, D, M, DT[dt], seed=seed, feature="normal", backward=backward)


@pytest.mark.parametrize("shape", FWD_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_feature_forward_against_oracle(shape):
    q, k, v, _ = _raw(shape, seed=sum(shape[:5]), backward=False)
    out = cp.causal_product_fwd_feature(q.to(DEV), k.to(DEV), v.to(DEV), "elu1")
    torch.cuda.synchronize()
    ref = oracle.fwd_feature(to_np(q), to_np(k), to_np(v), "elu1")
    assert row_rel_err(to_np(out), ref) <= TOL[shape[5]]


@pytest.mark.parametrize("shape", BWD_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_feature_backward_against_oracle(shape):
    q, k, v, g = _raw(shape, seed=sum(shape[:5]) + 7, backward=True)
    dq, dk, dv = cp.causal_product_bwd_feature(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), "elu1")
    torch.cuda.synchronize()
    r = oracle.bwd_feature(to_np(q), to_np(k), to_np(v), to_np(g), "elu1")
    for got, ref in zip((dq, dk, dv), r):
        assert row_rel_err(to_np(got), ref) <= TOL[shape[5]]


def test_feature_none_is_the_plain_product():
    q, k, v = (t.to(DEV) for t in _raw((2, 4, 600, 64, 64, "bf16"), 3, False)[:3])
    a = cp.causal_product_fwd_feature(q, k, v, "none")
    b = cp.causal_product_fwd(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_feature_autograd(dt):
    q, k, v, g = _raw((2, 4, 300, 32 if dt == "f32" else 64, 32 if dt == "f32" else 64, dt), 11,
                      True)
    qd, kd, vd = (t.to(DEV).requires_grad_() for t in (q, k, v))
    out = cp.causal_product(qd, kd, vd, feature="elu1")
    out.backward(g.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.fwd_feature(to_np(q), to_np(k), to_np(v))
    r = oracle.bwd_feature(to_np(q), to_np(k), to_np(v), to_np(g))
    assert row_rel_err(to_np(out), ref) <= TOL[dt]
    for t, rr in zip((qd, kd, vd), r):
        assert row_rel_err(to_np(t.grad), rr) <= TOL[dt]


def test_feature_matches_mapped_inputs():
    """The fused map equals mapping the inputs first (phi rounded to bf16
    once, as the fused kernels do) up to the rounding of e^x."""
    q, k, v, _ = _raw((2, 4, 1000, 64, 64, "bf16"), 5, False)
    phi = lambda x: torch.where(x > 0, x + 1, torch.exp(x)).to(torch.bfloat16)
    fused = cp.causal_product_fwd_feature(q.to(DEV), k.to(DEV), v.to(DEV), "elu1")
    mapped = cp.causal_product_fwd(phi(q.float()).to(DEV), phi(k.float()).to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    assert row_rel_err(to_np(fused), to_np(mapped)) <= 1e-2
