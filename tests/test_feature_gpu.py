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
# bf16 maps phi on the loaded tiles and applies phi' to the stored gradients.
# D, M <= 64: the fused dk/dv scan and the dq scan, in one launch on unsplit
# problems fewer than the SMs, else as a dq product and a dk/dv launch (more
# problems than SMs; segmented scans, whose aggregate passes map their
# tiles).  Wider: three products, every tile geometry of dq/dk (D' = M,
# M' = D) and dv (D' = D, M' = M), value blocks (D = 256).  Padded widths on
# either side, ragged tails.
BWD_SHAPES = [
    (2, 4, 1000, 64, 64, "bf16"),
    (8, 16, 1024, 64, 64, "bf16"),
    (16, 16, 300, 64, 64, "bf16"),
    (1, 2, 777, 128, 128, "bf16"),
    (2, 2, 400, 40, 64, "bf16"),
    (2, 3, 300, 64, 24, "bf16"),
    (1, 2, 700, 256, 64, "bf16"),
    (2, 2, 300, 192, 64, "bf16"),
    (3, 5, 129, 64, 128, "bf16"),
    (1, 2, 5000, 64, 64, "bf16"),
    (1, 2, 8229, 128, 128, "bf16"),
    (1, 3, 1, 64, 64, "bf16"),
    (2, 3, 200, 16, 16, "f32"),
    (1, 2, 300, 40, 24, "f16"),
]
DT["f16"] = torch.float16


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


def test_feature_backward_bf16_workspace_holds_no_features():
    """bf16 maps inside the kernels: the feature backward needs no more
    workspace than the plain backward, and runs in a caller's workspace of
    exactly that size."""
    B, H, N, D, M = 2, 4, 1000, 64, 64
    plain = cp.causal_product_workspace_size(B, H, N, D, M, torch.bfloat16, backward=True)
    feat = cp.causal_product_feature_workspace_size(B, H, N, D, M, torch.bfloat16, backward=True)
    assert feat == plain
    q, k, v, g = _raw((B, H, N, D, M, "bf16"), 9, True)
    ws = torch.zeros(feat, dtype=torch.uint8, device=DEV)
    dq, dk, dv = cp.causal_product_bwd_feature(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV), "elu1",
                                               workspace=ws)
    dq2, dk2, dv2 = cp.causal_product_bwd_feature(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV),
                                                  "elu1")
    torch.cuda.synchronize()
    assert cp.causal_product_status(ws) == 0
    for a, b in ((dq, dq2), (dk, dk2), (dv, dv2)):
        assert torch.equal(a, b)


def test_feature_backward_bf16_matches_mapped_inputs():
    """The fused bf16 backward agrees with the plain backward on phi(q),
    phi(k) (phi rounded to bf16 once, as the kernels do) followed by the
    chain rule in fp32, within the bf16 tolerance: the two differ by the
    fused path's bf16 phi' (e^min(x, 0) from a bf16 exponent) and product,
    the composed path's bf16 rounding of the unscaled gradients, and the
    plain backward's own order of summation (its one-launch dk/dv scan)."""
    q, k, v, g = _raw((2, 4, 1000, 64, 64, "bf16"), 13, True)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    phi = lambda x: torch.where(x > 0, x + 1, torch.exp(x)).to(torch.bfloat16)
    dphi = lambda x: torch.where(x > 0, torch.ones_like(x), torch.exp(x))
    dq, dk, dv = cp.causal_product_bwd_feature(qd, kd, vd, gd, "elu1")
    fq, fk, fv = cp.causal_product_bwd(phi(qd.float()), phi(kd.float()), vd, gd)
    torch.cuda.synchronize()
    assert row_rel_err(to_np(dv), to_np(fv)) <= 1e-2
    for got, mapped, x in ((dq, fq, q), (dk, fk, k)):
        ref = (mapped.float() * dphi(x.to(DEV).float())).cpu().numpy()
        assert row_rel_err(to_np(got), ref) <= TOL["bf16"]
