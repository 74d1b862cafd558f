"""Normaliser of causal linear attention on the GPU (``-m gpu``):
z_i = q_i . sum_{j<=i} k_j and its backward, against the fp64 oracle.

z is fp32 for both input dtypes and its arithmetic is fp32 on exact
inputs, so its bound is 1e-4 relative to the sum of absolute terms
(the oracle's normaliser of |q| and |k|: the scale fp32 summation error is
proportional to).  dq and dk are written in the input dtype and take the
causal product's row-relative bounds.
"""
import numpy as np
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import make_norm_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
Z_TOL = 1e-4

# (B, H, N, D, dtype, feature): segmented and unsplit problems, every lane
# layout (D/8 lanes per row for bf16; 16-byte or scalar f32 rows), ragged
# tails, one tile, many segments of one tile
SHAPES = [
    (2, 3, 1000, 64, "bf16", "elu"),
    (8, 16, 4096, 64, "bf16", "elu"),
    (1, 1, 65536, 64, "bf16", "elu"),
    (2, 2, 8229, 256, "bf16", "favor"),
    (1, 2, 300, 256, "bf16", "normal"),
    (2, 2, 77, 8, "bf16", "elu"),
    (1, 1, 5000, 48, "bf16", "elu"),
    (2, 3, 1000, 64, "f32", "elu"),
    (1, 2, 513, 36, "f32", "normal"),
    (1, 2, 700, 200, "f32", "elu"),
    (3, 1, 2000, 130, "f32", "elu"),
    (1, 2, 900, 256, "f32", "elu"),
    (1, 1, 333, 7, "f32", "elu"),
    (1, 1, 1, 1, "f32", "elu"),
    # D = 64 with at least half as many problems as SMs: one CTA per problem
    (8, 16, 1000, 64, "f32", "elu"),
    (4, 20, 129, 64, "bf16", "normal"),
    (4, 19, 77, 64, "bf16", "elu"),
    (4, 20, 300, 64, "f16", "elu"),
]


def _inputs(shape, seed):
    B, H, N, D, dt, feature = shape
    q, k, gz = make_norm_inputs(B, H, N, D, DT[dt], seed=seed, feature=feature)
    return q, k, gz


def _z_err(got, q, k):
    ref = oracle.norm(to_np(q), to_np(k))
    scale = oracle.norm(np.abs(to_np(q)), np.abs(to_np(k)))
    return float(np.max(np.abs(got - ref) / np.maximum(scale, 1e-30))) if ref.size else 0.0


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_normalizer_forward_against_oracle(shape):
    q, k, _ = _inputs(shape, seed=sum(shape[:4]))
    z = cp.causal_product_normalizer(q.to(DEV), k.to(DEV))
    torch.cuda.synchronize()
    assert _z_err(to_np(z), q, k) <= Z_TOL


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_normalizer_backward_against_oracle(shape):
    dt = shape[4]
    q, k, gz = _inputs(shape, seed=sum(shape[:4]) + 1)
    dq, dk = cp.causal_product_normalizer_bwd(q.to(DEV), k.to(DEV), gz.to(DEV))
    torch.cuda.synchronize()
    r_dq, r_dk = oracle.norm_bwd(to_np(q), to_np(k), gz.numpy())
    assert dq.dtype == q.dtype and dk.dtype == q.dtype
    assert row_rel_err(to_np(dq), r_dq) <= TOL[dt]
    assert row_rel_err(to_np(dk), r_dk) <= TOL[dt]


@pytest.mark.parametrize("shape", [(2, 2, 20000, 64, "bf16", "elu"),
                                   (8, 16, 2000, 64, "bf16", "elu")],
                         ids=lambda s: "x".join(map(str, s)))
def test_normalizer_is_bitwise_reproducible(shape):
    q, k, gz = (t.to(DEV) for t in _inputs(shape, seed=5))
    z1 = cp.causal_product_normalizer(q, k)
    z2 = cp.causal_product_normalizer(q, k)
    a = cp.causal_product_normalizer_bwd(q, k, gz)
    b = cp.causal_product_normalizer_bwd(q, k, gz)
    torch.cuda.synchronize()
    assert torch.equal(z1, z2) and torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_normalizer_empty_sequence():
    q = torch.empty((2, 3, 0, 64), dtype=torch.bfloat16, device=DEV)
    z = cp.causal_product_normalizer(q, q.clone())
    dq, dk = cp.causal_product_normalizer_bwd(q, q.clone(),
                                              torch.empty((2, 3, 0), device=DEV))
    torch.cuda.synchronize()
    assert z.shape == (2, 3, 0) and dq.shape == q.shape and dk.shape == q.shape


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_normalizer_autograd(dt):
    q, k, gz = _inputs((2, 4, 600, 64, dt, "elu"), seed=9)
    qd = q.to(DEV).requires_grad_()
    kd = k.to(DEV).requires_grad_()
    z = cp.normalizer(qd, kd)
    z.backward(gz.to(DEV))
    torch.cuda.synchronize()
    r_dq, r_dk = oracle.norm_bwd(to_np(q), to_np(k), gz.numpy())
    assert _z_err(to_np(z), q, k) <= Z_TOL
    assert row_rel_err(to_np(qd.grad), r_dq) <= TOL[dt]
    assert row_rel_err(to_np(kd.grad), r_dk) <= TOL[dt]


def test_normalised_attention_composes():
    """Causal linear attention as "Transformers are RNNs" writes it, the
    causal product divided by the normaliser, from the two entry points."""
    B, H, N, D, M = 2, 4, 700, 64, 64
    from prefix_sum_outer_gb300.workloads import make_inputs
    q, k, v, _ = make_inputs(B, H, N, D, M, torch.bfloat16, seed=13, backward=False)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    att = cp.causal_product_fwd(qd, kd, vd).float() / cp.causal_product_normalizer(qd, kd)[..., None]
    torch.cuda.synchronize()
    ref = oracle.fwd(to_np(q), to_np(k), to_np(v)) / oracle.norm(to_np(q), to_np(k))[..., None]
    assert row_rel_err(to_np(att), ref) <= TOL["bf16"]


# ---- the normaliser of mapped features from raw inputs (phi = elu + 1 in the
# kernel); phi > 0, so z itself is the scale of its summation error
FEAT_SHAPES = [
    (2, 3, 1000, 64, "bf16"),
    (8, 16, 1000, 64, "bf16"),
    (4, 19, 77, 64, "f32"),
    (4, 20, 300, 64, "f16"),
    (1, 1, 20000, 128, "bf16"),
    (2, 2, 300, 256, "f32"),
    (2, 3, 500, 36, "f32"),
]


@pytest.mark.parametrize("shape", FEAT_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_normalizer_feature_against_oracle(shape):
    B, H, N, D, dt = shape
    q, k, gz = make_norm_inputs(B, H, N, D, DT[dt], seed=N + D, feature="normal")
    z = cp.causal_product_normalizer(q.to(DEV), k.to(DEV), feature="elu1")
    dq, dk = cp.causal_product_normalizer_bwd(q.to(DEV), k.to(DEV), gz.to(DEV), feature="elu1")
    torch.cuda.synchronize()
    ref = oracle.norm_feature(to_np(q), to_np(k))
    assert float(np.max(np.abs(to_np(z) - ref) / ref)) <= Z_TOL
    r_dq, r_dk = oracle.norm_bwd_feature(to_np(q), to_np(k), gz.numpy())
    assert row_rel_err(to_np(dq), r_dq) <= TOL[dt]
    assert row_rel_err(to_np(dk), r_dk) <= TOL[dt]


def test_normalised_attention_from_raw_inputs():
    """out / z with phi applied inside both the product and the normaliser."""
    B, H, N, D, M = 2, 4, 700, 64, 64
    from prefix_sum_outer_gb300.workloads import make_inputs
    x_q, x_k, v, _ = make_inputs(B, H, N, D, M, torch.bfloat16, seed=21, feature="normal",
                                 backward=False)
    xq, xk, vd = x_q.to(DEV), x_k.to(DEV), v.to(DEV)
    att = (cp.causal_product(xq, xk, vd, feature="elu1").float()
           / cp.normalizer(xq, xk, feature="elu1")[..., None])
    torch.cuda.synchronize()
    ref = (oracle.fwd_feature(to_np(x_q), to_np(x_k), to_np(v))
           / oracle.norm_feature(to_np(x_q), to_np(x_k))[..., None])
    assert row_rel_err(to_np(att), ref) <= TOL["bf16"]


def test_normalizer_feature_autograd():
    q, k, gz = make_norm_inputs(2, 2, 400, 64, torch.bfloat16, seed=4, feature="normal")
    qd, kd = q.to(DEV).requires_grad_(), k.to(DEV).requires_grad_()
    z = cp.normalizer(qd, kd, feature="elu1")
    z.backward(gz.to(DEV))
    torch.cuda.synchronize()
    r_dq, r_dk = oracle.norm_bwd_feature(to_np(q), to_np(k), gz.numpy())
    assert row_rel_err(to_np(qd.grad), r_dq) <= TOL["bf16"]
    assert row_rel_err(to_np(kd.grad), r_dk) <= TOL["bf16"]


def test_normalizer_feature_needs_16_byte_rows():
    q = torch.zeros((1, 1, 16, 7), device=DEV)
    with pytest.raises(cp.CausalProductError):
        cp.causal_product_normalizer(q, q.clone(), feature="elu1")
