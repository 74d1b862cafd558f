"""The forward product and its normaliser in one call (``-m gpu``).

causal_product_fwd_norm returns out = causal product and z_i = q_i .
sum_{j<=i} k_j.  On bf16 with D, M <= 64 and unsplit problems z comes out of
the product kernel itself (one launch); elsewhere the call runs the product,
then the normaliser kernel.  Both results are compared with the fp64 oracle
(out row-normalised; z against the scale q . sum |k|, as the normaliser
tests do), and out with causal_product_fwd bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
Z_TOL = 1e-4


def _z_err(got, q, k):
    nq, nk = to_np(q), to_np(k)
    ref = oracle.norm(nq, nk)
    scale = oracle.norm(np.abs(nq), np.abs(nk))
    return float(np.max(np.abs(got - ref) / np.maximum(scale, 1e-30))) if ref.size else 0.0


# (B, H, N, D, M, dtype, fused)
SHAPES = [
    (3, 40, 1000, 64, 64, torch.bfloat16, True),    # ragged tail, 120 problems
    (4, 30, 700, 32, 48, torch.bfloat16, True),     # padded widths
    (1, 120, 1, 64, 64, torch.bfloat16, True),      # a single row
    (1, 128, 129, 16, 64, torch.bfloat16, True),    # two tiles, the second of one row
    (2, 100, 300, 64, 8, torch.bfloat16, True),     # more problems than SMs
    (1, 2, 5000, 64, 64, torch.bfloat16, False),    # split into segments: product + normaliser
    (1, 4, 700, 128, 128, torch.bfloat16, False),   # wide tiles
    (2, 3, 500, 64, 64, torch.float32, False),      # fp32
    (2, 3, 300, 40, 24, torch.float16, False),      # fp16
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s[:5])) + f"_{s[5]}")
def test_fwd_norm_matches_oracle(shape):
    B, H, N, D, M, dt, fused = shape
    q, k, v, _ = make_inputs(B, H, N, D, M, dt, seed=B * H + N + D + M, backward=False)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    assert (cp.causal_product_launch_count(B, H, N, D, M, dt, norm=True) == 1) == fused
    out, z = cp.causal_product_fwd_norm(qd, kd, vd)
    plain = cp.causal_product_fwd(qd, kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(out, plain)
    tol = {torch.bfloat16: TOL["bf16"], torch.float32: TOL["f32"], torch.float16: TOL["f16"]}[dt]
    assert row_rel_err(to_np(out), oracle.fwd(to_np(q), to_np(k), to_np(v))) <= tol
    assert _z_err(to_np(z), q, k) <= Z_TOL


def test_fwd_norm_full_size_and_deterministic():
    """B=8 H=16 N=4096 D=M=64 bf16: one launch; repeated calls give the same
    bits; z agrees with the separate normaliser kernel to fp32 rounding."""
    B, H, N, D, M = 8, 16, 4096, 64, 64
    q, k, v, _ = make_inputs(B, H, N, D, M, torch.bfloat16, seed=3, backward=False)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    assert cp.causal_product_launch_count(B, H, N, D, M, norm=True) == 1
    out, z = cp.causal_product_fwd_norm(qd, kd, vd)
    out, z = out.clone(), z.clone()
    for _ in range(2):
        o2, z2 = cp.causal_product_fwd_norm(qd, kd, vd)
        assert torch.equal(out, o2) and torch.equal(z, z2)
    zsep = cp.causal_product_normalizer(qd, kd)
    torch.cuda.synchronize()
    assert torch.equal(out, cp.causal_product_fwd(qd, kd, vd))
    assert _z_err(to_np(z), q, k) <= Z_TOL
    nq, nk = to_np(q), to_np(k)
    scale = oracle.norm(np.abs(nq), np.abs(nk))
    assert float(np.max(np.abs(to_np(z) - to_np(zsep)) / np.maximum(scale, 1e-30))) <= 1e-5


def test_fwd_norm_rejects():
    B, H, N, D, M = 1, 2, 64, 64, 64
    q = torch.zeros((B, H, N, D), dtype=torch.bfloat16, device=DEV)
    v = torch.zeros((B, H, N, M), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        cp.causal_product_fwd_norm(q, q, v, z=torch.empty((B, H, N + 1), device=DEV))
    with pytest.raises(ValueError):
        cp.causal_product_fwd_norm(q, q, v, z=torch.empty((B, H, N), dtype=torch.float16,
                                                          device=DEV))
