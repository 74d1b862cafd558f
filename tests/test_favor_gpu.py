"""Positive random features (FAVOR+) computed in the kernels (``-m gpu``).

causal_product_fwd_favor / _bwd_favor take the raw rows xq, xk and the
projection W and compute phi(x) = exp(W x - |x|^2 / 2) / sqrt(D) on the GPU.
Their results are compared element by element (row-normalised error) with
the oracle's fp64 fwd_favor / bwd_favor on the same bf16 values, up to the
full size of the D = 256 workload (B=4 H=8 N=8229 D=256 M=64, r = 64).
"""
import numpy as np
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import favor_raw_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def favor_inputs(B, H, N, R, D, M, seed):
    """bf16 xq, xk [B,H,N,R], v, g [B,H,N,M] and W [D,R] (the workload's draw
    with r = 64, cut to R input features)."""
    W, xq, xk = favor_raw_inputs(B, H, N, D, seed)
    W, xq, xk = W[:, :R].contiguous(), xq[..., :R].contiguous(), xk[..., :R].contiguous()
    gen = torch.Generator().manual_seed(seed + 1)
    v = torch.randn((B, H, N, M), generator=gen)
    g = torch.randn((B, H, N, M), generator=gen)
    bf = lambda t: t.to(torch.bfloat16)
    return bf(xq), bf(xk), bf(v), bf(g), bf(W)


def check(B, H, N, R, D, M, seed, backward=True):
    xq, xk, v, g, W = favor_inputs(B, H, N, R, D, M, seed)
    d = [t.to(DEV) for t in (xq, xk, v, g, W)]
    out = cp.causal_product_fwd_favor(d[0], d[1], d[2], d[4])
    torch.cuda.synchronize()
    nx = [to_np(t) for t in (xq, xk, v, g, W)]
    ref = oracle.fwd_favor(nx[0], nx[1], nx[2], nx[4])
    errs = {"out": row_rel_err(to_np(out), ref)}
    if backward:
        dxq, dxk, dv = cp.causal_product_bwd_favor(d[0], d[1], d[2], d[4], d[3])
        torch.cuda.synchronize()
        rq, rk, rv = oracle.bwd_favor(nx[0], nx[1], nx[2], nx[4], nx[3])
        errs.update(dxq=row_rel_err(to_np(dxq), rq), dxk=row_rel_err(to_np(dxk), rk),
                    dv=row_rel_err(to_np(dv), rv))
    for name, e in errs.items():
        assert np.isfinite(e) and e <= TOL["bf16"], f"{name}: row-rel err {e:.3e}"
    return errs


@pytest.mark.parametrize("shape", [
    (1, 2, 300, 64, 256, 64),    # the workload's widths, three tiles with a ragged tail
    (1, 3, 1000, 32, 128, 64),   # fewer input features (zero-padded to 64)
    (2, 2, 129, 64, 64, 32),     # D = 64, a one-row second tile
    (1, 2, 200, 16, 192, 128),   # D = 192, two value blocks
    (1, 1, 1, 8, 64, 8),         # one row
], ids=lambda s: "x".join(map(str, s)))
def test_favor_matches_oracle(shape):
    check(*shape, seed=sum(shape))


def test_favor_workload_full_size():
    """The D = 256 workload at full size, forward and backward."""
    check(4, 8, 8229, 64, 256, 64, seed=5)


def test_favor_autograd_and_rejects():
    xq, xk, v, g, W = (t.to(DEV) for t in favor_inputs(1, 2, 260, 64, 128, 64, 7))
    a = [t.clone().requires_grad_(True) for t in (xq, xk, v)]
    out = cp.causal_product_favor(a[0], a[1], a[2], W)
    out.backward(g)
    dxq, dxk, dv = cp.causal_product_bwd_favor(xq, xk, v, W, g)
    torch.cuda.synchronize()
    for got, want in zip((a[0].grad, a[1].grad, a[2].grad), (dxq, dxk, dv)):
        assert torch.equal(got, want)
    with pytest.raises(cp.CausalProductError):
        cp.causal_product_fwd_favor(xq.float(), xk.float(), v.float(), W.float())
