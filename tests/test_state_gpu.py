"""Carried state on the GPU (``-m gpu``): the scan started from S_0 with the
final state S_N handed on, and its backward with dL/dS_N in and dL/dS_0
out, against the fp64 oracle; chunked runs against whole-sequence runs."""
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
# states are fp32 sums of exact products: far tighter than the outputs
STATE_TOL = {"f32": 1e-5, "bf16": 1e-4}

SHAPES = [
    # (B, H, N, D, M, dtype): fused and unfused backward, one segment and
    # several, D != M, value-column blocks, ragged tails
    (2, 3, 1000, 64, 64, "bf16"),
    (8, 16, 640, 64, 64, "bf16"),
    (1, 2, 5000, 64, 64, "bf16"),
    (2, 2, 300, 64, 128, "bf16"),
    (1, 2, 260, 256, 64, "bf16"),
    (2, 1, 777, 32, 48, "bf16"),
    (1, 2, 500, 64, 64, "f32"),
    (2, 1, 99, 80, 24, "f32"),
]


def _states(B, H, D, M, seed):
    g = torch.Generator().manual_seed(seed)
    s0 = torch.randn((B, H, D, M), generator=g) * 4
    ds = torch.randn((B, H, D, M), generator=g)
    return s0, ds


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_state_fwd_bwd_against_oracle(shape):
    B, H, N, D, M, dt = shape
    q, k, v, g = make_inputs(B, H, N, D, M, DT[dt], seed=N + D + M)
    s0, ds = _states(B, H, D, M, seed=N)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    out, s_n = cp.causal_product_fwd(qd, kd, vd, state_in=s0.to(DEV), return_state=True)
    dq, dk, dv, ds0 = cp.causal_product_bwd(qd, kd, vd, gd, state_in=s0.to(DEV),
                                            grad_state_out=ds.to(DEV), return_state_grad=True)
    torch.cuda.synchronize()
    r_out, r_sn = oracle.fwd_state(to_np(q), to_np(k), to_np(v), state_in=s0.numpy())
    r_dq, r_dk, r_dv, r_ds0 = oracle.bwd_state(to_np(q), to_np(k), to_np(v), to_np(g),
                                               state_in=s0.numpy(), grad_state_out=ds.numpy())
    for name, got, ref, tol in (("out", out, r_out, TOL[dt]), ("dq", dq, r_dq, TOL[dt]),
                                ("dk", dk, r_dk, TOL[dt]), ("dv", dv, r_dv, TOL[dt]),
                                ("S_N", s_n, r_sn, STATE_TOL[dt]),
                                ("dS_0", ds0, r_ds0, STATE_TOL[dt])):
        err = row_rel_err(to_np(got), ref)
        assert np.isfinite(err) and err <= tol, f"{name} row-rel err {err:.3e} > {tol}"


def test_state_chunking_is_exact_on_tile_boundaries():
    """One segment per problem (B*H = 128) and a split on a 128-row tile
    boundary: handing the fp32 state across the split reproduces the whole
    sequence bit for bit, forward and backward."""
    B, H, N, D, M, cut = 8, 16, 1024, 64, 64, 512
    q, k, v, g = (t.to(DEV) for t in make_inputs(B, H, N, D, M, torch.bfloat16, seed=21))
    s0, ds = (t.to(DEV) for t in _states(B, H, D, M, seed=22))
    part = lambda t, a, b: t[:, :, a:b].contiguous()
    out, s_n = cp.causal_product_fwd(q, k, v, state_in=s0, return_state=True)
    o1, s1 = cp.causal_product_fwd(part(q, 0, cut), part(k, 0, cut), part(v, 0, cut),
                                   state_in=s0, return_state=True)
    o2, s2 = cp.causal_product_fwd(part(q, cut, N), part(k, cut, N), part(v, cut, N),
                                   state_in=s1, return_state=True)
    assert torch.equal(torch.cat([o1, o2], dim=2), out)
    assert torch.equal(s2, s_n)
    full = cp.causal_product_bwd(q, k, v, g, state_in=s0, grad_state_out=ds,
                                 return_state_grad=True)
    dq2, dk2, dv2, ds_mid = cp.causal_product_bwd(
        part(q, cut, N), part(k, cut, N), part(v, cut, N), part(g, cut, N), state_in=s1,
        grad_state_out=ds, return_state_grad=True)
    dq1, dk1, dv1, ds0 = cp.causal_product_bwd(
        part(q, 0, cut), part(k, 0, cut), part(v, 0, cut), part(g, 0, cut), state_in=s0,
        grad_state_out=ds_mid, return_state_grad=True)
    for a, b, ref in ((dq1, dq2, full[0]), (dk1, dk2, full[1]), (dv1, dv2, full[2])):
        assert torch.equal(torch.cat([a, b], dim=2), ref)
    assert torch.equal(ds0, full[3])


def test_state_zero_rows_passes_state_through():
    B, H, D, M = 2, 3, 64, 64
    e = torch.empty((B, H, 0, D), dtype=torch.bfloat16, device=DEV)
    ev = torch.empty((B, H, 0, M), dtype=torch.bfloat16, device=DEV)
    s0, ds = (t.to(DEV) for t in _states(B, H, D, M, seed=23))
    _, s_n = cp.causal_product_fwd(e, e, ev, state_in=s0, return_state=True)
    _, _, _, ds0 = cp.causal_product_bwd(e, e, ev, ev, state_in=s0, grad_state_out=ds,
                                         return_state_grad=True)
    _, s_zero = cp.causal_product_fwd(e, e, ev, return_state=True)
    torch.cuda.synchronize()
    assert torch.equal(s_n, s0) and torch.equal(ds0, ds)
    assert torch.count_nonzero(s_zero).item() == 0


def test_state_autograd_matches_oracle():
    B, H, N, D, M = 1, 2, 300, 64, 64
    q, k, v, g = make_inputs(B, H, N, D, M, torch.bfloat16, seed=24)
    s0, ds = _states(B, H, D, M, seed=25)
    qd, kd, vd = (t.to(DEV).requires_grad_(True) for t in (q, k, v))
    sd = s0.to(DEV).requires_grad_(True)
    out, s_n = cp.causal_product(qd, kd, vd, state=sd, return_state=True)
    loss = (out.float() * g.to(DEV).float()).sum() + (s_n * ds.to(DEV)).sum()
    loss.backward()
    r = oracle.bwd_state(to_np(q), to_np(k), to_np(v), to_np(g), state_in=s0.numpy(),
                         grad_state_out=ds.numpy())
    for got, ref, tol in ((qd.grad, r[0], TOL["bf16"]), (kd.grad, r[1], TOL["bf16"]),
                          (vd.grad, r[2], TOL["bf16"]), (sd.grad, r[3], STATE_TOL["bf16"])):
        assert row_rel_err(to_np(got), ref) <= tol
