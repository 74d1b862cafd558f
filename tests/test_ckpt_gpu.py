"""Forward checkpoints and the backward seeded from them (``-m gpu``).

causal_product_fwd_ckpt writes the state at fixed tile boundaries;
causal_product_bwd_ckpt starts every dq segment from one of them.  Every
call goes through the C ABI; results are compared with the fp64 oracle
element by element (row-normalised error), and the checkpoints themselves
with the oracle's state after the same rows.  Shapes whose backward does not
split dq use no checkpoints (size 0): the calls are then the plain ones, and
are checked all the same.
"""
import numpy as np
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def ckpt_bwd(q, k, v, g):
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    out, ckpt = cp.causal_product_fwd_ckpt(qd, kd, vd)
    dq, dk, dv = cp.causal_product_bwd_ckpt(qd, kd, vd, gd, ckpt)
    torch.cuda.synchronize()
    return out, ckpt, dq, dk, dv


def check(q, k, v, g, tol):
    out, _, dq, dk, dv = ckpt_bwd(q, k, v, g)
    nq, nk, nv, ng = (to_np(t) for t in (q, k, v, g))
    ref = oracle.fwd(nq, nk, nv)
    rq, rk, rv = oracle.bwd(nq, nk, nv, ng)
    errs = {"out": row_rel_err(to_np(out), ref), "dq": row_rel_err(to_np(dq), rq),
            "dk": row_rel_err(to_np(dk), rk), "dv": row_rel_err(to_np(dv), rv)}
    for name, e in errs.items():
        assert np.isfinite(e) and e <= tol, f"{name}: row-rel err {e:.3e} > {tol}"
    return errs


# shapes: (B, H, N, D, M); which backward each exercises is noted
SHAPES = [
    (8, 15, 1000, 64, 64),   # one-launch backward (no checkpoints), ragged tail
    (1, 120, 300, 64, 64),   # one-launch backward, 3 tiles
    (1, 151, 1100, 64, 64),  # one-launch backward, one spare SM
    (2, 57, 777, 48, 40),    # one-launch backward, padded widths
    (1, 130, 100, 64, 64),   # one-launch backward, one tile
    (1, 4, 3000, 64, 64),    # split fused backward: dq seeded, dk/dv two-pass
    (2, 3, 2000, 32, 48),    # padded widths, split
    (1, 2, 4100, 128, 64),   # general backward (D > 64), dq seeded
    (1, 3, 2500, 64, 192),   # dq with two value blocks of 128 (D' = 192 rows)
    (1, 2, 1500, 256, 64),   # D = 256: dq's value blocks of 128 columns
    (2, 2, 129, 64, 64),     # two tiles, the second of one row
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_ckpt_backward_matches_oracle(shape):
    B, H, N, D, M = shape
    q, k, v, g = make_inputs(B, H, N, D, M, torch.bfloat16, seed=sum(shape))
    check(q, k, v, g, TOL["bf16"])


@pytest.mark.parametrize("name", ["bf16_b8h16_n4096_d64", "bf16_long_n32768_d128",
                                  "bf16_favor_n8229_d256_m64"])
def test_ckpt_workloads_full_size(name):
    w = WORKLOADS[name]
    q, k, v, g = workload_inputs(w)
    check(q, k, v, g, TOL[w.dtype])


@pytest.mark.parametrize("shape", [(1, 3, 2500, 64, 192), (2, 4, 3000, 128, 128)],
                         ids=lambda s: "x".join(map(str, s)))
def test_ckpt_forward_is_the_forward_and_states_are_exact(shape):
    """The checkpoint forward's output is the plain forward's, bit for bit,
    and checkpoint s (fp32 [B, H, G - 1, D, M]) is the oracle's state before
    the first row of dq segment s.  On D = 64, M = 192 the dq segments are
    half the forward's, so most checkpoints come from inside a forward
    segment (written from the hi + lo state copy, 16 significant bits); on
    D = M = 128 they fall on forward segment ends (exact)."""
    B, H, N, D, M = shape
    q, k, v, g = make_inputs(B, H, N, D, M, torch.bfloat16, seed=5)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    out, ckpt = cp.causal_product_fwd_ckpt(qd, kd, vd)
    plain = cp.causal_product_fwd(qd, kd, vd)
    torch.cuda.synchronize()
    assert torch.equal(out, plain)
    n_bytes = cp.causal_product_checkpoint_size(B, H, N, D, M)
    assert n_bytes > 0 and n_bytes % (4 * B * H * D * M) == 0
    G = n_bytes // (4 * B * H * D * M) + 1
    n_tiles = -(-N // 128)
    tiles = -(-n_tiles // G)
    while -(-n_tiles // tiles) != G:  # the library's segment length
        tiles += 1
    slots = ckpt[: B * H * (G - 1) * D * M].view(B * H, G - 1, D, M).cpu().double().numpy()
    nq, nk, nv = (to_np(t).reshape(B * H, N, -1) for t in (q, k, v))
    for s in range(1, G):
        rows = s * tiles * 128
        _, want = oracle.fwd_state(nq[:, :rows], nk[:, :rows], nv[:, :rows])
        got = slots[:, s - 1]
        # fp32 sums carry an error proportional to the sum of the terms'
        # magnitudes; the hi + lo copy adds at most 2^-17 of the value
        terms = np.einsum("bnd,bnm->bdm", np.abs(nk[:, :rows]).astype(np.float64),
                          np.abs(nv[:, :rows]).astype(np.float64))
        assert np.all(np.abs(got - want) <= 2e-5 * np.abs(want) + 2e-7 * terms), s


def test_ckpt_backward_is_deterministic_and_matches_plain():
    """Repeats give the same bits; dk and dv equal the plain backward's, dq
    agrees with it to rounding."""
    B, H, N, D, M = 8, 16, 2048, 64, 64
    q, k, v, g = make_inputs(B, H, N, D, M, torch.bfloat16, seed=11)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    _, ckpt = cp.causal_product_fwd_ckpt(qd, kd, vd)
    first = cp.causal_product_bwd_ckpt(qd, kd, vd, gd, ckpt)
    first = [t.clone() for t in first]
    for _ in range(3):
        again = cp.causal_product_bwd_ckpt(qd, kd, vd, gd, ckpt)
        for a, b in zip(first, again):
            assert torch.equal(a, b)
    plain = cp.causal_product_bwd(qd, kd, vd, gd)
    torch.cuda.synchronize()
    assert torch.equal(first[1], plain[1]) and torch.equal(first[2], plain[2])
    assert row_rel_err(to_np(first[0]), to_np(plain[0]).astype(np.float64)) <= TOL["bf16"]


def test_ckpt_status_and_launch_counts():
    """A caller workspace stays clear across calls; the library reports one
    launch for the one-launch backward and a seeded dq launch elsewhere."""
    w = WORKLOADS["bf16_b8h16_n4096_d64"]
    assert cp.causal_product_launch_count(w.B, w.H, w.N, w.D, w.M, backward=True, ckpt=True) == 1
    B, H, N, D, M = 1, 2, 4100, 128, 64
    plain = cp.causal_product_launch_count(B, H, N, D, M, backward=True)
    seeded = cp.causal_product_launch_count(B, H, N, D, M, backward=True, ckpt=True)
    assert seeded == plain - 2  # dq's segment sums and their prefix
    q, k, v, g = make_inputs(w.B, w.H, 1024, w.D, w.M, torch.bfloat16, seed=3)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    ws = torch.zeros(cp.causal_product_workspace_size(w.B, w.H, 1024, w.D, w.M, backward=True),
                     dtype=torch.uint8, device=DEV)
    _, ckpt = cp.causal_product_fwd_ckpt(qd, kd, vd)
    for _ in range(3):
        cp.causal_product_bwd_ckpt(qd, kd, vd, gd, ckpt, workspace=ws)
    assert cp.causal_product_status(ws) == cp.CP_OK


def test_autograd_uses_checkpoints():
    B, H, N, D, M = 2, 60, 700, 64, 64
    q, k, v, g = make_inputs(B, H, N, D, M, torch.bfloat16, seed=9)
    qd, kd, vd = (t.to(DEV).requires_grad_(True) for t in (q, k, v))
    out = cp.causal_product(qd, kd, vd)
    out.backward(g.to(DEV))
    torch.cuda.synchronize()
    nq, nk, nv, ng = (to_np(t) for t in (q, k, v, g))
    rq, rk, rv = oracle.bwd(nq, nk, nv, ng)
    for got, ref in ((qd.grad, rq), (kd.grad, rk), (vd.grad, rv)):
        assert row_rel_err(to_np(got), ref) <= TOL["bf16"]
