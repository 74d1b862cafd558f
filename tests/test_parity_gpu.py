"""GPU path vs the fp64 oracle, element by element (``-m gpu``).

Every call goes through the C ABI (via the ctypes binding).  Inputs are the
seeded synthetic workloads; the oracle reads exactly the values the GPU
receives.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def run_fwd(q, k, v):
    out = cp.causal_product_fwd(q.to(DEV), k.to(DEV), v.to(DEV))
    torch.cuda.synchronize()
    return out


def run_bwd(q, k, v, g):
    r = cp.causal_product_bwd(q.to(DEV), k.to(DEV), v.to(DEV), g.to(DEV))
    torch.cuda.synchronize()
    return r


def _log(kind, shape, errs):
    """Append measured errors to $CP_PARITY_LOG (JSON lines) when set."""
    path = os.environ.get("CP_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"kind": kind, "shape": list(shape), "errs": errs}) + "\n")


def check_fwd(q, k, v, dtype):
    out = run_fwd(q, k, v)
    ref = oracle.fwd(to_np(q), to_np(k), to_np(v))
    err = row_rel_err(to_np(out), ref)
    _log("fwd_" + dtype, tuple(q.shape) + (v.shape[-1],), {"out": err})
    assert np.isfinite(err) and err <= TOL[dtype], f"fwd row-rel err {err:.3e} > {TOL[dtype]}"
    return err


def check_bwd(q, k, v, g, dtype):
    dq, dk, dv = run_bwd(q, k, v, g)
    rq, rk, rv = oracle.bwd(to_np(q), to_np(k), to_np(v), to_np(g))
    errs = {}
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        errs[name] = row_rel_err(to_np(got), ref)
    _log("bwd_" + dtype, tuple(q.shape) + (v.shape[-1],), errs)
    for name in ("dq", "dk", "dv"):
        assert np.isfinite(errs[name]) and errs[name] <= TOL[dtype], \
            f"{name} row-rel err {errs[name]:.3e} > {TOL[dtype]}"
    return errs


# ---------------------------------------------------------------- workloads
@pytest.mark.parametrize("name", ["tiny_f32_fwd", "mid_f32_fwd"])
def test_fp32_workloads(name):
    w = WORKLOADS[name]
    q, k, v, _ = workload_inputs(w)
    check_fwd(q, k, v, w.dtype)


@pytest.mark.parametrize("name", ["tiny_f32_fwd", "mid_f32_fwd"])
def test_fp32_workloads_backward(name):
    """The fp32 workloads' backward, on the inputs the bench's fwd + bwd step
    uses (the same draw with g)."""
    w = WORKLOADS[name]
    q, k, v, g = make_inputs(w.B, w.H, w.N, w.D, w.M, w.torch_dtype, w.seed,
                             feature=w.feature, x_std=w.x_std, backward=True)
    check_bwd(q, k, v, g, w.dtype)


@pytest.mark.parametrize("name", ["bf16_b8h16_n4096_d64", "bf16_long_n32768_d128",
                                  "bf16_favor_n8229_d256_m64"])
def test_bf16_workloads_full_size(name):
    """The three bf16 workloads at full size, forward and backward, against
    the oracle on every element."""
    w = WORKLOADS[name]
    q, k, v, g = workload_inputs(w)
    check_fwd(q, k, v, w.dtype)
    check_bwd(q, k, v, g, w.dtype)


# ---------------------------------------------------------------- shapes
SHAPES = [
    # (B, H, N, D, M): tiles of 128 rows, ragged tails, D != M, padded widths
    (1, 1, 1, 64, 64),
    (1, 2, 17, 64, 64),
    (2, 1, 127, 64, 64),
    (1, 1, 128, 64, 64),
    (1, 3, 129, 64, 64),
    (2, 2, 300, 64, 128),
    (1, 2, 385, 128, 64),
    (1, 1, 513, 128, 128),
    (1, 2, 260, 256, 64),
    (1, 1, 200, 192, 64),
    (1, 1, 140, 16, 16),
    (1, 1, 140, 32, 48),
    (2, 1, 99, 80, 24),
]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_shapes_fwd_bwd(shape, dtype):
    B, H, N, D, M = shape
    q, k, v, g = make_inputs(B, H, N, D, M, DT[dtype], seed=sum(shape))
    check_fwd(q, k, v, dtype)
    check_bwd(q, k, v, g, dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("shape", [(1, 1, 300, 256, 256), (1, 2, 200, 64, 256),
                                   (1, 1, 150, 256, 8)],
                         ids=lambda s: "x".join(map(str, s)))
def test_widest_shapes(shape, dtype):
    """D = M = 256 is the widest the boundary takes: four 64-column value
    blocks on the tensor-core path, 256-row states on the fp32 path."""
    B, H, N, D, M = shape
    q, k, v, g = make_inputs(B, H, N, D, M, DT[dtype], seed=N + D + M)
    check_fwd(q, k, v, "bf16" if dtype == "bf16" else "f32")
    check_bwd(q, k, v, g, "bf16" if dtype == "bf16" else "f32")


@pytest.mark.parametrize("shape", [(1, 1, 100, 1, 1), (2, 1, 333, 3, 5), (1, 1, 257, 33, 130)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fp32_odd_widths(shape):
    """fp32 takes any width from 1 to 256: widths that are not a multiple of
    4 pad the shared-memory tiles with zeros, and M = 130 leaves a value block
    two columns wide."""
    B, H, N, D, M = shape
    q, k, v, g = make_inputs(B, H, N, D, M, torch.float32, seed=N + 31 * D + M)
    check_fwd(q, k, v, "f32")
    check_bwd(q, k, v, g, "f32")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("N", [1000, 4096, 5000])
def test_segmented_scan(N, dtype):
    """Few problems, long sequences: the sequence is split into segments and
    the two-pass scan carries the state across them."""
    q, k, v, g = make_inputs(1, 2, N, 64, 64, DT[dtype], seed=N)
    check_fwd(q, k, v, dtype)
    check_bwd(q, k, v, g, dtype)


@pytest.mark.parametrize("shape", [(1, 1, 3000, 48, 32), (1, 3, 1111, 64, 40), (3, 5, 257, 8, 64),
                                   (2, 2, 640, 64, 64), (10, 13, 300, 64, 64),
                                   (1, 151, 256, 48, 64), (10, 16, 300, 64, 56)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fused_dkdv_shapes(shape):
    """bf16 backward with D, M <= 64 computes dk and dv in one pass over a
    shared reverse state: D != M, ragged tails, the two-pass scan across
    segments, and unsplit problems in one launch with dq scans on the
    spare SMs (130 and 151 problems) or as separate launches (160)."""
    B, H, N, D, M = shape
    q, k, v, g = make_inputs(B, H, N, D, M, torch.bfloat16, seed=N + D)
    check_bwd(q, k, v, g, "bf16")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_signed_features(dtype):
    """q, k with both signs (no positive feature map)."""
    q, k, v, g = make_inputs(2, 3, 777, 64, 64, DT[dtype], seed=11, feature="normal")
    check_fwd(q, k, v, dtype)
    check_bwd(q, k, v, g, dtype)


# ---------------------------------------------------------------- properties
def test_zero_value_gives_zero_every_column():
    """v = 0 must give exactly zero output in every column (column 0 too)."""
    q, k, v, _ = make_inputs(1, 2, 300, 64, 64, torch.bfloat16, seed=5)
    out = run_fwd(q * 100, k, torch.zeros_like(v))
    assert torch.count_nonzero(out).item() == 0


def test_first_row_closed_form():
    q, k, v, _ = make_inputs(2, 2, 257, 64, 64, torch.bfloat16, seed=6)
    out = to_np(run_fwd(q, k, v))[..., 0, :]
    qk = np.sum(to_np(q)[..., 0, :].astype(np.float64) * to_np(k)[..., 0, :], axis=-1)
    ref = qk[..., None] * to_np(v)[..., 0, :]
    assert row_rel_err(out, ref) <= TOL["bf16"]


def test_causality_on_gpu():
    """Changing rows j > i of k and v leaves rows <= i of the output bitwise
    unchanged (the kernels combine partial sums in a fixed order)."""
    q, k, v, _ = make_inputs(1, 2, 1000, 64, 64, torch.bfloat16, seed=7)
    base = run_fwd(q, k, v).cpu()
    cut = 600
    k2, v2 = k.clone(), v.clone()
    k2[..., cut + 1:, :] = k2[..., cut + 1:, :].flip(-2)
    v2[..., cut + 1:, :] = -v2[..., cut + 1:, :]
    pert = run_fwd(q, k2, v2).cpu()
    assert torch.equal(base[..., :cut + 1, :], pert[..., :cut + 1, :])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_deterministic(dtype):
    q, k, v, g = make_inputs(1, 2, 3000, 64, 64, DT[dtype], seed=8)
    a = run_fwd(q, k, v).cpu()
    b = run_fwd(q, k, v).cpu()
    assert torch.equal(a, b)
    ga = [t.cpu() for t in run_bwd(q, k, v, g)]
    gb = [t.cpu() for t in run_bwd(q, k, v, g)]
    assert all(torch.equal(x, y) for x, y in zip(ga, gb))


def test_output_guard_bands():
    """Nothing outside the output tensor is written (ragged tail included)."""
    B, H, N, D, M = 1, 3, 333, 64, 64
    q, k, v, g = make_inputs(B, H, N, D, M, torch.bfloat16, seed=9)
    pad = 4096  # elements
    n_out = B * H * N * M
    buf = torch.full((pad + n_out + pad,), 12345.0, dtype=torch.bfloat16, device=DEV)
    out = buf[pad:pad + n_out].view(B, H, N, M)
    cp.causal_product_fwd(q.to(DEV), k.to(DEV), v.to(DEV), out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345.0) and torch.all(buf[pad + n_out:] == 12345.0)
    ref = oracle.fwd(to_np(q), to_np(k), to_np(v))
    assert row_rel_err(to_np(out), ref) <= TOL["bf16"]


def test_autograd_matches_oracle():
    q, k, v, g = make_inputs(1, 2, 200, 64, 64, torch.bfloat16, seed=10)
    qd, kd, vd = (t.to(DEV).requires_grad_(True) for t in (q, k, v))
    out = cp.causal_product(qd, kd, vd)
    out.backward(g.to(DEV))
    rq, rk, rv = oracle.bwd(to_np(q), to_np(k), to_np(v), to_np(g))
    for got, ref in ((qd.grad, rq), (kd.grad, rk), (vd.grad, rv)):
        assert row_rel_err(to_np(got), ref) <= TOL["bf16"]


def test_status_word_is_clear_after_normal_calls():
    q, k, v, g = make_inputs(1, 1, 600, 64, 64, torch.bfloat16, seed=12)
    q, k, v, g = (t.to(DEV) for t in (q, k, v, g))
    ws = torch.zeros(cp.causal_product_workspace_size(1, 1, 600, 64, 64, torch.bfloat16, True),
                     dtype=torch.uint8, device=DEV)
    cp.causal_product_fwd(q, k, v, workspace=ws)
    cp.causal_product_bwd(q, k, v, g, workspace=ws)
    assert cp.causal_product_status(ws) == cp.CP_OK


def test_streams_are_respected():
    """Work is enqueued on the given stream."""
    q, k, v, _ = make_inputs(2, 2, 1024, 64, 64, torch.bfloat16, seed=13)
    q, k, v = (t.to(DEV) for t in (q, k, v))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = cp.causal_product_fwd(q, k, v, stream=s)
    s.synchronize()
    ref = oracle.fwd(to_np(q), to_np(k), to_np(v))
    assert row_rel_err(to_np(out), ref) <= TOL["bf16"]
