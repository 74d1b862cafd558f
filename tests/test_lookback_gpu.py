"""The split forward scan in one launch (``-m gpu``): with
CP_SPLIT_SCAN=lookback every segment sums itself, publishes the sum, forms
its prefix from the earlier segments' sums and scans, in one kernel.  The
prefix is added in the order the two-pass form adds it, so both forms give
the same bits; both are checked against the fp64 oracle too."""
import numpy as np
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"

# (B, H, N, D, M): every tile geometry of a split forward scan, ragged tails,
# the 16-problem N = 32768 D = M = 128 and 32-problem D = 256 M = 64 shapes
SHAPES = [
    (1, 2, 5000, 64, 64),
    (1, 3, 8229, 128, 128),
    (1, 2, 4100, 128, 64),
    (1, 2, 3000, 64, 128),
    (1, 2, 2000, 192, 64),
    (2, 2, 3333, 256, 64),
    (2, 8, 32768, 128, 128),
    (4, 8, 8229, 256, 64),
]


def _both(fn, monkeypatch):
    monkeypatch.setenv("CP_SPLIT_SCAN", "twopass")
    a = fn()
    torch.cuda.synchronize()
    monkeypatch.setenv("CP_SPLIT_SCAN", "lookback")
    b = fn()
    torch.cuda.synchronize()
    return a, b


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_lookback_forward_matches_two_pass_and_oracle(shape, monkeypatch):
    B, H, N, D, M = shape
    q, k, v, _ = make_inputs(B, H, N, D, M, torch.bfloat16, seed=sum(shape), backward=False)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    monkeypatch.setenv("CP_SPLIT_SCAN", "lookback")
    assert cp.causal_product_launch_count(B, H, N, D, M) == 1
    two, one = _both(lambda: cp.causal_product_fwd(qd, kd, vd), monkeypatch)
    assert torch.equal(two, one)
    if B * H * N <= 2 * 3 * 8229:
        assert row_rel_err(to_np(one), oracle.fwd(to_np(q), to_np(k), to_np(v))) <= TOL["bf16"]


def test_lookback_checkpoints_and_backward(monkeypatch):
    """The checkpoint-writing forward in one launch: the same output and the
    same checkpoints; the backward from them is unchanged, and a dq product
    that runs as a split forward scan gives the same bits too."""
    B, H, N, D, M = 1, 2, 4100, 128, 64
    q, k, v, g = make_inputs(B, H, N, D, M, torch.bfloat16, seed=7, backward=True)
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    (o2, c2), (o1, c1) = _both(lambda: cp.causal_product_fwd_ckpt(qd, kd, vd), monkeypatch)
    assert torch.equal(o2, o1) and torch.equal(c2, c1)
    b2, b1 = _both(lambda: cp.causal_product_bwd(qd, kd, vd, gd), monkeypatch)
    for x, y in zip(b2, b1):
        assert torch.equal(x, y)
    r = oracle.bwd(to_np(q), to_np(k), to_np(v), to_np(g))
    for got, ref in zip(b1, r):
        assert row_rel_err(to_np(got), ref) <= TOL["bf16"]


def test_lookback_status_stays_clear_and_deterministic(monkeypatch):
    B, H, N, D, M = 2, 8, 32768, 128, 128
    q, k, v, _ = make_inputs(B, H, N, D, M, torch.bfloat16, seed=5, backward=False)
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    monkeypatch.setenv("CP_SPLIT_SCAN", "lookback")
    ws = torch.zeros(cp.causal_product_workspace_size(B, H, N, D, M), dtype=torch.uint8,
                     device=DEV)
    first = cp.causal_product_fwd(qd, kd, vd, workspace=ws).clone()
    for _ in range(3):
        assert torch.equal(first, cp.causal_product_fwd(qd, kd, vd, workspace=ws))
    assert cp.causal_product_status(ws) == cp.CP_OK
