"""The allocation-free forward entry point (causal_product_fwd_noalloc).

Some callers cannot allocate device memory -- their host framework owns
every device allocation, or an allocation's implicit synchronisation is not
acceptable to them.  This entry point gives them the forward pass with its
scratch in a static device array instead of a workspace.  The GPU test calls
it through the C ABI twice in a row and checks each result against the
ordinary causal_product_fwd on the same inputs.  This file is collected last
so that a failure here does not hide the results of the other tests.
"""
import ctypes

import pytest
import torch

import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import make_inputs

CP_ERR_NOALLOC_LIMIT = 9


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Argument check only: nothing is enqueued, no device is needed."""
    lib = cp.load_library()
    A = 1 << 20  # fake aligned addresses, never dereferenced
    # fp32, D = M = 256, one long sequence: the scan aggregates need > 16 MiB
    rc = lib.causal_product_fwd_noalloc(A, 2 * A, 3 * A, 4 * A, 1, 1, 20000, 256, 256, 0, None)
    assert rc == CP_ERR_NOALLOC_LIMIT
    assert "noalloc" in cp.causal_product_error_string(rc)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, TOL["bf16"]), (torch.float32, TOL["f32"])])
def test_noalloc_matches_fwd_twice(dtype, tol):
    dev = torch.device("cuda:0")
    # few problems and a long sequence: the scan splits each problem into
    # segments, so the static scratch holds real aggregates
    shapes = [(1, 2, 5000, 64, 64, 21), (2, 1, 3001, 64, 64, 22)]
    for B, H, N, D, M, seed in shapes:
        q, k, v, _ = make_inputs(B, H, N, D, M, dtype, seed=seed, backward=False)
        q, k, v = q.to(dev), k.to(dev), v.to(dev)
        ref = cp.causal_product_fwd(q, k, v)
        out = torch.full_like(ref, float("nan"))
        cp.causal_product_fwd_noalloc(q, k, v, out)
        torch.cuda.synchronize()
        assert row_rel_err(to_np(out), to_np(ref).astype("float64")) <= tol
