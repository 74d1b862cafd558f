"""The failure path on the GPU (``-m gpu``), without a fault: a bounded wait
that runs out records CP_ERR_TIMEOUT in the workspace status word, the host
reads it, and the context stays usable."""
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def test_timeout_is_reported_and_sticky_then_cleared():
    q, k, v, _ = make_inputs(1, 2, 300, 64, 64, torch.bfloat16, seed=41, backward=False)
    ws = torch.zeros(cp.causal_product_workspace_size(1, 2, 300, 64, 64, torch.bfloat16, False),
                     dtype=torch.uint8, device=DEV)
    cp.causal_product_selftest_timeout(ws, wait_ns=20_000_000)   # a 20 ms wait runs out
    # a normal call afterwards leaves the recorded error in place (sticky)
    out = cp.causal_product_fwd(q.to(DEV), k.to(DEV), v.to(DEV), workspace=ws)
    assert cp.causal_product_status(ws) == cp.CP_ERR_TIMEOUT
    # reading clears it
    assert cp.causal_product_status(ws) == cp.CP_OK
    # the context is still usable and the call that ran after the timeout is right
    ref = oracle.fwd(to_np(q), to_np(k), to_np(v))
    assert row_rel_err(to_np(out), ref) <= TOL["bf16"]
    out2 = cp.causal_product_fwd(q.to(DEV), k.to(DEV), v.to(DEV), workspace=ws)
    torch.cuda.synchronize()
    assert cp.causal_product_status(ws) == cp.CP_OK
    assert torch.equal(out, out2)
