"""Decoding step on the GPU (``-m gpu``): S <- S + k v^T, out = S^T q per
(b,h), against the fp64 oracle's carried-state forward with N = 1, and
token-by-token decoding against the sequence forward."""
import numpy as np
import pytest
import torch

import oracle
import prefix_sum_outer_gb300 as cp
from parity_util import TOL, row_rel_err, to_np
from prefix_sum_outer_gb300.workloads import make_inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
DT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
STATE_TOL = {"f32": 1e-5, "bf16": 1e-4, "f16": 1e-4}


@pytest.mark.parametrize("shape", [(8, 16, 64, 64, "bf16"), (3, 5, 128, 32, "bf16"),
                                   (2, 2, 16, 256, "bf16"), (1, 4, 256, 64, "bf16"),
                                   (2, 3, 8, 8, "bf16"), (2, 3, 64, 64, "f32"),
                                   (1, 2, 80, 24, "f32"), (1, 1, 5, 3, "f32"),
                                   # a 128 MiB state, larger than the L2: the
                                   # streaming variant
                                   (512, 16, 64, 64, "bf16"),
                                   # fp16 rows, plain and streaming
                                   (2, 3, 64, 64, "f16"), (512, 16, 64, 64, "f16")],
                         ids=lambda s: "x".join(map(str, s)))
def test_decode_step_against_oracle(shape):
    B, H, D, M, dt = shape
    q, k, v, _ = make_inputs(B, H, 1, D, M, DT[dt], seed=D * M + B, backward=False)
    s0 = torch.randn((B, H, D, M), generator=torch.Generator().manual_seed(D + M)) * 3
    state = s0.to(DEV)
    out = cp.causal_product_decode(q[:, :, 0].to(DEV), k[:, :, 0].to(DEV), v[:, :, 0].to(DEV),
                                   state)
    torch.cuda.synchronize()
    r_out, r_state = oracle.fwd_state(to_np(q), to_np(k), to_np(v), state_in=s0.numpy())
    assert row_rel_err(to_np(out), r_out[:, :, 0]) <= TOL[dt]
    assert row_rel_err(to_np(state), r_state) <= STATE_TOL[dt]


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_decode_token_by_token_matches_sequence(dt):
    """Decoding the rows of a sequence one at a time gives the sequence
    forward's outputs and final state."""
    B, H, N, D, M = 2, 4, 40, 64, 64
    q, k, v, _ = (t.to(DEV) if t is not None else None
                  for t in make_inputs(B, H, N, D, M, DT[dt], seed=31, backward=False))
    s0 = torch.randn((B, H, D, M), generator=torch.Generator().manual_seed(32)).to(DEV)
    ref_out, ref_state = cp.causal_product_fwd(q, k, v, state_in=s0, return_state=True)
    state = s0.clone()
    rows = [cp.causal_product_decode(q[:, :, i].contiguous(), k[:, :, i].contiguous(),
                                     v[:, :, i].contiguous(), state) for i in range(N)]
    torch.cuda.synchronize()
    got = torch.stack(rows, dim=2)
    r_out, r_state = oracle.fwd_state(to_np(q), to_np(k), to_np(v), state_in=to_np(s0))
    assert row_rel_err(to_np(got), r_out) <= TOL[dt]
    assert row_rel_err(to_np(ref_out), r_out) <= TOL[dt]
    assert row_rel_err(to_np(state), r_state) <= STATE_TOL[dt]
    assert row_rel_err(to_np(ref_state), r_state) <= STATE_TOL[dt]
