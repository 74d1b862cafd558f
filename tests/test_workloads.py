"""The synthetic input recipe against independent definitions (CPU only)."""
import numpy as np
import torch

import oracle
from parity_util import row_rel_err
from prefix_sum_outer_gb300.workloads import WORKLOADS, favor_raw_inputs, make_inputs


def test_favor_workload_features_match_the_oracle_map():
    """The D = 256 workload's q and k are positive random features of raw
    rows: its generator (float32 torch, rounded to bf16) and the oracle's
    fp64 map of the same raw rows and projection must give the same causal
    product up to the bf16 rounding of the features (2^-9 relative)."""
    w = WORKLOADS["bf16_favor_n8229_d256_m64"]
    B, H, N = 1, 2, 60
    q, k, v, _ = make_inputs(B, H, N, w.D, w.M, torch.bfloat16, w.seed, feature="favor",
                             backward=False)
    W, xq, xk = favor_raw_inputs(B, H, N, w.D, w.seed)
    f = lambda t: t.float().numpy()
    want = oracle.fwd_favor(f(xq), f(xk), f(v), f(W))
    got = oracle.fwd(f(q), f(k), f(v))
    assert row_rel_err(got, want) < 1e-2


def test_favor_features_are_positive_and_heavy_tailed():
    """The recipe's claim for the D = 256 workload: every feature is
    positive, and the largest is orders of magnitude above the median."""
    w = WORKLOADS["bf16_favor_n8229_d256_m64"]
    q, k, _, _ = make_inputs(1, 2, 512, w.D, w.M, torch.float32, w.seed, feature="favor",
                             backward=False)
    x = np.concatenate([q.numpy().ravel(), k.numpy().ravel()])
    assert np.all(x > 0)
    assert x.max() / np.median(x) > 100
