"""Error metrics shared by the GPU parity tests.

The tolerance is a maximum relative error, taken per output row: for each
(b, h, i) the largest absolute deviation over the row's columns is divided
by the largest magnitude of the oracle's row (floored at 1e-30).  An
element-wise relative error is meaningless here because the values
v ~ N(0, 1) make individual outputs cancel towards zero; the row scale is
the scale the arithmetic works at.  Bounds: 1e-4 for fp32 inputs, 2e-2 for
bf16 inputs (fp32 accumulation and state), and 2e-3 for fp16 inputs: they
are computed in fp32 and rounded to fp16 once, a relative error of 2^-11
(4.9e-4) per element, with a factor of four to spare.
"""
import numpy as np

TOL = {"f32": 1e-4, "bf16": 2e-2, "f16": 2e-3}


def row_rel_err(got, ref) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0
    scale = np.maximum(np.max(np.abs(ref), axis=-1), 1e-30)
    return float(np.max(np.max(np.abs(got - ref), axis=-1) / scale))


def to_np(t):
    """torch tensor (any device, f32/bf16) -> float32 numpy (exact for bf16)."""
    return t.detach().float().cpu().numpy()
