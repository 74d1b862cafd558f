"""The allocation-free forward entry point (causal_product_fwd_noalloc).

Some callers cannot allocate device memory -- their host framework owns
every device allocation, or an allocation's implicit synchronisation is not
acceptable to them.  This entry point gives them the forward pass with its
scratch in a static device array instead of a workspace.  The GPU test calls
it through the C ABI twice in a row on each shape, reads the shared status
word after each call, checks both results against the oracle and against the
ordinary causal_product_fwd on the same inputs, and checks that the calls
allocated no device memory.  This file is collected last so that a failure
here does not hide the results of the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
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


def _pool_used_bytes(dev_index):
    """Bytes in use in the device's default stream-ordered memory pool (the
    pool cudaMallocAsync draws from), or None if the runtime cannot be asked."""
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            continue
    else:
        return None
    pool = ctypes.c_void_p()
    if rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), ctypes.c_int(dev_index)) != 0:
        return None
    used = ctypes.c_uint64()
    cuda_mem_pool_attr_used_mem_current = 7
    if rt.cudaMemPoolGetAttribute(pool, cuda_mem_pool_attr_used_mem_current,
                                  ctypes.byref(used)) != 0:
        return None
    return used.value


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,tol", [(torch.bfloat16, TOL["bf16"]), (torch.float32, TOL["f32"])])
def test_noalloc_matches_fwd_twice(dtype, tol):
    dev = torch.device("cuda:0")
    # few problems and a long sequence: the scan splits each problem into
    # segments, so the static scratch holds real aggregates; the second shape
    # has a different segment count and a ragged tail
    shapes = [(1, 2, 5000, 64, 64, 21), (2, 1, 3001, 64, 64, 22)]
    lib = cp.load_library()
    stream = torch.cuda.current_stream(dev)
    for B, H, N, D, M, seed in shapes:
        q, k, v, _ = make_inputs(B, H, N, D, M, dtype, seed=seed, backward=False)
        ref = oracle.fwd(to_np(q), to_np(k), to_np(v))
        q, k, v = q.to(dev), k.to(dev), v.to(dev)
        ordinary = cp.causal_product_fwd(q, k, v)
        outs = [torch.full_like(ordinary, float("nan")) for _ in range(2)]
        torch.cuda.synchronize()
        stats0 = torch.cuda.memory_stats(dev).get("allocation.all.allocated", 0)
        pool0 = _pool_used_bytes(dev.index)
        for out in outs:
            # the C ABI directly, then the shared status word after the call
            rc = lib.causal_product_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                out.data_ptr(), B, H, N, D, M,
                                                cp._DTYPES[dtype], stream.cuda_stream)
            assert rc == cp.CP_OK, cp.causal_product_error_string(rc)
            assert cp.causal_product_noalloc_status(stream) == cp.CP_OK
        # neither call allocated through torch or from the stream-ordered pool
        assert torch.cuda.memory_stats(dev).get("allocation.all.allocated", 0) == stats0
        pool1 = _pool_used_bytes(dev.index)
        if pool0 is not None and pool1 is not None:
            assert pool1 == pool0
        for out in outs:
            got = to_np(out)
            assert np.isfinite(got).all()
            assert row_rel_err(got, ref) <= tol
            assert row_rel_err(got, to_np(ordinary).astype(np.float64)) <= tol
