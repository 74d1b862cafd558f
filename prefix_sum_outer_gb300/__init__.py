"""GB300-native causal dot product (causal linear attention's prefix sum).

Python face of ``libcausal_product.so`` (C ABI in ``include/causal_product.h``).
This module only marshals arguments: every step of the computation runs in
the library's CUDA kernels.  PyTorch supplies device memory and streams.

    out = causal_product(q, k, v)              # autograd-aware
    causal_product_fwd(q, k, v, out)           # raw entry points, same names
    causal_product_bwd(q, k, v, g, dq, dk, dv) #   as the C ABI

q, k: [B, H, N, D]; v: [B, H, N, M]; all contiguous, on one CUDA device,
dtype float32, bfloat16 or float16 (fp16 runs on the fp32 path, widened on
load).  out_i = sum_{j<=i} (q_i . k_j) v_j.

There is no fallback: if the library cannot be built or loaded, every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "CP_OK", "CausalProductError", "causal_product", "causal_product_fwd", "causal_product_bwd",
    "causal_product_fwd_noalloc", "causal_product_noalloc_status", "causal_product_decode",
    "causal_product_normalizer", "causal_product_normalizer_bwd", "normalizer",
    "causal_product_fwd_norm",
    "causal_product_fwd_feature", "causal_product_bwd_feature", "FEATURES",
    "causal_product_workspace_size", "causal_product_feature_workspace_size",
    "causal_product_launch_count", "causal_product_status",
    "causal_product_checkpoint_size", "causal_product_fwd_ckpt", "causal_product_bwd_ckpt",
    "causal_product_fwd_favor", "causal_product_bwd_favor", "causal_product_favor",
    "causal_product_error_string", "library_path", "load_library",
]

CP_DTYPE_F32, CP_DTYPE_BF16, CP_DTYPE_F16 = 0, 1, 2
CP_OK = 0
CP_ERR_TIMEOUT = 7
_DTYPES = {torch.float32: CP_DTYPE_F32, torch.bfloat16: CP_DTYPE_BF16,
           torch.float16: CP_DTYPE_F16}
# feature maps applied to q and k inside the kernels (cp_feature_t)
FEATURES = {None: 0, "none": 0, "elu1": 1}


def _feature_code(feature) -> int:
    if feature not in FEATURES:
        raise ValueError(f"unknown feature map {feature!r}; expected one of {list(FEATURES)}")
    return FEATURES[feature]

_lib = None
_lock = threading.Lock()


class CausalProductError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {causal_product_error_string(code)}")


def library_path() -> str:
    return _build.LIB


def load_library(rebuild: bool = True) -> ctypes.CDLL:
    """Load the C ABI library (building it first if its sources changed)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if rebuild else _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libcausal_product.so not found at {path}")
            lib = ctypes.CDLL(path)
            p, i64, c_int, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            lib.causal_product_workspace_size.argtypes = [i64, i64, i64, i64, i64, c_int, c_int]
            lib.causal_product_workspace_size.restype = sz
            lib.causal_product_launch_count.argtypes = [i64, i64, i64, i64, i64, c_int, c_int]
            lib.causal_product_launch_count.restype = c_int
            lib.causal_product_fwd.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, c_int, p, sz, p]
            lib.causal_product_fwd.restype = c_int
            lib.causal_product_bwd.argtypes = [p, p, p, p, p, p, p, i64, i64, i64, i64, i64, c_int,
                                               p, sz, p]
            lib.causal_product_bwd.restype = c_int
            lib.causal_product_checkpoint_size.argtypes = [i64, i64, i64, i64, i64, c_int]
            lib.causal_product_checkpoint_size.restype = sz
            lib.causal_product_fwd_ckpt.argtypes = [p, p, p, p, p, sz, i64, i64, i64, i64, i64,
                                                    c_int, p, sz, p]
            lib.causal_product_fwd_ckpt.restype = c_int
            lib.causal_product_bwd_ckpt.argtypes = [p, p, p, p, p, sz, p, p, p, i64, i64, i64,
                                                    i64, i64, c_int, p, sz, p]
            lib.causal_product_bwd_ckpt.restype = c_int
            lib.causal_product_fwd_state.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                                     c_int, p, sz, p]
            lib.causal_product_fwd_state.restype = c_int
            lib.causal_product_bwd_state.argtypes = [p, p, p, p, p, p, p, p, p, p, i64, i64, i64,
                                                     i64, i64, c_int, p, sz, p]
            lib.causal_product_bwd_state.restype = c_int
            lib.causal_product_selftest_timeout.argtypes = [p, ctypes.c_uint64, p]
            lib.causal_product_selftest_timeout.restype = c_int
            lib.causal_product_decode.argtypes = [p, p, p, p, p, i64, i64, i64, i64, c_int, p]
            lib.causal_product_decode.restype = c_int
            lib.causal_product_fwd_noalloc.argtypes = [p, p, p, p, i64, i64, i64, i64, i64, c_int,
                                                       p]
            lib.causal_product_fwd_noalloc.restype = c_int
            lib.causal_product_noalloc_status.argtypes = [p]
            lib.causal_product_noalloc_status.restype = c_int
            lib.causal_product_normalizer_workspace_size.argtypes = [i64, i64, i64, i64, c_int]
            lib.causal_product_normalizer_workspace_size.restype = sz
            lib.causal_product_fwd_norm_workspace_size.argtypes = [i64, i64, i64, i64, i64, c_int]
            lib.causal_product_fwd_norm_workspace_size.restype = sz
            lib.causal_product_fwd_norm.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, c_int,
                                                    p, sz, p]
            lib.causal_product_fwd_norm.restype = c_int
            lib.causal_product_normalizer.argtypes = [p, p, p, i64, i64, i64, i64, c_int, p, sz, p]
            lib.causal_product_normalizer.restype = c_int
            lib.causal_product_normalizer_bwd.argtypes = [p, p, p, p, p, i64, i64, i64, i64, c_int,
                                                          p, sz, p]
            lib.causal_product_normalizer_bwd.restype = c_int
            lib.causal_product_fwd_feature.argtypes = [p, p, p, p, c_int, i64, i64, i64, i64, i64,
                                                       c_int, p, sz, p]
            lib.causal_product_fwd_feature.restype = c_int
            lib.causal_product_bwd_feature.argtypes = [p, p, p, p, p, p, p, c_int, i64, i64, i64,
                                                       i64, i64, c_int, p, sz, p]
            lib.causal_product_bwd_feature.restype = c_int
            lib.causal_product_feature_workspace_size.argtypes = [i64, i64, i64, i64, i64, c_int,
                                                                  c_int]
            lib.causal_product_feature_workspace_size.restype = sz
            lib.causal_product_normalizer_feature.argtypes = [p, p, p, c_int, i64, i64, i64, i64,
                                                              c_int, p, sz, p]
            lib.causal_product_normalizer_feature.restype = c_int
            lib.causal_product_normalizer_bwd_feature.argtypes = [p, p, p, p, p, c_int, i64, i64,
                                                                  i64, i64, c_int, p, sz, p]
            lib.causal_product_normalizer_bwd_feature.restype = c_int
            lib.causal_product_favor_workspace_size.argtypes = [i64, i64, i64, i64, i64, i64,
                                                                c_int, c_int]
            lib.causal_product_favor_workspace_size.restype = sz
            lib.causal_product_fwd_favor.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64,
                                                     c_int, p, sz, p]
            lib.causal_product_fwd_favor.restype = c_int
            lib.causal_product_bwd_favor.argtypes = [p, p, p, p, p, p, p, p, i64, i64, i64, i64,
                                                     i64, i64, c_int, p, sz, p]
            lib.causal_product_bwd_favor.restype = c_int
            lib.causal_product_status.argtypes = [p, p]
            lib.causal_product_status.restype = c_int
            lib.causal_product_error_string.argtypes = [c_int]
            lib.causal_product_error_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def causal_product_error_string(code: int) -> str:
    return load_library().causal_product_error_string(int(code)).decode()


def _dims(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor):
    if q.dim() != 4 or k.shape != q.shape or v.dim() != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError(f"expected q,k [B,H,N,D] and v [B,H,N,M]; got {tuple(q.shape)}, "
                         f"{tuple(k.shape)}, {tuple(v.shape)}")
    B, H, N, D = q.shape
    return B, H, N, D, v.shape[3]


def _dtype_code(*ts: torch.Tensor) -> int:
    dt = ts[0].dtype
    if dt not in _DTYPES or any(t.dtype != dt for t in ts):
        raise TypeError(f"all tensors must share one dtype in {list(_DTYPES)}; "
                        f"got {[t.dtype for t in ts]}")
    return _DTYPES[dt]


def _check_device(*ts: torch.Tensor):
    dev = ts[0].device
    if dev.type != "cuda":
        raise RuntimeError("causal_product runs on CUDA tensors only (no CPU path)")
    for t in ts:
        if t.device != dev:
            raise RuntimeError("all tensors must be on the same CUDA device")
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def _check_like(t: torch.Tensor, shape, dtype: torch.dtype, name: str):
    """A caller-provided output must have exactly the shape and dtype the
    kernels write: the C ABI receives only its pointer, so a smaller buffer
    would be written past its end."""
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} of shape {tuple(shape)}; "
                         f"got {t.dtype} {tuple(t.shape)}")


def _stream_ptr(stream: Optional[torch.cuda.Stream], device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return int(s.cuda_stream)


def causal_product_workspace_size(B: int, H: int, N: int, D: int, M: int,
                                  dtype: torch.dtype = torch.bfloat16,
                                  backward: bool = False) -> int:
    return int(load_library().causal_product_workspace_size(B, H, N, D, M, _DTYPES[dtype],
                                                            int(bool(backward))))


def causal_product_feature_workspace_size(B: int, H: int, N: int, D: int, M: int,
                                          dtype: torch.dtype = torch.bfloat16,
                                          backward: bool = False) -> int:
    """Workspace bytes of causal_product_fwd_feature / _bwd_feature."""
    return int(load_library().causal_product_feature_workspace_size(
        B, H, N, D, M, _DTYPES[dtype], int(bool(backward))))


def causal_product_launch_count(B: int, H: int, N: int, D: int, M: int,
                                dtype: torch.dtype = torch.bfloat16,
                                backward: bool = False, ckpt: bool = False,
                                norm: bool = False) -> int:
    """Kernels one causal_product_fwd (or, with ``backward``, _bwd; with
    ``ckpt``, the checkpoint calls; with ``norm``, causal_product_fwd_norm)
    launches for this shape; -1 for a shape the entry points reject."""
    mode = 4 if norm else int(bool(backward)) + (2 if ckpt else 0)
    return int(load_library().causal_product_launch_count(B, H, N, D, M, _DTYPES[dtype], mode))


def causal_product_checkpoint_size(B: int, H: int, N: int, D: int, M: int,
                                   dtype: torch.dtype = torch.bfloat16) -> int:
    """Bytes of the checkpoint buffer of causal_product_fwd_ckpt (0: none)."""
    return int(load_library().causal_product_checkpoint_size(B, H, N, D, M, _DTYPES[dtype]))


def _ckpt_buffer(B, H, N, D, M, dtype, device, ckpt):
    n = causal_product_checkpoint_size(B, H, N, D, M, dtype)
    if ckpt is None:
        ckpt = torch.empty(max(n // 4, 1), dtype=torch.float32, device=device)
    if ckpt.dtype != torch.float32 or ckpt.numel() * 4 < n or not ckpt.is_contiguous():
        raise ValueError(f"ckpt must be a contiguous float32 tensor of at least {n} bytes")
    return ckpt


def causal_product_fwd_ckpt(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                            out: Optional[torch.Tensor] = None,
                            ckpt: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None):
    """The forward that also writes checkpoints of the state for the
    backward (causal_product_bwd_ckpt); returns (out, ckpt)."""
    B, H, N, D, M = _dims(q, k, v)
    code = _dtype_code(q, k, v)
    if out is None:
        out = torch.empty((B, H, N, M), dtype=q.dtype, device=q.device)
    _check_like(out, (B, H, N, M), q.dtype, "out")
    _check_device(q, k, v, out)
    ckpt = _ckpt_buffer(B, H, N, D, M, q.dtype, q.device, ckpt)
    _check_device(q, ckpt)
    lib = load_library()
    need = lib.causal_product_workspace_size(B, H, N, D, M, code, 0)
    if workspace is None:
        workspace = _workspace(need, q.device)
    rc = lib.causal_product_fwd_ckpt(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                     ckpt.data_ptr(), ckpt.numel() * 4, B, H, N, D, M, code,
                                     workspace.data_ptr(), workspace.numel(),
                                     _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_fwd_ckpt")
    return out, ckpt


def causal_product_bwd_ckpt(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                            grad_out: torch.Tensor, ckpt: torch.Tensor,
                            grad_q: Optional[torch.Tensor] = None,
                            grad_k: Optional[torch.Tensor] = None,
                            grad_v: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None):
    """(dq, dk, dv) of L = <grad_out, out>, the dq scans seeded from the
    checkpoints causal_product_fwd_ckpt wrote for the same q, k, v."""
    B, H, N, D, M = _dims(q, k, v)
    code = _dtype_code(q, k, v, grad_out)
    if grad_out.shape != v.shape:
        raise ValueError("grad_out must have v's shape")
    grad_q = torch.empty_like(q) if grad_q is None else grad_q
    grad_k = torch.empty_like(k) if grad_k is None else grad_k
    grad_v = torch.empty_like(v) if grad_v is None else grad_v
    for t, ref, name in ((grad_q, q, "grad_q"), (grad_k, k, "grad_k"), (grad_v, v, "grad_v")):
        _check_like(t, ref.shape, ref.dtype, name)
    _check_device(q, k, v, grad_out, grad_q, grad_k, grad_v)
    ckpt = _ckpt_buffer(B, H, N, D, M, q.dtype, q.device, ckpt)
    _check_device(q, ckpt)
    lib = load_library()
    need = lib.causal_product_workspace_size(B, H, N, D, M, code, 1)
    if workspace is None:
        workspace = _workspace(need, q.device)
    rc = lib.causal_product_bwd_ckpt(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                     grad_out.data_ptr(), ckpt.data_ptr(), ckpt.numel() * 4,
                                     grad_q.data_ptr(), grad_k.data_ptr(), grad_v.data_ptr(),
                                     B, H, N, D, M, code, workspace.data_ptr(),
                                     workspace.numel(), _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_bwd_ckpt")
    return grad_q, grad_k, grad_v


def _workspace(nbytes: int, device) -> torch.Tensor:
    # the status word at its start must begin at zero (it is sticky)
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _state_arg(t: Optional[torch.Tensor], shape, device, name: str) -> int:
    """Device pointer of an optional fp32 [B,H,D,M] state tensor (0 if None)."""
    if t is None:
        return 0
    if t.dtype != torch.float32 or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be float32 of shape {tuple(shape)}; "
                         f"got {t.dtype} {tuple(t.shape)}")
    if t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor on {device}")
    return t.data_ptr()


def causal_product_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                       out: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None,
                       state_in: Optional[torch.Tensor] = None,
                       return_state: bool = False,
                       state_out: Optional[torch.Tensor] = None):
    """out[b,h,i] = (S_0 + sum_{j<=i} k[b,h,j] v[b,h,j]^T)^T q[b,h,i], enqueued
    on ``stream``.  ``state_in`` is S_0 (float32 [B,H,D,M], None = zero);
    with ``return_state`` the result is (out, S_N), S_N the state after the
    last row (written into ``state_out`` when given)."""
    B, H, N, D, M = _dims(q, k, v)
    code = _dtype_code(q, k, v)
    if out is None:
        out = torch.empty((B, H, N, M), dtype=q.dtype, device=q.device)
    _check_like(out, (B, H, N, M), q.dtype, "out")
    _check_device(q, k, v, out)
    if return_state and state_out is None:
        state_out = torch.empty((B, H, D, M), dtype=torch.float32, device=q.device)
    lib = load_library()
    need = lib.causal_product_workspace_size(B, H, N, D, M, code, 0)
    if workspace is None:
        workspace = _workspace(need, q.device)
    rc = lib.causal_product_fwd_state(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
        _state_arg(state_in, (B, H, D, M), q.device, "state_in"),
        _state_arg(state_out, (B, H, D, M), q.device, "state_out"),
        B, H, N, D, M, code, workspace.data_ptr(), workspace.numel(),
        _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_fwd")
    return (out, state_out) if return_state else out


def causal_product_fwd_feature(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                               feature: str = "elu1", out: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None,
                               stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """out_i = sum_{j<=i} (phi(q_i) . phi(k_j)) v_j with phi applied inside the
    kernels (``feature="elu1"``: phi(x) = elu(x) + 1); q and k are the raw
    inputs."""
    B, H, N, D, M = _dims(q, k, v)
    code = _dtype_code(q, k, v)
    if out is None:
        out = torch.empty((B, H, N, M), dtype=q.dtype, device=q.device)
    _check_like(out, (B, H, N, M), q.dtype, "out")
    _check_device(q, k, v, out)
    lib = load_library()
    need = lib.causal_product_feature_workspace_size(B, H, N, D, M, code, 0)
    if workspace is None:
        workspace = _workspace(need, q.device)
    rc = lib.causal_product_fwd_feature(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                        _feature_code(feature), B, H, N, D, M, code,
                                        workspace.data_ptr(), workspace.numel(),
                                        _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_fwd_feature")
    return out


def causal_product_bwd_feature(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                               grad_out: torch.Tensor, feature: str = "elu1",
                               grad_q: Optional[torch.Tensor] = None,
                               grad_k: Optional[torch.Tensor] = None,
                               grad_v: Optional[torch.Tensor] = None,
                               workspace: Optional[torch.Tensor] = None,
                               stream: Optional[torch.cuda.Stream] = None):
    """(dq, dk, dv) of L = <grad_out, out> for causal_product_fwd_feature,
    with respect to the raw q, k and v."""
    B, H, N, D, M = _dims(q, k, v)
    code = _dtype_code(q, k, v, grad_out)
    if grad_out.shape != v.shape:
        raise ValueError("grad_out must have v's shape")
    grad_q = torch.empty_like(q) if grad_q is None else grad_q
    grad_k = torch.empty_like(k) if grad_k is None else grad_k
    grad_v = torch.empty_like(v) if grad_v is None else grad_v
    for t, ref, name in ((grad_q, q, "grad_q"), (grad_k, k, "grad_k"), (grad_v, v, "grad_v")):
        _check_like(t, ref.shape, ref.dtype, name)
    _check_device(q, k, v, grad_out, grad_q, grad_k, grad_v)
    lib = load_library()
    need = lib.causal_product_feature_workspace_size(B, H, N, D, M, code, 1)
    if workspace is None:
        workspace = _workspace(need, q.device)
    rc = lib.causal_product_bwd_feature(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                        grad_out.data_ptr(), grad_q.data_ptr(), grad_k.data_ptr(),
                                        grad_v.data_ptr(), _feature_code(feature), B, H, N, D, M,
                                        code, workspace.data_ptr(), workspace.numel(),
                                        _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_bwd_feature")
    return grad_q, grad_k, grad_v


def causal_product_fwd_noalloc(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                               out: torch.Tensor,
                               stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Forward pass through the library's allocation-free entry point.

    For callers that must not allocate device memory (their host framework
    owns all device allocations, or they cannot afford an implicit device
    synchronisation): the library uses a fixed static scratch array instead
    of a workspace, so ``out`` must be provided.  Calls that overlap on the
    GPU share that array and race; order them on one stream.
    """
    B, H, N, D, M = _dims(q, k, v)
    code = _dtype_code(q, k, v, out)
    _check_like(out, (B, H, N, M), q.dtype, "out")
    _check_device(q, k, v, out)
    rc = load_library().causal_product_fwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                   out.data_ptr(), B, H, N, D, M, code,
                                                   _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_fwd_noalloc")
    return out


def _favor_dims(xq: torch.Tensor, xk: torch.Tensor, v: torch.Tensor, W: torch.Tensor):
    if (xq.dim() != 4 or xk.shape != xq.shape or v.dim() != 4 or v.shape[:3] != xq.shape[:3]
            or W.dim() != 2 or W.shape[1] != xq.shape[3]):
        raise ValueError(f"expected xq, xk [B,H,N,R], v [B,H,N,M], W [D,R]; got {tuple(xq.shape)}, "
                         f"{tuple(xk.shape)}, {tuple(v.shape)}, {tuple(W.shape)}")
    B, H, N, R = xq.shape
    return B, H, N, R, W.shape[0], v.shape[3]


def causal_product_fwd_favor(xq: torch.Tensor, xk: torch.Tensor, v: torch.Tensor,
                             W: torch.Tensor, out: Optional[torch.Tensor] = None,
                             workspace: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """out_i = sum_{j<=i} (phi(xq_i) . phi(xk_j)) v_j with the positive random
    features phi(x) = exp(W x - |x|^2 / 2) / sqrt(D), computed in the kernels
    from the raw rows xq, xk [B,H,N,R] and the projection W [D,R] (bf16)."""
    B, H, N, R, D, M = _favor_dims(xq, xk, v, W)
    code = _dtype_code(xq, xk, v, W)
    if out is None:
        out = torch.empty((B, H, N, M), dtype=v.dtype, device=v.device)
    _check_like(out, (B, H, N, M), v.dtype, "out")
    _check_device(xq, xk, v, W, out)
    lib = load_library()
    need = lib.causal_product_favor_workspace_size(B, H, N, R, D, M, code, 0)
    if workspace is None:
        workspace = _workspace(need, v.device)
    rc = lib.causal_product_fwd_favor(xq.data_ptr(), xk.data_ptr(), v.data_ptr(), W.data_ptr(),
                                      out.data_ptr(), B, H, N, R, D, M, code,
                                      workspace.data_ptr(), workspace.numel(),
                                      _stream_ptr(stream, v.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_fwd_favor")
    return out


def causal_product_bwd_favor(xq: torch.Tensor, xk: torch.Tensor, v: torch.Tensor,
                             W: torch.Tensor, grad_out: torch.Tensor,
                             grad_xq: Optional[torch.Tensor] = None,
                             grad_xk: Optional[torch.Tensor] = None,
                             grad_v: Optional[torch.Tensor] = None,
                             workspace: Optional[torch.Tensor] = None,
                             stream: Optional[torch.cuda.Stream] = None):
    """(dxq, dxk, dv) of L = <grad_out, out> for causal_product_fwd_favor (W
    fixed)."""
    B, H, N, R, D, M = _favor_dims(xq, xk, v, W)
    code = _dtype_code(xq, xk, v, W, grad_out)
    if grad_out.shape != v.shape:
        raise ValueError("grad_out must have v's shape")
    grad_xq = torch.empty_like(xq) if grad_xq is None else grad_xq
    grad_xk = torch.empty_like(xk) if grad_xk is None else grad_xk
    grad_v = torch.empty_like(v) if grad_v is None else grad_v
    for t, ref, name in ((grad_xq, xq, "grad_xq"), (grad_xk, xk, "grad_xk"), (grad_v, v, "grad_v")):
        _check_like(t, ref.shape, ref.dtype, name)
    _check_device(xq, xk, v, W, grad_out, grad_xq, grad_xk, grad_v)
    lib = load_library()
    need = lib.causal_product_favor_workspace_size(B, H, N, R, D, M, code, 1)
    if workspace is None:
        workspace = _workspace(need, v.device)
    rc = lib.causal_product_bwd_favor(xq.data_ptr(), xk.data_ptr(), v.data_ptr(), W.data_ptr(),
                                      grad_out.data_ptr(), grad_xq.data_ptr(), grad_xk.data_ptr(),
                                      grad_v.data_ptr(), B, H, N, R, D, M, code,
                                      workspace.data_ptr(), workspace.numel(),
                                      _stream_ptr(stream, v.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_bwd_favor")
    return grad_xq, grad_xk, grad_v


def causal_product_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, grad_out: torch.Tensor,
                       grad_q: Optional[torch.Tensor] = None,
                       grad_k: Optional[torch.Tensor] = None,
                       grad_v: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None,
                       state_in: Optional[torch.Tensor] = None,
                       grad_state_out: Optional[torch.Tensor] = None,
                       return_state_grad: bool = False,
                       grad_state_in: Optional[torch.Tensor] = None):
    """(dq, dk, dv) of L = <grad_out, out> + <grad_state_out, S_N> for the
    forward from ``state_in`` (S_0; both float32 [B,H,D,M], None = zero).
    With ``return_state_grad`` the result is (dq, dk, dv, dL/dS_0), the last
    written into ``grad_state_in`` when given."""
    B, H, N, D, M = _dims(q, k, v)
    code = _dtype_code(q, k, v, grad_out)
    if grad_out.shape != v.shape:
        raise ValueError("grad_out must have v's shape")
    grad_q = torch.empty_like(q) if grad_q is None else grad_q
    grad_k = torch.empty_like(k) if grad_k is None else grad_k
    grad_v = torch.empty_like(v) if grad_v is None else grad_v
    for t, ref, name in ((grad_q, q, "grad_q"), (grad_k, k, "grad_k"), (grad_v, v, "grad_v")):
        _check_like(t, ref.shape, ref.dtype, name)
    _check_device(q, k, v, grad_out, grad_q, grad_k, grad_v)
    if return_state_grad and grad_state_in is None:
        grad_state_in = torch.empty((B, H, D, M), dtype=torch.float32, device=q.device)
    lib = load_library()
    need = lib.causal_product_workspace_size(B, H, N, D, M, code, 1)
    if workspace is None:
        workspace = _workspace(need, q.device)
    shape = (B, H, D, M)
    rc = lib.causal_product_bwd_state(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), grad_out.data_ptr(),
        _state_arg(state_in, shape, q.device, "state_in"),
        _state_arg(grad_state_out, shape, q.device, "grad_state_out"),
        grad_q.data_ptr(), grad_k.data_ptr(), grad_v.data_ptr(),
        _state_arg(grad_state_in, shape, q.device, "grad_state_in"),
        B, H, N, D, M, code, workspace.data_ptr(), workspace.numel(),
        _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_bwd")
    if return_state_grad:
        return grad_q, grad_k, grad_v, grad_state_in
    return grad_q, grad_k, grad_v


def causal_product_decode(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                          state: torch.Tensor, out: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """One decoding step: state <- state + k v^T (in place), out = state^T q.

    q, k: [B,H,D]; v: [B,H,M]; state: float32 [B,H,D,M]."""
    if q.dim() != 3 or k.shape != q.shape or v.dim() != 3 or v.shape[:2] != q.shape[:2]:
        raise ValueError(f"expected q,k [B,H,D] and v [B,H,M]; got {tuple(q.shape)}, "
                         f"{tuple(k.shape)}, {tuple(v.shape)}")
    B, H, D = q.shape
    M = v.shape[2]
    code = _dtype_code(q, k, v)
    if out is None:
        out = torch.empty((B, H, M), dtype=q.dtype, device=q.device)
    _check_like(out, (B, H, M), q.dtype, "out")
    _check_device(q, k, v, out, state)
    _state_arg(state, (B, H, D, M), q.device, "state")
    rc = load_library().causal_product_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                              out.data_ptr(), state.data_ptr(), B, H, D, M, code,
                                              _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_decode")
    return out


def _qk_dims(q: torch.Tensor, k: torch.Tensor):
    if q.dim() != 4 or k.shape != q.shape:
        raise ValueError(f"expected q,k [B,H,N,D]; got {tuple(q.shape)}, {tuple(k.shape)}")
    return tuple(q.shape)


def causal_product_normalizer(q: torch.Tensor, k: torch.Tensor,
                              z: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None,
                              stream: Optional[torch.cuda.Stream] = None,
                              feature: Optional[str] = None) -> torch.Tensor:
    """z[b,h,i] = q[b,h,i] . sum_{j<=i} k[b,h,j] (float32 [B,H,N]): the
    denominator of causal linear attention.  With ``feature="elu1"`` q and k
    are raw inputs mapped by phi(x) = elu(x) + 1 inside the kernel."""
    B, H, N, D = _qk_dims(q, k)
    code = _dtype_code(q, k)
    if z is None:
        z = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if z.dtype != torch.float32 or tuple(z.shape) != (B, H, N):
        raise ValueError(f"z must be float32 of shape {(B, H, N)}")
    _check_device(q, k, z)
    lib = load_library()
    need = lib.causal_product_normalizer_workspace_size(B, H, N, D, code)
    if workspace is None:
        workspace = _workspace(need, q.device)
    rc = lib.causal_product_normalizer_feature(q.data_ptr(), k.data_ptr(), z.data_ptr(),
                                               _feature_code(feature), B, H, N, D, code,
                                               workspace.data_ptr(), workspace.numel(),
                                               _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_normalizer")
    return z


def causal_product_fwd_norm(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                            out: Optional[torch.Tensor] = None,
                            z: Optional[torch.Tensor] = None,
                            workspace: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None):
    """(out, z): the causal product and its normaliser z[b,h,i] = q[b,h,i] .
    sum_{j<=i} k[b,h,j] (float32 [B,H,N]) in one call; one kernel launch for
    bf16 with D, M <= 64 on unsplit problems."""
    B, H, N, D, M = _dims(q, k, v)
    code = _dtype_code(q, k, v)
    if out is None:
        out = torch.empty((B, H, N, M), dtype=q.dtype, device=q.device)
    _check_like(out, (B, H, N, M), q.dtype, "out")
    if z is None:
        z = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_like(z, (B, H, N), torch.float32, "z")
    _check_device(q, k, v, out, z)
    lib = load_library()
    need = lib.causal_product_fwd_norm_workspace_size(B, H, N, D, M, code)
    if workspace is None:
        workspace = _workspace(need, q.device)
    rc = lib.causal_product_fwd_norm(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                     z.data_ptr(), B, H, N, D, M, code, workspace.data_ptr(),
                                     workspace.numel(), _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_fwd_norm")
    return out, z


def causal_product_normalizer_bwd(q: torch.Tensor, k: torch.Tensor, grad_z: torch.Tensor,
                                  grad_q: Optional[torch.Tensor] = None,
                                  grad_k: Optional[torch.Tensor] = None,
                                  workspace: Optional[torch.Tensor] = None,
                                  stream: Optional[torch.cuda.Stream] = None,
                                  feature: Optional[str] = None):
    """(dq, dk) of L = <grad_z, z>: dq_i = grad_z_i sum_{j<=i} k_j,
    dk_j = sum_{i>=j} grad_z_i q_i, in q's dtype (with ``feature``, with
    respect to the raw q, k: times phi')."""
    B, H, N, D = _qk_dims(q, k)
    code = _dtype_code(q, k)
    if grad_z.dtype != torch.float32 or tuple(grad_z.shape) != (B, H, N):
        raise ValueError(f"grad_z must be float32 of shape {(B, H, N)}")
    grad_q = torch.empty_like(q) if grad_q is None else grad_q
    grad_k = torch.empty_like(k) if grad_k is None else grad_k
    for t, ref, name in ((grad_q, q, "grad_q"), (grad_k, k, "grad_k")):
        _check_like(t, ref.shape, ref.dtype, name)
    _check_device(q, k, grad_z, grad_q, grad_k)
    lib = load_library()
    need = lib.causal_product_normalizer_workspace_size(B, H, N, D, code)
    if workspace is None:
        workspace = _workspace(need, q.device)
    rc = lib.causal_product_normalizer_bwd_feature(q.data_ptr(), k.data_ptr(), grad_z.data_ptr(),
                                                   grad_q.data_ptr(), grad_k.data_ptr(),
                                                   _feature_code(feature), B, H, N, D, code,
                                                   workspace.data_ptr(), workspace.numel(),
                                                   _stream_ptr(stream, q.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_normalizer_bwd")
    return grad_q, grad_k


def causal_product_selftest_timeout(workspace: torch.Tensor, wait_ns: int = 20_000_000,
                                    stream: Optional[torch.cuda.Stream] = None) -> None:
    """Enqueue the failure-path self-test: a bounded wait that runs out and
    records CP_ERR_TIMEOUT in ``workspace``'s status word (read it with
    causal_product_status)."""
    rc = load_library().causal_product_selftest_timeout(workspace.data_ptr(), int(wait_ns),
                                                        _stream_ptr(stream, workspace.device))
    if rc != CP_OK:
        raise CausalProductError(rc, "causal_product_selftest_timeout")


def causal_product_status(workspace: torch.Tensor,
                          stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise ``stream`` and return (and clear) the workspace status word."""
    return int(load_library().causal_product_status(workspace.data_ptr(),
                                                    _stream_ptr(stream, workspace.device)))


def causal_product_noalloc_status(stream: Optional[torch.cuda.Stream] = None,
                                  device=None) -> int:
    """Synchronise ``stream`` and return (and clear) the status word that
    every causal_product_fwd_noalloc call on the current device shares."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    return int(load_library().causal_product_noalloc_status(_stream_ptr(stream, dev)))


class CausalProduct(torch.autograd.Function):
    """Autograd wrapper: forward and backward both call the C ABI; the
    forward keeps checkpoints of the state for the backward's dq scans."""

    @staticmethod
    def forward(ctx, q, k, v):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        out, ckpt = causal_product_fwd_ckpt(q, k, v)
        ctx.save_for_backward(q, k, v, ckpt)
        return out

    @staticmethod
    def backward(ctx, g):
        q, k, v, ckpt = ctx.saved_tensors
        return causal_product_bwd_ckpt(q, k, v, g.contiguous().to(q.dtype), ckpt)


class Normalizer(torch.autograd.Function):
    """Autograd wrapper of the normaliser: (q, k) -> z."""

    @staticmethod
    def forward(ctx, q, k, feature):
        q, k = q.contiguous(), k.contiguous()
        ctx.save_for_backward(q, k)
        ctx.feature = feature
        return causal_product_normalizer(q, k, feature=feature)

    @staticmethod
    def backward(ctx, gz):
        q, k = ctx.saved_tensors
        dq, dk = causal_product_normalizer_bwd(q, k, gz.contiguous().float(), feature=ctx.feature)
        return dq, dk, None


def normalizer(q: torch.Tensor, k: torch.Tensor, feature: Optional[str] = None) -> torch.Tensor:
    """z_i = q_i . sum_{j<=i} k_j (float32 [B,H,N]) with autograd support;
    ``feature="elu1"`` maps raw q, k by phi(x) = elu(x) + 1 in the kernel."""
    return Normalizer.apply(q, k, feature)


class CausalProductFeature(torch.autograd.Function):
    """Autograd wrapper with the feature map applied inside the kernels."""

    @staticmethod
    def forward(ctx, q, k, v, feature):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        ctx.save_for_backward(q, k, v)
        ctx.feature = feature
        return causal_product_fwd_feature(q, k, v, feature)

    @staticmethod
    def backward(ctx, g):
        q, k, v = ctx.saved_tensors
        dq, dk, dv = causal_product_bwd_feature(q, k, v, g.contiguous().to(q.dtype), ctx.feature)
        return dq, dk, dv, None


class CausalProductState(torch.autograd.Function):
    """Autograd wrapper with a carried state: (q, k, v, S_0) -> (out, S_N)."""

    @staticmethod
    def forward(ctx, q, k, v, state):
        q, k, v = q.contiguous(), k.contiguous(), v.contiguous()
        state = None if state is None else state.contiguous()
        ctx.save_for_backward(q, k, v, state)
        ctx.has_state = state is not None
        return causal_product_fwd(q, k, v, state_in=state, return_state=True)

    @staticmethod
    def backward(ctx, g, g_state):
        q, k, v, state = ctx.saved_tensors
        g = torch.zeros_like(v) if g is None else g.contiguous().to(q.dtype)
        g_state = None if g_state is None else g_state.contiguous().float()
        dq, dk, dv, ds = causal_product_bwd(q, k, v, g, state_in=state if ctx.has_state else None,
                                            grad_state_out=g_state, return_state_grad=True)
        return dq, dk, dv, (ds if ctx.has_state else None)


class CausalProductFavor(torch.autograd.Function):
    """Autograd wrapper of the positive-random-feature product: (xq, xk, v)
    -> out for a fixed projection W (no gradient for W)."""

    @staticmethod
    def forward(ctx, xq, xk, v, W):
        xq, xk, v, W = xq.contiguous(), xk.contiguous(), v.contiguous(), W.contiguous()
        ctx.save_for_backward(xq, xk, v, W)
        return causal_product_fwd_favor(xq, xk, v, W)

    @staticmethod
    def backward(ctx, g):
        xq, xk, v, W = ctx.saved_tensors
        dxq, dxk, dv = causal_product_bwd_favor(xq, xk, v, W, g.contiguous().to(v.dtype))
        return dxq, dxk, dv, None


def causal_product_favor(xq: torch.Tensor, xk: torch.Tensor, v: torch.Tensor,
                         W: torch.Tensor) -> torch.Tensor:
    """Causal product of the positive random features phi(x) = exp(W x -
    |x|^2 / 2) / sqrt(D) of the raw rows xq, xk, with autograd support for
    xq, xk and v (W is treated as a constant)."""
    return CausalProductFavor.apply(xq, xk, v, W)


def causal_product(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                   state: Optional[torch.Tensor] = None, return_state: bool = False,
                   feature: Optional[str] = None):
    """Causal dot product with autograd support (no normaliser, no scale).

    ``state`` (float32 [B,H,D,M]) is the state before the first row; with
    ``return_state`` the result is (out, state after the last row), both
    differentiable.  ``feature="elu1"`` applies phi(x) = elu(x) + 1 to q and
    k inside the kernels (no carried state in that mode)."""
    if _feature_code(feature) != 0:
        if state is not None or return_state:
            raise ValueError("a feature map is not combined with a carried state")
        return CausalProductFeature.apply(q, k, v, feature)
    if state is None and not return_state:
        return CausalProduct.apply(q, k, v)
    out, s_n = CausalProductState.apply(q, k, v, state)
    return (out, s_n) if return_state else out
