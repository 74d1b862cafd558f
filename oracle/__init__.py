"""Oracle for the causal dot product -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg (and its ``--impl reference`` arm) may import this package.  The CUDA
product path never imports it, and this package imports nothing from the
product package.

The arithmetic lives in ``causal_product_oracle.c`` (plain C, fp64, the
serial recurrence of triton-lang/triton issue #217, "Dot Product Computes
Wrong Values": state += k v^T, then out = state^T q).  This module compiles
it with gcc and exposes it through ctypes:

    fwd(q, k, v)        -> out            (float64 [..., N, M])
    bwd(q, k, v, g)     -> (dq, dk, dv)   (float64)
    fwd_state(q, k, v, state_in=None)
                        -> (out, state_out)           with carried state
    bwd_state(q, k, v, g, state_in=None, grad_state_out=None)
                        -> (dq, dk, dv, grad_state_in)
    norm(q, k)          -> z = q_i . sum_{j<=i} k_j   (float64 [..., N])
    norm_bwd(q, k, g)   -> (dq, dk)                   (g = dL/dz, [..., N])
    fwd_feature(q, k, v, feature="elu1")   -> out of phi(q), phi(k), v
    norm_feature(q, k, feature="elu1")     -> z of phi(q), phi(k)
    norm_bwd_feature(q, k, g, feature="elu1") -> (dq, dk) w.r.t. raw q, k
    bwd_feature(q, k, v, g, feature="elu1") -> (dq, dk, dv) w.r.t. raw q, k, v
    fwd_favor(xq, xk, v, W)    -> out of phi(xq), phi(xk), v with positive
                                  random features phi(x) = exp(W x - |x|^2/2)/sqrt(D)
    bwd_favor(xq, xk, v, W, g) -> (dxq, dxk, dv) w.r.t. xq, xk, v (W fixed)
    norm_favor(xq, xk, W)      -> z of phi(xq), phi(xk)
    norm_bwd_favor(xq, xk, W, g) -> (dxq, dxk) w.r.t. xq, xk (g = dL/dz)

States are [..., D, M] arrays; they may be float64 (the oracle's own
states) as well as float32 or bfloat16 values, all exact in double.

Inputs are numpy arrays of shape [B, H, N, D] / [B, H, N, M] (any leading
shape works; the last two axes are N and the feature axis).  They are
converted to float32, which is exact for bfloat16 and float32 inputs; a
float64 input is rejected because narrowing it would silently change the
values under test.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "causal_product_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libcpo.so")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libcpo.so`` (gcc, OpenMP).

    No fast-math and no architecture-specific flags: the fp64 arithmetic is
    evaluated exactly in source order on x86_64 and aarch64 alike.
    """
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fopenmp",
           "-shared", "-fPIC", "-std=c11", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, p, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            lib.cpo_fwd.argtypes = [p, p, p, p, i64, i64, i64, i64, c_int]
            lib.cpo_fwd.restype = c_int
            lib.cpo_bwd.argtypes = [p, p, p, p, p, p, p, i64, i64, i64, i64, c_int]
            lib.cpo_bwd.restype = c_int
            lib.cpo_fwd_state.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, c_int]
            lib.cpo_fwd_state.restype = c_int
            lib.cpo_bwd_state.argtypes = [p, p, p, p, p, p, p, p, p, p, i64, i64, i64, i64,
                                          c_int]
            lib.cpo_bwd_state.restype = c_int
            lib.cpo_norm.argtypes = [p, p, p, i64, i64, i64, c_int]
            lib.cpo_norm.restype = c_int
            lib.cpo_norm_bwd.argtypes = [p, p, p, p, p, i64, i64, i64, c_int]
            lib.cpo_norm_bwd.restype = c_int
            lib.cpo_fwd_feature.argtypes = [p, p, p, p, c_int, i64, i64, i64, i64, c_int]
            lib.cpo_fwd_feature.restype = c_int
            lib.cpo_bwd_feature.argtypes = [p, p, p, p, p, p, p, c_int, i64, i64, i64, i64,
                                            c_int]
            lib.cpo_bwd_feature.restype = c_int
            lib.cpo_norm_feature.argtypes = [p, p, p, c_int, i64, i64, i64, c_int]
            lib.cpo_norm_feature.restype = c_int
            lib.cpo_norm_bwd_feature.argtypes = [p, p, p, p, p, c_int, i64, i64, i64, c_int]
            lib.cpo_norm_bwd_feature.restype = c_int
            lib.cpo_fwd_favor.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, c_int]
            lib.cpo_fwd_favor.restype = c_int
            lib.cpo_bwd_favor.argtypes = [p, p, p, p, p, p, p, p, i64, i64, i64, i64, i64,
                                          c_int]
            lib.cpo_bwd_favor.restype = c_int
            lib.cpo_norm_favor.argtypes = [p, p, p, p, i64, i64, i64, i64, c_int]
            lib.cpo_norm_favor.restype = c_int
            lib.cpo_norm_bwd_favor.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, c_int]
            lib.cpo_norm_bwd_favor.restype = c_int
            lib.cpo_threads.argtypes = [c_int]
            lib.cpo_threads.restype = c_int
            _lib = lib
    return _lib


def _as_f32(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.float64:
        raise TypeError("oracle inputs must hold float32/bfloat16 values; "
                        "pass float32 arrays (bf16 -> f32 is exact)")
    return np.ascontiguousarray(x, dtype=np.float32)


def _dims(q, k, v):
    if q.ndim < 2 or q.shape != k.shape or q.shape[:-1] != v.shape[:-1]:
        raise ValueError(f"shape mismatch: q{q.shape} k{k.shape} v{v.shape}")
    lead = q.shape[:-2]
    BH = int(np.prod(lead)) if lead else 1
    return lead, BH, q.shape[-2], q.shape[-1], v.shape[-1]


def threads(nthreads: int = 0) -> int:
    """Threads the oracle uses for ``nthreads`` (0 = OpenMP default)."""
    return int(_load().cpo_threads(int(nthreads)))


def fwd(q, k, v, nthreads: int = 0) -> np.ndarray:
    """out_i = sum_{j<=i} (q_i . k_j) v_j per leading slice, in fp64."""
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    lead, BH, N, D, M = _dims(q, k, v)
    out = np.zeros(lead + (N, M), dtype=np.float64)
    rc = _load().cpo_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, out.ctypes.data,
                         BH, N, D, M, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle fwd failed ({rc})")
    return out


def bwd(q, k, v, g, nthreads: int = 0):
    """(dq, dk, dv) of L = <g, out> for the causal product, in fp64."""
    q, k, v, g = _as_f32(q), _as_f32(k), _as_f32(v), _as_f32(g)
    lead, BH, N, D, M = _dims(q, k, v)
    if g.shape != v.shape:
        raise ValueError(f"grad shape {g.shape} != out shape {v.shape}")
    dq = np.zeros(lead + (N, D), dtype=np.float64)
    dk = np.zeros(lead + (N, D), dtype=np.float64)
    dv = np.zeros(lead + (N, M), dtype=np.float64)
    rc = _load().cpo_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data,
                         dq.ctypes.data, dk.ctypes.data, dv.ctypes.data,
                         BH, N, D, M, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle bwd failed ({rc})")
    return dq, dk, dv


def _state(x, lead, D, M, name):
    if x is None:
        return None
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if x.shape != lead + (D, M):
        raise ValueError(f"{name} shape {x.shape} != {lead + (D, M)}")
    return x


def _ptr(x):
    return None if x is None else x.ctypes.data


def fwd_state(q, k, v, state_in=None, nthreads: int = 0):
    """(out, state_out) with the scan started from state_in ([..., D, M],
    None = zero): out_i = (S_0 + sum_{j<=i} k_j v_j^T)^T q_i and
    state_out = S_0 + sum_j k_j v_j^T, in fp64."""
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    lead, BH, N, D, M = _dims(q, k, v)
    s0 = _state(state_in, lead, D, M, "state_in")
    out = np.zeros(lead + (N, M), dtype=np.float64)
    s_n = np.zeros(lead + (D, M), dtype=np.float64)
    rc = _load().cpo_fwd_state(q.ctypes.data, k.ctypes.data, v.ctypes.data, out.ctypes.data,
                               _ptr(s0), s_n.ctypes.data, BH, N, D, M, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle fwd_state failed ({rc})")
    return out, s_n


def bwd_state(q, k, v, g, state_in=None, grad_state_out=None, nthreads: int = 0):
    """(dq, dk, dv, grad_state_in) of L = <g, out> + <grad_state_out, S_N>
    for the scan started from state_in (None = zero), in fp64."""
    q, k, v, g = _as_f32(q), _as_f32(k), _as_f32(v), _as_f32(g)
    lead, BH, N, D, M = _dims(q, k, v)
    if g.shape != v.shape:
        raise ValueError(f"grad shape {g.shape} != out shape {v.shape}")
    s0 = _state(state_in, lead, D, M, "state_in")
    ds_n = _state(grad_state_out, lead, D, M, "grad_state_out")
    dq = np.zeros(lead + (N, D), dtype=np.float64)
    dk = np.zeros(lead + (N, D), dtype=np.float64)
    dv = np.zeros(lead + (N, M), dtype=np.float64)
    ds0 = np.zeros(lead + (D, M), dtype=np.float64)
    rc = _load().cpo_bwd_state(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data,
                               _ptr(s0), _ptr(ds_n), dq.ctypes.data, dk.ctypes.data,
                               dv.ctypes.data, ds0.ctypes.data, BH, N, D, M, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle bwd_state failed ({rc})")
    return dq, dk, dv, ds0


def _qk_dims(q, k):
    if q.ndim < 2 or q.shape != k.shape:
        raise ValueError(f"shape mismatch: q{q.shape} k{k.shape}")
    lead = q.shape[:-2]
    BH = int(np.prod(lead)) if lead else 1
    return lead, BH, q.shape[-2], q.shape[-1]


def norm(q, k, nthreads: int = 0) -> np.ndarray:
    """Normaliser z_i = q_i . sum_{j<=i} k_j per leading slice, in fp64."""
    q, k = _as_f32(q), _as_f32(k)
    lead, BH, N, D = _qk_dims(q, k)
    z = np.zeros(lead + (N,), dtype=np.float64)
    rc = _load().cpo_norm(q.ctypes.data, k.ctypes.data, z.ctypes.data, BH, N, D, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle norm failed ({rc})")
    return z


def norm_bwd(q, k, g, nthreads: int = 0):
    """(dq, dk) of L = sum_i g_i z_i: dq_i = g_i sum_{j<=i} k_j,
    dk_j = sum_{i>=j} g_i q_i, in fp64."""
    q, k, g = _as_f32(q), _as_f32(k), _as_f32(g)
    lead, BH, N, D = _qk_dims(q, k)
    if g.shape != lead + (N,):
        raise ValueError(f"grad shape {g.shape} != z shape {lead + (N,)}")
    dq = np.zeros(lead + (N, D), dtype=np.float64)
    dk = np.zeros(lead + (N, D), dtype=np.float64)
    rc = _load().cpo_norm_bwd(q.ctypes.data, k.ctypes.data, g.ctypes.data, dq.ctypes.data,
                              dk.ctypes.data, BH, N, D, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle norm_bwd failed ({rc})")
    return dq, dk


_FEATURES = {"none": 0, "elu1": 1}


def fwd_feature(q, k, v, feature: str = "elu1", nthreads: int = 0) -> np.ndarray:
    """out_i = sum_{j<=i} (phi(q_i) . phi(k_j)) v_j with phi(x) = elu(x) + 1
    evaluated in fp64 from the raw q, k."""
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    lead, BH, N, D, M = _dims(q, k, v)
    out = np.zeros(lead + (N, M), dtype=np.float64)
    rc = _load().cpo_fwd_feature(q.ctypes.data, k.ctypes.data, v.ctypes.data, out.ctypes.data,
                                 _FEATURES[feature], BH, N, D, M, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle fwd_feature failed ({rc})")
    return out


def bwd_feature(q, k, v, g, feature: str = "elu1", nthreads: int = 0):
    """(dq, dk, dv) of L = <g, out> for fwd_feature, with respect to the raw
    q, k and v, in fp64."""
    q, k, v, g = _as_f32(q), _as_f32(k), _as_f32(v), _as_f32(g)
    lead, BH, N, D, M = _dims(q, k, v)
    if g.shape != v.shape:
        raise ValueError(f"grad shape {g.shape} != out shape {v.shape}")
    dq = np.zeros(lead + (N, D), dtype=np.float64)
    dk = np.zeros(lead + (N, D), dtype=np.float64)
    dv = np.zeros(lead + (N, M), dtype=np.float64)
    rc = _load().cpo_bwd_feature(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data,
                                 dq.ctypes.data, dk.ctypes.data, dv.ctypes.data,
                                 _FEATURES[feature], BH, N, D, M, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle bwd_feature failed ({rc})")
    return dq, dk, dv


def norm_feature(q, k, feature: str = "elu1", nthreads: int = 0) -> np.ndarray:
    """z_i = phi(q_i) . sum_{j<=i} phi(k_j) from the raw q, k, in fp64."""
    q, k = _as_f32(q), _as_f32(k)
    lead, BH, N, D = _qk_dims(q, k)
    z = np.zeros(lead + (N,), dtype=np.float64)
    rc = _load().cpo_norm_feature(q.ctypes.data, k.ctypes.data, z.ctypes.data,
                                  _FEATURES[feature], BH, N, D, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle norm_feature failed ({rc})")
    return z


def norm_bwd_feature(q, k, g, feature: str = "elu1", nthreads: int = 0):
    """(dq, dk) of L = sum_i g_i z_i for norm_feature, with respect to the
    raw q and k, in fp64."""
    q, k, g = _as_f32(q), _as_f32(k), _as_f32(g)
    lead, BH, N, D = _qk_dims(q, k)
    if g.shape != lead + (N,):
        raise ValueError(f"grad shape {g.shape} != z shape {lead + (N,)}")
    dq = np.zeros(lead + (N, D), dtype=np.float64)
    dk = np.zeros(lead + (N, D), dtype=np.float64)
    rc = _load().cpo_norm_bwd_feature(q.ctypes.data, k.ctypes.data, g.ctypes.data,
                                      dq.ctypes.data, dk.ctypes.data, _FEATURES[feature], BH, N,
                                      D, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle norm_bwd_feature failed ({rc})")
    return dq, dk


def _favor_dims(xq, xk, v, W):
    if (xq.ndim < 2 or xq.shape != xk.shape or xq.shape[:-1] != v.shape[:-1] or W.ndim != 2
            or W.shape[1] != xq.shape[-1]):
        raise ValueError(f"shape mismatch: xq{xq.shape} xk{xk.shape} v{v.shape} W{W.shape}")
    lead = xq.shape[:-2]
    BH = int(np.prod(lead)) if lead else 1
    return lead, BH, xq.shape[-2], xq.shape[-1], W.shape[0], v.shape[-1]


def fwd_favor(xq, xk, v, W, nthreads: int = 0) -> np.ndarray:
    """out_i = sum_{j<=i} (phi(xq_i) . phi(xk_j)) v_j with the positive random
    features phi(x)_d = exp(w_d . x - |x|^2 / 2) / sqrt(D), evaluated in fp64.
    xq, xk: [..., N, r]; W: [D, r] (one projection for every slice);
    v: [..., N, M]."""
    xq, xk, v, W = _as_f32(xq), _as_f32(xk), _as_f32(v), _as_f32(W)
    lead, BH, N, r, D, M = _favor_dims(xq, xk, v, W)
    out = np.zeros(lead + (N, M), dtype=np.float64)
    rc = _load().cpo_fwd_favor(xq.ctypes.data, xk.ctypes.data, v.ctypes.data, W.ctypes.data,
                               out.ctypes.data, BH, N, r, D, M, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle fwd_favor failed ({rc})")
    return out


def bwd_favor(xq, xk, v, W, g, nthreads: int = 0):
    """(dxq, dxk, dv) of L = <g, out> for fwd_favor, with respect to xq, xk
    and v (W is fixed), in fp64."""
    xq, xk, v, W, g = _as_f32(xq), _as_f32(xk), _as_f32(v), _as_f32(W), _as_f32(g)
    lead, BH, N, r, D, M = _favor_dims(xq, xk, v, W)
    if g.shape != v.shape:
        raise ValueError(f"grad shape {g.shape} != out shape {v.shape}")
    dxq = np.zeros(lead + (N, r), dtype=np.float64)
    dxk = np.zeros(lead + (N, r), dtype=np.float64)
    dv = np.zeros(lead + (N, M), dtype=np.float64)
    rc = _load().cpo_bwd_favor(xq.ctypes.data, xk.ctypes.data, v.ctypes.data, W.ctypes.data,
                               g.ctypes.data, dxq.ctypes.data, dxk.ctypes.data, dv.ctypes.data,
                               BH, N, r, D, M, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle bwd_favor failed ({rc})")
    return dxq, dxk, dv


def _favor_qk_dims(xq, xk, W):
    if xq.ndim < 2 or xq.shape != xk.shape or W.ndim != 2 or W.shape[1] != xq.shape[-1]:
        raise ValueError(f"shape mismatch: xq{xq.shape} xk{xk.shape} W{W.shape}")
    lead = xq.shape[:-2]
    BH = int(np.prod(lead)) if lead else 1
    return lead, BH, xq.shape[-2], xq.shape[-1], W.shape[0]


def norm_favor(xq, xk, W, nthreads: int = 0) -> np.ndarray:
    """z_i = phi(xq_i) . sum_{j<=i} phi(xk_j) with the positive random
    features of fwd_favor, in fp64."""
    xq, xk, W = _as_f32(xq), _as_f32(xk), _as_f32(W)
    lead, BH, N, r, D = _favor_qk_dims(xq, xk, W)
    z = np.zeros(lead + (N,), dtype=np.float64)
    rc = _load().cpo_norm_favor(xq.ctypes.data, xk.ctypes.data, W.ctypes.data, z.ctypes.data,
                                BH, N, r, D, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle norm_favor failed ({rc})")
    return z


def norm_bwd_favor(xq, xk, W, g, nthreads: int = 0):
    """(dxq, dxk) of L = sum_i g_i z_i for norm_favor (W fixed), in fp64."""
    xq, xk, W, g = _as_f32(xq), _as_f32(xk), _as_f32(W), _as_f32(g)
    lead, BH, N, r, D = _favor_qk_dims(xq, xk, W)
    if g.shape != lead + (N,):
        raise ValueError(f"grad shape {g.shape} != z shape {lead + (N,)}")
    dxq = np.zeros(lead + (N, r), dtype=np.float64)
    dxk = np.zeros(lead + (N, r), dtype=np.float64)
    rc = _load().cpo_norm_bwd_favor(xq.ctypes.data, xk.ctypes.data, W.ctypes.data, g.ctypes.data,
                                    dxq.ctypes.data, dxk.ctypes.data, BH, N, r, D, int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle norm_bwd_favor failed ({rc})")
    return dxq, dxk
