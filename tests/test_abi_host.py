"""Host-side checks of the C ABI library (no GPU needed).

The library must load, export every function include/causal_product.h
declares, and reject bad arguments before it touches the device.  Only
calls that return before any CUDA work are made here.
"""
import ctypes
import os
import re

import pytest

import prefix_sum_outer_gb300 as cp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")

F32, BF16 = 0, 1
(OK, INVALID_ARG, UNSUPPORTED_SHAPE, UNSUPPORTED_DTYPE, MISALIGNED, WS_TOO_SMALL, CUDA_ERR,
 TIMEOUT, NO_DEVICE) = range(9)


def declared_functions():
    names = set()
    for fname in os.listdir(HEADER_DIR):
        if not fname.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fname)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(causal_product\w*)\s*\(", text, re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    return cp.load_library()


def test_header_declares_entry_points():
    names = declared_functions()
    for required in ("causal_product_fwd", "causal_product_bwd", "causal_product_workspace_size",
                     "causal_product_status", "causal_product_error_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_library_is_in_tree(lib):
    path = cp.library_path()
    assert os.path.exists(path)
    assert os.path.commonpath([os.path.abspath(path), ROOT]) == ROOT


def test_error_strings(lib):
    for code in range(9):
        s = cp.causal_product_error_string(code)
        assert s and isinstance(s, str)
    assert cp.causal_product_error_string(0) == "CP_OK"
    assert "unknown" in cp.causal_product_error_string(99)


def test_workspace_size(lib):
    ws = lib.causal_product_workspace_size
    # large batch x heads: one segment per problem, status word only
    assert ws(8, 16, 4096, 64, 64, BF16, 0) == 256
    assert ws(8, 16, 4096, 64, 64, BF16, 1) == 256
    # few long problems: split into segments, aggregates needed
    n = ws(2, 8, 32768, 128, 128, BF16, 1)
    assert n > 256 and n % 256 == 0
    assert ws(4, 8, 8229, 256, 64, BF16, 1) > 256
    assert ws(1, 2, 64, 16, 16, F32, 0) >= 256
    # rejected shapes give 0
    assert ws(1, 1, 16, 0, 16, F32, 0) == 0
    assert ws(1, 1, 16, 16, 300, F32, 0) == 0
    assert ws(1, 1, 16, 12, 16, BF16, 0) == 0
    assert ws(0, 1, 16, 16, 16, F32, 0) == 0
    assert ws(1, 1, -1, 16, 16, F32, 0) == 0
    assert ws(1, 1, 16, 16, 16, 5, 0) == 0


def test_launch_count(lib):
    """The plan's launch counts for the five workloads (152 SMs when no GPU
    is present, as on the target part)."""
    import torch
    if torch.cuda.is_available():
        n_sm = torch.cuda.get_device_properties(0).multi_processor_count
        if n_sm != 152:
            pytest.skip("counts below are for a 152-SM device")
    lc = lib.causal_product_launch_count
    # B=8 H=16 N=4096 D=M=64: 128 unsplit problems, fwd 1 launch, the
    # whole backward in 1
    assert lc(8, 16, 4096, 64, 64, BF16, 0) == 1
    assert lc(8, 16, 4096, 64, 64, BF16, 1) == 1
    # 16 problems of 32768 rows: every scan split (sums, prefix, scan),
    # three products in the backward, dk seeded from dv's segment prefixes
    # (one launch); with checkpoints dq is one seeded launch
    assert lc(2, 8, 32768, 128, 128, BF16, 0) == 3
    assert lc(2, 8, 32768, 128, 128, BF16, 1) == 7
    assert lc(2, 8, 32768, 128, 128, BF16, 2) == 3
    assert lc(2, 8, 32768, 128, 128, BF16, 3) == 5
    assert lc(4, 8, 8229, 256, 64, BF16, 0) == 3
    assert lc(4, 8, 8229, 256, 64, BF16, 1) == 7
    assert lc(4, 8, 8229, 256, 64, BF16, 3) == 5
    assert lc(8, 16, 4096, 64, 64, BF16, 3) == 1
    # the forward with the normaliser: one launch on the fused shapes, else
    # the product and the normaliser kernel
    assert lc(8, 16, 4096, 64, 64, BF16, 4) == 1
    assert lc(2, 8, 32768, 128, 128, BF16, 4) == 4
    assert lc(8, 16, 4096, 64, 64, BF16, 5) == -1
    # fp32: 32 problems of 32 tiles split 16 ways; one 64-row tile unsplit
    assert lc(4, 8, 1024, 64, 64, F32, 0) == 3
    assert lc(4, 8, 1024, 64, 64, F32, 1) == 9
    assert lc(1, 2, 64, 16, 16, F32, 0) == 1
    assert lc(1, 2, 64, 16, 16, F32, 1) == 3
    # bf16 D = M = 64 split: dq product (3), reverse sums + prefix, dk/dv scan;
    # with checkpoints dq is one seeded launch
    assert lc(1, 2, 8192, 64, 64, BF16, 1) == 6
    assert lc(1, 2, 8192, 64, 64, BF16, 3) == 4
    # many problems: fused dk/dv scan on its own launch after dq
    assert lc(16, 16, 1024, 64, 64, BF16, 1) == 2
    assert lc(1, 1, 0, 64, 64, BF16, 1) == 0
    assert lc(1, 1, 16, 12, 16, BF16, 0) == -1


A = 1 << 20  # a 16-byte-aligned fake device address; never dereferenced here


def fwd(lib, q=A, k=2 * A, v=3 * A, out=4 * A, B=1, H=1, N=16, D=16, M=16, dtype=F32,
        ws=None, ws_bytes=0):
    return lib.causal_product_fwd(q, k, v, out, B, H, N, D, M, dtype, ws, ws_bytes, None)


def test_checkpoint_calls(lib):
    """Checkpoint sizes and the argument checks of the checkpoint calls."""
    size = lib.causal_product_checkpoint_size
    # split dq (16 problems of 256 tiles, 9 segments): 8 checkpoints of D x M
    assert size(2, 8, 32768, 128, 128, BF16) == 4 * 16 * 8 * 128 * 128
    # the one-launch backward keeps whole dq scans; fp32 has none; rejects: 0
    assert size(8, 16, 4096, 64, 64, BF16) == 0
    assert size(1, 2, 8192, 64, 64, F32) == 0
    assert size(1, 1, 16, 12, 16, BF16) == 0
    n = size(1, 2, 8192, 64, 64, BF16)
    assert n > 0 and n % (4 * 2 * 64 * 64) == 0
    fck, bck = lib.causal_product_fwd_ckpt, lib.causal_product_bwd_ckpt
    args = (1, 2, 8192, 64, 64, BF16, None, 0, None)
    assert fck(A, 2 * A, 3 * A, 4 * A, None, 0, *args) == INVALID_ARG
    assert fck(A, 2 * A, 3 * A, 4 * A, 5 * A, n - 16, *args) == WS_TOO_SMALL
    assert fck(A, 2 * A, 3 * A, 4 * A, 5 * A + 4, n, *args) == MISALIGNED
    # the checkpoints may not overlap the output
    assert fck(A, 2 * A, 3 * A, 4 * A, 4 * A + 64, n, *args) == INVALID_ARG
    assert bck(A, 2 * A, 3 * A, 4 * A, None, 0, 5 * A, 6 * A, 7 * A, *args) == INVALID_ARG
    assert bck(A, 2 * A, 3 * A, 4 * A, 8 * A, n - 16, 5 * A, 6 * A, 7 * A, *args) == WS_TOO_SMALL
    # ... nor a gradient
    assert bck(A, 2 * A, 3 * A, 4 * A, 5 * A, n, 5 * A, 6 * A, 7 * A, *args) == INVALID_ARG
    # without rows nothing is needed
    assert fck(A, 2 * A, 3 * A, 4 * A, None, 0, 1, 2, 0, 64, 64, BF16, None, 0, None) == OK


def test_fwd_argument_checks(lib):
    assert fwd(lib, q=None) == INVALID_ARG
    assert fwd(lib, out=None) == INVALID_ARG
    assert fwd(lib, B=0) == INVALID_ARG
    assert fwd(lib, N=-3) == INVALID_ARG
    assert fwd(lib, D=0) == UNSUPPORTED_SHAPE
    assert fwd(lib, M=257) == UNSUPPORTED_SHAPE
    assert fwd(lib, D=12, dtype=BF16) == UNSUPPORTED_SHAPE
    assert fwd(lib, dtype=9) == UNSUPPORTED_DTYPE
    assert fwd(lib, q=A + 4) == MISALIGNED
    assert fwd(lib, out=4 * A + 8) == MISALIGNED
    # out overlapping an input
    assert fwd(lib, out=A + 256) == INVALID_ARG
    # caller workspace too small
    assert fwd(lib, ws=8 * A, ws_bytes=16) == WS_TOO_SMALL
    # N = 0: nothing to do, nothing touched
    assert fwd(lib, N=0) == OK


def test_bwd_argument_checks(lib):
    def bwd(**kw):
        args = dict(q=A, k=2 * A, v=3 * A, g=4 * A, dq=5 * A, dk=6 * A, dv=7 * A, B=1, H=1, N=16,
                    D=16, M=16, dtype=F32, ws=None, ws_bytes=0)
        args.update(kw)
        return lib.causal_product_bwd(args["q"], args["k"], args["v"], args["g"], args["dq"],
                                      args["dk"], args["dv"], args["B"], args["H"], args["N"],
                                      args["D"], args["M"], args["dtype"], args["ws"],
                                      args["ws_bytes"], None)
    assert bwd(g=None) == INVALID_ARG
    assert bwd(dk=None) == INVALID_ARG
    assert bwd(dv=7 * A + 2) == MISALIGNED
    assert bwd(dq=A) == INVALID_ARG            # grad aliases q
    assert bwd(dk=5 * A) == INVALID_ARG        # two grads alias
    assert bwd(D=20, dtype=BF16) == UNSUPPORTED_SHAPE
    assert bwd(ws=8 * A, ws_bytes=1) == WS_TOO_SMALL
    assert bwd(N=0) == OK


def test_python_binding_refuses_cpu_tensors():
    """Every compute entry point of the binding refuses host tensors with an
    error: there is no CPU path to fall back to."""
    import torch
    q = torch.ones(1, 1, 4, 16)
    z = torch.ones(1, 1, 4)
    q1 = torch.ones(1, 1, 16)
    st = torch.zeros(1, 1, 16, 16)
    calls = [
        lambda: cp.causal_product_fwd(q, q, q),
        lambda: cp.causal_product_bwd(q, q, q, q),
        lambda: cp.causal_product_fwd_noalloc(q, q, q, torch.empty_like(q)),
        lambda: cp.causal_product_fwd_feature(q, q, q),
        lambda: cp.causal_product_bwd_feature(q, q, q, q),
        lambda: cp.causal_product_normalizer(q, q),
        lambda: cp.causal_product_normalizer_bwd(q, q, z),
        lambda: cp.causal_product_decode(q1, q1, q1, st),
        lambda: cp.causal_product(q, q, q),
        lambda: cp.normalizer(q, q),
    ]
    for call in calls:
        with pytest.raises(RuntimeError, match="CUDA tensors only"):
            call()


def test_python_binding_refuses_misshaped_outputs():
    """A caller's output buffer must match the shape and dtype the kernels
    write; the C ABI only sees its pointer, so the binding checks it before
    anything else (here on host tensors, which are refused later anyway)."""
    import torch
    q = torch.ones(1, 1, 4, 16)
    short = torch.empty(1, 1, 3, 16)
    wrong = torch.empty(1, 1, 4, 16, dtype=torch.float16)
    z = torch.ones(1, 1, 4)
    q1 = torch.ones(1, 1, 16)
    st = torch.zeros(1, 1, 16, 16)
    calls = [
        lambda: cp.causal_product_fwd(q, q, q, out=short),
        lambda: cp.causal_product_fwd(q, q, q, out=wrong),
        lambda: cp.causal_product_fwd_noalloc(q, q, q, short),
        lambda: cp.causal_product_fwd_feature(q, q, q, out=short),
        lambda: cp.causal_product_bwd(q, q, q, q, grad_q=short),
        lambda: cp.causal_product_bwd(q, q, q, q, grad_k=short),
        lambda: cp.causal_product_bwd(q, q, q, q, grad_v=wrong),
        lambda: cp.causal_product_bwd_feature(q, q, q, q, grad_v=short),
        lambda: cp.causal_product_normalizer_bwd(q, q, z, grad_k=short),
        lambda: cp.causal_product_decode(q1, q1, q1, st, out=torch.empty(1, 1, 8)),
    ]
    for call in calls:
        with pytest.raises(ValueError):
            call()


def test_state_argument_checks(lib):
    def fwd_state(**kw):
        args = dict(q=A, k=2 * A, v=3 * A, out=4 * A, s_in=None, s_out=None, B=1, H=1, N=16,
                    D=16, M=16, dtype=F32)
        args.update(kw)
        return lib.causal_product_fwd_state(args["q"], args["k"], args["v"], args["out"],
                                            args["s_in"], args["s_out"], args["B"], args["H"],
                                            args["N"], args["D"], args["M"], args["dtype"],
                                            None, 0, None)
    assert fwd_state(s_in=5 * A + 4) == MISALIGNED
    assert fwd_state(s_out=5 * A + 8) == MISALIGNED
    # the final state may not overlap an input, the output or the initial state
    assert fwd_state(s_out=A + 64) == INVALID_ARG
    assert fwd_state(s_out=4 * A + 64) == INVALID_ARG
    assert fwd_state(s_in=5 * A, s_out=5 * A + 256) == INVALID_ARG
    # the output may not overlap the initial state
    assert fwd_state(s_in=4 * A + 512) == INVALID_ARG
    assert fwd_state(N=0) == OK

    def bwd_state(**kw):
        args = dict(q=A, k=2 * A, v=3 * A, g=4 * A, s_in=None, gs_out=None, dq=5 * A, dk=6 * A,
                    dv=7 * A, gs_in=None, B=1, H=1, N=16, D=16, M=16, dtype=F32)
        args.update(kw)
        return lib.causal_product_bwd_state(args["q"], args["k"], args["v"], args["g"],
                                            args["s_in"], args["gs_out"], args["dq"], args["dk"],
                                            args["dv"], args["gs_in"], args["B"], args["H"],
                                            args["N"], args["D"], args["M"], args["dtype"],
                                            None, 0, None)
    assert bwd_state(gs_in=8 * A + 4) == MISALIGNED
    assert bwd_state(s_in=8 * A + 12) == MISALIGNED
    # dL/dS_0 may not overlap a gradient or any input state
    assert bwd_state(gs_in=5 * A + 16) == INVALID_ARG
    assert bwd_state(s_in=8 * A, gs_in=8 * A + 32) == INVALID_ARG
    assert bwd_state(gs_out=8 * A, gs_in=8 * A) == INVALID_ARG
    # a gradient may not overlap an input state
    assert bwd_state(s_in=6 * A + 128) == INVALID_ARG
    assert bwd_state(N=0) == OK


def test_decode_argument_checks(lib):
    def dec(**kw):
        args = dict(q=A, k=2 * A, v=3 * A, out=4 * A, st=5 * A, B=1, H=1, D=16, M=16, dtype=F32)
        args.update(kw)
        return lib.causal_product_decode(args["q"], args["k"], args["v"], args["out"], args["st"],
                                         args["B"], args["H"], args["D"], args["M"],
                                         args["dtype"], None)
    assert dec(st=None) == INVALID_ARG
    assert dec(q=None) == INVALID_ARG
    assert dec(st=5 * A + 4) == MISALIGNED
    assert dec(D=12, dtype=BF16) == UNSUPPORTED_SHAPE
    assert dec(M=300) == UNSUPPORTED_SHAPE
    assert dec(dtype=7) == UNSUPPORTED_DTYPE
    # the state or the output may not overlap an input or each other
    assert dec(st=A + 32) == INVALID_ARG
    assert dec(out=3 * A + 16) == INVALID_ARG
    assert dec(out=5 * A + 64) == INVALID_ARG


def test_selftest_argument_checks(lib):
    st = lib.causal_product_selftest_timeout
    assert st(None, 1000, None) == INVALID_ARG
    assert st(A + 8, 1000, None) == MISALIGNED
    assert st(A, 0, None) == INVALID_ARG
    assert st(A, 2_000_000_000, None) == INVALID_ARG


def test_normalizer_argument_checks(lib):
    ws = lib.causal_product_normalizer_workspace_size
    assert ws(8, 16, 4096, 64, BF16) >= 256 and ws(8, 16, 4096, 64, BF16) % 256 == 0
    assert ws(1, 1, 65536, 64, BF16) > 256      # few long problems: segment sums
    assert ws(8, 16, 0, 64, BF16) == 256
    assert ws(0, 16, 4096, 64, BF16) == 0
    assert ws(1, 1, 16, 12, BF16) == 0
    assert ws(1, 1, 16, 257, F32) == 0

    def fwd(**kw):
        a = dict(q=A, k=2 * A, z=3 * A, B=1, H=2, N=64, D=16, dtype=F32, ws=None, wsb=0)
        a.update(kw)
        return lib.causal_product_normalizer(a["q"], a["k"], a["z"], a["B"], a["H"], a["N"],
                                             a["D"], a["dtype"], a["ws"], a["wsb"], None)

    assert fwd(z=None) == INVALID_ARG
    assert fwd(q=A + 8) == MISALIGNED
    assert fwd(D=0) == UNSUPPORTED_SHAPE
    assert fwd(D=12, dtype=BF16) == UNSUPPORTED_SHAPE
    assert fwd(dtype=3) == UNSUPPORTED_DTYPE
    assert fwd(B=-1) == INVALID_ARG
    assert fwd(z=A + 64) == INVALID_ARG                 # z inside q
    assert fwd(ws=8 * A, wsb=16) == WS_TOO_SMALL
    assert fwd(N=0) == OK and fwd(N=0, q=None, k=None, z=None) == OK

    def bwd(**kw):
        a = dict(q=A, k=2 * A, g=3 * A, dq=4 * A, dk=5 * A, B=1, H=2, N=64, D=16, dtype=F32)
        a.update(kw)
        return lib.causal_product_normalizer_bwd(a["q"], a["k"], a["g"], a["dq"], a["dk"],
                                                 a["B"], a["H"], a["N"], a["D"], a["dtype"],
                                                 None, 0, None)

    assert bwd(dk=None) == INVALID_ARG
    assert bwd(g=3 * A + 4) == MISALIGNED
    assert bwd(D=300) == UNSUPPORTED_SHAPE
    assert bwd(dq=5 * A) == INVALID_ARG                 # dq and dk alias
    assert bwd(dk=3 * A + 16) == INVALID_ARG            # dk over grad_z
    assert bwd(dq=2 * A + 32) == INVALID_ARG            # dq over k
    assert bwd(N=0) == OK


def test_feature_argument_checks(lib):
    ws = lib.causal_product_feature_workspace_size
    plain_f = lib.causal_product_workspace_size(8, 16, 4096, 64, 64, BF16, 0)
    plain_b = lib.causal_product_workspace_size(8, 16, 4096, 64, 64, BF16, 1)
    assert ws(8, 16, 4096, 64, 64, BF16, 0) == plain_f
    # bf16 maps inside the product kernels: the plain backward's workspace
    assert ws(8, 16, 4096, 64, 64, BF16, 1) == plain_b
    # fp32 and fp16 keep phi(q) and phi(k) next to the backward's workspace
    plain_b32 = lib.causal_product_workspace_size(8, 16, 4096, 64, 64, F32, 1)
    assert ws(8, 16, 4096, 64, 64, F32, 1) == plain_b32 + 2 * 8 * 16 * 4096 * 64 * 4
    assert ws(8, 16, 4096, 12, 64, BF16, 1) == 0

    def fwd(**kw):
        a = dict(q=A, k=2 * A, v=3 * A, out=4 * A, feat=1, B=1, H=2, N=64, D=16, M=16, dtype=F32)
        a.update(kw)
        return lib.causal_product_fwd_feature(a["q"], a["k"], a["v"], a["out"], a["feat"], a["B"],
                                              a["H"], a["N"], a["D"], a["M"], a["dtype"], None, 0,
                                              None)

    assert fwd(feat=7) == INVALID_ARG
    assert fwd(q=A + 4) == MISALIGNED
    assert fwd(out=2 * A + 64) == INVALID_ARG          # out over k
    assert fwd(D=12, dtype=BF16) == UNSUPPORTED_SHAPE
    assert fwd(N=0) == OK

    def bwd(**kw):
        a = dict(q=A, k=2 * A, v=3 * A, g=4 * A, dq=5 * A, dk=6 * A, dv=7 * A, feat=1, B=1, H=2,
                 N=64, D=16, M=16, dtype=F32, ws=None, wsb=0)
        a.update(kw)
        return lib.causal_product_bwd_feature(a["q"], a["k"], a["v"], a["g"], a["dq"], a["dk"],
                                              a["dv"], a["feat"], a["B"], a["H"], a["N"], a["D"],
                                              a["M"], a["dtype"], a["ws"], a["wsb"], None)

    assert bwd(feat=7) == INVALID_ARG
    assert bwd(dq=None) == INVALID_ARG
    assert bwd(k=2 * A + 8) == MISALIGNED
    assert bwd(dq=A + 256) == INVALID_ARG              # dq over q
    assert bwd(dk=5 * A) == INVALID_ARG                # dq and dk alias
    assert bwd(ws=8 * A, wsb=1024) == WS_TOO_SMALL
    assert bwd(N=0) == OK


def test_f16_dtype_checks(lib):
    F16 = 2
    # fp16 runs on the fp32 path: any D, M in [1, 256]
    assert lib.causal_product_workspace_size(1, 2, 64, 12, 7, F16, 1) >= 256
    assert lib.causal_product_workspace_size(1, 2, 64, 257, 7, F16, 0) == 0
    # the normaliser moves 16-bit rows in 16-byte vectors
    assert lib.causal_product_normalizer_workspace_size(1, 2, 64, 16, F16) >= 256
    assert lib.causal_product_normalizer_workspace_size(1, 2, 64, 12, F16) == 0
    assert lib.causal_product_fwd(A, 2 * A, 3 * A, 4 * A, 1, 1, 64, 16, 16, 3, None, 0,
                                  None) == UNSUPPORTED_DTYPE


def test_normalizer_feature_argument_checks(lib):
    f = lib.causal_product_normalizer_feature
    args = lambda **kw: dict(dict(q=A, k=2 * A, z=3 * A, feat=1, B=1, H=2, N=64, D=16, dtype=F32), **kw)

    def call(**kw):
        a = args(**kw)
        return f(a["q"], a["k"], a["z"], a["feat"], a["B"], a["H"], a["N"], a["D"], a["dtype"],
                 None, 0, None)

    assert call(feat=5) == INVALID_ARG
    assert call(D=7) == UNSUPPORTED_SHAPE        # fp32 rows of 28 bytes: no feature map
    assert call(N=0) == OK
    assert call(N=0, D=7, feat=0) == OK          # the plain normaliser takes any fp32 D
    b = lib.causal_product_normalizer_bwd_feature
    assert b(A, 2 * A, 3 * A, 4 * A, 5 * A, 5, 1, 2, 64, 16, F32, None, 0, None) == INVALID_ARG
    assert b(A, 2 * A, 3 * A, 4 * A, 5 * A, 1, 1, 2, 64, 12, BF16, None, 0, None) == UNSUPPORTED_SHAPE


def test_launch_count_one_launch_split_scan(lib, monkeypatch):
    """CP_SPLIT_SCAN=lookback: a bf16 forward split scan whose grid fits the
    SMs is one launch (each segment's sum, its prefix, its scan); reverse
    scans keep three."""
    import torch
    if torch.cuda.is_available() and torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("counts below are for a 152-SM device")
    lc = lib.causal_product_launch_count
    monkeypatch.setenv("CP_SPLIT_SCAN", "lookback")
    assert lc(2, 8, 32768, 128, 128, BF16, 0) == 1
    assert lc(2, 8, 32768, 128, 128, BF16, 2) == 1
    # backward: dq (forward, one launch), dv (reverse, three), dk seeded (one)
    assert lc(2, 8, 32768, 128, 128, BF16, 1) == 5
    assert lc(4, 8, 8229, 256, 64, BF16, 0) == 1
    assert lc(1, 2, 8192, 64, 64, BF16, 1) == 4
    # fp32 keeps its two passes
    assert lc(4, 8, 1024, 64, 64, F32, 0) == 3
    monkeypatch.setenv("CP_SPLIT_SCAN", "twopass")
    assert lc(2, 8, 32768, 128, 128, BF16, 0) == 3
