"""Pins for the causal-product oracle.

Each pin checks an implementation ``impl`` (an object with ``fwd(q,k,v)``,
``bwd(q,k,v,g)``, ``fwd_state(q,k,v,s0)``, ``bwd_state(q,k,v,g,s0,ds_n)``,
``norm(q,k)``, ``norm_bwd(q,k,g)``, ``fwd_feature(q,k,v)``,
``bwd_feature(q,k,v,g)``, ``norm_feature(q,k)``, ``norm_bwd_feature(q,k,g)``,
``fwd_favor(xq,xk,v,W)``, ``bwd_favor(xq,xk,v,W,g)``, ``norm_favor(xq,xk,W)``
and ``norm_bwd_favor(xq,xk,W,g)`` returning float64 numpy arrays, like
``oracle``)
against something other than the recurrence itself: hand-worked values,
a brute-force quadratic form, closed forms, textbook special cases,
linearity, causality and finite differences.  ``tests/test_oracle.py``
runs them on the oracle; ``tests/test_oracle_mutants.py`` checks that each
planted mistake in a copy of the oracle trips at least one of them.

Every pin raises AssertionError on failure.
"""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "hand_examples.json")


def _rng(seed):
    return np.random.default_rng(seed)


def _pos(rng, shape):
    """elu(x)+1 features drawn in float32 (positive, like the workloads)."""
    x = rng.standard_normal(shape).astype(np.float32)
    return np.where(x > 0, x + 1, np.exp(x)).astype(np.float32)


def _dyadic(rng, shape, lo=-4, hi=4, denom=16):
    """Values k/denom in [lo, hi]: exact in float32, and sums of their
    products are exact in float64 for the small shapes used here."""
    return (rng.integers(lo * denom, hi * denom + 1, size=shape) / denom).astype(np.float32)


def _rel(a, b):
    scale = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / scale)


# --------------------------------------------------------------------------
# forward pins
# --------------------------------------------------------------------------

def pin_golden(impl):
    """Hand-worked examples in tests/golden/hand_examples.json."""
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = np.array(c["q"], np.float32)[None]
        k = np.array(c["k"], np.float32)[None]
        v = np.array(c["v"], np.float32)[None]
        out = impl.fwd(q, k, v)[0]
        assert np.array_equal(out, np.array(c["out"], np.float64)), (c["name"], out)
        if "g" in c:
            g = np.array(c["g"], np.float32)[None]
            dq, dk, dv = impl.bwd(q, k, v, g)
            for name, got in (("dq", dq), ("dk", dk), ("dv", dv)):
                assert np.array_equal(got[0], np.array(c[name], np.float64)), (c["name"], name, got[0])


def brute_force_fwd(q, k, v):
    """(Q K^T masked to j <= i) V, in float64 -- quadratic, no recurrence."""
    q, k, v = (np.asarray(t, np.float64) for t in (q, k, v))
    N = q.shape[-2]
    A = q @ np.swapaxes(k, -1, -2)
    A = A * np.tril(np.ones((N, N)))
    return A @ v


def brute_force_bwd(q, k, v, g):
    """Matrix-calculus form of the gradient of <g, (QK^T * tril) V>."""
    q, k, v, g = (np.asarray(t, np.float64) for t in (q, k, v, g))
    N = q.shape[-2]
    L = np.tril(np.ones((N, N)))
    T = lambda x: np.swapaxes(x, -1, -2)
    GV = (g @ T(v)) * L          # [i, j] = g_i . v_j for j <= i
    QK = (q @ T(k)) * L          # [i, j] = q_i . k_j for j <= i
    return GV @ k, T(GV) @ q, T(QK) @ g


def pin_brute_force(impl, shapes=((1, 1, 1, 1, 1), (2, 2, 17, 16, 16), (1, 3, 64, 8, 5),
                                  (2, 1, 33, 3, 12))):
    for s, (B, H, N, D, M) in enumerate(shapes):
        rng = _rng(100 + s)
        q, k = _pos(rng, (B, H, N, D)), _pos(rng, (B, H, N, D))
        v = rng.standard_normal((B, H, N, M)).astype(np.float32)
        got = impl.fwd(q, k, v)
        ref = brute_force_fwd(q, k, v)
        assert got.shape == ref.shape
        assert _rel(got, ref) <= 1e-12, ("brute force", (B, H, N, D, M), _rel(got, ref))


def pin_first_row_closed_form(impl):
    """out_0 = (q_0 . k_0) v_0."""
    rng = _rng(7)
    q, k = _pos(rng, (2, 3, 9, 6)), _pos(rng, (2, 3, 9, 6))
    v = rng.standard_normal((2, 3, 9, 4)).astype(np.float32)
    out = impl.fwd(q, k, v)
    qk = np.sum(q[..., 0, :].astype(np.float64) * k[..., 0, :], axis=-1)
    ref = qk[..., None] * v[..., 0, :].astype(np.float64)
    assert np.allclose(out[..., 0, :], ref, rtol=1e-14, atol=0), "first row"


def pin_last_row_is_noncausal(impl):
    """out_{N-1} = q_{N-1}^T (K^T V): the last row sees every key, so it is
    non-causal linear attention, a plain matrix product."""
    rng = _rng(8)
    q, k = _pos(rng, (1, 2, 40, 7)), _pos(rng, (1, 2, 40, 7))
    v = rng.standard_normal((1, 2, 40, 5)).astype(np.float32)
    out = impl.fwd(q, k, v)
    KV = np.einsum("bhnd,bhnm->bhdm", k.astype(np.float64), v.astype(np.float64))
    ref = np.einsum("bhd,bhdm->bhm", q[..., -1, :].astype(np.float64), KV)
    assert _rel(out[..., -1, :], ref) <= 1e-12, "last row"


def pin_scalar_cumsum(impl):
    """D = M = 1: out = q * cumsum(k * v), a textbook prefix sum."""
    rng = _rng(9)
    q = rng.standard_normal((3, 2, 50, 1)).astype(np.float32)
    k = rng.standard_normal((3, 2, 50, 1)).astype(np.float32)
    v = rng.standard_normal((3, 2, 50, 1)).astype(np.float32)
    out = impl.fwd(q, k, v)
    ref = q.astype(np.float64) * np.cumsum(k.astype(np.float64) * v, axis=-2)
    assert _rel(out, ref) <= 1e-13, "D=M=1 cumsum"


def pin_ones_cumsum(impl):
    """q = k = 1: out_i = D * sum_{j<=i} v_j."""
    rng = _rng(10)
    D = 6
    q = np.ones((1, 2, 30, D), np.float32)
    v = rng.standard_normal((1, 2, 30, 4)).astype(np.float32)
    out = impl.fwd(q, q.copy(), v)
    ref = D * np.cumsum(v.astype(np.float64), axis=-2)
    assert _rel(out, ref) <= 1e-13, "q=k=1 cumsum"


def pin_zero_value(impl):
    """v = 0 gives exactly 0 in every column (column 0 included)."""
    rng = _rng(11)
    q, k = _pos(rng, (1, 2, 20, 4)), _pos(rng, (1, 2, 20, 4))
    v = np.zeros((1, 2, 20, 4), np.float32)
    assert np.all(impl.fwd(q * 100, k, v) == 0.0), "v=0"
    assert np.all(impl.fwd(q, k * 0, _pos(rng, (1, 2, 20, 4))) == 0.0), "k=0"


def pin_linearity(impl):
    """Linear in v and in q (dyadic inputs and scalars keep it exact)."""
    rng = _rng(12)
    q, k = _dyadic(rng, (1, 2, 24, 5)), _dyadic(rng, (1, 2, 24, 5))
    v1, v2 = _dyadic(rng, (1, 2, 24, 3)), _dyadic(rng, (1, 2, 24, 3))
    a, b = 0.5, -2.0
    lhs = impl.fwd(q, k, (a * v1 + b * v2).astype(np.float32))
    rhs = a * impl.fwd(q, k, v1) + b * impl.fwd(q, k, v2)
    assert np.allclose(lhs, rhs, rtol=1e-13, atol=1e-13), "linear in v"
    q2 = _dyadic(rng, (1, 2, 24, 5))
    lhs = impl.fwd((a * q + b * q2).astype(np.float32), k, v1)
    rhs = a * impl.fwd(q, k, v1) + b * impl.fwd(q2, k, v1)
    assert np.allclose(lhs, rhs, rtol=1e-13, atol=1e-13), "linear in q"


def pin_causality(impl):
    """Changing k_j, v_j for j > i leaves out_i bitwise unchanged, and
    changing q_j leaves every other row unchanged."""
    rng = _rng(13)
    N, cut = 32, 19
    q, k = _pos(rng, (1, 1, N, 4)), _pos(rng, (1, 1, N, 4))
    v = rng.standard_normal((1, 1, N, 3)).astype(np.float32)
    base = impl.fwd(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[..., cut + 1:, :] = _pos(rng, k2[..., cut + 1:, :].shape)
    v2[..., cut + 1:, :] = rng.standard_normal(v2[..., cut + 1:, :].shape)
    pert = impl.fwd(q, k2, v2)
    assert np.array_equal(base[..., :cut + 1, :], pert[..., :cut + 1, :]), "future leaked"
    assert not np.array_equal(base[..., cut + 1:, :], pert[..., cut + 1:, :]), "future ignored"
    q3 = q.copy()
    q3[..., cut, :] += 1.0
    pert = impl.fwd(q3, k, v)
    mask = np.ones(N, bool)
    mask[cut] = False
    assert np.array_equal(base[..., mask, :], pert[..., mask, :]), "q_i leaked to other rows"


# --------------------------------------------------------------------------
# backward pins
# --------------------------------------------------------------------------

def pin_finite_differences(impl, shape=(1, 2, 7, 3, 2)):
    """dL/dx for L = <g, out> by central differences in every coordinate.

    out is linear in each of q, k and v separately, so the central
    difference with any step is exact up to rounding; dyadic inputs and a
    unit step make it exact in float64.
    """
    B, H, N, D, M = shape
    rng = _rng(14)
    q, k = _dyadic(rng, (B, H, N, D)), _dyadic(rng, (B, H, N, D))
    v, g = _dyadic(rng, (B, H, N, M)), _dyadic(rng, (B, H, N, M))
    dq, dk, dv = impl.bwd(q, k, v, g)
    g64 = g.astype(np.float64)

    def loss(qq, kk, vv):
        return float(np.sum(impl.fwd(qq, kk, vv) * g64))

    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        fd = np.zeros(x.shape, np.float64)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += 1.0
            xm[idx] -= 1.0
            args_p = {"q": q, "k": k, "v": v}
            args_m = dict(args_p)
            args_p[name], args_m[name] = xp, xm
            fd[idx] = (loss(args_p["q"], args_p["k"], args_p["v"])
                       - loss(args_m["q"], args_m["k"], args_m["v"])) / 2.0
        assert np.allclose(grad, fd, rtol=1e-12, atol=1e-12), ("finite differences", name)


def pin_bwd_brute_force(impl, shapes=((2, 2, 19, 8, 6), (1, 1, 64, 16, 16), (1, 2, 5, 1, 3))):
    for s, (B, H, N, D, M) in enumerate(shapes):
        rng = _rng(200 + s)
        q, k = _pos(rng, (B, H, N, D)), _pos(rng, (B, H, N, D))
        v = rng.standard_normal((B, H, N, M)).astype(np.float32)
        g = rng.standard_normal((B, H, N, M)).astype(np.float32)
        got = impl.bwd(q, k, v, g)
        ref = brute_force_bwd(q, k, v, g)
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert _rel(a, b) <= 1e-12, ("bwd brute force", name, (B, H, N, D, M), _rel(a, b))


def pin_bwd_identities(impl):
    """The gradients are causal products themselves:
    dQ = fwd(g, v, k); dV = flip(fwd(flip k, flip q, flip g));
    dK = flip(fwd(flip v, flip g, flip q)), flip = reverse the sequence."""
    rng = _rng(15)
    B, H, N, D, M = 1, 2, 23, 6, 4
    q, k = _pos(rng, (B, H, N, D)), _pos(rng, (B, H, N, D))
    v = rng.standard_normal((B, H, N, M)).astype(np.float32)
    g = rng.standard_normal((B, H, N, M)).astype(np.float32)
    dq, dk, dv = impl.bwd(q, k, v, g)
    f = lambda x: np.ascontiguousarray(x[..., ::-1, :])
    assert _rel(dq, impl.fwd(g, v, k)) <= 1e-13, "dq identity"
    assert _rel(dv, f(impl.fwd(f(k), f(q), f(g)))) <= 1e-13, "dv identity"
    assert _rel(dk, f(impl.fwd(f(v), f(g), f(q)))) <= 1e-13, "dk identity"


# --------------------------------------------------------------------------
# carried-state pins: impl.fwd_state(q, k, v, s0) -> (out, s_n) and
# impl.bwd_state(q, k, v, g, s0, ds_n) -> (dq, dk, dv, ds0)
# --------------------------------------------------------------------------

def _state_case(seed, shape=(1, 2, 23, 6, 4)):
    B, H, N, D, M = shape
    rng = _rng(seed)
    q, k = _pos(rng, (B, H, N, D)), _pos(rng, (B, H, N, D))
    v = rng.standard_normal((B, H, N, M)).astype(np.float32)
    g = rng.standard_normal((B, H, N, M)).astype(np.float32)
    s0 = rng.standard_normal((B, H, D, M)).astype(np.float32)
    ds_n = rng.standard_normal((B, H, D, M)).astype(np.float32)
    return q, k, v, g, s0, ds_n


def pin_state_closed_forms(impl):
    """With an initial state S_0 and a final-state gradient dS_N (numpy
    products in float64 on the right-hand sides):
      S_N = S_0 + K^T V;  out(S_0) = out(0) + Q S_0 row by row;
      dS_0 = dS_N + Q^T G;  dq(S_0) = dq(0) + G S_0^T;
      dk(dS_N) = dk(0) + V dS_N^T;  dv(dS_N) = dv(0) + K dS_N."""
    q, k, v, g, s0, ds_n = _state_case(16)
    f64 = lambda x: x.astype(np.float64)
    out, s_n = impl.fwd_state(q, k, v, s0)
    assert _rel(s_n, f64(s0) + np.einsum("bhnd,bhnm->bhdm", f64(k), f64(v))) <= 1e-12, "S_N"
    assert _rel(out, impl.fwd(q, k, v) + np.einsum("bhnd,bhdm->bhnm", f64(q), f64(s0))) <= 1e-12, \
        "out with S_0"
    dq, dk, dv, ds0 = impl.bwd_state(q, k, v, g, s0, ds_n)
    dq0, dk0, dv0 = impl.bwd(q, k, v, g)
    assert _rel(ds0, f64(ds_n) + np.einsum("bhnd,bhnm->bhdm", f64(q), f64(g))) <= 1e-12, "dS_0"
    assert _rel(dq, dq0 + np.einsum("bhnm,bhdm->bhnd", f64(g), f64(s0))) <= 1e-12, "dq with S_0"
    assert _rel(dk, dk0 + np.einsum("bhdm,bhnm->bhnd", f64(ds_n), f64(v))) <= 1e-12, "dk with dS_N"
    assert _rel(dv, dv0 + np.einsum("bhdm,bhnd->bhnm", f64(ds_n), f64(k))) <= 1e-12, "dv with dS_N"


def pin_state_chunking(impl, cut=16):
    """Splitting the sequence and handing the state on reproduces the whole
    sequence exactly: the forward runs chunk 1 then chunk 2 from its final
    state; the backward runs chunk 2 (final-state gradient dS_N) then chunk
    1 with chunk 2's dS_0 as its final-state gradient."""
    q, k, v, g, s0, ds_n = _state_case(17)
    parts = lambda x: (np.ascontiguousarray(x[..., :cut, :]), np.ascontiguousarray(x[..., cut:, :]))
    (q1, q2), (k1, k2), (v1, v2), (g1, g2) = parts(q), parts(k), parts(v), parts(g)
    out, s_n = impl.fwd_state(q, k, v, s0)
    o1, s1 = impl.fwd_state(q1, k1, v1, s0)
    o2, s2 = impl.fwd_state(q2, k2, v2, s1)
    assert np.array_equal(np.concatenate([o1, o2], axis=-2), out), "chunked out"
    assert np.array_equal(s2, s_n), "chunked S_N"
    full = impl.bwd_state(q, k, v, g, s0, ds_n)
    dq2, dk2, dv2, ds_mid = impl.bwd_state(q2, k2, v2, g2, s1, ds_n)
    dq1, dk1, dv1, ds0 = impl.bwd_state(q1, k1, v1, g1, s0, ds_mid)
    for name, a, b in (("dq", (dq1, dq2), full[0]), ("dk", (dk1, dk2), full[1]),
                       ("dv", (dv1, dv2), full[2])):
        assert np.array_equal(np.concatenate(a, axis=-2), b), ("chunked", name)
    assert np.array_equal(ds0, full[3]), "chunked dS_0"


def pin_state_finite_differences(impl, shape=(1, 1, 6, 3, 2)):
    """Central differences of L = <g, out> + <dS_N, S_N> in every coordinate
    of S_0, k and v (L is linear in each, dyadic inputs: exact)."""
    B, H, N, D, M = shape
    rng = _rng(18)
    q, k = _dyadic(rng, (B, H, N, D)), _dyadic(rng, (B, H, N, D))
    v, g = _dyadic(rng, (B, H, N, M)), _dyadic(rng, (B, H, N, M))
    s0, ds_n = _dyadic(rng, (B, H, D, M)), _dyadic(rng, (B, H, D, M))
    dq, dk, dv, ds0 = impl.bwd_state(q, k, v, g, s0, ds_n)

    def loss(kk, vv, ss):
        out, s_n = impl.fwd_state(q, kk, vv, ss)
        return float(np.sum(out * g.astype(np.float64)) + np.sum(s_n * ds_n.astype(np.float64)))

    for name, x, grad in (("k", k, dk), ("v", v, dv), ("s0", s0, ds0)):
        fd = np.zeros(x.shape, np.float64)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += 1.0
            xm[idx] -= 1.0
            args = {"k": k, "v": v, "s0": s0}
            ap, am = dict(args), dict(args)
            ap[name], am[name] = xp, xm
            fd[idx] = (loss(ap["k"], ap["v"], ap["s0"]) - loss(am["k"], am["v"], am["s0"])) / 2.0
        assert np.allclose(grad, fd, rtol=1e-12, atol=1e-12), ("state finite differences", name)


FWD_PINS = [pin_golden, pin_brute_force, pin_first_row_closed_form, pin_last_row_is_noncausal,
            pin_scalar_cumsum, pin_ones_cumsum, pin_zero_value, pin_linearity, pin_causality]
BWD_PINS = [pin_finite_differences, pin_bwd_brute_force, pin_bwd_identities]
def pin_state_token_by_token(impl, n=9):
    """Feeding the rows one at a time (N = 1 per call, the decoding step)
    and handing the state on reproduces the whole sequence exactly."""
    q, k, v, g, s0, ds_n = _state_case(19, shape=(1, 2, n, 5, 3))
    out, s_n = impl.fwd_state(q, k, v, s0)
    state = s0.astype(np.float64)
    rows = []
    for i in range(n):
        o, state = impl.fwd_state(q[..., i:i + 1, :], k[..., i:i + 1, :], v[..., i:i + 1, :], state)
        rows.append(o)
    assert np.array_equal(np.concatenate(rows, axis=-2), out), "token-by-token out"
    assert np.array_equal(state, s_n), "token-by-token state"


STATE_PINS = [pin_state_closed_forms, pin_state_chunking, pin_state_finite_differences,
              pin_state_token_by_token]


# --------------------------------------------------------------------------
# normaliser pins: z_i = q_i . sum_{j<=i} k_j and its backward
# --------------------------------------------------------------------------

def _norm_case(seed, shape=(2, 2, 13, 5)):
    rng = _rng(seed)
    q = _dyadic(rng, shape, -2, 2, 8)
    k = _dyadic(rng, shape, -2, 2, 8)
    g = _dyadic(rng, shape[:-1], -2, 2, 8)
    return q, k, g


def pin_norm_quadratic_form(impl):
    """z = rowsum(tril(Q K^T)) and, for L = g . z, dq = diag(g) A K and
    dk = A^T diag(g) Q with A the lower-triangular matrix of ones: the
    quadratic form written with dense matrices (exact for dyadic inputs)."""
    for seed, shape in ((31, (2, 2, 13, 5)), (32, (1, 1, 1, 1)), (33, (1, 3, 40, 8))):
        q, k, g = _norm_case(seed, shape)
        N = shape[-2]
        A = np.tril(np.ones((N, N)))
        qd, kd, gd = (x.astype(np.float64) for x in (q, k, g))
        z_ref = np.einsum("...ij,...ij->...i", A * (qd @ np.swapaxes(kd, -1, -2)), np.ones((N, N)))
        assert np.array_equal(impl.norm(q, k), z_ref), "norm quadratic form"
        dq, dk = impl.norm_bwd(q, k, g)
        assert np.array_equal(dq, gd[..., None] * (A @ kd)), "norm dq quadratic form"
        assert np.array_equal(dk, A.T @ (gd[..., None] * qd)), "norm dk quadratic form"


def pin_norm_is_product_with_ones(impl):
    """The normaliser is the causal product with a single value column of
    ones, and its gradients are the product's with grad_out = g."""
    q, k, g = _norm_case(34, (2, 3, 21, 6))
    ones = np.ones(q.shape[:-1] + (1,), np.float32)
    assert np.array_equal(impl.norm(q, k), impl.fwd(q, k, ones)[..., 0]), "norm vs product"
    dq, dk = impl.norm_bwd(q, k, g)
    pq, pk, _ = impl.bwd(q, k, ones, g[..., None])
    assert np.array_equal(dq, pq) and np.array_equal(dk, pk), "norm bwd vs product bwd"


def pin_norm_closed_forms(impl):
    """Row 0 is q_0 . k_0, the last row is q_{N-1} . sum_j k_j; dk of the
    first row is sum_i g_i q_i, of the last row g_{N-1} q_{N-1}; dq of the
    last row is g_{N-1} sum_j k_j."""
    q, k, g = _norm_case(35, (1, 2, 17, 7))
    qd, kd, gd = (x.astype(np.float64) for x in (q, k, g))
    z = impl.norm(q, k)
    assert np.array_equal(z[..., 0], np.sum(qd[..., 0, :] * kd[..., 0, :], -1)), "norm row 0"
    assert np.array_equal(z[..., -1], np.sum(qd[..., -1, :] * kd.sum(-2), -1)), "norm last row"
    dq, dk = impl.norm_bwd(q, k, g)
    assert np.array_equal(dk[..., 0, :], (gd[..., None] * qd).sum(-2)), "norm dk row 0"
    assert np.array_equal(dk[..., -1, :], gd[..., -1, None] * qd[..., -1, :]), "norm dk last row"
    assert np.array_equal(dq[..., -1, :], gd[..., -1, None] * kd.sum(-2)), "norm dq last row"


def pin_norm_finite_differences(impl, shape=(1, 1, 6, 3)):
    """L = g . z is linear in q for fixed k (and in k for fixed q), so a
    central difference with a unit step is exact for dyadic inputs."""
    q, k, g = _norm_case(36, shape)
    gd = g.astype(np.float64)
    dq, dk = impl.norm_bwd(q, k, g)
    for name, x, grad in (("q", q, dq), ("k", k, dk)):
        fd = np.zeros(x.shape)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += 1.0
            xm[idx] -= 1.0
            if name == "q":
                lp, lm = (np.sum(gd * impl.norm(a, k)) for a in (xp, xm))
            else:
                lp, lm = (np.sum(gd * impl.norm(q, a)) for a in (xp, xm))
            fd[idx] = (lp - lm) / 2.0
        assert np.allclose(grad, fd, rtol=1e-12, atol=1e-12), ("norm finite differences", name)


NORM_PINS = [pin_norm_quadratic_form, pin_norm_is_product_with_ones, pin_norm_closed_forms,
             pin_norm_finite_differences]


# --------------------------------------------------------------------------
# feature-map pins: phi(x) = elu(x) + 1 applied to q and k
# --------------------------------------------------------------------------

def _elu1(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def pin_feature_positive_is_shift(impl):
    """For x > 0, phi(x) = x + 1 (exact in float32 for these dyadic values)
    and phi'(x) = 1: the feature forward and backward equal the plain ones on
    x + 1."""
    rng = _rng(41)
    shape = (1, 2, 19, 5)
    q = _dyadic(rng, shape, 0, 4, 16) + np.float32(1 / 16)
    k = _dyadic(rng, shape, 0, 4, 16) + np.float32(1 / 16)
    v = _dyadic(rng, shape[:-1] + (3,), -2, 2, 16)
    g = _dyadic(rng, shape[:-1] + (3,), -2, 2, 16)
    assert np.array_equal(impl.fwd_feature(q, k, v), impl.fwd(q + 1, k + 1, v)), "feature fwd shift"
    a = impl.bwd_feature(q, k, v, g)
    b = impl.bwd(q + 1, k + 1, v, g)
    for x, y, name in zip(a, b, ("dq", "dk", "dv")):
        assert np.array_equal(x, y), ("feature bwd shift", name)


def pin_feature_quadratic_form(impl):
    """out = tril(phi(Q) phi(K)^T) V with phi from numpy in fp64; the
    gradients from the same dense form: dphi(Q) = tril(G V^T) phi(K),
    dphi(K) = tril(G V^T)^T phi(Q), dV = tril(phi(Q) phi(K)^T)^T G, and
    dQ = dphi(Q) * phi'(Q), dK = dphi(K) * phi'(K)."""
    rng = _rng(42)
    shape = (2, 1, 23, 6)
    q = rng.standard_normal(shape).astype(np.float32)
    k = rng.standard_normal(shape).astype(np.float32)
    v = rng.standard_normal(shape[:-1] + (4,)).astype(np.float32)
    g = rng.standard_normal(shape[:-1] + (4,)).astype(np.float32)
    qd, kd, vd, gd = (x.astype(np.float64) for x in (q, k, v, g))
    fq, fk = _elu1(qd), _elu1(kd)
    A = np.tril(np.ones((shape[-2], shape[-2])))
    T = lambda x: np.swapaxes(x, -1, -2)
    P = A * (fq @ T(fk))
    out = P @ vd
    assert _rel(impl.fwd_feature(q, k, v), out) < 1e-12, "feature fwd dense form"
    GV = A * (gd @ T(vd))
    dfq, dfk, dv = GV @ fk, T(GV) @ fq, T(P) @ gd
    dq = dfq * np.where(qd > 0, 1.0, np.exp(np.minimum(qd, 0.0)))
    dk = dfk * np.where(kd > 0, 1.0, np.exp(np.minimum(kd, 0.0)))
    got = impl.bwd_feature(q, k, v, g)
    for x, y, name in zip(got, (dq, dk, dv), ("dq", "dk", "dv")):
        assert _rel(x, y) < 1e-12, ("feature bwd dense form", name)


def pin_feature_finite_differences(impl, shape=(1, 1, 5, 3)):
    """Central differences of L = <g, out> with respect to the raw q and k
    (step 2^-12, exact in float32 for these inputs) agree with the feature
    backward to the O(h^2) truncation error.  The inputs are odd multiples of
    1/32, away from the kink of phi'' at 0."""
    rng = _rng(43)
    q = _dyadic(rng, shape, -2, 2, 16) + np.float32(1 / 32)
    k = _dyadic(rng, shape, -2, 2, 16) + np.float32(1 / 32)
    v = _dyadic(rng, shape[:-1] + (2,), -2, 2, 16)
    g = _dyadic(rng, shape[:-1] + (2,), -2, 2, 16)
    gd = g.astype(np.float64)
    dq, dk, _ = impl.bwd_feature(q, k, v, g)
    h = np.float32(2.0 ** -12)
    for name, x, grad in (("q", q, dq), ("k", k, dk)):
        fd = np.zeros(x.shape)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = (xp, k) if name == "q" else (q, xp)
            args_m = (xm, k) if name == "q" else (q, xm)
            lp = np.sum(gd * impl.fwd_feature(*args_p, v))
            lm = np.sum(gd * impl.fwd_feature(*args_m, v))
            fd[idx] = (lp - lm) / (2.0 * float(h))
        assert np.allclose(grad, fd, rtol=1e-5, atol=1e-6), ("feature finite differences", name)


def pin_norm_feature(impl):
    """The normaliser of mapped features: for x > 0 it is the plain
    normaliser of x + 1 (exact); in general z = rowsum(tril(phi(Q) phi(K)^T))
    with numpy's fp64 exp, and the gradients are the dense forms times
    phi' (dq = phi'(Q) * diag(g) A phi(K), dk = phi'(K) * A^T diag(g) phi(Q))."""
    rng = _rng(44)
    shape = (1, 2, 17, 6)
    qp = _dyadic(rng, shape, 0, 3, 16) + np.float32(1 / 16)
    kp = _dyadic(rng, shape, 0, 3, 16) + np.float32(1 / 16)
    g = _dyadic(rng, shape[:-1], -2, 2, 8)
    assert np.array_equal(impl.norm_feature(qp, kp), impl.norm(qp + 1, kp + 1)), "norm feature shift"
    a, b = impl.norm_bwd_feature(qp, kp, g), impl.norm_bwd(qp + 1, kp + 1, g)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]), "norm feature bwd shift"
    q = rng.standard_normal(shape).astype(np.float32)
    k = rng.standard_normal(shape).astype(np.float32)
    qd, kd, gd = (x.astype(np.float64) for x in (q, k, g))
    fq, fk = _elu1(qd), _elu1(kd)
    dfq = np.where(qd > 0, 1.0, np.exp(np.minimum(qd, 0.0)))
    dfk = np.where(kd > 0, 1.0, np.exp(np.minimum(kd, 0.0)))
    A = np.tril(np.ones((shape[-2], shape[-2])))
    z = np.sum(A * (fq @ np.swapaxes(fk, -1, -2)), axis=-1)
    assert _rel(impl.norm_feature(q, k), z) < 1e-12, "norm feature dense form"
    dq, dk = impl.norm_bwd_feature(q, k, g)
    assert _rel(dq, dfq * (gd[..., None] * (A @ fk))) < 1e-12, "norm feature dq"
    assert _rel(dk, dfk * (A.T @ (gd[..., None] * fq))) < 1e-12, "norm feature dk"


FEATURE_PINS = [pin_feature_positive_is_shift, pin_feature_quadratic_form,
                pin_feature_finite_differences, pin_norm_feature]


# --------------------------------------------------------------------------
# positive random features: phi(x)_d = exp(w_d . x - |x|^2 / 2) / sqrt(D)
# --------------------------------------------------------------------------

def pin_favor_zero_projection(impl):
    """W = 0 makes every feature exp(-|x|^2 / 2) / sqrt(D), so
    phi(x) . phi(y) = exp(-(|x|^2 + |y|^2) / 2) whatever D is: with
    a_i = exp(-|xq_i|^2 / 2) and b_j = exp(-|xk_j|^2 / 2) the product is the
    scaled cumulative sum out_i = a_i sum_{j<=i} b_j v_j.  Its gradients in
    closed form: dxq_i = -xq_i a_i (g_i . c_i) with c_i = sum_{j<=i} b_j v_j;
    with e_j = sum_{i>=j} a_i g_i, dv_j = b_j e_j and dxk_j = -xk_j b_j (v_j . e_j)."""
    rng = _rng(51)
    lead, N, r, D, M = (2, 1), 11, 3, 6, 4
    xq = (rng.standard_normal(lead + (N, r)) * 0.7).astype(np.float32)
    xk = (rng.standard_normal(lead + (N, r)) * 0.7).astype(np.float32)
    v = rng.standard_normal(lead + (N, M)).astype(np.float32)
    g = rng.standard_normal(lead + (N, M)).astype(np.float32)
    W = np.zeros((D, r), np.float32)
    qd, kd, vd, gd = (x.astype(np.float64) for x in (xq, xk, v, g))
    a = np.exp(-0.5 * np.sum(qd * qd, axis=-1))
    b = np.exp(-0.5 * np.sum(kd * kd, axis=-1))
    c = np.cumsum(b[..., None] * vd, axis=-2)
    assert _rel(impl.fwd_favor(xq, xk, v, W), a[..., None] * c) < 1e-12, "favor W=0 fwd"
    e = np.flip(np.cumsum(np.flip(a[..., None] * gd, axis=-2), axis=-2), axis=-2)
    dxq = -qd * (a * np.sum(gd * c, axis=-1))[..., None]
    dxk = -kd * (b * np.sum(vd * e, axis=-1))[..., None]
    dv = b[..., None] * e
    got = impl.bwd_favor(xq, xk, v, W, g)
    for x, y, name in zip(got, (dxq, dxk, dv), ("dxq", "dxk", "dv")):
        assert _rel(x, y) < 1e-12, ("favor W=0 bwd", name)


def pin_favor_unbiased(impl):
    """Positive random features estimate the softmax kernel without bias:
    for w ~ N(0, I), E[exp(w.x - |x|^2/2) exp(w.y - |y|^2/2)] = exp(x . y).
    With D = 2^15 Gaussian rows of W and v = 1, out_i = sum_{j<=i}
    phi(xq_i) . phi(xk_j) must come within a few standard errors (about 1 %
    here) of sum_{j<=i} exp(xq_i . xk_j)."""
    rng = _rng(52)
    N, r, D = 4, 4, 1 << 15
    xq = (rng.standard_normal((1, 1, N, r)) * 0.25).astype(np.float32)
    xk = (rng.standard_normal((1, 1, N, r)) * 0.25).astype(np.float32)
    W = rng.standard_normal((D, r)).astype(np.float32)
    v = np.ones((1, 1, N, 1), np.float32)
    got = impl.fwd_favor(xq, xk, v, W)[0, 0, :, 0]
    K = np.exp(xq[0, 0].astype(np.float64) @ xk[0, 0].astype(np.float64).T)
    want = np.array([np.sum(K[i, :i + 1]) for i in range(N)])
    assert np.all(np.abs(got / want - 1.0) < 0.05), ("favor unbiased", got, want)


def pin_favor_finite_differences(impl, shape=(1, 1, 5, 3)):
    """Central differences of L = <g, out> with respect to xq and xk (step
    2^-12, exact in float32 for these dyadic inputs) agree with the backward
    to the O(h^2) truncation error."""
    rng = _rng(53)
    D, M = 4, 2
    xq = _dyadic(rng, shape, -2, 2, 16) / np.float32(2)
    xk = _dyadic(rng, shape, -2, 2, 16) / np.float32(2)
    W = _dyadic(rng, (D, shape[-1]), -2, 2, 8)
    v = _dyadic(rng, shape[:-1] + (M,), -2, 2, 16)
    g = _dyadic(rng, shape[:-1] + (M,), -2, 2, 16)
    gd = g.astype(np.float64)
    dxq, dxk, _ = impl.bwd_favor(xq, xk, v, W, g)
    h = np.float32(2.0 ** -12)
    for name, x, grad in (("xq", xq, dxq), ("xk", xk, dxk)):
        fd = np.zeros(x.shape)
        for idx in np.ndindex(*x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args_p = (xp, xk) if name == "xq" else (xq, xp)
            args_m = (xm, xk) if name == "xq" else (xq, xm)
            lp = np.sum(gd * impl.fwd_favor(*args_p, v, W))
            lm = np.sum(gd * impl.fwd_favor(*args_m, v, W))
            fd[idx] = (lp - lm) / (2.0 * float(h))
        assert np.allclose(grad, fd, rtol=1e-5, atol=1e-6), ("favor finite differences", name)


def pin_norm_favor(impl):
    """The normaliser of positive random features.  With W = 0 (features
    exp(-|x|^2 / 2) / sqrt(D)) it is a scaled cumulative sum, z_i = a_i
    sum_{j<=i} b_j, with gradients dxq_i = -xq_i a_i g_i sum_{j<=i} b_j and
    dxk_j = -xk_j b_j sum_{i>=j} g_i a_i.  For a random W it is the product
    with v = 1, forward and backward (the product is pinned above)."""
    rng = _rng(54)
    lead, N, r, D = (1, 2), 13, 3, 5
    xq = (rng.standard_normal(lead + (N, r)) * 0.7).astype(np.float32)
    xk = (rng.standard_normal(lead + (N, r)) * 0.7).astype(np.float32)
    g = rng.standard_normal(lead + (N,)).astype(np.float32)
    qd, kd, gd = (x.astype(np.float64) for x in (xq, xk, g))
    W0 = np.zeros((D, r), np.float32)
    a = np.exp(-0.5 * np.sum(qd * qd, axis=-1))
    b = np.exp(-0.5 * np.sum(kd * kd, axis=-1))
    cb = np.cumsum(b, axis=-1)
    ea = np.flip(np.cumsum(np.flip(a * gd, axis=-1), axis=-1), axis=-1)
    assert _rel(impl.norm_favor(xq, xk, W0), a * cb) < 1e-12, "norm favor W=0"
    dxq, dxk = impl.norm_bwd_favor(xq, xk, W0, g)
    assert _rel(dxq, -qd * (a * gd * cb)[..., None]) < 1e-12, "norm favor W=0 dxq"
    assert _rel(dxk, -kd * (b * ea)[..., None]) < 1e-12, "norm favor W=0 dxk"
    W = rng.standard_normal((D, r)).astype(np.float32)
    ones = np.ones(lead + (N, 1), np.float32)
    assert _rel(impl.norm_favor(xq, xk, W), impl.fwd_favor(xq, xk, ones, W)[..., 0]) < 1e-12, \
        "norm favor = product with v = 1"
    got = impl.norm_bwd_favor(xq, xk, W, g)
    ref = impl.bwd_favor(xq, xk, ones, W, g[..., None])
    assert _rel(got[0], ref[0]) < 1e-12 and _rel(got[1], ref[1]) < 1e-12, \
        "norm favor bwd = product bwd with v = 1"


FAVOR_PINS = [pin_favor_zero_projection, pin_favor_unbiased, pin_favor_finite_differences,
              pin_norm_favor]
ALL_PINS = FWD_PINS + BWD_PINS + STATE_PINS + NORM_PINS + FEATURE_PINS + FAVOR_PINS
