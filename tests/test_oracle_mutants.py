"""Planted mistakes in a copy of the oracle must trip at least one pin.

Each mutant is the oracle's C source with one plausible mistake (a dropped
term, a wrong operand, a wrong index, an exclusive instead of inclusive
prefix, a transposed state) compiled into a temporary library and run
through the same pins as the real oracle.  Nothing here touches the real
oracle's build.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "causal_product_oracle.c")

MUTANTS = {
    # readout with the key instead of the query (the listing's own TODO)
    "readout_uses_key": [("double qd = qi[d];", "double qd = ki[d];")],
    # half-weight state update (a scaled term)
    "scaled_update": [("for (int64_t m = 0; m < M; ++m) Sd[m] += kd * vi[m];\n        }\n        /* readout",
                       "for (int64_t m = 0; m < M; ++m) Sd[m] += 0.5 * kd * vi[m];\n        }\n        /* readout")],
    # query of the previous row
    "query_off_by_one": [("*qi = q + i * D;", "*qi = q + (i > 0 ? i - 1 : 0) * D;")],
    # exclusive prefix: row i is taken out of the state for its own readout
    "exclusive_prefix": [
        ("/* readout: out_i = S^T q_i */",
         "for (int64_t d = 0; d < D; ++d) for (int64_t m = 0; m < M; ++m) S[d * M + m] -= ki[d] * vi[m];"),
        ("for (int64_t m = 0; m < M; ++m) oi[m] += qd * Sd[m];\n        }\n    }\n    if (SN)",
         "for (int64_t m = 0; m < M; ++m) oi[m] += qd * Sd[m];\n        }\n"
         "        for (int64_t d = 0; d < D; ++d) for (int64_t m = 0; m < M; ++m) S[d * M + m] += ki[d] * vi[m];\n    }\n    if (SN)")],
    # dq with the value instead of the output gradient
    "dq_uses_v": [("acc += Sd[m] * gi[m];", "acc += Sd[m] * vi[m];")],
    # reverse sweep skips row 0
    "reverse_drops_row0": [("for (int64_t j = N - 1; j >= 0; --j) {", "for (int64_t j = N - 1; j >= 1; --j) {")],
    # dv with the query instead of the key
    "dv_uses_q": [("double kd = kj[d];", "double kd = qj[d];")],
    # reverse state accumulates k g^T instead of q g^T
    "reverse_state_uses_k": [("double qd = qj[d];", "double qd = kj[d];")],
    # dk reads the state transposed (indices kept in bounds for any D, M)
    "dk_transposed": [("for (int64_t m = 0; m < M; ++m) acc += Rd[m] * vj[m];",
                       "for (int64_t m = 0; m < M; ++m) acc += R[(m % D) * M + (d % M)] * vj[m];")],
    # the forward ignores the initial state
    "fwd_ignores_state_in": [("/* start from the initial state */\n    if (S0)",
                              "/* start from the initial state */\n    if (0)")],
    # dq's forward sweep ignores the initial state
    "dq_ignores_state_in": [("dq_i = S_i g_i */\n    if (S0)", "dq_i = S_i g_i */\n    if (0)")],
    # the reverse sweep ignores the final-state gradient
    "reverse_ignores_grad_state": [("if (dSN) memcpy(R, dSN,", "if (0) memcpy(R, dSN,")],
    # the final state is the sum without the initial state
    "state_out_drops_state_in": [("    if (SN) memcpy(SN, S, sizeof(double) * (size_t)(D * M));",
                                  "    if (SN) { memcpy(SN, S, sizeof(double) * (size_t)(D * M));"
                                  " if (S0) for (int64_t e = 0; e < D * M; ++e) SN[e] -= S0[e]; }")],
    # dS_0 is taken before the last row of the reverse sweep
    "grad_state_in_misses_row0": [("    /* dS_0 = R_0 */\n    if (dS0) memcpy(dS0, R, sizeof(double) * (size_t)(D * M));",
                                   "    /* dS_0 = R_0 */\n    if (dS0) { memcpy(dS0, R, sizeof(double) * (size_t)(D * M));"
                                   " for (int64_t d = 0; d < D; ++d) for (int64_t m = 0; m < M; ++m)"
                                   " dS0[d * M + m] -= q[d] * g[m]; }")],
    # the normaliser reads the running sum before adding row i (exclusive)
    "norm_exclusive": [("/* c += k_i, then z_i = q_i . c */\n"
                        "            for (int64_t d = 0; d < D; ++d) c[d] += (double)ks[i * D + d];\n"
                        "            double acc = 0.0;\n"
                        "            for (int64_t d = 0; d < D; ++d) acc += (double)qs[i * D + d] * c[d];",
                        "double acc = 0.0;\n"
                        "            for (int64_t d = 0; d < D; ++d) acc += (double)qs[i * D + d] * c[d];\n"
                        "            for (int64_t d = 0; d < D; ++d) c[d] += (double)ks[i * D + d];")],
    # the normaliser's readout uses k instead of q
    "norm_reads_k": [("acc += (double)qs[i * D + d] * c[d];", "acc += (double)ks[i * D + d] * c[d];")],
    # dq of the normaliser without the gradient factor
    "norm_dq_drops_g": [("dqs[i * D + d] = (double)gs[i] * c[d];", "dqs[i * D + d] = c[d];")],
    # dk of the normaliser summed forwards instead of backwards
    "norm_dk_forward": [("for (int64_t j = N - 1; j >= 0; j--) {\n            for (int64_t d = 0; d < D; ++d) {\n"
                         "                c[d] += (double)gs[j]",
                         "for (int64_t j = 0; j < N; ++j) {\n            for (int64_t d = 0; d < D; ++d) {\n"
                         "                c[d] += (double)gs[j]")],
    # dk of the normaliser uses k instead of q
    "norm_dk_uses_k": [("c[d] += (double)gs[j] * (double)qs[j * D + d];",
                        "c[d] += (double)gs[j] * (double)ks[j * D + d];")],
    # the feature map without its exponential branch
    "feature_no_exp": [("if (feature == 1) return x > 0.0 ? x + 1.0 : exp(x);",
                        "if (feature == 1) return x + 1.0;")],
    # the backward without the chain rule through phi
    "feature_no_chain_rule": [("dqs[e] *= dphi(feature, (double)qs[e]);", "(void)0;")],
    # phi' taken as phi
    "feature_dphi_is_phi": [("if (feature == 1) return x > 0.0 ? 1.0 : exp(x);",
                             "if (feature == 1) return x > 0.0 ? x + 1.0 : exp(x);")],
    # the normaliser of mapped features without phi' on dq
    "norm_feature_dq_no_dphi": [("dqs[i * D + d] = dphi(feature, qx) * ((double)gs[i] * c[d]);",
                                 "dqs[i * D + d] = (double)gs[i] * c[d];")],
    # the normaliser of mapped features reading phi(k) for the readout
    "norm_feature_reads_k": [("acc += phi(feature, (double)qs[i * D + d]) * c[d];",
                              "acc += phi(feature, (double)ks[i * D + d]) * c[d];")],
    # positive random features with the norm term's sign flipped
    "favor_norm_sign": [("phi[i * D + d] = exp(wx - 0.5 * n2) * scale;",
                         "phi[i * D + d] = exp(wx + 0.5 * n2) * scale;")],
    # positive random features without the 1/sqrt(D) normalisation
    "favor_no_scale": [("const double scale = 1.0 / sqrt((double)D);", "const double scale = 1.0;")],
    # the projection read transposed (still in bounds: t < r, d < D)
    "favor_w_transposed": [("wx += (double)W[d * r + t] * (double)xi[t];",
                            "wx += (double)W[t * D + d] * (double)xi[t];")],
    # the chain rule without the -x (a . phi) term of the norm
    "favor_grad_drops_norm_term": [("dx[i * r + t] = acc - (double)x[i * r + t] * s;",
                                    "dx[i * r + t] = acc;")],
    # the chain rule without the phi factor on the projection term
    "favor_grad_unweighted": [("acc += (double)W[d * r + t] * (ai[d] * pi[d]);",
                               "acc += (double)W[d * r + t] * ai[d];")],
    # the normaliser of positive random features reading phi(k) for the readout
    "norm_favor_reads_k": [("acc += pq[i * D + d] * c[d];", "acc += pk[i * D + d] * c[d];")],
    # its backward without the gradient factor on dq
    "norm_bwd_favor_drops_g": [("aq[i * D + d] = (double)gs[i] * c[d];", "aq[i * D + d] = c[d];")],
}


class _Impl:
    def __init__(self, path):
        lib = ctypes.CDLL(path)
        i64, p, c_int = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.cpo_fwd.argtypes = [p, p, p, p, i64, i64, i64, i64, c_int]
        lib.cpo_bwd.argtypes = [p, p, p, p, p, p, p, i64, i64, i64, i64, c_int]
        lib.cpo_fwd_state.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, c_int]
        lib.cpo_bwd_state.argtypes = [p, p, p, p, p, p, p, p, p, p, i64, i64, i64, i64, c_int]
        lib.cpo_norm.argtypes = [p, p, p, i64, i64, i64, c_int]
        lib.cpo_fwd_feature.argtypes = [p, p, p, p, c_int, i64, i64, i64, i64, c_int]
        lib.cpo_norm_feature.argtypes = [p, p, p, c_int, i64, i64, i64, c_int]
        lib.cpo_norm_bwd_feature.argtypes = [p, p, p, p, p, c_int, i64, i64, i64, c_int]
        lib.cpo_bwd_feature.argtypes = [p, p, p, p, p, p, p, c_int, i64, i64, i64, i64, c_int]
        lib.cpo_norm_bwd.argtypes = [p, p, p, p, p, i64, i64, i64, c_int]
        lib.cpo_fwd_favor.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, c_int]
        lib.cpo_bwd_favor.argtypes = [p, p, p, p, p, p, p, p, i64, i64, i64, i64, i64, c_int]
        lib.cpo_norm_favor.argtypes = [p, p, p, p, i64, i64, i64, i64, c_int]
        lib.cpo_norm_bwd_favor.argtypes = [p, p, p, p, p, p, i64, i64, i64, i64, c_int]
        self.lib = lib

    def norm_favor(self, xq, xk, W):
        xq, xk, W = (np.ascontiguousarray(x, np.float32) for x in (xq, xk, W))
        lead = xq.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, r, D = xq.shape[-2], xq.shape[-1], W.shape[0]
        z = np.zeros(lead + (N,))
        assert self.lib.cpo_norm_favor(xq.ctypes.data, xk.ctypes.data, W.ctypes.data,
                                       z.ctypes.data, BH, N, r, D, 1) == 0
        return z

    def norm_bwd_favor(self, xq, xk, W, g):
        xq, xk, W, g = (np.ascontiguousarray(x, np.float32) for x in (xq, xk, W, g))
        lead = xq.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, r, D = xq.shape[-2], xq.shape[-1], W.shape[0]
        dxq, dxk = np.zeros(lead + (N, r)), np.zeros(lead + (N, r))
        assert self.lib.cpo_norm_bwd_favor(xq.ctypes.data, xk.ctypes.data, W.ctypes.data,
                                           g.ctypes.data, dxq.ctypes.data, dxk.ctypes.data, BH,
                                           N, r, D, 1) == 0
        return dxq, dxk

    def fwd_favor(self, xq, xk, v, W):
        xq, xk, v, W = (np.ascontiguousarray(x, np.float32) for x in (xq, xk, v, W))
        lead = xq.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, r, D, M = xq.shape[-2], xq.shape[-1], W.shape[0], v.shape[-1]
        out = np.zeros(lead + (N, M))
        assert self.lib.cpo_fwd_favor(xq.ctypes.data, xk.ctypes.data, v.ctypes.data,
                                      W.ctypes.data, out.ctypes.data, BH, N, r, D, M, 1) == 0
        return out

    def bwd_favor(self, xq, xk, v, W, g):
        xq, xk, v, W, g = (np.ascontiguousarray(x, np.float32) for x in (xq, xk, v, W, g))
        lead = xq.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, r, D, M = xq.shape[-2], xq.shape[-1], W.shape[0], v.shape[-1]
        dxq, dxk, dv = np.zeros(lead + (N, r)), np.zeros(lead + (N, r)), np.zeros(lead + (N, M))
        assert self.lib.cpo_bwd_favor(xq.ctypes.data, xk.ctypes.data, v.ctypes.data,
                                      W.ctypes.data, g.ctypes.data, dxq.ctypes.data,
                                      dxk.ctypes.data, dv.ctypes.data, BH, N, r, D, M, 1) == 0
        return dxq, dxk, dv

    def fwd_feature(self, q, k, v):
        q, k, v = (np.ascontiguousarray(x, np.float32) for x in (q, k, v))
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, D, M = q.shape[-2], q.shape[-1], v.shape[-1]
        out = np.zeros(lead + (N, M))
        assert self.lib.cpo_fwd_feature(q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                        out.ctypes.data, 1, BH, N, D, M, 1) == 0
        return out

    def bwd_feature(self, q, k, v, g):
        q, k, v, g = (np.ascontiguousarray(x, np.float32) for x in (q, k, v, g))
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, D, M = q.shape[-2], q.shape[-1], v.shape[-1]
        dq, dk, dv = np.zeros(lead + (N, D)), np.zeros(lead + (N, D)), np.zeros(lead + (N, M))
        assert self.lib.cpo_bwd_feature(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data,
                                        dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, 1, BH, N,
                                        D, M, 1) == 0
        return dq, dk, dv

    def norm_feature(self, q, k):
        q, k = (np.ascontiguousarray(x, np.float32) for x in (q, k))
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, D = q.shape[-2], q.shape[-1]
        z = np.zeros(lead + (N,))
        assert self.lib.cpo_norm_feature(q.ctypes.data, k.ctypes.data, z.ctypes.data, 1, BH, N,
                                         D, 1) == 0
        return z

    def norm_bwd_feature(self, q, k, g):
        q, k, g = (np.ascontiguousarray(x, np.float32) for x in (q, k, g))
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, D = q.shape[-2], q.shape[-1]
        dq, dk = np.zeros(lead + (N, D)), np.zeros(lead + (N, D))
        assert self.lib.cpo_norm_bwd_feature(q.ctypes.data, k.ctypes.data, g.ctypes.data,
                                             dq.ctypes.data, dk.ctypes.data, 1, BH, N, D, 1) == 0
        return dq, dk

    def norm(self, q, k):
        q, k = (np.ascontiguousarray(x, np.float32) for x in (q, k))
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, D = q.shape[-2], q.shape[-1]
        z = np.zeros(lead + (N,))
        assert self.lib.cpo_norm(q.ctypes.data, k.ctypes.data, z.ctypes.data, BH, N, D, 1) == 0
        return z

    def norm_bwd(self, q, k, g):
        q, k, g = (np.ascontiguousarray(x, np.float32) for x in (q, k, g))
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, D = q.shape[-2], q.shape[-1]
        dq, dk = np.zeros(lead + (N, D)), np.zeros(lead + (N, D))
        assert self.lib.cpo_norm_bwd(q.ctypes.data, k.ctypes.data, g.ctypes.data, dq.ctypes.data,
                                     dk.ctypes.data, BH, N, D, 1) == 0
        return dq, dk

    def fwd(self, q, k, v):
        q, k, v = (np.ascontiguousarray(x, np.float32) for x in (q, k, v))
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, D, M = q.shape[-2], q.shape[-1], v.shape[-1]
        out = np.zeros(lead + (N, M))
        rc = self.lib.cpo_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, out.ctypes.data,
                              BH, N, D, M, 1)
        assert rc == 0
        return out

    def bwd(self, q, k, v, g):
        q, k, v, g = (np.ascontiguousarray(x, np.float32) for x in (q, k, v, g))
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, D, M = q.shape[-2], q.shape[-1], v.shape[-1]
        dq, dk, dv = np.zeros(lead + (N, D)), np.zeros(lead + (N, D)), np.zeros(lead + (N, M))
        rc = self.lib.cpo_bwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data,
                              dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, BH, N, D, M, 1)
        assert rc == 0
        return dq, dk, dv


    def fwd_state(self, q, k, v, s0):
        q, k, v = (np.ascontiguousarray(x, np.float32) for x in (q, k, v))
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, D, M = q.shape[-2], q.shape[-1], v.shape[-1]
        s0 = np.ascontiguousarray(s0, np.float64)
        out, s_n = np.zeros(lead + (N, M)), np.zeros(lead + (D, M))
        rc = self.lib.cpo_fwd_state(q.ctypes.data, k.ctypes.data, v.ctypes.data, out.ctypes.data,
                                    s0.ctypes.data, s_n.ctypes.data, BH, N, D, M, 1)
        assert rc == 0
        return out, s_n

    def bwd_state(self, q, k, v, g, s0, ds_n):
        q, k, v, g = (np.ascontiguousarray(x, np.float32) for x in (q, k, v, g))
        lead = q.shape[:-2]
        BH = int(np.prod(lead)) if lead else 1
        N, D, M = q.shape[-2], q.shape[-1], v.shape[-1]
        s0, ds_n = (np.ascontiguousarray(x, np.float64) for x in (s0, ds_n))
        dq, dk, dv = np.zeros(lead + (N, D)), np.zeros(lead + (N, D)), np.zeros(lead + (N, M))
        ds0 = np.zeros(lead + (D, M))
        rc = self.lib.cpo_bwd_state(q.ctypes.data, k.ctypes.data, v.ctypes.data, g.ctypes.data,
                                    s0.ctypes.data, ds_n.ctypes.data, dq.ctypes.data,
                                    dk.ctypes.data, dv.ctypes.data, ds0.ctypes.data,
                                    BH, N, D, M, 1)
        assert rc == 0
        return dq, dk, dv, ds0


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    src = open(SRC).read()
    for old, new in MUTANTS[name]:
        assert src.count(old) == 1, f"mutation site for {name} not unique/present"
        src = src.replace(old, new)
    mpath = tmp_path / f"{name}.c"
    mpath.write_text(src)
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-shared", "-fPIC", "-std=c11", "-o", str(lib),
                    str(mpath), "-lm"], check=True)
    impl = _Impl(str(lib))
    caught = []
    for pin in pins.ALL_PINS:
        try:
            pin(impl)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"mutant {name} passed every pin"
