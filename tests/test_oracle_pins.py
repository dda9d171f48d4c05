"""Pins for the fp64 oracle against what the recurrence itself fixes.

None of these compares the oracle with a copy of itself: each uses a closed
form, an invariant, a hand-worked example, a dense brute-force operator, an
independent algorithm (the chunked WY form) or finite differences.  The
update being pinned is the Gated DeltaNet recurrence
S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t,
a_t = exp(g_t), used by the recurrent kernel of "Defending Against the
Training-Inference Numeric Mismatch in RL (Especially Linear Attention)",
section 3.2.
"""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def rand_case(rng, lengths, HK=1, HV=2, dk=4, dv=3, s0_scale=0.5):
    T = sum(lengths)
    q = rng.standard_normal((T, HK, dk))
    k = rng.standard_normal((T, HK, dk))
    v = rng.standard_normal((T, HV, dv))
    g = -np.log1p(np.exp(rng.standard_normal((T, HV))))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, HV))))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64)
    s0 = rng.standard_normal((len(lengths), HV, dv, dk)) * s0_scale
    return q, k, v, g, beta, cu, s0


def unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def test_hand_worked_example():
    fx = json.load(open(os.path.join(HERE, "golden", "hand_worked_2x2.json")))
    a = {n: np.array(fx[n], dtype=np.float64) for n in ("q", "k", "v", "g", "beta")}
    o, fs = oracle.gdn_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], fx["cu_seqlens"],
                           use_qk_l2norm=False)
    np.testing.assert_allclose(o, np.array(fx["expected_o"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(fs, np.array(fx["expected_final_state"]), rtol=0, atol=1e-15)


def test_identity_gate_keeps_state():
    # a = 1 (g = 0) and b = 0: S_t = S_0 for every t, o_t = S_0 q_t
    rng = np.random.default_rng(1)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [9, 4], HK=1, HV=2, dk=5, dv=3)
    g[:] = 0.0
    beta[:] = 0.0
    o, fs = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0, use_qk_l2norm=False)
    assert np.array_equal(fs, s0)
    for n in range(2):
        for t in range(cu[n], cu[n + 1]):
            for h in range(2):
                np.testing.assert_allclose(o[t, h], s0[n, h] @ q[t, 0], rtol=1e-13, atol=1e-14)


def test_delta_rule_projection():
    # b = 1 with a unit key: the updated state maps k_t to v_t exactly
    rng = np.random.default_rng(2)
    T, dk, dv = 7, 6, 4
    q, k, v, g, beta, cu, s0 = rand_case(rng, [T], HK=1, HV=1, dk=dk, dv=dv)
    k = unit(k)
    beta[:] = 1.0
    for t in range(1, T + 1):
        _, fs = oracle.gdn_fwd(q[:t], k[:t], v[:t], g[:t], beta[:t], [0, t], init_state=s0,
                               use_qk_l2norm=False)
        np.testing.assert_allclose(fs[0, 0] @ k[t - 1, 0], v[t - 1, 0], rtol=1e-12, atol=1e-12)


def test_full_forget():
    # a = 0 (g = -inf): S_t = b v_t k_t^T and o_t = b v_t (k_t . q_t)
    rng = np.random.default_rng(3)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [5], HK=1, HV=1, dk=4, dv=3)
    g[:] = -np.inf
    o, fs = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0, use_qk_l2norm=False)
    for t in range(5):
        np.testing.assert_allclose(o[t, 0], beta[t, 0] * v[t, 0] * (k[t, 0] @ q[t, 0]),
                                   rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(fs[0, 0], beta[4, 0] * np.outer(v[4, 0], k[4, 0]), rtol=1e-14)


def test_associative_recall_and_overwrite():
    # a = 1, b = 1, keys are basis vectors: slot j holds the LAST value written to it
    # (a plain linear-attention sum would hold the sum of all of them).
    rng = np.random.default_rng(4)
    dk, dv = 8, 5
    slots = [3, 0, 6, 3, 1, 6]
    T = len(slots)
    k = np.zeros((T, 1, dk))
    for t, j in enumerate(slots):
        k[t, 0, j] = 1.0
    v = rng.standard_normal((T, 1, dv))
    q = np.zeros((T, 1, dk))
    q[:, 0, 3] = 1.0
    g = np.zeros((T, 1))
    beta = np.ones((T, 1))
    o, fs = oracle.gdn_fwd(q, k, v, g, beta, [0, T], use_qk_l2norm=False)
    last = {}
    for t, j in enumerate(slots):
        last[j] = v[t, 0]
    for j in range(dk):
        expect = last.get(j, np.zeros(dv))
        assert np.array_equal(fs[0, 0][:, j], expect)
    # o_t reads slot 3: v_0 until t=3 overwrites it with v_3
    assert np.array_equal(o[0, 0], v[0, 0]) and np.array_equal(o[2, 0], v[0, 0])
    assert np.array_equal(o[3, 0], v[3, 0]) and np.array_equal(o[5, 0], v[3, 0])


@pytest.mark.parametrize("l2", [False, True])
def test_kronecker_brute_force(l2):
    # vec_r(S_t) = a_t (I_dv kron P_t^T) vec_r(S_{t-1}) + b_t vec_r(v_t k_t^T),
    # P_t = I - b_t k_t k_t^T, assembled as dense matrices (row-major vec).
    rng = np.random.default_rng(5)
    T, dk, dv = 8, 4, 3
    q, k, v, g, beta, cu, s0 = rand_case(rng, [T], HK=1, HV=1, dk=dk, dv=dv)
    o, fs = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0, use_qk_l2norm=l2)
    x = s0[0, 0].reshape(-1)
    for t in range(T):
        kk, qq = k[t, 0], q[t, 0]
        if l2:
            kk = kk / np.sqrt(kk @ kk + oracle.oracle.EPS)
            qq = qq / np.sqrt(qq @ qq + oracle.oracle.EPS)
        P = np.eye(dk) - beta[t, 0] * np.outer(kk, kk)
        x = np.exp(g[t, 0]) * (np.kron(np.eye(dv), P.T) @ x) + beta[t, 0] * np.outer(v[t, 0], kk).reshape(-1)
        np.testing.assert_allclose(o[t, 0], x.reshape(dv, dk) @ qq, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(fs[0, 0], x.reshape(dv, dk), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("chunk", [1, 7, 64])
def test_recurrent_matches_chunked_wy(chunk):
    rng = np.random.default_rng(6)
    lengths = [1, 13, 64, 70, 130]
    q, k, v, g, beta, cu, s0 = rand_case(rng, lengths, HK=2, HV=4, dk=8, dv=6)
    o1, f1 = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0)
    o2, f2 = oracle.gdn_fwd_chunked(q, k, v, g, beta, cu, init_state=s0, chunk=chunk)
    scale_o, scale_f = np.abs(o1).max(), np.abs(f1).max()
    assert np.abs(o1 - o2).max() <= 1e-10 * scale_o
    assert np.abs(f1 - f2).max() <= 1e-10 * scale_f


def test_split_resume_is_exact():
    rng = np.random.default_rng(7)
    T = 40
    q, k, v, g, beta, cu, s0 = rand_case(rng, [T], HK=1, HV=2, dk=5, dv=4)
    o, fs = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0)
    for m in (1, 17, 39):
        oa, fa = oracle.gdn_fwd(q[:m], k[:m], v[:m], g[:m], beta[:m], [0, m], init_state=s0)
        ob, fb = oracle.gdn_fwd(q[m:], k[m:], v[m:], g[m:], beta[m:], [0, T - m], init_state=fa)
        assert np.array_equal(np.concatenate([oa, ob]), o)
        assert np.array_equal(fb, fs)


def test_linear_in_value_and_state():
    rng = np.random.default_rng(8)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [6, 11], HK=1, HV=2, dk=4, dv=3)
    o, fs = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0)
    o2, fs2 = oracle.gdn_fwd(q, k, 2 * v, g, beta, cu, init_state=2 * s0)
    assert np.array_equal(o2, 2 * o) and np.array_equal(fs2, 2 * fs)


def test_gqa_head_map_consecutive():
    # v-heads 2j and 2j+1 read k-head j (consecutive sharing), checked against
    # single-head runs fed that k-head's q/k.
    rng = np.random.default_rng(9)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [5, 7], HK=2, HV=4, dk=4, dv=3)
    o, fs = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0)
    for h in range(4):
        hk = h // 2
        o1, f1 = oracle.gdn_fwd(q[:, hk:hk + 1], k[:, hk:hk + 1], v[:, h:h + 1], g[:, h:h + 1],
                                beta[:, h:h + 1], cu, init_state=s0[:, h:h + 1])
        assert np.array_equal(o1[:, 0], o[:, h]) and np.array_equal(f1[:, 0], fs[:, h])


def test_l2norm_scale_invariance():
    # with the in-kernel L2 norm, scaling q and k by c > 0 changes nothing beyond the eps term
    rng = np.random.default_rng(10)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [12], HK=1, HV=1, dk=6, dv=3)
    o, fs = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0)
    o2, fs2 = oracle.gdn_fwd(8.0 * q, 8.0 * k, v, g, beta, cu, init_state=s0)
    np.testing.assert_allclose(o2, o, rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(fs2, fs, rtol=1e-5, atol=1e-6)


def test_zero_length_sequence_passes_state_through():
    rng = np.random.default_rng(11)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [3, 0, 4], HK=1, HV=2, dk=4, dv=3)
    o, fs = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0)
    assert np.array_equal(fs[1], s0[1])


# ---------------------------------------------------------------- backward pins

def _loss(args, cu, dO, dsT, l2):
    q, k, v, g, beta, s0 = args
    o, fs = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0, use_qk_l2norm=l2)
    return float(np.sum(o * dO) + np.sum(fs * dsT))


@pytest.mark.parametrize("l2", [True, False])
def test_backward_finite_differences(l2):
    rng = np.random.default_rng(12)
    lengths = [9, 16]
    q, k, v, g, beta, cu, s0 = rand_case(rng, lengths, HK=1, HV=2, dk=5, dv=4)
    T = sum(lengths)
    dO = rng.standard_normal((T, 2, 4))
    dsT = rng.standard_normal(s0.shape)
    gr = oracle.gdn_bwd(q, k, v, g, beta, cu, dO, init_state=s0, d_final_state=dsT,
                        use_qk_l2norm=l2)
    names = ["dq", "dk", "dv", "dg", "dbeta", "d_init_state"]
    base = [q, k, v, g, beta, s0]
    h = 1e-6
    for i, name in enumerate(names):
        # directional derivatives along random directions, plus single coordinates
        dirs = [rng.standard_normal(base[i].shape) for _ in range(3)]
        for j in rng.choice(base[i].size, size=4, replace=False):
            e = np.zeros(base[i].size)
            e[j] = 1.0
            dirs.append(e.reshape(base[i].shape))
        for d in dirs:
            plus = [a.copy() for a in base]
            minus = [a.copy() for a in base]
            plus[i] = plus[i] + h * d
            minus[i] = minus[i] - h * d
            fd = (_loss(plus, cu, dO, dsT, l2) - _loss(minus, cu, dO, dsT, l2)) / (2 * h)
            an = float(np.sum(gr[name] * d))
            scale = max(1.0, abs(an), float(np.abs(gr[name]).max()))
            assert abs(fd - an) <= 1e-6 * scale, (name, fd, an)


def test_backward_special_cases():
    rng = np.random.default_rng(13)
    q, k, v, g, beta, cu, s0 = rand_case(rng, [6], HK=1, HV=1, dk=4, dv=3)
    dO = rng.standard_normal((6, 1, 3))
    beta0 = np.zeros_like(beta)
    gr = oracle.gdn_bwd(q, k, v, g, beta0, cu, dO, init_state=s0)
    assert np.all(gr["dv"] == 0.0)
    # one token from a zero state: o = b (k.q) v does not depend on g
    gr1 = oracle.gdn_bwd(q[:1], k[:1], v[:1], g[:1], beta[:1], [0, 1], dO[:1],
                         init_state=np.zeros((1, 1, 3, 4)))
    assert np.all(gr1["dg"] == 0.0)


def test_replay_state_pins():
    """The chunk-replay cache: rebuilding the state from it (S_P = exp(gam_r) S0 +
    sum_i exp(gam_r - gam_i) d_i k_i^T) gives the C recurrence's final state, and
    its d rows are the chunked WY form's U rows (an independent algorithm)."""
    rng = np.random.default_rng(11)
    lengths = [70, 64, 5, 0, 130]
    cu = np.concatenate([[0], np.cumsum(lengths)])
    T, HK, HV, dk, dv = int(cu[-1]), 1, 2, 8, 6
    q, k = rng.standard_normal((T, HK, dk)), rng.standard_normal((T, HK, dk))
    v = rng.standard_normal((T, HV, dv))
    g = -np.log1p(np.exp(rng.standard_normal((T, HV))))
    beta = 1 / (1 + np.exp(-rng.standard_normal((T, HV))))
    s0 = rng.standard_normal((len(lengths), HV, dv, dk)) * 0.3
    states, d_all = oracle.gdn_replay_state(q, k, v, g, beta, cu, init_state=s0, chunk=64)
    _, fs = oracle.gdn_fwd(q, k, v, g, beta, cu, init_state=s0)
    for n, st in enumerate(states):
        assert st["r"] == lengths[n] % 64
        for h in range(HV):
            S = st["S0"][h].copy()
            if st["r"]:
                gam = st["gam"][:, h]
                S = np.exp(gam[-1]) * S + sum(np.exp(gam[-1] - gam[i]) * np.outer(st["D"][i, h], st["K"][i, h])
                                              for i in range(st["r"]))
            np.testing.assert_allclose(S, fs[n, h], rtol=1e-12, atol=1e-12)
    # d rows against the chunked form's U = T diag(b) V - W S0^T, computed independently
    kn = k / np.sqrt((k * k).sum(-1, keepdims=True) + 1e-6)
    n, h = 4, 1
    a = int(cu[n])
    S = s0[n, h].copy()
    for c0 in range(a, int(cu[n + 1]), 64):
        c1 = min(c0 + 64, int(cu[n + 1]))
        K, V, b = kn[c0:c1, 0], v[c0:c1, h], beta[c0:c1, h]
        gam = np.cumsum(g[c0:c1, h])
        E = np.exp(gam[:, None] - gam[None, :])
        A = np.tril(b[:, None] * E * (K @ K.T), -1)
        Tm = np.linalg.inv(np.eye(c1 - c0) + A)
        U = Tm @ (b[:, None] * V) - (Tm @ ((b * np.exp(gam))[:, None] * K)) @ S.T
        np.testing.assert_allclose(d_all[c0:c1, h], U, rtol=1e-11, atol=1e-12)
        S = np.exp(gam[-1]) * S + U.T @ (np.exp(gam[-1] - gam)[:, None] * K)
