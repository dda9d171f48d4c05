"""Pins for the layer-op oracle (gates, causal conv, gated RMSNorm) against
closed forms, special cases and invariants of their definitions."""
import numpy as np

from oracle import layer_ops as L


def test_gates_closed_forms():
    a = np.array([[0.0, -40.0, 3.0]])
    b = np.array([[0.0, 2.0, -2.0]])
    A_log = np.array([np.log(2.0), 0.0, 0.0])
    dt_bias = np.zeros(3)
    g, beta = L.gates(a, b, A_log, dt_bias)
    assert g[0, 0] == -2.0 * np.log(2.0)                          # softplus(0) = ln 2
    assert 0.0 > g[0, 1] > -1e-17                                 # softplus(-40) ~ e^-40
    np.testing.assert_allclose(g[0, 2], -np.log1p(np.exp(3.0)), rtol=1e-15)
    assert beta[0, 0] == 0.5
    np.testing.assert_allclose(beta[0, 1] + beta[0, 2], 1.0, rtol=1e-15)  # sigmoid(x) + sigmoid(-x) = 1
    # dt_bias shifts the softplus argument per head, A_log scales per head
    g2, _ = L.gates(np.zeros((1, 3)), b, np.array([0.0, np.log(3.0), 0.0]), np.array([0.0, 0.0, 3.0]))
    np.testing.assert_allclose(g2[0], [-np.log(2.0), -3.0 * np.log(2.0), -np.log1p(np.exp(3.0))], rtol=1e-15)


def test_gated_rmsnorm_invariants():
    rng = np.random.default_rng(1)
    o = rng.standard_normal((5, 2, 16))
    z = rng.standard_normal((5, 2, 16))
    w = rng.standard_normal(16)
    y = L.gated_rmsnorm(o, z, w, eps=0.0)
    # scale invariance of the normalisation (exact with eps = 0: sqrt(4x) = 2 sqrt(x))
    assert np.array_equal(L.gated_rmsnorm(2.0 * o, z, w, eps=0.0), y)
    # z = 0 closes the gate
    assert np.all(L.gated_rmsnorm(o, np.zeros_like(z), w) == 0.0)
    # unit weight, large gate: the normalised vector has rms 1 and silu(z) ~ z
    big = np.full_like(z, 40.0)
    yy = L.gated_rmsnorm(o, big, np.ones(16), eps=0.0) / 40.0
    np.testing.assert_allclose(np.sqrt(np.mean(yy * yy, axis=-1)), 1.0, rtol=1e-12)
    # a row of equal entries c normalises to sign(c) exactly (eps = 0)
    flat = np.full((1, 1, 8), -3.0)
    np.testing.assert_allclose(L.gated_rmsnorm(flat, np.full_like(flat, 40.0), np.ones(8), eps=0.0) / 40.0,
                               -1.0, rtol=1e-15)


def test_conv_identity_and_shift_taps():
    rng = np.random.default_rng(2)
    T, C, W = 9, 3, 4
    x = rng.standard_normal((T, C))
    cu = [0, 4, 9]
    ident = np.zeros((C, W))
    ident[:, -1] = 1.0
    y, _ = L.causal_conv1d(x, ident, cu)
    np.testing.assert_allclose(y, L.silu(x), rtol=0, atol=0)
    shift = np.zeros((C, W))
    shift[:, -2] = 1.0                                             # y_t = silu(x_{t-1})
    st = rng.standard_normal((2, W - 1, C))
    y2, fin = L.causal_conv1d(x, shift, cu, conv_state=st)
    assert np.array_equal(y2[0], L.silu(st[0][-1]))               # first token sees the cached input
    assert np.array_equal(y2[1:4], L.silu(x[0:3]))
    assert np.array_equal(y2[4], L.silu(st[1][-1]))               # sequence 2 never sees sequence 1
    assert np.array_equal(y2[5:9], L.silu(x[4:8]))
    assert np.array_equal(fin[0], x[1:4]) and np.array_equal(fin[1], x[6:9])


def test_conv_prefill_then_updates_equals_one_pass():
    rng = np.random.default_rng(3)
    T, C, W = 12, 5, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    bias = rng.standard_normal(C)
    st0 = rng.standard_normal((1, W - 1, C))
    y, fin = L.causal_conv1d(x, w, [0, T], bias=bias, conv_state=st0)
    P = 7
    ya, fa = L.causal_conv1d(x[:P], w, [0, P], bias=bias, conv_state=st0)
    st = fa
    ys = [ya]
    for t in range(P, T):
        yt, st = L.causal_conv1d_update(x[t:t + 1], w, st, bias=bias)
        ys.append(yt)
    assert np.array_equal(np.concatenate(ys), y)
    assert np.array_equal(st, fin)


def test_conv_brute_force_matches_explicit_sum():
    # short sequence, explicit formula with hand-indexed taps (no window concatenation)
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 2))
    w = rng.standard_normal((2, 4))
    st = rng.standard_normal((1, 3, 2))
    y, _ = L.causal_conv1d(x, w, [0, 3], conv_state=st, activation=False)
    past = st[0]
    for c in range(2):
        seq = [past[0, c], past[1, c], past[2, c], x[0, c], x[1, c], x[2, c]]
        for t in range(3):
            expect = sum(w[c, i] * seq[t + i] for i in range(4))
            np.testing.assert_allclose(y[t, c], expect, rtol=1e-14)


def test_conv_matches_numpy_convolve():
    # one sequence, zero state: the conv is numpy's full convolution with the reversed taps
    rng = np.random.default_rng(7)
    x = rng.standard_normal((20, 1))
    w = rng.standard_normal((1, 5))
    y, _ = L.causal_conv1d(x, w, [0, 20], activation=False)
    want = np.convolve(x[:, 0], w[0, ::-1])[:20]
    np.testing.assert_allclose(y[:, 0], want, rtol=1e-13, atol=1e-14)


def test_conv_short_sequence_keeps_part_of_the_old_state():
    # a sequence shorter than W-1 leaves the oldest cached rows in the final state
    rng = np.random.default_rng(5)
    C, W = 3, 4
    st = rng.standard_normal((2, W - 1, C))
    x = rng.standard_normal((1, C))
    _, fin = L.causal_conv1d(x, rng.standard_normal((C, W)), [0, 1, 1], conv_state=st)
    assert np.array_equal(fin[0], np.concatenate([st[0][1:], x]))
    assert np.array_equal(fin[1], st[1])                           # empty sequence: state unchanged


def test_conv_update_skips_negative_slot():
    rng = np.random.default_rng(6)
    C, W = 2, 3
    st = rng.standard_normal((3, W - 1, C))
    x = rng.standard_normal((2, C))
    y, st2 = L.causal_conv1d_update(x, rng.standard_normal((C, W)), st, state_indices=[-1, 2])
    assert np.all(y[0] == 0) and np.array_equal(st2[:2], st[:2])
    assert np.array_equal(st2[2], np.concatenate([st[2][1:], x[1:2]]))
