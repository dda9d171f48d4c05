"""GPU parity and invariance of the layer ops around the recurrence (gate
activations, short causal conv with its conv state cache, gated RMSNorm)
against the fp64 oracle in oracle/layer_ops.py.

Tolerances.  The forward bound of the recurrence (normwise 2e-3, bf16 rounding net of
2^-8 per element) is asserted on every output; on top of it each test checks
the tighter per-element bound that fp32 arithmetic gives these ops:
  * gates: a few correctly rounded or 2-ulp fp32 operations per element
    (add, exp, log1p, multiply; exp, add, divide): relative error below
    16 ulp = 1e-6; asserted 4e-6.
  * RMSNorm: the fp32 sum of d <= 256 squares (relative error <= d * 2^-24
    <= 1.6e-5), rsqrt, three products and the SiLU gate (hardware exponential
    and fast divide, <= 20 ulp for |z| < 10; all relative, no cancellation):
    asserted 4e-5 relative, plus the output's own rounding.
  * conv: W + 1 fused multiply-adds (absolute error <= (W + 1) 2^-24 *
    (|bias| + sum |w x|)), then SiLU (slope <= 1.1) through the hardware
    exponential and the fast divide: relative error <= (2 + 1.2 |acc|) ulp
    for the exponential plus 2 ulp for the divide and 2 for the add; asserted
    4x the sum part and 2x the SiLU part, plus the output's own rounding.
The conv state is pure data movement: compared bit for bit.
"""
import numpy as np
import pytest
import torch

import invariant_linear_attention_gb300 as gdn
from invariant_linear_attention_gb300 import inputs
from oracle import layer_ops as ref
from helpers import FWD_TOL, BF16_ROUND, bf16_err, normwise, to_np

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
U32 = 2.0 ** -24


def rounding(t):
    return BF16_ROUND if t.dtype == torch.bfloat16 else U32


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


# ---------------------------------------------------------------- gates

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_gates_vs_oracle(dtype):
    L = inputs.make_layer_inputs([1000, 3, 37], HK=2, HV=32, dk=16, dv=16, dtype=dtype, seed=61).to(DEV)
    g, beta = gdn.gdn_gates(L.a, L.b, L.A_log, L.dt_bias)
    gr, br = ref.gates(L.a, L.b, L.A_log, L.dt_bias)
    for got, want in ((to_np(g), gr), (to_np(beta), br)):
        assert normwise(got, want) < FWD_TOL
        assert np.all(np.abs(got - want) <= 4e-6 * np.abs(want))
    # no dt_bias, an odd head count (scalar path), and extreme inputs (softplus
    # switches to x above 20; sigmoid saturates)
    a = torch.tensor([[-80.0, -20.0, 0.0, 19.9, 20.1, 60.0]], device=DEV).repeat(4, 1).to(dtype)
    A_log = torch.zeros(6, device=DEV)
    g2, b2 = gdn.gdn_gates(a, a.clone(), A_log)
    gr2, br2 = ref.gates(a, a, A_log, np.zeros(6))
    assert np.all(np.abs(to_np(g2) - gr2) <= 4e-6 * np.abs(gr2) + 1e-38)
    assert np.all(np.abs(to_np(b2) - br2) <= 4e-6 * np.abs(br2) + 1e-38)


def test_gates_batch_invariant_and_paths_agree():
    L = inputs.make_layer_inputs([512, 77], HK=2, HV=32, dk=16, dv=16, seed=62).to(DEV)
    g, beta = gdn.gdn_gates(L.a, L.b, L.A_log, L.dt_bias)
    g1, b1 = gdn.gdn_gates(L.a[512:].contiguous(), L.b[512:].contiguous(), L.A_log, L.dt_bias)
    assert torch.equal(bits(g[512:]), bits(g1)) and torch.equal(bits(beta[512:]), bits(b1))
    # an output that is not 16-byte aligned takes the scalar kernel: same bits
    gs = torch.empty(L.a.numel() + 1, device=DEV)[1:].view(L.a.shape)
    bs = torch.empty(L.a.numel() + 1, device=DEV)[1:].view(L.a.shape)
    gdn.gdn_gates(L.a, L.b, L.A_log, L.dt_bias, g=gs, beta=bs)
    assert torch.equal(bits(gs), bits(g)) and torch.equal(bits(bs), bits(beta))


# ---------------------------------------------------------------- gated RMSNorm

@pytest.mark.parametrize("dtype,dv,gate", [(torch.bfloat16, 128, True), (torch.float32, 128, True),
                                           (torch.bfloat16, 64, False), (torch.bfloat16, 256, True),
                                           (torch.float32, 40, True), (torch.bfloat16, 8, True)])
def test_rmsnorm_vs_oracle(dtype, dv, gate):
    L = inputs.make_layer_inputs([203, 1, 54], HK=1, HV=6, dk=16, dv=dv, dtype=dtype, seed=63).to(DEV)
    z = L.z if gate else None
    y = gdn.gdn_gated_rmsnorm(L.o, z, L.norm_w, eps=1e-6)
    want = ref.gated_rmsnorm(L.o, L.z if gate else np.full(L.o.shape, 60.0), L.norm_w, eps=1e-6)
    if not gate:
        want = want / 60.0  # silu(60) = 60 to double precision: undo the stand-in gate
    got = to_np(y)
    err = bf16_err(got, want) if dtype == torch.bfloat16 else normwise(got, want)
    assert err < FWD_TOL
    assert np.all(np.abs(got - want) <= (rounding(y) + 4e-5) * np.abs(want) + 1e-30)


def test_rmsnorm_in_place_and_batch_invariant():
    L = inputs.make_layer_inputs([300, 5], HK=1, HV=32, dk=16, dv=128, seed=64).to(DEV)
    y = gdn.gdn_gated_rmsnorm(L.o, L.z, L.norm_w)
    part = gdn.gdn_gated_rmsnorm(L.o[300:].contiguous(), L.z[300:].contiguous(), L.norm_w)
    assert torch.equal(bits(y[300:]), bits(part))
    o2 = L.o.clone()
    gdn.gdn_gated_rmsnorm(o2, L.z, L.norm_w, out=o2)
    assert torch.equal(bits(o2), bits(y))


# ---------------------------------------------------------------- causal conv

LENS = [0, 1, 2, 3, 5, 127, 128, 129, 255, 256, 257, 300, 1000, 4]


def conv_bound(x, w, b, y_ref, W, out_dtype, cu, state):
    """Per-element error bound of the conv output (see the module docstring)."""
    xn, wn, bn, sn = to_np(x), to_np(w), to_np(b), to_np(state)
    mag, _ = ref.causal_conv1d(np.abs(xn), np.abs(wn), cu, bias=np.abs(bn), conv_state=np.abs(sn), activation=False)
    acc, _ = ref.causal_conv1d(xn, wn, cu, bias=bn, conv_state=sn, activation=False)
    silu_ulps = 2 * (6 + 1.2 * np.abs(acc))
    return 4 * (W + 1) * U32 * 1.1 * mag + (silu_ulps * U32 + (BF16_ROUND if out_dtype == torch.bfloat16 else U32)) \
        * np.abs(y_ref) + 1e-30


@pytest.mark.parametrize("dtype,W,C", [(torch.bfloat16, 4, 512), (torch.float32, 4, 256), (torch.bfloat16, 2, 24),
                                       (torch.bfloat16, 8, 1032), (torch.float32, 3, 12)])
def test_conv_fwd_vs_oracle(dtype, W, C):
    L = inputs.make_layer_inputs(LENS, HK=1, HV=1, dk=16, dv=16, W=W, dtype=dtype, seed=65, C=C).to(DEV)
    N = len(LENS)
    # slots permuted over a larger pool; every other sequence starts from zeros
    slots = torch.randperm(N + 3, generator=torch.Generator().manual_seed(1))[:N].to(torch.int32)
    pool = torch.randn(N + 3, W - 1, C, generator=torch.Generator().manual_seed(2)).to(dtype).to(DEV)
    pool[slots.long()] = L.conv_state
    has_init = torch.tensor([1, 0] * (N // 2) + [1] * (N % 2), dtype=torch.int32, device=DEV)
    pool0 = pool.clone()
    y = gdn.gdn_causal_conv1d_fwd(L.x, L.conv_w, L.cu_seqlens, bias=L.conv_b, conv_state=pool,
                                  state_indices=slots.to(DEV), has_initial_state=has_init)
    torch.cuda.synchronize()
    init = L.conv_state.clone()
    init[has_init == 0] = 0
    y_ref, fin_ref = ref.causal_conv1d(L.x, L.conv_w, L.cu_seqlens.cpu(), bias=L.conv_b, conv_state=init)
    got = to_np(y)
    cu = L.cu_seqlens.cpu().tolist()
    for n in range(N):
        a, b = cu[n], cu[n + 1]
        if b > a:
            e = bf16_err(got[a:b], y_ref[a:b]) if dtype == torch.bfloat16 else normwise(got[a:b], y_ref[a:b])
            assert e < FWD_TOL, (n, e)
    bound = conv_bound(L.x, L.conv_w, L.conv_b, y_ref, W, dtype, L.cu_seqlens.cpu(), init)
    assert np.all(np.abs(got - y_ref) <= bound)
    # final states: exact; slots no sequence uses keep their bits
    for n in range(N):
        assert np.array_equal(to_np(pool[slots[n]]), fin_ref[n]), n
    spare = sorted(set(range(N + 3)) - set(slots.tolist()))
    assert torch.equal(bits(pool[spare]), bits(pool0[spare]))


def test_conv_without_state_and_without_activation():
    L = inputs.make_layer_inputs([130, 7], HK=1, HV=1, dk=16, dv=16, seed=66, C=64).to(DEV)
    y = gdn.gdn_causal_conv1d_fwd(L.x, L.conv_w, L.cu_seqlens, activation=False)
    y_ref, _ = ref.causal_conv1d(L.x, L.conv_w, L.cu_seqlens.cpu(), activation=False)
    assert bf16_err(to_np(y), y_ref) < FWD_TOL
    # slot indices outside the pool: zero initial state, pool untouched
    pool = torch.randn(1, 3, 64, device=DEV).to(torch.bfloat16)
    p0 = pool.clone()
    y2 = gdn.gdn_causal_conv1d_fwd(L.x, L.conv_w, L.cu_seqlens, conv_state=pool,
                                   state_indices=torch.tensor([-1, 5], dtype=torch.int32, device=DEV),
                                   activation=False)
    assert torch.equal(bits(y2), bits(y)) and torch.equal(bits(pool), bits(p0))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_conv_batch_and_mode_invariance(dtype):
    """A sequence's outputs and final state have the same bits alone or in a batch,
    in one prefill, in two chained prefills, or as a prefill followed by decode
    updates one token at a time (batched with other sequences)."""
    W, C = 4, 512
    lens = [700, 33, 129, 2]
    L = inputs.make_layer_inputs(lens, HK=1, HV=1, dk=16, dv=16, W=W, dtype=dtype, seed=67, C=C).to(DEV)
    pool = L.conv_state.clone()
    y = gdn.gdn_causal_conv1d_fwd(L.x, L.conv_w, L.cu_seqlens, bias=L.conv_b, conv_state=pool)
    Ln = lens[0]
    seq = L.x[:Ln]
    one = lambda m: inputs.cu_from_lengths([m]).to(DEV)  # noqa: E731
    # alone
    st = L.conv_state[0:1].clone()
    y1 = gdn.gdn_causal_conv1d_fwd(seq.contiguous(), L.conv_w, one(Ln), bias=L.conv_b, conv_state=st)
    assert torch.equal(bits(y1), bits(y[:Ln])) and torch.equal(bits(st[0]), bits(pool[0]))
    # two chained prefills (split off a tile boundary) and then decode updates
    P1, P2 = 257, 600
    st = L.conv_state[0:1].clone()
    ya = gdn.gdn_causal_conv1d_fwd(seq[:P1].contiguous(), L.conv_w, one(P1), bias=L.conv_b, conv_state=st)
    yb = gdn.gdn_causal_conv1d_fwd(seq[P1:P2].contiguous(), L.conv_w, one(P2 - P1), bias=L.conv_b, conv_state=st)
    outs = [ya, yb]
    # decode: the same sequence in slot 2 of a 3-slot pool, batched with two other sequences
    dpool = torch.randn(3, W - 1, C, device=DEV).to(dtype)
    dpool[2] = st[0]
    idx = torch.tensor([0, 2, 1], dtype=torch.int32, device=DEV)
    for t in range(P2, Ln):
        xb = torch.randn(3, C, device=DEV).to(dtype)
        xb[1] = seq[t]
        yt = gdn.gdn_causal_conv1d_update(xb, L.conv_w, dpool, state_indices=idx, bias=L.conv_b)
        outs.append(yt[1:2])
    assert torch.equal(bits(torch.cat(outs)), bits(y[:Ln]))
    assert torch.equal(bits(dpool[2]), bits(pool[0]))


def test_conv_update_vs_oracle_and_skips():
    C, W, B = 264, 4, 9
    L = inputs.make_layer_inputs([1] * B, HK=1, HV=1, dk=16, dv=16, W=W, seed=68, C=C).to(DEV)
    pool = torch.randn(12, W - 1, C, device=DEV).to(torch.bfloat16)
    idx = torch.tensor([3, -1, 0, 11, 7, 12, 5, 1, 2], dtype=torch.int32, device=DEV)  # -1 and 12: skipped
    y = torch.full((B, C), 7.0, device=DEV).to(torch.bfloat16)
    p0 = pool.clone()
    gdn.gdn_causal_conv1d_update(L.x, L.conv_w, pool, state_indices=idx, bias=L.conv_b, out=y)
    torch.cuda.synchronize()
    idx_ref = [i if 0 <= i < 12 else -1 for i in idx.tolist()]
    y_ref, st_ref = ref.causal_conv1d_update(L.x, L.conv_w, p0, state_indices=idx_ref, bias=L.conv_b)
    got = to_np(y)
    for b, s in enumerate(idx_ref):
        if s < 0:
            assert np.all(got[b] == 7.0)
        else:
            assert bf16_err(got[b], y_ref[b]) < FWD_TOL
    assert np.array_equal(to_np(pool), st_ref)


def test_conv_full_size_sampled():
    """The bench's prefill shape (C = 2*16*128 + 32*128 = 8192 channels) on a
    lognormal length mix, checked at sampled (token, channel) points."""
    lengths = inputs.lognormal_lengths(16, 4096, 16384, seed=4)
    L = inputs.make_layer_inputs(lengths, HK=16, HV=32, dk=128, dv=128, seed=69, device=DEV)
    pool = L.conv_state.clone()
    y = gdn.gdn_causal_conv1d_fwd(L.x, L.conv_w, L.cu_seqlens, bias=L.conv_b, conv_state=pool)
    torch.cuda.synchronize()
    rng = np.random.default_rng(0)
    T, C = L.x.shape
    cu = L.cu_seqlens.cpu().numpy()
    S = 4000
    ts = rng.integers(0, T, S)
    cs = rng.integers(0, C, S)
    ns = np.searchsorted(cu, ts, side="right") - 1
    cc = torch.from_numpy(cs).to(DEV)
    # the 4 input rows each sample sees: rows of its own sequence, else its conv state rows
    xw = np.zeros((S, 4))
    for j in range(4):
        r = ts - 3 + j
        inside = r >= cu[ns]
        fromx = to_np(L.x[torch.from_numpy(np.where(inside, r, 0)).to(DEV), cc])
        srow = torch.from_numpy(np.where(inside, 0, r - cu[ns] + 3)).to(DEV)
        fromst = to_np(L.conv_state[torch.from_numpy(ns).to(DEV), srow, cc])
        xw[:, j] = np.where(inside, fromx, fromst)
    w, bb = to_np(L.conv_w)[cs], to_np(L.conv_b)[cs]
    got = to_np(y[torch.from_numpy(ts).to(DEV), cc])
    for i in range(S):
        want = ref.causal_conv1d(xw[i][:, None], w[i:i + 1], [0, 4], bias=bb[i:i + 1])[0][3, 0]
        mag = abs(bb[i]) + np.abs(w[i] * xw[i]).sum()
        assert abs(got[i] - want) <= (BF16_ROUND + 40 * U32) * abs(want) + 4 * 5 * U32 * 1.1 * mag + 1e-30, i
    # final states: the last 3 rows of every sequence (all are longer than 3 tokens)
    assert min(lengths) >= 3
    last = torch.cat([L.x[int(cu[n + 1]) - 3:int(cu[n + 1])][None] for n in range(len(lengths))])
    assert torch.equal(bits(pool), bits(last))


def test_conv_all_sequences_empty():
    # T_total = 0 with N > 0: every slot keeps its state (initial state on) or is zeroed (off)
    C, W = 64, 4
    x = torch.empty(0, C, dtype=torch.bfloat16, device=DEV)
    w = torch.randn(C, W, device=DEV)
    pool = torch.randn(3, W - 1, C, device=DEV).to(torch.bfloat16)
    p0 = pool.clone()
    cu = torch.zeros(4, dtype=torch.int32, device=DEV)
    has = torch.tensor([1, 0, 1], dtype=torch.int32, device=DEV)
    y = gdn.gdn_causal_conv1d_fwd(x, w, cu, conv_state=pool, has_initial_state=has)
    torch.cuda.synchronize()
    assert y.shape == (0, C)
    assert torch.equal(bits(pool[0]), bits(p0[0])) and torch.equal(bits(pool[2]), bits(p0[2]))
    assert torch.all(pool[1] == 0)


def test_norm_and_gates_full_size_sampled():
    """The bench's shapes (T = 68,535 tokens here, HV = 32, dv = 128, bf16) at sampled rows."""
    lengths = inputs.lognormal_lengths(16, 4096, 16384, seed=4)
    L = inputs.make_layer_inputs(lengths, HK=16, HV=32, dk=128, dv=128, seed=70, device=DEV, C=16)
    y = gdn.gdn_gated_rmsnorm(L.o, L.z, L.norm_w)
    g, beta = gdn.gdn_gates(L.a, L.b, L.A_log, L.dt_bias)
    torch.cuda.synchronize()
    rng = np.random.default_rng(1)
    T = L.o.shape[0]
    ts = torch.from_numpy(rng.integers(0, T, 512)).to(DEV)
    want = ref.gated_rmsnorm(L.o[ts], L.z[ts], L.norm_w)
    got = to_np(y[ts])
    assert np.all(np.abs(got - want) <= (BF16_ROUND + 4e-5) * np.abs(want) + 1e-30)
    gr, br = ref.gates(L.a[ts], L.b[ts], L.A_log, L.dt_bias)
    assert np.all(np.abs(to_np(g[ts]) - gr) <= 4e-6 * np.abs(gr))
    assert np.all(np.abs(to_np(beta[ts]) - br) <= 4e-6 * np.abs(br))
