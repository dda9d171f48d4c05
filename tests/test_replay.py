"""Chunk-order-replaying prefill and decode (include/gdn_replay.h).

The Nemotron experiment makes decode agree with prefill by replaying the
chunked computation order instead of running the recurrent kernel everywhere
("Finish RL Training Faster: Bitwise-Consistent, High-Performance,
Agent-Driven").  Checked here: outputs and the replay cache against the fp64
oracle (within the forward tolerance; bf16 outputs net of their own
rounding), and bit-identical outputs and cache however a sequence's tokens are
split between prefill calls and decode steps and whatever shares its batch.
"""
import numpy as np
import pytest
import torch

import invariant_linear_attention_gb300 as gdn
from invariant_linear_attention_gb300 import inputs
import oracle
from helpers import FWD_TOL, bf16_err, normwise, to_np

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
C = gdn.binding.REPLAY_CHUNK


def bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)


def one(x, n, a, b):
    """Tokens a..b-1 of sequence n of x (an input set) as a one-sequence input set on the device."""
    c0 = int(x.cu_seqlens[n])
    sl = slice(c0 + a, c0 + b)
    return inputs.GDNInputs(x.q[sl].contiguous(), x.k[sl].contiguous(), x.v[sl].contiguous(), x.g[sl].contiguous(),
                            x.beta[sl].contiguous(), inputs.cu_from_lengths([b - a]).to(DEV), None, [b - a])


def pos(vals):
    return torch.tensor(vals, dtype=torch.int32, device=DEV)


@pytest.mark.parametrize("dtype,dk", [(torch.float32, 64), (torch.bfloat16, 128), (torch.float32, 32),
                                      (torch.float32, 16)])
def test_replay_prefill_vs_oracle(dtype, dk):
    lengths = [1, 63, 64, 65, 130, 200, 0, 7]
    N, HK, HV = len(lengths), 2, 4
    x = inputs.make_inputs(lengths, HK=HK, HV=HV, dk=dk, dv=dk, dtype=dtype, seed=81, init_scale=0.3)
    d = x.to(DEV)
    rs = gdn.replay_state_new(N, HV, dk, dk, init_state=d.init_state, device=DEV)
    out = gdn.gdn_replay_prefill(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, rs)
    torch.cuda.synchronize()
    o_ref, _ = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, init_state=x.init_state)
    got = to_np(out)
    cu = x.cu_seqlens.tolist()
    for n in range(N):
        for h in range(HV):
            a, b = cu[n], cu[n + 1]
            if b > a:
                err = (bf16_err if dtype == torch.bfloat16 else normwise)(got[a:b, h], o_ref[a:b, h])
                assert err < FWD_TOL, (n, h, err)
    # the cache: chunk-start state, k^ rows, d rows, cumulative log-decays
    states, _ = oracle.gdn_replay_state(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, init_state=x.init_state, chunk=C)
    views = gdn.replay_views(rs, dk, dk)
    for n, st in enumerate(states):
        r = st["r"]
        for h in range(HV):
            assert normwise(to_np(views["S0"][n, h]), st["S0"][h]) < FWD_TOL, (n, h)
            if r:
                assert normwise(to_np(views["K"][n, h, :r]), st["K"][:, h]) < 1e-5
                assert normwise(to_np(views["D"][n, h, :r]), st["D"][:, h]) < FWD_TOL, (n, h)
                assert np.allclose(to_np(views["gam"][n, h, :r]), st["gam"][:, h], rtol=1e-5, atol=1e-6)


@pytest.mark.parametrize("dtype,dk", [(torch.bfloat16, 64), (torch.float32, 64), (torch.float32, 16)])
def test_replay_decode_bitwise_equals_prefill(dtype, dk):
    """Prefill of P tokens then decode steps (batched with other sequences, in
    permuted slots) gives the bits of one prefill over the whole sequence."""
    L = 150
    HK, HV = 2, 4
    x = inputs.make_inputs([L], HK=HK, HV=HV, dk=dk, dv=dk, dtype=dtype, seed=82, init_scale=0.2, device=DEV)
    full_rs = gdn.replay_state_new(1, HV, dk, dk, init_state=x.init_state, device=DEV)
    full = gdn.gdn_replay_prefill(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, full_rs)
    others = inputs.make_inputs([L] * 2, HK=HK, HV=HV, dk=dk, dv=dk, dtype=dtype, seed=83, init_scale=0.2,
                                device=DEV)
    for P in (0, 1, 63, 64, 100):
        rs = gdn.replay_state_new(5, HV, dk, dk, device=DEV)
        gdn.replay_views(rs, dk, dk)["S0"][3].copy_(x.init_state[0])
        outs = []
        if P:
            pre = one(x, 0, 0, P)
            outs.append(gdn.gdn_replay_prefill(pre.q, pre.k, pre.v, pre.g, pre.beta, pre.cu_seqlens, rs,
                                               state_indices=pos([3]), seq_pos=pos([0])))
        # two other sequences decode alongside, in slots 0 and 4 (their own states)
        idx = pos([0, 3, 4])
        for t in range(P, L):
            sl = [int(others.cu_seqlens[0]) + t, t, int(others.cu_seqlens[1]) + t]
            src = [others, x, others]
            q = torch.stack([s.q[i] for s, i in zip(src, sl)])
            k = torch.stack([s.k[i] for s, i in zip(src, sl)])
            v = torch.stack([s.v[i] for s, i in zip(src, sl)])
            g = torch.stack([s.g[i] for s, i in zip(src, sl)])
            b = torch.stack([s.beta[i] for s, i in zip(src, sl)])
            o = gdn.gdn_replay_decode(q, k, v, g, b, rs, pos([t, t, t]), state_indices=idx)
            outs.append(o[1:2])
        torch.cuda.synchronize()
        assert torch.equal(bits(torch.cat(outs)), bits(full)), P
        assert _same_live_rows(rs[3], full_rs[0], L, dk), P


def _same_live_rows(a, b, L, dk):
    """Replay states agree on everything a continuation reads: S0 and rows 0 .. L mod C - 1."""
    va, vb = gdn.replay_views(a[None], dk, dk), gdn.replay_views(b[None], dk, dk)
    r = L % C
    return (torch.equal(bits(va["S0"]), bits(vb["S0"])) and torch.equal(bits(va["K"][..., :r, :]), bits(vb["K"][..., :r, :]))
            and torch.equal(bits(va["D"][..., :r, :]), bits(vb["D"][..., :r, :]))
            and torch.equal(bits(va["gam"][..., :r]), bits(vb["gam"][..., :r])))


def test_replay_chained_prefills_and_batch_invariance():
    lengths = [300, 17, 64, 129]
    HK, HV, dk = 2, 4, 128
    x = inputs.make_inputs(lengths, HK=HK, HV=HV, dk=dk, dv=dk, dtype=torch.bfloat16, seed=84, init_scale=0.1,
                           device=DEV)
    rs = gdn.replay_state_new(4, HV, dk, dk, init_state=x.init_state, device=DEV)
    out = gdn.gdn_replay_prefill(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, rs)
    for n, Ln in enumerate(lengths):
        c0 = int(x.cu_seqlens[n])
        # alone
        rs1 = gdn.replay_state_new(1, HV, dk, dk, init_state=x.init_state[n:n + 1], device=DEV)
        s = one(x, n, 0, Ln)
        o1 = gdn.gdn_replay_prefill(s.q, s.k, s.v, s.g, s.beta, s.cu_seqlens, rs1)
        assert torch.equal(bits(o1), bits(out[c0:c0 + Ln])), n
        assert _same_live_rows(rs1[0], rs[n], Ln, dk), n
        # split into two prefill calls at a point inside a chunk
        P = Ln // 3 + 1
        rs2 = gdn.replay_state_new(1, HV, dk, dk, init_state=x.init_state[n:n + 1], device=DEV)
        a, b = one(x, n, 0, P), one(x, n, P, Ln)
        oa = gdn.gdn_replay_prefill(a.q, a.k, a.v, a.g, a.beta, a.cu_seqlens, rs2)
        ob = gdn.gdn_replay_prefill(b.q, b.k, b.v, b.g, b.beta, b.cu_seqlens, rs2, seq_pos=pos([P]))
        assert torch.equal(bits(torch.cat([oa, ob])), bits(out[c0:c0 + Ln])), n
        assert _same_live_rows(rs2[0], rs[n], Ln, dk), n


def test_replay_skips_invalid_slots():
    x = inputs.make_inputs([5, 5], HK=1, HV=2, dk=32, dv=32, dtype=torch.float32, seed=85, device=DEV)
    rs = gdn.replay_state_new(1, 2, 32, 32, device=DEV)
    rs0 = rs.clone()
    out = torch.full_like(x.v, 7.0)
    gdn.gdn_replay_prefill(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, rs, state_indices=pos([-1, 9]), out=out)
    torch.cuda.synchronize()
    assert torch.all(out == 7.0) and torch.equal(rs, rs0)
    d = inputs.make_inputs([1, 1], HK=1, HV=2, dk=32, dv=32, dtype=torch.float32, seed=86, device=DEV)
    o = torch.full_like(d.v, 7.0)
    gdn.gdn_replay_decode(d.q, d.k, d.v, d.g, d.beta, rs, pos([0, 0]), state_indices=pos([-1, 0]), out=o)
    torch.cuda.synchronize()
    assert torch.all(o[0] == 7.0) and not torch.all(o[1] == 7.0)


def test_replay_bench_shape_vs_oracle():
    """The bench's head shape (HK=16, HV=32, dk=dv=128, bf16) on two long sequences."""
    lengths = [4096, 1000]
    x = inputs.make_inputs(lengths, HK=16, HV=32, dk=128, dv=128, dtype=torch.bfloat16, seed=87, init_scale=0.05)
    d = x.to(DEV)
    rs = gdn.replay_state_new(2, 32, 128, 128, init_state=d.init_state, device=DEV)
    out = gdn.gdn_replay_prefill(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, rs)
    torch.cuda.synchronize()
    o_ref, _ = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, init_state=x.init_state)
    errs = [bf16_err(to_np(out[a:b, h]), o_ref[a:b, h]) for a, b in ((0, 4096), (4096, 5096)) for h in range(32)]
    assert max(errs) < FWD_TOL
