"""Prefix-cache state snapshots (gdn_recurrent_fwd_snapshots).

The pages keep prefix caching working with the recurrent kernel by reusing the
serving engine's state snapshots ("Defending Against the Training-Inference
Numeric Mismatch in RL (Especially Linear Attention)", section 3.2).  A
snapshot after m * snap_every tokens must be bit for bit the final state of
the forward over that prefix, and resuming from it must reproduce the rest of
the sequence bit for bit; against the fp64 oracle it sits within the forward
tolerance like any final state.
"""
import numpy as np
import pytest
import torch

import invariant_linear_attention_gb300 as gdn
from invariant_linear_attention_gb300 import inputs
import oracle
from helpers import FWD_TOL, normwise, to_np

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def seq_slice(x, n, a, b):
    """Tokens a..b-1 of sequence n as a one-sequence input set."""
    c0 = int(x.cu_seqlens[n])
    sl = slice(c0 + a, c0 + b)
    return inputs.GDNInputs(x.q[sl], x.k[sl], x.v[sl], x.g[sl], x.beta[sl], inputs.cu_from_lengths([b - a]).to(DEV),
                            None, [b - a])


@pytest.mark.parametrize("snap_every", [32, 64, 128])
def test_snapshots_equal_prefix_states_and_resume(snap_every):
    lengths = [300, 64, 31, 256, 0, 513]
    x = inputs.make_inputs(lengths, HK=16, HV=32, dk=128, dv=128, dtype=torch.bfloat16, seed=41, init_scale=0.1,
                           device=DEV)
    out, fs, snaps, snap_cu = gdn.gdn_recurrent_fwd_snapshots(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, snap_every,
                                                              init_state=x.init_state)
    torch.cuda.synchronize()
    cu = snap_cu.cpu().tolist()
    assert cu == [0] + list(np.cumsum([L // snap_every for L in lengths]))
    # the plain forward gives the same outputs and final states
    out0, fs0 = gdn.gdn_recurrent_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, init_state=x.init_state)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
    assert torch.equal(fs.view(torch.int32), fs0.view(torch.int32))
    for n, L in enumerate(lengths):
        for m in range(1, L // snap_every + 1):
            P = m * snap_every
            pre = seq_slice(x, n, 0, P)
            _, fp = gdn.gdn_recurrent_fwd(pre.q, pre.k, pre.v, pre.g, pre.beta, pre.cu_seqlens,
                                          init_state=x.init_state[n:n + 1].contiguous())
            torch.cuda.synchronize()
            snap = snaps[cu[n] + m - 1]
            assert torch.equal(snap.view(torch.int32), fp[0].view(torch.int32)), (n, m)
            if m == 1 and P < L:
                # resume from the snapshot: the rest of the sequence comes out bit for bit
                rest = seq_slice(x, n, P, L)
                o_r, f_r = gdn.gdn_recurrent_fwd(rest.q, rest.k, rest.v, rest.g, rest.beta, rest.cu_seqlens,
                                                 init_state=snap[None].contiguous())
                torch.cuda.synchronize()
                c0 = int(x.cu_seqlens[n])
                assert torch.equal(o_r.view(torch.int16), out[c0 + P:c0 + L].view(torch.int16)), (n, m)
                assert torch.equal(f_r.view(torch.int32), fs[n:n + 1].view(torch.int32)), (n, m)


def test_snapshot_vs_oracle():
    lengths = [192, 97]
    x = inputs.make_inputs(lengths, HK=2, HV=4, dk=64, dv=64, dtype=torch.float32, seed=42, init_scale=0.2)
    d = x.to(DEV)
    _, _, snaps, snap_cu = gdn.gdn_recurrent_fwd_snapshots(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, 64,
                                                           init_state=d.init_state)
    torch.cuda.synchronize()
    cu = snap_cu.cpu().tolist()
    for n, L in enumerate(lengths):
        c0 = int(x.cu_seqlens[n])
        for m in range(1, L // 64 + 1):
            P = 64 * m
            _, f_ref = oracle.gdn_fwd(x.q[c0:c0 + P], x.k[c0:c0 + P], x.v[c0:c0 + P], x.g[c0:c0 + P],
                                      x.beta[c0:c0 + P], [0, P], init_state=x.init_state[n:n + 1])
            for h in range(4):
                assert normwise(to_np(snaps[cu[n] + m - 1, h]), f_ref[0, h]) < FWD_TOL


def test_snapshot_interval_must_align_with_chunks():
    x = inputs.make_inputs([64], HK=1, HV=1, dk=32, dv=32, dtype=torch.float32, seed=43, device=DEV)
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_recurrent_fwd_snapshots(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, 48)
    assert ei.value.code == -2


def test_snapshot_slots_bounded():
    # fewer slots than snapshots: the extra ones are dropped, nothing is written out of range
    lengths = [256]
    x = inputs.make_inputs(lengths, HK=1, HV=2, dk=32, dv=32, dtype=torch.float32, seed=44, device=DEV)
    snap_cu = torch.tensor([0, 4], dtype=torch.int32, device=DEV)
    snaps = torch.full((2 + 1, 2, 32, 32), float("nan"), device=DEV)
    view = snaps[:2]
    gdn.gdn_recurrent_fwd_snapshots(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, 64, snap_cu=snap_cu,
                                    snap_states=view)
    torch.cuda.synchronize()
    assert not torch.isnan(snaps[:2]).any()
    assert torch.isnan(snaps[2]).all()


def test_decode_resumes_from_snapshot_bitwise():
    """A snapshot taken by the prefill, continued by decode steps, gives the bits
    of the full prefill (prefix caching followed by generation)."""
    L, every = 200, 64
    x = inputs.make_inputs([L], HK=2, HV=4, dk=64, dv=64, dtype=torch.bfloat16, seed=45, init_scale=0.1, device=DEV)
    out, fs, snaps, snap_cu = gdn.gdn_recurrent_fwd_snapshots(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, every,
                                                              init_state=x.init_state)
    P = 2 * every
    pool = torch.zeros(3, 4, 64, 64, device=DEV)
    pool[1] = snaps[1]  # the state after 128 tokens
    idx = torch.tensor([1], dtype=torch.int32, device=DEV)
    for t in range(P, L):
        o = gdn.gdn_decode_step(x.q[t:t + 1], x.k[t:t + 1], x.v[t:t + 1], x.g[t:t + 1], x.beta[t:t + 1], pool,
                                state_indices=idx)
        assert torch.equal(o.view(torch.int16), out[t:t + 1].view(torch.int16)), t
    torch.cuda.synchronize()
    assert torch.equal(pool[1].view(torch.int32), fs[0].view(torch.int32))
