"""Bitwise batch invariance and prefill/decode parity.

The order follows the pages' verification order: first a request alone vs in
mixed batches, then whole-prompt prefill vs token-by-token decode
("Finish RL Training Faster: Bitwise-Consistent, High-Performance,
Agent-Driven" as summarised in "train-inference-consistency", section
"Consistency has several layers"; the split point is part of the
computation: "bitwise parity / linear attention", section "Why linear
attention is the next wall").  Every comparison is byte equality.
"""
import numpy as np
import pytest
import torch

import invariant_linear_attention_gb300 as gdn
from invariant_linear_attention_gb300 import inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
SHAPE = dict(HK=16, HV=32, dk=128, dv=128, dtype=torch.bfloat16)


def fwd(x, dv_slice=0):
    d = x.to(DEV)
    out, fs = gdn.gdn_recurrent_fwd(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, init_state=d.init_state,
                                    dv_slice=dv_slice)
    torch.cuda.synchronize()
    return out.cpu(), fs.cpu()


def seq(x, i):
    return inputs.GDNInputs(*(t for t in (
        x.q[x.cu_seqlens[i]:x.cu_seqlens[i + 1]], x.k[x.cu_seqlens[i]:x.cu_seqlens[i + 1]],
        x.v[x.cu_seqlens[i]:x.cu_seqlens[i + 1]], x.g[x.cu_seqlens[i]:x.cu_seqlens[i + 1]],
        x.beta[x.cu_seqlens[i]:x.cu_seqlens[i + 1]])),
        cu_seqlens=inputs.cu_from_lengths([x.lengths[i]]),
        init_state=None if x.init_state is None else x.init_state[i:i + 1].clone(),
        lengths=[x.lengths[i]])


@pytest.mark.parametrize("init_scale", [0.0, 0.1])
def test_batch_invariance(init_scale):
    lengths = inputs.uniform_lengths(8, 1, 512, seed=1)
    targets = inputs.make_inputs(lengths, seed=1, init_scale=init_scale, **SHAPE)
    comp_lengths = inputs.uniform_lengths(63, 1, 512, seed=2)
    pool = inputs.make_inputs(comp_lengths, seed=2, init_scale=init_scale, **SHAPE)
    companions = [seq(pool, j) for j in range(63)]
    rng = np.random.default_rng(2)
    for i in range(8):
        alone = seq(targets, i)
        ref_o, ref_s = fwd(alone)
        for bsz in (1, 8, 64):
            parts = [companions[j] for j in rng.permutation(63)[:bsz - 1]]
            pos = int(rng.integers(0, bsz))
            parts.insert(pos, alone)
            batch = inputs.concat(parts)
            for dv_slice in (128, 64, 32):
                out, fs = fwd(batch, dv_slice=dv_slice)
                a, b = int(batch.cu_seqlens[pos]), int(batch.cu_seqlens[pos + 1])
                assert torch.equal(out[a:b].view(torch.int16), ref_o.view(torch.int16)), (i, bsz, dv_slice)
                assert torch.equal(fs[pos:pos + 1].view(torch.int32), ref_s.view(torch.int32)), (i, bsz, dv_slice)


def test_per_length_slices_are_bit_neutral():
    """The scheduler splits the heads of a sequence longer than 1.5 (3) times the
    average work per CTA slot over 2 (4) CTAs, with fewer rows per thread.  With
    152 SMs (304 slots) and HV = 32 these lengths give one 4-way split (3000
    tokens), one 2-way split (1200) and 18 whole heads (100); any other device
    splits differently, and the bits must not change either way: automatic
    slices, forced whole heads, forced quarter heads and each sequence alone
    agree."""
    lengths = [100] * 9 + [3000] + [100] * 9 + [1200]
    x = inputs.make_inputs(lengths, seed=11, init_scale=0.1, **SHAPE)
    auto_o, auto_s = fwd(x)
    for dv_slice in (128, 32):
        o, s = fwd(x, dv_slice=dv_slice)
        assert torch.equal(o.view(torch.int16), auto_o.view(torch.int16)), dv_slice
        assert torch.equal(s.view(torch.int32), auto_s.view(torch.int32)), dv_slice
    cu = x.cu_seqlens.tolist()
    for i in (9, 19, 0):
        o, s = fwd(seq(x, i))
        assert torch.equal(o.view(torch.int16), auto_o[cu[i]:cu[i + 1]].view(torch.int16)), i
        assert torch.equal(s.view(torch.int32), auto_s[i:i + 1].view(torch.int32)), i


def _decode_tokens(x, n_prompt, state, graph=False):
    """Run tokens n_prompt.. of every sequence (all the same length) through gdn_decode_step."""
    N = len(x.lengths)
    L = x.lengths[0]
    d = x.to(DEV)
    cu = x.cu_seqlens.tolist()
    idx = torch.tensor([cu[n] for n in range(N)], dtype=torch.long, device=DEV)
    outs = []
    if not graph:
        for t in range(n_prompt, L):
            sel = idx + t
            outs.append(gdn.gdn_decode_step(d.q[sel].contiguous(), d.k[sel].contiguous(), d.v[sel].contiguous(),
                                            d.g[sel].contiguous(), d.beta[sel].contiguous(), state))
        torch.cuda.synchronize()
        return torch.stack(outs, 1).cpu()
    # CUDA-graph capture of the whole decode loop on static buffers
    steps = L - n_prompt
    sel_all = (idx[:, None] + torch.arange(n_prompt, L, device=DEV)[None, :])  # [N, steps]
    qs = d.q[sel_all].transpose(0, 1).contiguous()
    ks = d.k[sel_all].transpose(0, 1).contiguous()
    vs = d.v[sel_all].transpose(0, 1).contiguous()
    gs = d.g[sel_all].transpose(0, 1).contiguous()
    bs = d.beta[sel_all].transpose(0, 1).contiguous()
    out = torch.empty(steps, N, *x.v.shape[1:], dtype=x.v.dtype, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph_obj = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph_obj, stream=s):
            for t in range(steps):
                gdn.gdn_decode_step(qs[t], ks[t], vs[t], gs[t], bs[t], state, out=out[t])
    torch.cuda.current_stream().wait_stream(s)
    graph_obj.replay()
    torch.cuda.synchronize()
    return out.transpose(0, 1).cpu()


@pytest.mark.parametrize("graph", [False, True])
def test_prefill_decode_parity(graph):
    N, L, P = 4, 2304, 2048
    x = inputs.make_inputs([L] * N, seed=3, init_scale=0.0, **SHAPE)
    full_o, full_s = fwd(x)
    # prompt through the recurrent forward
    prompt = inputs.GDNInputs(
        *(torch.cat([t[n * L:n * L + P] for n in range(N)]) for t in (x.q, x.k, x.v, x.g, x.beta)),
        cu_seqlens=inputs.cu_from_lengths([P] * N), init_state=x.init_state, lengths=[P] * N)
    p_o, p_s = fwd(prompt)
    state = p_s.to(DEV).contiguous()
    dec = _decode_tokens(x, P, state, graph=graph)  # [N, L-P, HV, dv]
    for n in range(N):
        assert torch.equal(p_o[n * P:(n + 1) * P].view(torch.int16), full_o[n * L:n * L + P].view(torch.int16))
        assert torch.equal(dec[n].view(torch.int16), full_o[n * L + P:(n + 1) * L].view(torch.int16)), n
    assert torch.equal(state.cpu().view(torch.int32), full_s.view(torch.int32))


def test_random_prefill_splits():
    N, L = 3, 700
    x = inputs.make_inputs([L] * N, seed=7, init_scale=0.1, **SHAPE)
    full_o, full_s = fwd(x)
    rng = np.random.default_rng(7)
    cuts = sorted(set(int(c) for c in rng.integers(1, L, size=4))) + [L]
    state = x.init_state.clone()
    start = 0
    pieces = []
    for c in cuts:
        part = inputs.GDNInputs(
            *(torch.cat([t[n * L + start:n * L + c] for n in range(N)]) for t in (x.q, x.k, x.v, x.g, x.beta)),
            cu_seqlens=inputs.cu_from_lengths([c - start] * N), init_state=state, lengths=[c - start] * N)
        o, state = fwd(part)
        pieces.append(o.view(N, c - start, *o.shape[1:]))
        start = c
    got = torch.cat(pieces, 1).reshape(full_o.shape)
    assert torch.equal(got.view(torch.int16), full_o.view(torch.int16))
    assert torch.equal(state.view(torch.int32), full_s.view(torch.int32))


def test_decode_pool_permutation_invariance():
    # the same sequences decoded through a permuted slot pool give the same bits
    B = 16
    x = inputs.make_inputs([1] * B, seed=8, **SHAPE)
    pool = inputs.random_states(B, 32, 128, 128, seed=9, scale=0.5)
    d = x.to(DEV)
    st_a = pool.to(DEV)
    out_a = gdn.gdn_decode_step(d.q, d.k, d.v, d.g, d.beta, st_a)
    perm = torch.randperm(B, generator=torch.Generator().manual_seed(9))
    pool_b = torch.empty(B + 5, *pool.shape[1:])
    pool_b[perm] = pool
    st_b = pool_b.to(DEV)
    out_b = gdn.gdn_decode_step(d.q, d.k, d.v, d.g, d.beta, st_b, state_indices=perm.to(torch.int32).to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(out_a.cpu().view(torch.int16), out_b.cpu().view(torch.int16))
    assert torch.equal(st_a.cpu()[torch.arange(B)].view(torch.int32), st_b.cpu()[perm].view(torch.int32))
