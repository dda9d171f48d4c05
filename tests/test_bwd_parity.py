"""GPU chunked (WY-form) backward vs the fp64 BPTT oracle (itself pinned by
finite differences in test_oracle_pins.py).  Tolerance: normwise-max
relative error 1e-2 per gradient tensor, per (sequence, head) where the
tensor has one.  Cases span partial and exact chunks (chunk = 64), empty
sequences, GQA folding, both dtypes, the l2norm switch, and sampled units of
the 8 x 4096-token workload."""
import dataclasses

import numpy as np
import pytest
import torch

import invariant_linear_attention_gb300 as gdn
from invariant_linear_attention_gb300 import inputs
import oracle
from helpers import GRAD_TOL, normwise, to_np

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "d_init_state")


def run(x, dO, dsT=None, use_qk_l2norm=True):
    d = x.to(DEV)
    got = gdn.gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, dO.to(DEV), init_state=d.init_state,
                            d_final_state=None if dsT is None else dsT.to(DEV), use_qk_l2norm=use_qk_l2norm)
    torch.cuda.synchronize()
    ref = oracle.gdn_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, dO, init_state=x.init_state,
                         d_final_state=dsT, use_qk_l2norm=use_qk_l2norm)
    return {k: to_np(v) for k, v in got.items() if v is not None}, ref


def check(got, ref, cu, skip=()):
    cu = [int(c) for c in cu]
    for name in NAMES:
        if name in skip:
            continue
        g, r = got[name], ref[name]
        if name == "d_init_state":
            for n in range(g.shape[0]):
                for h in range(g.shape[1]):
                    e = normwise(g[n, h], r[n, h])
                    assert e < GRAD_TOL, (name, n, h, e)
            continue
        for n in range(len(cu) - 1):
            a, b = cu[n], cu[n + 1]
            if a == b:
                continue
            for h in range(g.shape[1]):
                e = normwise(g[a:b, h], r[a:b, h])
                assert e < GRAD_TOL, (name, n, h, e)


def test_tiny_config_fp32():
    x = inputs.tiny_config(seed=0)
    dO = inputs.grad_out(64, 2, 16, dtype=torch.float32, seed=6)
    got, ref = run(x, dO)
    check(got, ref, x.cu_seqlens)
    assert max(normwise(got[k], ref[k]) for k in NAMES) < 1e-4  # fp32 end to end


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (32, 128), (64, 32), (32, 64)])
def test_varlen_chunks(dtype, dk, dv):
    lengths = [65, 1, 0, 64, 130, 37]
    x = inputs.make_inputs(lengths, HK=2, HV=4, dk=dk, dv=dv, dtype=dtype, seed=21, init_scale=0.2)
    T = sum(lengths)
    dO = inputs.grad_out(T, 4, dv, dtype=dtype, seed=22)
    dsT = inputs.random_states(len(lengths), 4, dv, dk, seed=23, scale=0.5)
    got, ref = run(x, dO, dsT)
    check(got, ref, x.cu_seqlens)


def test_no_init_no_dfinal_no_l2norm():
    lengths = [100, 29]
    x = inputs.make_inputs(lengths, HK=1, HV=2, dk=64, dv=64, dtype=torch.float32, seed=24)
    dO = inputs.grad_out(sum(lengths), 2, 64, dtype=torch.float32, seed=25)
    got, ref = run(x, dO, None, use_qk_l2norm=False)
    check(got, ref, x.cu_seqlens)


def test_no_l2norm_bf16_head128():
    """use_qk_l2norm off (inputs drawn unit-norm, then rounded to bf16) through the tcgen05
    kernels (bf16, dk = dv = 128)."""
    lengths = [150, 64, 9]
    x = inputs.make_inputs(lengths, HK=1, HV=2, dk=128, dv=128, dtype=torch.bfloat16, seed=28, init_scale=0.1)
    dO = inputs.grad_out(sum(lengths), 2, 128, seed=29)
    got, ref = run(x, dO, None, use_qk_l2norm=False)
    check(got, ref, x.cu_seqlens)


@pytest.mark.parametrize("lengths", [[9, 20], [1], [63]])
def test_short_batch_head128(lengths):
    """A packed batch shorter than one chunk through the tcgen05 kernels (bf16, dk = dv = 128):
    the tensor copies' 64-row boxes reach past T_total (read as zeros) and past each sequence."""
    x = inputs.make_inputs(lengths, HK=2, HV=4, dk=128, dv=128, dtype=torch.bfloat16, seed=31, init_scale=0.2)
    dO = inputs.grad_out(sum(lengths), 4, 128, seed=32)
    dsT = inputs.random_states(len(lengths), 4, 128, 128, seed=33, scale=0.5)
    got, ref = run(x, dO, dsT)
    check(got, ref, x.cu_seqlens)


def test_backward_workload_sampled():
    """gdn_chunk_bwd on 8 x 4096 tokens, HK=16, HV=32, dk=dv=128, bf16, as the
    benchmark launches it; the oracle recomputes sampled (sequence, k-head)
    groups (both value heads of the k-head, so the GQA fold is covered)."""
    N, L = 8, 4096
    d = inputs.make_inputs([L] * N, HK=16, HV=32, dk=128, dv=128, dtype=torch.bfloat16, seed=6, device=DEV)
    dO = inputs.grad_out(N * L, 32, 128, seed=6, device=DEV)
    got = gdn.gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, dO)
    torch.cuda.synchronize()
    x = d.cpu()
    dOc = dO.cpu()
    for n, hk in ((0, 0), (5, 11)):
        a, b = n * L, (n + 1) * L
        hs = slice(2 * hk, 2 * hk + 2)
        ref = oracle.gdn_bwd(x.q[a:b, hk:hk + 1], x.k[a:b, hk:hk + 1], x.v[a:b, hs], x.g[a:b, hs],
                             x.beta[a:b, hs], [0, L], dOc[a:b, hs])
        pairs = {"dq": (got["dq"][a:b, hk], ref["dq"][:, 0]), "dk": (got["dk"][a:b, hk], ref["dk"][:, 0])}
        for j in range(2):
            h = 2 * hk + j
            pairs[f"dv{j}"] = (got["dv"][a:b, h], ref["dv"][:, j])
            pairs[f"dg{j}"] = (got["dg"][a:b, h], ref["dg"][:, j])
            pairs[f"dbeta{j}"] = (got["dbeta"][a:b, h], ref["dbeta"][:, j])
            pairs[f"dS0{j}"] = (got["d_init_state"][n, h], ref["d_init_state"][0, j])
        for name, (g, r) in pairs.items():
            e = normwise(to_np(g), r)
            assert e < GRAD_TOL, (n, hk, name, e)


def test_deterministic():
    x = inputs.make_inputs([200, 77], HK=2, HV=4, dk=128, dv=128, dtype=torch.bfloat16, seed=26, init_scale=0.1)
    dO = inputs.grad_out(277, 4, 128, seed=27)
    d = x.to(DEV)
    a = gdn.gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, dO.to(DEV), init_state=d.init_state)
    b = gdn.gdn_chunk_bwd(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, dO.to(DEV), init_state=d.init_state)
    torch.cuda.synchronize()
    for k in NAMES:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("dtype,dk,dv", [(torch.bfloat16, 128, 128), (torch.float32, 64, 64)])
def test_strong_decay(dtype, dk, dv):
    """Log-decays about eight times the usual draw (a chunk's cumulative decay reaches several
    hundred): the decay factors between two positions of a chunk are only ever taken in the
    decaying direction, so no exp overflows into a NaN.  Both the tcgen05 and the mma.sync
    kernels."""
    lengths = [130, 64, 21]
    x = inputs.make_inputs(lengths, HK=1, HV=2, dk=dk, dv=dv, dtype=dtype, seed=34, init_scale=0.2)
    x = dataclasses.replace(x, g=(x.g * 8.0).contiguous())
    assert float(x.g[:64].sum()) < -300.0
    dO = inputs.grad_out(sum(lengths), 2, dv, dtype=dtype, seed=35)
    dsT = inputs.random_states(len(lengths), 2, dv, dk, seed=36, scale=0.5)
    got, ref = run(x, dO, dsT)
    for name, v in got.items():
        assert np.isfinite(v).all(), name
    check(got, ref, x.cu_seqlens)


@pytest.mark.parametrize("HK,HV", [(2, 2), (1, 4)])
def test_fold_group_sizes_head128(HK, HV):
    """G = HV / HK value heads per k-head of 1 and 4 through the tcgen05 kernels (bf16, dk = dv =
    128), whose last value-head CTA of each (chunk, k-head) folds dq and dk on chip."""
    lengths = [130, 7, 64]
    x = inputs.make_inputs(lengths, HK=HK, HV=HV, dk=128, dv=128, dtype=torch.bfloat16, seed=37, init_scale=0.2)
    dO = inputs.grad_out(sum(lengths), HV, 128, seed=38)
    dsT = inputs.random_states(len(lengths), HV, 128, 128, seed=39, scale=0.5)
    got, ref = run(x, dO, dsT)
    check(got, ref, x.cu_seqlens)


def test_deterministic_many_ctas():
    """Bitwise-equal gradients over three calls with thousands of CTAs in flight (4 x 1024 tokens,
    32 value heads): which value-head CTA folds a (chunk, k-head) changes from run to run, the sums
    it takes do not."""
    x = inputs.make_inputs([1024] * 4, HK=16, HV=32, dk=128, dv=128, dtype=torch.bfloat16, seed=40, device=DEV)
    dO = inputs.grad_out(4096, 32, 128, seed=41, device=DEV)
    runs = [gdn.gdn_chunk_bwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, dO) for _ in range(3)]
    torch.cuda.synchronize()
    for k in ("dq", "dk", "dv", "dg", "dbeta"):
        assert torch.equal(runs[0][k], runs[1][k]) and torch.equal(runs[0][k], runs[2][k]), k


def test_many_ragged_sequences_head128():
    """Forty sequences of 0 to 190 tokens (many partial chunks, some empty, some a single token)
    through the tcgen05 kernels (bf16, dk = dv = 128), against the oracle per (sequence, head)."""
    rng = np.random.default_rng(42)
    lengths = [int(v) for v in rng.integers(0, 191, size=40)]
    lengths[3], lengths[7], lengths[11] = 0, 1, 64
    x = inputs.make_inputs(lengths, HK=2, HV=4, dk=128, dv=128, dtype=torch.bfloat16, seed=43, init_scale=0.2)
    dO = inputs.grad_out(sum(lengths), 4, 128, seed=44)
    dsT = inputs.random_states(len(lengths), 4, 128, 128, seed=45, scale=0.5)
    got, ref = run(x, dO, dsT)
    check(got, ref, x.cu_seqlens)


@pytest.mark.parametrize("scale", [1e5, 1e-6])
def test_state_magnitudes_head128(scale):
    """Values and output gradients scaled so that the chunk states reach far above fp16's largest
    value (1e5) or far below its smallest normal one (1e-6) through
    the tcgen05 kernels (bf16, dk = dv = 128), which store S and D as fp16 with a power-of-two
    factor per 32 x 32 tile: the relative errors stay those of unscaled inputs."""
    lengths = [200, 64, 37]
    x = inputs.make_inputs(lengths, HK=1, HV=2, dk=128, dv=128, dtype=torch.bfloat16, seed=46, init_scale=0.2)
    x = dataclasses.replace(x, v=(x.v.float() * scale).to(x.v.dtype), init_state=x.init_state * scale)
    dO = (inputs.grad_out(sum(lengths), 2, 128, seed=47).float() * scale).to(torch.bfloat16)
    dsT = inputs.random_states(len(lengths), 2, 128, 128, seed=48, scale=0.5) * scale
    got, ref = run(x, dO, dsT)
    for name, v in got.items():
        assert np.isfinite(v).all(), name
    check(got, ref, x.cu_seqlens)
