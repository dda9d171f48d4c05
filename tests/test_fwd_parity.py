"""GPU recurrent forward and decode step vs the fp64 oracle, element by element.

Tolerance: normwise-max relative error 2e-3 per (sequence, head) for out and
final_state.  Cases span several 16-token chunks and ragged tails, empty
sequences, every supported dk/dv, fp32 and bf16, the l2norm switch, all
dv slices, and at the end the full-size throughput workload on sampled units.
"""
import numpy as np
import pytest
import torch

import invariant_linear_attention_gb300 as gdn
from invariant_linear_attention_gb300 import inputs
import oracle
from helpers import FWD_TOL, bf16_err, normwise, per_unit_errors, to_np

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def fp32_twin(x):
    """The same inputs widened exactly to fp32 (bf16 values are fp32 values)."""
    return inputs.GDNInputs(x.q.float(), x.k.float(), x.v.float(), x.g, x.beta, x.cu_seqlens, x.init_state,
                            list(x.lengths))


def run_both(x, use_qk_l2norm=True, dv_slice=0):
    """Run the kernel; for bf16 also its fp32 twin, check the bit relation between
    the two, and return the fp32 values for the oracle comparison."""
    d = x.to(DEV)
    out, fs = gdn.gdn_recurrent_fwd(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, init_state=d.init_state,
                                    use_qk_l2norm=use_qk_l2norm, dv_slice=dv_slice)
    torch.cuda.synchronize()
    o_ref, fs_ref = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, init_state=x.init_state,
                                   use_qk_l2norm=use_qk_l2norm)
    if x.q.dtype == torch.bfloat16:
        f = fp32_twin(x).to(DEV)
        out32, fs32 = gdn.gdn_recurrent_fwd(f.q, f.k, f.v, f.g, f.beta, f.cu_seqlens, init_state=f.init_state,
                                            use_qk_l2norm=use_qk_l2norm, dv_slice=dv_slice)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), out32.to(torch.bfloat16).view(torch.int16)), \
            "bf16 output is not the fp32 twin rounded to nearest"
        assert torch.equal(fs.view(torch.int32), fs32.view(torch.int32)), "state differs from the fp32 twin"
        e = bf16_err(to_np(out), o_ref)
        assert e < FWD_TOL * (1 + 2.0 ** -8), f"bf16 out vs oracle, net of output rounding: {e:.3e}"
        out = out32
    return to_np(out), to_np(fs), o_ref, fs_ref


def assert_close(out, fs, o_ref, fs_ref, cu):
    e = per_unit_errors(out, o_ref, cu)
    assert e.size == 0 or e.max() < FWD_TOL, f"out normwise error {e.max():.3e}"
    for n in range(fs.shape[0]):
        for h in range(fs.shape[1]):
            err = normwise(fs[n, h], fs_ref[n, h])
            assert err < FWD_TOL, f"final_state[{n},{h}] normwise error {err:.3e}"


def test_tiny_config_fp32():
    x = inputs.tiny_config(seed=0)
    out, fs, o_ref, fs_ref = run_both(x)
    assert_close(out, fs, o_ref, fs_ref, x.cu_seqlens)
    # fp32 path: far inside the tolerance
    assert normwise(out, o_ref) < 1e-5


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (32, 16), (16, 32)])
def test_varlen_ragged(dtype, dk, dv):
    lengths = [37, 0, 1, 16, 17, 100, 5]
    x = inputs.make_inputs(lengths, HK=2, HV=4, dk=dk, dv=dv, dtype=dtype, seed=11, init_scale=0.1)
    out, fs, o_ref, fs_ref = run_both(x)
    assert_close(out, fs, o_ref, fs_ref, x.cu_seqlens)
    # the empty sequence passes its initial state through bit for bit
    assert np.array_equal(fs[1], x.init_state[1].numpy())


@pytest.mark.parametrize("dv_slice", [16, 32, 64, 128])
def test_dv_slices_match_oracle(dv_slice):
    x = inputs.make_inputs([50, 130], HK=1, HV=2, dk=128, dv=128, dtype=torch.bfloat16, seed=12, init_scale=0.1)
    out, fs, o_ref, fs_ref = run_both(x, dv_slice=dv_slice)
    assert_close(out, fs, o_ref, fs_ref, x.cu_seqlens)


def test_without_l2norm():
    x = inputs.make_inputs([70, 33], HK=2, HV=4, dk=64, dv=64, dtype=torch.float32, seed=13, init_scale=0.1)
    out, fs, o_ref, fs_ref = run_both(x, use_qk_l2norm=False)
    assert_close(out, fs, o_ref, fs_ref, x.cu_seqlens)


def test_unnormalised_inputs_with_l2norm():
    # q/k far from unit norm: the in-kernel normalisation does the work
    x = inputs.make_inputs([45], HK=1, HV=2, dk=128, dv=128, dtype=torch.bfloat16, seed=14, init_scale=0.0,
                           normalise_qk=False)
    out, fs, o_ref, fs_ref = run_both(x)
    assert_close(out, fs, o_ref, fs_ref, x.cu_seqlens)


def test_no_init_no_final():
    x = inputs.make_inputs([20, 9], HK=1, HV=2, dk=32, dv=32, dtype=torch.float32, seed=15)
    d = x.to(DEV)
    out, fs = gdn.gdn_recurrent_fwd(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, output_final_state=False)
    torch.cuda.synchronize()
    assert fs is None
    o_ref, _ = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens)
    assert per_unit_errors(to_np(out), o_ref, x.cu_seqlens).max() < FWD_TOL


def test_in_place_state():
    x = inputs.make_inputs([40, 3], HK=1, HV=2, dk=64, dv=64, dtype=torch.bfloat16, seed=16, init_scale=0.2)
    d = x.to(DEV)
    st = d.init_state.clone()
    out, fs = gdn.gdn_recurrent_fwd(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, init_state=st, final_state=st)
    torch.cuda.synchronize()
    assert fs.data_ptr() == st.data_ptr()
    o_ref, fs_ref = oracle.gdn_fwd(x.q, x.k, x.v, x.g, x.beta, x.cu_seqlens, init_state=x.init_state)
    e = max(bf16_err(to_np(out)[a:b], o_ref[a:b]) for a, b in ((0, 40), (40, 43)))
    assert e < FWD_TOL * (1 + 2.0 ** -8)
    for n in range(2):
        for h in range(2):
            assert normwise(to_np(st)[n, h], fs_ref[n, h]) < FWD_TOL


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_step_vs_oracle(dtype):
    B, HK, HV, dk, dv = 6, 2, 4, 128, 128
    x = inputs.make_inputs([1] * B, HK=HK, HV=HV, dk=dk, dv=dv, dtype=dtype, seed=17)
    pool = inputs.random_states(9, HV, dv, dk, seed=18, scale=0.3)
    idx = torch.tensor([4, 0, 8, 2, -1, 7], dtype=torch.int32)
    d = x.to(DEV)
    st = pool.to(DEV)
    out = torch.full_like(d.v, float("nan"))
    gdn.gdn_decode_step(d.q, d.k, d.v, d.g, d.beta, st, state_indices=idx.to(DEV), out=out)
    torch.cuda.synchronize()
    valid = [b for b in range(B) if idx[b] >= 0]
    s0 = pool[idx[valid].long()]
    sel = torch.tensor(valid)
    o_ref, fs_ref = oracle.gdn_fwd(x.q[sel], x.k[sel], x.v[sel], x.g[sel], x.beta[sel],
                                   np.arange(len(valid) + 1), init_state=s0)
    got = to_np(out)
    err = bf16_err if dtype == torch.bfloat16 else normwise
    for i, b in enumerate(valid):
        for h in range(HV):
            assert err(got[b, h], o_ref[i, h]) < FWD_TOL * (1 + 2.0 ** -8)
            assert normwise(to_np(st[int(idx[b])])[h], fs_ref[i, h]) < FWD_TOL
    # skipped row untouched, untouched slots unchanged
    assert torch.isnan(out[4]).all()
    for slot in (1, 3, 5, 6):
        assert torch.equal(st[slot].cpu(), pool[slot])


def test_throughput_workload_sampled():
    """The 64-sequence lognormal workload at full size, as the benchmark launches
    it; the oracle checks sampled (sequence, head) units one by one."""
    lengths = inputs.lognormal_lengths(64, 4096, 16384, seed=4)
    d = inputs.make_inputs(lengths, HK=16, HV=32, dk=128, dv=128, dtype=torch.bfloat16, seed=4, device=DEV)
    out, fs = gdn.gdn_recurrent_fwd(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens)
    torch.cuda.synchronize()
    x = d.cpu()
    order = np.argsort(lengths)
    picks = [(int(order[0]), 0), (int(order[1]), 31), (int(order[32]), 7), (int(order[-1]), 18)]
    cu = x.cu_seqlens.numpy()
    for n, h in picks:
        a, b = int(cu[n]), int(cu[n + 1])
        hk = h // 2
        o_ref, fs_ref = oracle.gdn_fwd(x.q[a:b, hk:hk + 1], x.k[a:b, hk:hk + 1], x.v[a:b, h:h + 1],
                                       x.g[a:b, h:h + 1], x.beta[a:b, h:h + 1], [0, b - a])
        assert bf16_err(to_np(out[a:b, h]), o_ref[:, 0]) < FWD_TOL * (1 + 2.0 ** -8), (n, h)
        assert normwise(to_np(fs[n, h]), fs_ref[0, 0]) < FWD_TOL, (n, h)
