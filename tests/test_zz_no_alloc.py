"""The allocation-free forward entry point (gdn_recurrent_fwd_noalloc).

It serves callers that cannot call cudaMalloc (device memory owned by another
allocator, or paths where allocating may synchronise the device): its scratch
is a fixed array inside the library.  Called here straight through the C ABI
(ctypes), twice in a row on different batches, and compared with
gdn_recurrent_fwd.  The kernels are the same, so the outputs must agree bit for
bit, which is inside the forward tolerance the other tests use.  This file is
collected last on purpose.
"""
import ctypes

import pytest
import torch

import invariant_linear_attention_gb300 as gdn
from invariant_linear_attention_gb300 import binding, inputs
from helpers import FWD_TOL, normwise, to_np

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def call_noalloc(d, out, fs):
    shape = gdn.make_shape(d.q, d.v, len(d.lengths))
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return gdn.lib().gdn_recurrent_fwd_noalloc(ctypes.byref(shape), p(d.q), p(d.k), p(d.v), p(d.g), p(d.beta),
                                               p(d.init_state), p(d.cu_seqlens), p(out), p(fs), stream)


def test_noalloc_matches_workspace_entry_two_calls():
    batches = [
        inputs.make_inputs([37, 0, 200, 16, 91], HK=16, HV=32, dk=128, dv=128, dtype=torch.bfloat16, seed=31,
                           init_scale=0.1, device=DEV),
        inputs.make_inputs([300, 5, 1], HK=2, HV=4, dk=64, dv=128, dtype=torch.float32, seed=32,
                           init_scale=0.2, device=DEV),
    ]
    for d in batches:  # two calls in a row: the second reuses the array the first left behind
        out = torch.full_like(d.v, float("nan"))
        fs = torch.full((len(d.lengths),) + tuple(d.v.shape[1:]) + (d.q.shape[2],), float("nan"),
                        dtype=torch.float32, device=DEV)
        rc = call_noalloc(d, out, fs)
        assert rc == binding.GDN_OK, gdn.status_string(rc)
        ref_out, ref_fs = gdn.gdn_recurrent_fwd(d.q, d.k, d.v, d.g, d.beta, d.cu_seqlens, init_state=d.init_state)
        torch.cuda.synchronize()
        assert normwise(to_np(out), to_np(ref_out)) <= FWD_TOL
        assert normwise(to_np(fs), to_np(ref_fs)) <= FWD_TOL
        assert torch.equal(out, ref_out) and torch.equal(fs, ref_fs)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # 2049 sequences x 32 heads x 1 slice = 65568 work units > 65536: refused on the host
    lengths = [1] * 2049
    d = inputs.make_inputs(lengths, HK=16, HV=32, dk=128, dv=128, dtype=torch.bfloat16, seed=33, device=DEV)
    out = torch.empty_like(d.v)
    rc = call_noalloc(d, out, None)
    assert rc == -3  # GDN_ERR_WORKSPACE
