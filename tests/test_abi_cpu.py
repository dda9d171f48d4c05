"""CPU-only checks of the C ABI: the library loads, exports every function
include/gdn.h declares, and rejects bad arguments on the host (these calls
return before any CUDA call, so no GPU is needed)."""
import ctypes
import os
import re

import pytest

import invariant_linear_attention_gb300 as gdn
from invariant_linear_attention_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = "".join(open(os.path.join(ROOT, "include", f)).read()
                   for f in sorted(os.listdir(os.path.join(ROOT, "include"))) if f.endswith(".h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from invariant_linear_attention_gb300 import build_lib
    build_lib.build()
    return gdn.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"gdn_recurrent_fwd", "gdn_decode_step", "gdn_chunk_bwd", "gdn_workspace_size"} <= set(names)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(binding.SYMBOLS) == set(names)


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4):
        assert gdn.status_string(code).startswith("GDN_")


def shape(**kw):
    base = dict(N=2, T_total=10, HK=2, HV=4, dk=128, dv=128, dtype=binding.GDN_BF16, use_qk_l2norm=1, dv_slice=0)
    base.update(kw)
    return binding.GdnShape(**base)


def test_workspace_sizes(lib):
    s = shape(N=64)
    fwd = gdn.gdn_workspace_size(s, binding.OP_FWD)
    # automatic slices may split every head of a long sequence in 4: room for 4 * N * HV items
    assert fwd >= 256 + 4 * 64 * 4 * 4
    assert gdn.gdn_workspace_size(s, binding.OP_DECODE) == 0
    assert gdn.gdn_workspace_size(shape(N=64, dv_slice=16), binding.OP_FWD) > fwd  # 8 slices per head
    # no automatic splitting below dv = 64 (units keep at least 16 rows): one item per head
    assert gdn.gdn_workspace_size(shape(N=64, dv=32), binding.OP_FWD) == 256 + 64 * 4 * 4
    assert gdn.gdn_workspace_size(shape(dk=48), binding.OP_FWD) == 0  # unsupported
    assert gdn.gdn_workspace_size(shape(HV=3), binding.OP_FWD) == 0   # HV % HK != 0


def call_fwd(lib, s, ptrs, ws_bytes=1 << 20):
    P = ctypes.c_void_p
    args = [P(p) if p else None for p in ptrs]
    return lib.gdn_recurrent_fwd(ctypes.byref(s), *args[:9], args[9], ctypes.c_size_t(ws_bytes), None)


FAKE = 0x10000  # never dereferenced: every case below fails validation first


@pytest.mark.parametrize("case,expect", [
    ("null_q", -1), ("null_cu", -1), ("misaligned_v", -1), ("out_aliases_q", -1),
    ("bad_dk", -2), ("bad_dtype", -2), ("bad_slice", -2), ("hv_not_multiple", -1),
    ("no_workspace", -3), ("small_workspace", -3), ("token_head_index_over_32_bits", -2),
])
def test_fwd_host_validation(lib, case, expect):
    s = shape()
    q, k, v, g, b, s0, cu, out, fs, ws = [FAKE + i * 0x1000 for i in range(10)]
    ws_bytes = 1 << 20
    if case == "null_q":
        q = 0
    elif case == "null_cu":
        cu = 0
    elif case == "misaligned_v":
        v += 4
    elif case == "out_aliases_q":
        out = q
    elif case == "bad_dk":
        s.dk = 96
    elif case == "bad_dtype":
        s.dtype = 7
    elif case == "bad_slice":
        s.dv_slice = 24
    elif case == "hv_not_multiple":
        s.HV = 3
    elif case == "no_workspace":
        ws = 0
    elif case == "small_workspace":
        ws_bytes = 16
    elif case == "token_head_index_over_32_bits":
        s.T_total, s.HV = 1 << 26, 32  # T_total * HV = 2^31
    assert call_fwd(lib, s, [q, k, v, g, b, s0, cu, out, fs, ws], ws_bytes) == expect


def call_bwd(lib, s, ptrs, ws_bytes):
    P = ctypes.c_void_p
    args = [P(p) if p else None for p in ptrs]
    return lib.gdn_chunk_bwd(ctypes.byref(s), *args[:16], ctypes.c_size_t(ws_bytes), None)


@pytest.mark.parametrize("case,expect", [
    ("null_q", -1), ("null_cu", -1), ("null_dg", -1), ("misaligned_dq", -1), ("dq_aliases_q", -1),
    ("dinit_aliases_init", -1), ("bad_dk", -2), ("bad_dtype", -2), ("hv_not_multiple", -1),
    ("no_workspace", -3), ("small_workspace", -3), ("no_sequences", 0), ("token_head_index_over_32_bits", -2),
])
def test_bwd_host_validation(lib, case, expect):
    """gdn_chunk_bwd rejects bad arguments before any CUDA call (N = 0 returns at once)."""
    s = shape()
    (q, k, v, g, b, s0, cu, dO, dsT, dq, dk, dv, dg, db, ds0, ws) = [FAKE + i * 0x1000 for i in range(16)]
    ws_bytes = 1 << 20
    if case == "null_q":
        q = 0
    elif case == "null_cu":
        cu = 0
    elif case == "null_dg":
        dg = 0
    elif case == "misaligned_dq":
        dq += 4
    elif case == "dq_aliases_q":
        dq = q
    elif case == "dinit_aliases_init":
        ds0 = s0
    elif case == "bad_dk":
        s.dk = 96
    elif case == "bad_dtype":
        s.dtype = 7
    elif case == "hv_not_multiple":
        s.HV = 3
    elif case == "no_workspace":
        ws = 0
    elif case == "small_workspace":
        ws_bytes = 16
    elif case == "no_sequences":
        s.N, s.T_total = 0, 0
    elif case == "token_head_index_over_32_bits":
        s.T_total, s.HV = 1 << 26, 32  # T_total * HV = 2^31
    assert call_bwd(lib, s, [q, k, v, g, b, s0, cu, dO, dsT, dq, dk, dv, dg, db, ds0, ws], ws_bytes) == expect


def test_decode_host_validation(lib):
    P = ctypes.c_void_p
    s = shape(N=4, T_total=4)
    ptr = [P(FAKE + i * 0x1000) for i in range(8)]
    # T_total != N
    bad = shape(N=4, T_total=5)
    assert lib.gdn_decode_step(ctypes.byref(bad), *ptr[:6], None, 4, ptr[7], None) == -1
    # no indices and too few slots
    assert lib.gdn_decode_step(ctypes.byref(s), *ptr[:6], None, 3, ptr[7], None) == -1
    # out aliases the state
    assert lib.gdn_decode_step(ctypes.byref(s), *ptr[:6], None, 4, ptr[5], None) == -1
    # unsupported dv
    assert lib.gdn_decode_step(ctypes.byref(shape(N=4, T_total=4, dv=20)), *ptr[:6], None, 4, ptr[7],
                               None) == -2


def test_snapshot_host_validation(lib):
    P = ctypes.c_void_p
    s = shape()
    q, k, v, g, b, s0, cu, out, fs, ws, sc, ss = [P(FAKE + i * 0x1000) for i in range(12)]
    f = lib.gdn_recurrent_fwd_snapshots
    # interval not a multiple of the 32-token chunk, or not positive
    assert f(ctypes.byref(s), q, k, v, g, b, s0, cu, out, fs, 48, sc, 4, ss, ws, 1 << 20, None) == -2
    assert f(ctypes.byref(s), q, k, v, g, b, s0, cu, out, fs, 0, sc, 4, ss, ws, 1 << 20, None) == -2
    # slots but no buffer; misaligned buffer; buffer aliasing the final state
    assert f(ctypes.byref(s), q, k, v, g, b, s0, cu, out, fs, 64, sc, 4, None, ws, 1 << 20, None) == -1
    assert f(ctypes.byref(s), q, k, v, g, b, s0, cu, out, fs, 64, sc, 4, P(FAKE + 8), ws, 1 << 20, None) == -1
    assert f(ctypes.byref(s), q, k, v, g, b, s0, cu, out, fs, 64, sc, 4, fs, ws, 1 << 20, None) == -1
    # workspace rules as for gdn_recurrent_fwd
    assert f(ctypes.byref(s), q, k, v, g, b, s0, cu, out, fs, 64, sc, 4, ss, None, 1 << 20, None) == -3


def conv_shape(**kw):
    base = dict(N=2, T_total=10, C=64, W=4, dtype=binding.GDN_BF16, activation=1)
    base.update(kw)
    return binding.ConvShape(**base)


def test_layer_ops_host_validation(lib):
    P = ctypes.c_void_p
    a, b, al, dt, g, be = [P(FAKE + i * 0x1000) for i in range(6)]
    # gates: bad dtype, null output, misaligned A_log; empty input launches nothing
    assert lib.gdn_gates(8, 4, 7, a, b, al, dt, g, be, None) == -2
    assert lib.gdn_gates(8, 4, binding.GDN_BF16, a, b, al, dt, None, be, None) == -1
    assert lib.gdn_gates(8, 4, binding.GDN_BF16, a, b, P(FAKE + 2), dt, g, be, None) == -1
    assert lib.gdn_gates(0, 4, binding.GDN_BF16, a, b, al, dt, g, be, None) == 0
    o, z, w, y = [P(FAKE + i * 0x1000) for i in range(4)]
    # rmsnorm: d not a multiple of the 16-byte vector, d too large, misaligned o, negative eps
    assert lib.gdn_gated_rmsnorm(4, 12, binding.GDN_BF16, o, z, w, 1e-6, y, None) == -2
    assert lib.gdn_gated_rmsnorm(4, 4096, binding.GDN_BF16, o, z, w, 1e-6, y, None) == -2
    assert lib.gdn_gated_rmsnorm(4, 128, binding.GDN_BF16, P(FAKE + 8), z, w, 1e-6, y, None) == -1
    assert lib.gdn_gated_rmsnorm(4, 128, binding.GDN_BF16, o, z, w, -1.0, y, None) == -1
    x, cw, cb, cu, st, idx, hi, cy = [P(FAKE + i * 0x1000) for i in range(8)]
    fwd = lib.gdn_causal_conv1d_fwd
    assert fwd(ctypes.byref(conv_shape(W=9)), x, cw, cb, cu, st, idx, 4, hi, cy, None) == -2
    assert fwd(ctypes.byref(conv_shape(C=60)), x, cw, cb, cu, st, idx, 4, hi, cy, None) == -2
    assert fwd(ctypes.byref(conv_shape()), x, cw, cb, cu, st, idx, 4, hi, x, None) == -1       # y aliases x
    assert fwd(ctypes.byref(conv_shape()), x, cw, cb, None, st, idx, 4, hi, cy, None) == -1    # no cu_seqlens
    assert fwd(ctypes.byref(conv_shape()), x, cw, cb, cu, st, None, 1, hi, cy, None) == -1     # slots < N
    assert fwd(ctypes.byref(conv_shape()), P(FAKE + 4), cw, cb, cu, st, idx, 4, hi, cy, None) == -1
    upd = lib.gdn_causal_conv1d_update
    assert upd(ctypes.byref(conv_shape(N=4, T_total=5)), x, cw, cb, st, idx, 4, cy, None) == -1
    assert upd(ctypes.byref(conv_shape(N=4, T_total=4)), x, cw, cb, None, idx, 4, cy, None) == -1
    assert upd(ctypes.byref(conv_shape(N=4, T_total=4)), x, cw, cb, st, None, 3, cy, None) == -1
    assert upd(ctypes.byref(conv_shape(N=4, T_total=4, dtype=3)), x, cw, cb, st, idx, 4, cy, None) == -2


def test_replay_host_validation(lib):
    P = ctypes.c_void_p
    assert lib.gdn_replay_block_floats(128, 128) == 128 * 128 + 64 * (128 + 128 + 1)
    assert lib.gdn_replay_block_floats(48, 128) == 0
    s = shape(N=4, T_total=4)
    assert lib.gdn_replay_workspace_size(ctypes.byref(s)) >= 256 + 4 * 4 * 4
    q, k, v, g, b, cu, sp, rs, idx, out, ws = [P(FAKE + i * 0x1000) for i in range(11)]
    pre = lib.gdn_replay_prefill
    assert pre(ctypes.byref(s), q, k, v, g, b, None, sp, rs, idx, 4, out, ws, 1 << 20, None) == -1   # no cu
    assert pre(ctypes.byref(s), q, k, v, g, b, cu, sp, None, idx, 4, out, ws, 1 << 20, None) == -1   # no state
    assert pre(ctypes.byref(s), q, k, v, g, b, cu, sp, rs, None, 3, out, ws, 1 << 20, None) == -1    # slots < N
    assert pre(ctypes.byref(s), q, k, v, g, b, cu, sp, rs, idx, 4, q, ws, 1 << 20, None) == -1      # out aliases q
    assert pre(ctypes.byref(s), q, k, v, g, b, cu, sp, rs, idx, 4, out, None, 1 << 20, None) == -3
    assert pre(ctypes.byref(shape(N=4, T_total=4, dk=96)), q, k, v, g, b, cu, sp, rs, idx, 4, out, ws, 1 << 20,
               None) == -2
    dec = lib.gdn_replay_decode
    assert dec(ctypes.byref(s), q, k, v, g, b, None, rs, idx, 4, out, None) == -1                    # no seq_pos
    assert dec(ctypes.byref(shape(N=4, T_total=5)), q, k, v, g, b, sp, rs, idx, 4, out, None) == -1
    assert dec(ctypes.byref(s), q, k, v, g, b, sp, P(FAKE + 8), idx, 4, out, None) == -1             # misaligned
