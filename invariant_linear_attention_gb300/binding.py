"""Thin ctypes binding over libgdn.so (include/gdn.h).

Argument marshalling only: tensors are checked for device, dtype, layout and
alignment, outputs and workspaces are allocated with PyTorch when the caller
does not pass them, and the raw device pointers plus the current CUDA stream
go to the C entry points, which run every step of the computation in the
library's own kernels.  There is no fallback: if the library is missing or a
call fails, a RuntimeError is raised.
"""
import ctypes
import os

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgdn.so")
_lib = None

GDN_OK = 0
GDN_F32, GDN_BF16 = 0, 1
OP_FWD, OP_DECODE, OP_BWD = 0, 1, 2
DEVERR_CU_SEQLENS, DEVERR_TIMEOUT, DEVERR_SMEM_ALIGN = 1, 2, 4

_P = ctypes.c_void_p

SYMBOLS = ("gdn_workspace_size", "gdn_recurrent_fwd", "gdn_decode_step", "gdn_chunk_bwd",
           "gdn_read_device_error", "gdn_status_string", "gdn_recurrent_fwd_noalloc",
           "gdn_recurrent_fwd_snapshots", "gdn_gates", "gdn_gated_rmsnorm", "gdn_causal_conv1d_fwd",
           "gdn_causal_conv1d_update", "gdn_replay_block_floats", "gdn_replay_workspace_size",
           "gdn_replay_prefill", "gdn_replay_decode")


class GdnShape(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("T_total", ctypes.c_int), ("HK", ctypes.c_int),
                ("HV", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
                ("dtype", ctypes.c_int), ("use_qk_l2norm", ctypes.c_int), ("dv_slice", ctypes.c_int)]


class ConvShape(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int), ("T_total", ctypes.c_int), ("C", ctypes.c_int), ("W", ctypes.c_int),
                ("dtype", ctypes.c_int), ("activation", ctypes.c_int)]


class GdnError(RuntimeError):
    def __init__(self, code, what):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} ({code})")


def lib():
    """Load libgdn.so once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with invariant_linear_attention_gb300."
                               "build_lib.build() (or __graft_entry__.build())")
        L = ctypes.CDLL(_LIB_PATH)
        L.gdn_workspace_size.argtypes = [ctypes.POINTER(GdnShape), ctypes.c_int]
        L.gdn_workspace_size.restype = ctypes.c_size_t
        L.gdn_recurrent_fwd.argtypes = [ctypes.POINTER(GdnShape)] + [_P] * 10 + [ctypes.c_size_t, _P]
        L.gdn_recurrent_fwd.restype = ctypes.c_int
        L.gdn_recurrent_fwd_noalloc.argtypes = [ctypes.POINTER(GdnShape)] + [_P] * 10
        L.gdn_recurrent_fwd_noalloc.restype = ctypes.c_int
        L.gdn_recurrent_fwd_snapshots.argtypes = ([ctypes.POINTER(GdnShape)] + [_P] * 9 +
                                                  [ctypes.c_int, _P, ctypes.c_int, _P, _P, ctypes.c_size_t, _P])
        L.gdn_recurrent_fwd_snapshots.restype = ctypes.c_int
        L.gdn_decode_step.argtypes = [ctypes.POINTER(GdnShape)] + [_P] * 7 + [ctypes.c_int, _P, _P]
        L.gdn_decode_step.restype = ctypes.c_int
        L.gdn_chunk_bwd.argtypes = [ctypes.POINTER(GdnShape)] + [_P] * 16 + [ctypes.c_size_t, _P]
        L.gdn_chunk_bwd.restype = ctypes.c_int
        L.gdn_read_device_error.argtypes = [_P, ctypes.POINTER(ctypes.c_uint), _P]
        L.gdn_read_device_error.restype = ctypes.c_int
        L.gdn_gates.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int] + [_P] * 7
        L.gdn_gates.restype = ctypes.c_int
        L.gdn_gated_rmsnorm.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, _P, _P, _P, ctypes.c_float,
                                        _P, _P]
        L.gdn_gated_rmsnorm.restype = ctypes.c_int
        L.gdn_causal_conv1d_fwd.argtypes = [ctypes.POINTER(ConvShape)] + [_P] * 6 + [ctypes.c_int, _P, _P, _P]
        L.gdn_causal_conv1d_fwd.restype = ctypes.c_int
        L.gdn_causal_conv1d_update.argtypes = [ctypes.POINTER(ConvShape)] + [_P] * 5 + [ctypes.c_int, _P, _P]
        L.gdn_causal_conv1d_update.restype = ctypes.c_int
        L.gdn_replay_block_floats.argtypes = [ctypes.c_int, ctypes.c_int]
        L.gdn_replay_block_floats.restype = ctypes.c_size_t
        L.gdn_replay_workspace_size.argtypes = [ctypes.POINTER(GdnShape)]
        L.gdn_replay_workspace_size.restype = ctypes.c_size_t
        L.gdn_replay_prefill.argtypes = [ctypes.POINTER(GdnShape)] + [_P] * 9 + [ctypes.c_int, _P, _P,
                                                                                ctypes.c_size_t, _P]
        L.gdn_replay_prefill.restype = ctypes.c_int
        L.gdn_replay_decode.argtypes = [ctypes.POINTER(GdnShape)] + [_P] * 8 + [ctypes.c_int, _P, _P]
        L.gdn_replay_decode.restype = ctypes.c_int
        L.gdn_status_string.argtypes = [ctypes.c_int]
        L.gdn_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().gdn_status_string(int(code)).decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _need(t, name, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def make_shape(q, v, N, use_qk_l2norm=True, dv_slice=0, T_total=None):
    T, HK, dk = q.shape
    HV, dv = v.shape[1], v.shape[2]
    return GdnShape(int(N), int(T if T_total is None else T_total), int(HK), int(HV), int(dk), int(dv),
                    _dtype_code(q), int(bool(use_qk_l2norm)), int(dv_slice))


def gdn_workspace_size(shape: GdnShape, op: int) -> int:
    return int(lib().gdn_workspace_size(ctypes.byref(shape), int(op)))


def _check(rc, what):
    if rc != GDN_OK:
        raise GdnError(rc, what)


def gdn_recurrent_fwd(q, k, v, g, beta, cu_seqlens, init_state=None, out=None, final_state=None,
                      workspace=None, use_qk_l2norm=True, dv_slice=0, output_final_state=True,
                      stream=None):
    """Batch-invariant recurrent forward over a packed varlen batch.

    q, k [T, HK, dk] and v [T, HV, dv] (bf16 or fp32, same dtype), g, beta
    [T, HV] fp32, cu_seqlens int32 [N+1] on the device, init_state
    [N, HV, dv, dk] fp32 or None.  Returns (out [T, HV, dv], final_state
    [N, HV, dv, dk] fp32 or None).  final_state may be init_state (in place).
    """
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    N = cu_seqlens.numel() - 1
    T, HK, dk = q.shape
    HV, dv = v.shape[1], v.shape[2]
    if k.shape != q.shape or v.shape[0] != T or g.shape != (T, HV) or beta.shape != (T, HV):
        raise ValueError("inconsistent shapes")
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, dev)
        if init_state.shape != (N, HV, dv, dk):
            raise ValueError("init_state must be [N, HV, dv, dk]")
    shape = make_shape(q, v, N, use_qk_l2norm, dv_slice)
    if out is None:
        out = torch.empty_like(v)
    _need(out, "out", q.dtype, dev)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, HV, dv, dk, dtype=torch.float32, device=dev)
    if final_state is not None:
        _need(final_state, "final_state", torch.float32, dev)
    need = gdn_workspace_size(shape, OP_FWD)
    if workspace is None:
        workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    with torch.cuda.device(dev):
        rc = lib().gdn_recurrent_fwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(init_state), _ptr(cu_seqlens), _ptr(out), _ptr(final_state),
                                     _ptr(workspace), ctypes.c_size_t(workspace.numel()), _stream(stream))
    _check(rc, "gdn_recurrent_fwd")
    return out, final_state


def gdn_recurrent_fwd_noalloc(q, k, v, g, beta, cu_seqlens, init_state=None, out=None, final_state=None,
                              use_qk_l2norm=True, dv_slice=0, output_final_state=True, stream=None):
    """gdn_recurrent_fwd through the entry point that needs no workspace (its
    scratch is a fixed array inside the library; calls must not overlap on the
    GPU).  Same arguments and results as gdn_recurrent_fwd minus `workspace`;
    out / final_state are allocated here only when the caller passes none."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    N = cu_seqlens.numel() - 1
    T, HK, dk = q.shape
    HV, dv = v.shape[1], v.shape[2]
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, dev)
    shape = make_shape(q, v, N, use_qk_l2norm, dv_slice)
    if out is None:
        out = torch.empty_like(v)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, HV, dv, dk, dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        rc = lib().gdn_recurrent_fwd_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                             _ptr(beta), _ptr(init_state), _ptr(cu_seqlens), _ptr(out),
                                             _ptr(final_state), _stream(stream))
    _check(rc, "gdn_recurrent_fwd_noalloc")
    return out, final_state


def snapshot_offsets(lengths, snap_every):
    """int32 [N+1] slot offsets giving each sequence floor(len / snap_every) snapshot slots."""
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n) // int(snap_every))
    return torch.tensor(cu, dtype=torch.int32)


def gdn_recurrent_fwd_snapshots(q, k, v, g, beta, cu_seqlens, snap_every, snap_cu=None, snap_states=None,
                                init_state=None, out=None, final_state=None, workspace=None,
                                use_qk_l2norm=True, dv_slice=0, stream=None):
    """gdn_recurrent_fwd plus fp32 state snapshots after every snap_every-th token of
    each sequence (prefix caching).  snap_cu: int32 [N+1] device slot offsets (built
    from cu_seqlens with a host copy when None).  Returns (out, final_state,
    snap_states [slots, HV, dv, dk], snap_cu)."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    N = cu_seqlens.numel() - 1
    T, HK, dk = q.shape
    HV, dv = v.shape[1], v.shape[2]
    if init_state is not None:
        _need(init_state, "init_state", torch.float32, dev)
    if snap_cu is None:
        cuh = cu_seqlens.cpu().tolist()
        snap_cu = snapshot_offsets([cuh[i + 1] - cuh[i] for i in range(N)], snap_every).to(dev)
    _need(snap_cu, "snap_cu", torch.int32, dev)
    slots = int(snap_cu[-1].item()) if snap_states is None else int(snap_states.shape[0])
    if snap_states is None:
        snap_states = torch.empty(max(slots, 0), HV, dv, dk, dtype=torch.float32, device=dev)
    _need(snap_states, "snap_states", torch.float32, dev)
    shape = make_shape(q, v, N, use_qk_l2norm, dv_slice)
    if out is None:
        out = torch.empty_like(v)
    if final_state is None:
        final_state = torch.empty(N, HV, dv, dk, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.zeros(max(gdn_workspace_size(shape, OP_FWD), 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = lib().gdn_recurrent_fwd_snapshots(
            ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(init_state),
            _ptr(cu_seqlens), _ptr(out), _ptr(final_state), int(snap_every), _ptr(snap_cu), slots,
            _ptr(snap_states) if slots > 0 else None, _ptr(workspace), ctypes.c_size_t(workspace.numel()),
            _stream(stream))
    _check(rc, "gdn_recurrent_fwd_snapshots")
    return out, final_state, snap_states, snap_cu


def gdn_decode_step(q, k, v, g, beta, state, state_indices=None, out=None, use_qk_l2norm=True,
                    dv_slice=0, stream=None):
    """One token per sequence on the cached fp32 state pool, updated in place.

    q, k [B, HK, dk], v [B, HV, dv], g, beta [B, HV]; state [slots, HV, dv, dk]
    fp32; state_indices int32 [B] or None (slot b).  Returns out [B, HV, dv].
    """
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(state, "state", torch.float32, dev)
    B = q.shape[0]
    if state_indices is not None:
        _need(state_indices, "state_indices", torch.int32, dev)
    shape = make_shape(q, v, B, use_qk_l2norm, dv_slice)
    if out is None:
        out = torch.empty_like(v)
    _need(out, "out", q.dtype, dev)
    with torch.cuda.device(dev):
        rc = lib().gdn_decode_step(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                   _ptr(state), _ptr(state_indices), int(state.shape[0]), _ptr(out),
                                   _stream(stream))
    _check(rc, "gdn_decode_step")
    return out


def gdn_chunk_bwd(q, k, v, g, beta, cu_seqlens, d_out, init_state=None, d_final_state=None,
                  workspace=None, use_qk_l2norm=True, need_d_init_state=True, stream=None):
    """Chunked (WY) backward.  Returns dict dq, dk, dv (dtype of q), dg, dbeta, d_init_state (fp32)."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (d_out, "d_out")):
        _need(t, n, q.dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    N = cu_seqlens.numel() - 1
    T, HK, dk = q.shape
    HV, dv = v.shape[1], v.shape[2]
    for t, n in ((init_state, "init_state"), (d_final_state, "d_final_state")):
        if t is not None:
            _need(t, n, torch.float32, dev)
    shape = make_shape(q, v, N, use_qk_l2norm, 0)
    res = dict(dq=torch.empty_like(q), dk=torch.empty_like(k), dv=torch.empty_like(v),
               dg=torch.empty(T, HV, dtype=torch.float32, device=dev),
               dbeta=torch.empty(T, HV, dtype=torch.float32, device=dev),
               d_init_state=torch.empty(N, HV, dv, dk, dtype=torch.float32, device=dev)
               if need_d_init_state else None)
    need = gdn_workspace_size(shape, OP_BWD)
    if workspace is None:
        workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    _need(workspace, "workspace", torch.uint8, dev)
    with torch.cuda.device(dev):
        rc = lib().gdn_chunk_bwd(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                 _ptr(init_state), _ptr(cu_seqlens), _ptr(d_out), _ptr(d_final_state),
                                 _ptr(res["dq"]), _ptr(res["dk"]), _ptr(res["dv"]), _ptr(res["dg"]),
                                 _ptr(res["dbeta"]), _ptr(res["d_init_state"]), _ptr(workspace),
                                 ctypes.c_size_t(workspace.numel()), _stream(stream))
    _check(rc, "gdn_chunk_bwd")
    return res


def read_device_error(workspace, stream=None) -> int:
    """Device error bits left in a FWD/BWD workspace (synchronises the stream)."""
    bits = ctypes.c_uint(0)
    rc = lib().gdn_read_device_error(_ptr(workspace), ctypes.byref(bits), _stream(stream))
    _check(rc, "gdn_read_device_error")
    return int(bits.value)


# ---------------------------------------------------------------- layer ops (include/gdn_layer.h)

def gdn_gates(a, b, A_log, dt_bias=None, g=None, beta=None, stream=None):
    """(g, beta) [T, HV] fp32 from the raw projections a, b [T, HV] (bf16 or fp32):
    g = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b)."""
    dev = a.device
    _need(a, "a", None, dev)
    _need(b, "b", a.dtype, dev)
    _need(A_log, "A_log", torch.float32, dev)
    if dt_bias is not None:
        _need(dt_bias, "dt_bias", torch.float32, dev)
    if a.dim() != 2 or b.shape != a.shape or A_log.shape != (a.shape[1],):
        raise ValueError("a, b must be [T, HV] and A_log [HV]")
    T, HV = a.shape
    g = torch.empty(T, HV, dtype=torch.float32, device=dev) if g is None else g
    beta = torch.empty(T, HV, dtype=torch.float32, device=dev) if beta is None else beta
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    with torch.cuda.device(dev):
        rc = lib().gdn_gates(int(T), int(HV), _dtype_code(a), _ptr(a), _ptr(b), _ptr(A_log), _ptr(dt_bias),
                             _ptr(g), _ptr(beta), _stream(stream))
    _check(rc, "gdn_gates")
    return g, beta


def gdn_gated_rmsnorm(o, z, weight, eps=1e-6, out=None, stream=None):
    """y = o / sqrt(mean(o^2, -1) + eps) * weight * silu(z) over the last axis of
    o [..., d] (bf16 or fp32); z like o or None; weight [d] fp32.  out may be o."""
    dev = o.device
    _need(o, "o", None, dev)
    if z is not None:
        _need(z, "z", o.dtype, dev)
        if z.shape != o.shape:
            raise ValueError("z must have o's shape")
    _need(weight, "weight", torch.float32, dev)
    d = o.shape[-1]
    if weight.shape != (d,):
        raise ValueError("weight must be [d]")
    out = torch.empty_like(o) if out is None else out
    _need(out, "out", o.dtype, dev)
    with torch.cuda.device(dev):
        rc = lib().gdn_gated_rmsnorm(int(o.numel() // d), int(d), _dtype_code(o), _ptr(o), _ptr(z), _ptr(weight),
                                     float(eps), _ptr(out), _stream(stream))
    _check(rc, "gdn_gated_rmsnorm")
    return out


def _conv_shape(x, weight, N, activation):
    T, C = x.shape
    if weight.dim() != 2 or weight.shape[0] != C:
        raise ValueError("weight must be [C, W]")
    return ConvShape(int(N), int(T), int(C), int(weight.shape[1]), _dtype_code(x), int(bool(activation)))


def gdn_causal_conv1d_fwd(x, weight, cu_seqlens, bias=None, conv_state=None, state_indices=None,
                          has_initial_state=None, activation=True, out=None, stream=None):
    """Causal depthwise conv over packed varlen x [T, C] with taps weight [C, W]
    fp32.  conv_state [slots, W-1, C] (dtype of x) is read as the initial state
    and overwritten with the final state of each sequence's slot (in place).
    Returns y [T, C]."""
    dev = x.device
    _need(x, "x", None, dev)
    _need(weight, "weight", torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    for t, n, dt in ((bias, "bias", torch.float32), (conv_state, "conv_state", x.dtype),
                     (state_indices, "state_indices", torch.int32),
                     (has_initial_state, "has_initial_state", torch.int32)):
        if t is not None:
            _need(t, n, dt, dev)
    N = cu_seqlens.numel() - 1
    shape = _conv_shape(x, weight, N, activation)
    if conv_state is not None and tuple(conv_state.shape[1:]) != (shape.W - 1, shape.C):
        raise ValueError("conv_state must be [slots, W-1, C]")
    out = torch.empty_like(x) if out is None else out
    _need(out, "out", x.dtype, dev)
    slots = 0 if conv_state is None else int(conv_state.shape[0])
    with torch.cuda.device(dev):
        rc = lib().gdn_causal_conv1d_fwd(ctypes.byref(shape), _ptr(x), _ptr(weight), _ptr(bias), _ptr(cu_seqlens),
                                         _ptr(conv_state), _ptr(state_indices), slots, _ptr(has_initial_state),
                                         _ptr(out), _stream(stream))
    _check(rc, "gdn_causal_conv1d_fwd")
    return out


def gdn_causal_conv1d_update(x, weight, conv_state, state_indices=None, bias=None, activation=True, out=None,
                             stream=None):
    """One decode token per sequence: x [B, C]; conv_state [slots, W-1, C]
    updated in place.  Returns y [B, C] (rows of skipped sequences untouched)."""
    dev = x.device
    _need(x, "x", None, dev)
    _need(weight, "weight", torch.float32, dev)
    _need(conv_state, "conv_state", x.dtype, dev)
    for t, n, dt in ((bias, "bias", torch.float32), (state_indices, "state_indices", torch.int32)):
        if t is not None:
            _need(t, n, dt, dev)
    shape = _conv_shape(x, weight, x.shape[0], activation)
    if tuple(conv_state.shape[1:]) != (shape.W - 1, shape.C):
        raise ValueError("conv_state must be [slots, W-1, C]")
    out = torch.empty_like(x) if out is None else out
    _need(out, "out", x.dtype, dev)
    with torch.cuda.device(dev):
        rc = lib().gdn_causal_conv1d_update(ctypes.byref(shape), _ptr(x), _ptr(weight), _ptr(bias),
                                            _ptr(conv_state), _ptr(state_indices), int(conv_state.shape[0]),
                                            _ptr(out), _stream(stream))
    _check(rc, "gdn_causal_conv1d_update")
    return out


# ---------------------------------------------------------------- chunk-replay variant (include/gdn_replay.h)

REPLAY_CHUNK = 64


def replay_block_floats(dk, dv):
    """Floats per (slot, head) in a replay-state pool."""
    return int(lib().gdn_replay_block_floats(int(dk), int(dv)))


def replay_state_new(slots, HV, dk, dv, init_state=None, device="cuda"):
    """A zeroed replay-state pool [slots, HV, B] fp32 whose chunk-start states are
    init_state [slots, HV, dv, dk] (zeros when None)."""
    rs = torch.zeros(slots, HV, replay_block_floats(dk, dv), dtype=torch.float32, device=device)
    if init_state is not None:
        replay_views(rs, dk, dv)["S0"].copy_(init_state)
    return rs


def replay_views(rs, dk, dv):
    """Views of a replay-state pool: S0 [slots, HV, dv, dk], K [.., C, dk], D [.., C, dv], gam [.., C]."""
    C = REPLAY_CHUNK
    a, b, c = dv * dk, dv * dk + C * dk, dv * dk + C * (dk + dv)
    sl, HV = rs.shape[0], rs.shape[1]
    return dict(S0=rs[..., :a].unflatten(-1, (dv, dk)), K=rs[..., a:b].unflatten(-1, (C, dk)),
                D=rs[..., b:c].unflatten(-1, (C, dv)), gam=rs[..., c:c + C])


def gdn_replay_prefill(q, k, v, g, beta, cu_seqlens, replay_state, seq_pos=None, state_indices=None, out=None,
                       workspace=None, use_qk_l2norm=True, stream=None):
    """Chunked prefill that continues every sequence from its replay state (at
    position seq_pos[n], int32 on the device; None: 0) and leaves the state
    after its last token.  Returns out [T, HV, dv]."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(cu_seqlens, "cu_seqlens", torch.int32, dev)
    _need(replay_state, "replay_state", torch.float32, dev)
    for t, n in ((seq_pos, "seq_pos"), (state_indices, "state_indices")):
        if t is not None:
            _need(t, n, torch.int32, dev)
    N = cu_seqlens.numel() - 1
    shape = make_shape(q, v, N, use_qk_l2norm, 0)
    if replay_state.shape[1:] != (shape.HV, replay_block_floats(shape.dk, shape.dv)):
        raise ValueError("replay_state must be [slots, HV, replay_block_floats(dk, dv)]")
    out = torch.empty_like(v) if out is None else out
    _need(out, "out", q.dtype, dev)
    if workspace is None:
        workspace = torch.zeros(max(int(lib().gdn_replay_workspace_size(ctypes.byref(shape))), 256),
                                dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        rc = lib().gdn_replay_prefill(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                      _ptr(cu_seqlens), _ptr(seq_pos), _ptr(replay_state), _ptr(state_indices),
                                      int(replay_state.shape[0]), _ptr(out), _ptr(workspace),
                                      ctypes.c_size_t(workspace.numel()), _stream(stream))
    _check(rc, "gdn_replay_prefill")
    return out


def gdn_replay_decode(q, k, v, g, beta, replay_state, seq_pos, state_indices=None, out=None, use_qk_l2norm=True,
                      stream=None):
    """One token per sequence replaying the chunked order; seq_pos [B] int32 (tokens
    already processed).  Returns out [B, HV, dv] (rows of skipped slots untouched)."""
    dev = q.device
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, n, q.dtype, dev)
    _need(g, "g", torch.float32, dev)
    _need(beta, "beta", torch.float32, dev)
    _need(replay_state, "replay_state", torch.float32, dev)
    _need(seq_pos, "seq_pos", torch.int32, dev)
    if state_indices is not None:
        _need(state_indices, "state_indices", torch.int32, dev)
    shape = make_shape(q, v, q.shape[0], use_qk_l2norm, 0)
    out = torch.empty_like(v) if out is None else out
    _need(out, "out", q.dtype, dev)
    with torch.cuda.device(dev):
        rc = lib().gdn_replay_decode(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                                     _ptr(seq_pos), _ptr(replay_state), _ptr(state_indices),
                                     int(replay_state.shape[0]), _ptr(out), _stream(stream))
    _check(rc, "gdn_replay_decode")
    return out
