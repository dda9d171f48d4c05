"""Python face of the fp64 CPU oracle -- TEST INFRASTRUCTURE ONLY.

``gdn_fwd`` / ``gdn_bwd`` call the plain C recurrence in ``gdn_oracle.c``
(built by ``build_oracle.py``).  ``gdn_fwd_chunked`` is an independent second
forward in numpy: the chunked WY ("UT") form of the gated delta rule, used only
to pin the recurrence against a different algorithm.

Inputs may be numpy arrays or torch tensors of any float dtype; they are
widened exactly to float64 (bf16 and fp32 values are representable), so the
oracle sees the very values a GPU kernel receives.  Layouts (row-major):

    q, k   [T, HK, dk]        v        [T, HV, dv]
    g, beta [T, HV]           state    [N, HV, dv, dk]   cu_seqlens [N+1]

Source for the method: "Defending Against the Training-Inference Numeric
Mismatch in RL (Especially Linear Attention)", section 3.2 (recurrent kernel
for forward, prefill and decode; chunked kernel for the backward only; fp32
state cache per the section 4.2 setup tables), with the Gated DeltaNet update
S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T, o_t = S_t q_t,
a_t = exp(g_t), L2-normalised q and k.
"""
import ctypes
import os

import numpy as np

from .build_oracle import LIB, build

_lib = None
_D = ctypes.POINTER(ctypes.c_double)
_LL = ctypes.POINTER(ctypes.c_longlong)

EPS = 1e-6


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(LIB)
        common = [ctypes.c_int, _LL, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, ctypes.c_double]
        lib.gdn_oracle_fwd.argtypes = common + [_D] * 8 + [ctypes.c_int]
        lib.gdn_oracle_fwd.restype = ctypes.c_int
        lib.gdn_oracle_bwd.argtypes = common + [_D] * 16 + [ctypes.c_int]
        lib.gdn_oracle_bwd.restype = ctypes.c_int
        lib.gdn_oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _p(a):
    return None if a is None else a.ctypes.data_as(_D)


def _shapes(q, v, cu):
    T, HK, dk = q.shape
    Tv, HV, dv = v.shape
    assert T == Tv and HV % HK == 0
    N = len(cu) - 1
    assert cu[0] == 0 and cu[-1] == T and np.all(np.diff(cu) >= 0)
    return T, N, HK, HV, dk, dv


def gdn_fwd(q, k, v, g, beta, cu_seqlens, init_state=None, use_qk_l2norm=True,
            eps=EPS, threads=0):
    """Plain fp64 recurrence.  Returns (o [T,HV,dv], final_state [N,HV,dv,dk])."""
    q, k, v, g, beta, s0 = map(_f64, (q, k, v, g, beta, init_state))
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    T, N, HK, HV, dk, dv = _shapes(q, v, cu)
    o = np.zeros((T, HV, dv))
    fs = np.zeros((N, HV, dv, dk))
    rc = _load().gdn_oracle_fwd(N, cu.ctypes.data_as(_LL), HK, HV, dk, dv, int(bool(use_qk_l2norm)),
                                float(eps), _p(q), _p(k), _p(v), _p(g), _p(beta), _p(s0),
                                _p(o), _p(fs), int(threads))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_fwd failed ({rc})")
    return o, fs


def gdn_bwd(q, k, v, g, beta, cu_seqlens, d_out, init_state=None, d_final_state=None,
            use_qk_l2norm=True, eps=EPS, threads=0):
    """fp64 backpropagation through time of L = sum <dO, o> + <dS_T, S_T>.

    Returns a dict with dq, dk [T,HK,dk], dv [T,HV,dv], dg, dbeta [T,HV] and
    d_init_state [N,HV,dv,dk].
    """
    q, k, v, g, beta, s0, dO, dsT = map(_f64, (q, k, v, g, beta, init_state, d_out, d_final_state))
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    T, N, HK, HV, dk, dv = _shapes(q, v, cu)
    dq_hat = np.zeros((T, HV, dk))
    dk_hat = np.zeros((T, HV, dk))
    out = dict(dq=np.zeros((T, HK, dk)), dk=np.zeros((T, HK, dk)), dv=np.zeros((T, HV, dv)),
               dg=np.zeros((T, HV)), dbeta=np.zeros((T, HV)), d_init_state=np.zeros((N, HV, dv, dk)))
    rc = _load().gdn_oracle_bwd(N, cu.ctypes.data_as(_LL), HK, HV, dk, dv, int(bool(use_qk_l2norm)),
                                float(eps), _p(q), _p(k), _p(v), _p(g), _p(beta), _p(s0), _p(dO),
                                _p(dsT), _p(dq_hat), _p(dk_hat), _p(out["dq"]), _p(out["dk"]),
                                _p(out["dv"]), _p(out["dg"]), _p(out["dbeta"]),
                                _p(out["d_init_state"]), int(threads))
    if rc != 0:
        raise RuntimeError(f"gdn_oracle_bwd failed ({rc})")
    return out


def _l2n(x, on, eps):
    if not on:
        return x
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def gdn_fwd_chunked(q, k, v, g, beta, cu_seqlens, init_state=None, chunk=64,
                    use_qk_l2norm=True, eps=EPS):
    """Second, independent fp64 forward: the chunked WY form.

    Per chunk of C tokens inside one sequence (chunks restart at every
    sequence start, the last one partial), with start state S0:
        gam = cumsum(g),  Gam = exp(gam),  E[r,s] = exp(gam_r - gam_s)
        A   = strictly-lower( diag(beta) (E * K K^T) ),   Tm = (I + A)^-1
        W   = Tm diag(beta Gam) K,   U~ = Tm diag(beta) V,   U = U~ - W S0^T
        O   = diag(Gam) Q S0^T + (lower-incl(E) * Q K^T) U
        S_C = Gam_C S0 + U^T diag(exp(gam_C - gam)) K
    which follows from unrolling u_r = beta_r (v_r - a_r S_{r-1} k_r) inside
    the chunk (the WY / UT representation of the delta rule: Yang et al.,
    "Parallelizing Linear Transformers with the Delta Rule over Sequence
    Length", 2024, and "Gated Delta Networks", ICLR 2025).  The pages call
    this "the chunked kernel" (section 3.2) and keep it for the backward.
    Library primitives only: matmul and a triangular solve.
    """
    q, k, v, g, beta, s0 = map(_f64, (q, k, v, g, beta, init_state))
    cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64)
    T, N, HK, HV, dk, dv = _shapes(q, v, cu)
    G = HV // HK
    qn = _l2n(q, use_qk_l2norm, eps)
    kn = _l2n(k, use_qk_l2norm, eps)
    o = np.zeros((T, HV, dv))
    fs = np.zeros((N, HV, dv, dk))
    for n in range(N):
        for h in range(HV):
            S = np.zeros((dv, dk)) if s0 is None else s0[n, h].copy()
            for c0 in range(cu[n], cu[n + 1], chunk):
                c1 = min(c0 + chunk, cu[n + 1])
                K = kn[c0:c1, h // G]
                Q = qn[c0:c1, h // G]
                V = v[c0:c1, h]
                b = beta[c0:c1, h]
                gam = np.cumsum(g[c0:c1, h])
                Gam = np.exp(gam)
                E = np.exp(gam[:, None] - gam[None, :])
                C = c1 - c0
                A = np.tril(b[:, None] * E * (K @ K.T), -1)
                Tm = np.linalg.solve(np.eye(C) + A, np.eye(C))
                W = Tm @ ((b * Gam)[:, None] * K)
                U = Tm @ (b[:, None] * V) - W @ S.T
                M = np.tril(E)
                o[c0:c1, h] = Gam[:, None] * (Q @ S.T) + (M * (Q @ K.T)) @ U
                S = Gam[-1] * S + U.T @ (np.exp(gam[-1] - gam)[:, None] * K)
            fs[n, h] = S
    return o, fs


def gdn_replay_state(q, k, v, g, beta, cu_seqlens, init_state=None, chunk=64, use_qk_l2norm=True, eps=EPS):
    """The chunk-replay cache of every sequence after all its tokens (fp64).

    The delta-rule step written as S_t = a_t S_{t-1} + d_t k^_t^T with
    d_t = b_t (v_t - a_t S_{t-1} k^_t) (expand a_t S_{t-1} (I - b_t k^ k^T) +
    b_t v_t k^T).  With chunks of `chunk` tokens from each sequence start, a
    sequence that has seen P tokens is described by the state at the start of
    its current chunk, S0 = S_{C*floor(P/C)}, plus, for the r = P mod C tokens
    of that chunk, k^_i, d_i and gam_i = g_{start} + ... + g_i (the chunk's
    cumulative log-decay).  This is the state a decode that replays the
    chunked computation order needs ("Finish RL Training Faster:
    Bitwise-Consistent, High-Performance, Agent-Driven", the Nemotron
    experiment: decode replays prefill's chunked order).

    Returns per sequence n: dict(S0 [HV,dv,dk], K [r,HV,dk], D [r,HV,dv],
    gam [r,HV], r) and the per-token d [T,HV,dv].
    """
    q, k, v, g, beta, s0 = map(_f64, (q, k, v, g, beta, init_state))
    cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64)
    T, N, HK, HV, dk, dv = _shapes(q, v, cu)
    G = HV // HK
    kn = _l2n(k, use_qk_l2norm, eps)
    d_all = np.zeros((T, HV, dv))
    res = []
    for n in range(N):
        a, e = int(cu[n]), int(cu[n + 1])
        P = e - a
        c0 = a + (P // chunk) * chunk  # first token of the current (partial) chunk
        S0 = np.zeros((HV, dv, dk))
        for h in range(HV):
            S = np.zeros((dv, dk)) if s0 is None else s0[n, h].copy()
            for t in range(a, e):
                if t == c0:
                    S0[h] = S
                kt = kn[t, h // G]
                at = np.exp(g[t, h])
                d = beta[t, h] * (v[t, h] - at * (S @ kt))
                d_all[t, h] = d
                S = at * S + np.outer(d, kt)
            if c0 == e:
                S0[h] = S
        r = e - c0
        gam = np.zeros((r, HV))
        for h in range(HV):
            gam[:, h] = np.cumsum(g[c0:e, h])
        res.append(dict(S0=S0, K=kn[c0:e][:, np.arange(HV) // G], D=d_all[c0:e].copy(), gam=gam, r=r))
    return res, d_all
