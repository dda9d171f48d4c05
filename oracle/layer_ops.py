"""fp64 oracle for the ops around the Gated DeltaNet recurrence -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU baseline may use this
module; the library never does.

These are the next steps either side of the recurrent kernel in a GDN layer:
the gate activations that produce (g, beta) from the layer's projections,
the short causal depthwise conv (with its per-sequence conv state cache)
applied to the q/k/v projections before the recurrence, and the gated
RMSNorm applied to the recurrence's output.  The pages name them as part of
what the unified model carries over (A_log kept in fp32 through the trainer's
bf16 wrapping; the serving engine's conv state and SSM state caches reused
unchanged: "Defending Against the Training-Inference Numeric Mismatch in RL
(Especially Linear Attention)", sections 3.1 and 3.2); their formulas are
the standard Gated DeltaNet layer's:

    g    = -exp(A_log[h]) * softplus(a + dt_bias[h])         beta = sigmoid(b)
    conv: y[t, c] = silu( sum_i w[c, i] * xw[t + i, c] + bias[c] ),  i = 0..W-1,
          xw = (conv state: the W-1 input rows before the sequence) ++ (the sequence's rows)
    norm: y = o / sqrt(mean(o^2) + eps) * weight * silu(z)     (per token and head, over dv)

Plain numpy in float64; library primitives only (exp, logaddexp, sqrt).
"""
import numpy as np


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def gates(a, b, A_log, dt_bias):
    """(g, beta) from the raw projections a, b [T, HV] and per-head A_log, dt_bias [HV]."""
    a, b, A_log, dt_bias = map(_f64, (a, b, A_log, dt_bias))
    g = -np.exp(A_log)[None, :] * np.logaddexp(0.0, a + dt_bias[None, :])
    beta = 1.0 / (1.0 + np.exp(-b))
    return g, beta


def silu(x):
    return x / (1.0 + np.exp(-x))


def gated_rmsnorm(o, z, weight, eps=1e-6):
    """y[t, h, :] = o / sqrt(mean(o^2) + eps) * weight * silu(z) over the last axis."""
    o, z, weight = map(_f64, (o, z, weight))
    r = np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps)
    return o / r * weight * silu(z)


def causal_conv1d(x, w, cu_seqlens, bias=None, conv_state=None, activation=True):
    """Depthwise causal conv over packed varlen x [T, C] with taps w [C, W].

    conv_state [N, W-1, C] holds, per sequence, the W-1 input rows before it
    (zeros when None).  Returns (y [T, C], final conv state [N, W-1, C]): the
    last W-1 rows of (conv state ++ the sequence's inputs).
    """
    x, w, bias, conv_state = map(_f64, (x, w, bias, conv_state))
    cu = [int(c) for c in (cu_seqlens.tolist() if hasattr(cu_seqlens, "tolist") else cu_seqlens)]
    T, C = x.shape
    W = w.shape[1]
    N = len(cu) - 1
    y = np.zeros((T, C))
    final = np.zeros((N, W - 1, C))
    for n in range(N):
        a, e = cu[n], cu[n + 1]
        past = np.zeros((W - 1, C)) if conv_state is None else conv_state[n]
        xw = np.concatenate([past, x[a:e]], axis=0)  # [W-1 + L, C]
        for t in range(e - a):
            acc = np.zeros(C)
            for i in range(W):
                acc = acc + w[:, i] * xw[t + i]
            if bias is not None:
                acc = acc + bias
            y[a + t] = silu(acc) if activation else acc
        final[n] = xw[len(xw) - (W - 1):]
    return y, final


def causal_conv1d_update(x, w, conv_state, state_indices=None, bias=None, activation=True):
    """One decode token per sequence: x [B, C]; conv_state [slots, W-1, C] updated
    (returned as a copy); a negative slot skips the sequence (its y row stays 0)."""
    x, w, bias, conv_state = map(_f64, (x, w, bias, conv_state))
    B, C = x.shape
    W = w.shape[1]
    st = conv_state.copy()
    idx = list(range(B)) if state_indices is None else [int(i) for i in state_indices]
    y = np.zeros((B, C))
    for b in range(B):
        s = idx[b]
        if s < 0:
            continue
        xw = np.concatenate([st[s], x[b:b + 1]], axis=0)  # [W, C]
        acc = np.zeros(C)
        for i in range(W):
            acc = acc + w[:, i] * xw[i]
        if bias is not None:
            acc = acc + bias
        y[b] = silu(acc) if activation else acc
        st[s] = xw[1:]
    return y, st
