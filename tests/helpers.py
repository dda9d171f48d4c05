"""Shared helpers for the parity and invariance tests."""
import numpy as np
import torch

# Tolerances (normwise-max relative error per (sequence, head, tensor)):
# forward 2e-3, gradients 1e-2, on fp32 values.  A bf16 output adds its own
# rounding, up to 2^-8 of the element (8 significant bits, round to nearest),
# which by itself can exceed 2e-3; bf16 outputs are therefore checked as
# (a) bit-identical to the fp32 kernel's output rounded to bf16 on the same
# inputs, and (b) against the oracle with the 2^-8 per-element rounding term
# added to the bound (bf16_err below).
FWD_TOL = 2e-3
GRAD_TOL = 1e-2
BF16_ROUND = 2.0 ** -8


def normwise(x, ref):
    """max |x - ref| / max |ref| (0 if both are all zero)."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max() if ref.size else 0.0
    num = np.abs(x - ref).max() if ref.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)


def per_unit_errors(out, ref, cu):
    """Normwise error of out vs ref [T, HV, dv] for every (sequence, head)."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    errs = []
    for n in range(len(cu) - 1):
        a, b = int(cu[n]), int(cu[n + 1])
        if b == a:
            continue
        for h in range(out.shape[1]):
            errs.append(normwise(out[a:b, h], ref[a:b, h]))
    return np.array(errs)


def to_np(t):
    return t.detach().cpu().to(torch.float64).numpy()


def bytes_equal(a, b):
    return a.shape == b.shape and a.dtype == b.dtype and torch.equal(a.view(torch.uint8) if a.dtype != torch.bool
                                                                      else a, b.view(torch.uint8))


def bf16_err(x, ref):
    """Normwise error of a bf16-rounded output, net of its own rounding:
    max_i (|x_i - r_i| - 2^-8 |r_i|)^+ / max |r| (compare with FWD_TOL * (1 + 2^-8))."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.abs(ref).max() if ref.size else 0.0
    if den == 0.0:
        return float(np.abs(x).max()) if x.size else 0.0
    return float(np.maximum(np.abs(x - ref) - BF16_ROUND * np.abs(ref), 0.0).max() / den)
