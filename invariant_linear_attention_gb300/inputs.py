"""Seeded synthetic inputs for the Gated DeltaNet kernels and their oracle.

This module is the ONE thing the CUDA path and the fp64 oracle share: it only
draws random numbers and shapes them; it holds none of the recurrence's
arithmetic.  Every tensor is drawn in fp32 with a seeded ``torch.Generator``
(on the host, or on the GPU for multi-GB workloads) and then cast; the oracle
receives a host copy of exactly the values the kernels read.

Recipe (the pages run RL on named datasets; these synthetic tensors stand in
for the activations a GDN layer receives there):

* q, k ~ randn, then L2-normalised per head row in fp32, then cast;
* v ~ randn;  b ~ randn and beta = sigmoid(b) (the kernels take beta already
  activated, in (0, 1));  g = -softplus(randn) (a log-decay, so a = exp(g) is
  in (0, 1));
* init_state = 0 or randn * init_scale (fp32);
* lengths: uniform in [lo, hi], or lognormal with the stated mean (before the
  cap) and sigma = 1, rounded and clipped to [1, cap].

Layouts: q, k [T, HK, dk]; v [T, HV, dv]; g, beta [T, HV] fp32;
state [N, HV, dv, dk] fp32; cu_seqlens int32 [N + 1].

The layer ops around the recurrence (make_layer_inputs) get: gate
projections a, b ~ randn [T, HV]; A_log = log(uniform(1, 16)) and
dt_bias ~ randn * 0.5 - 2 per head (fp32); conv input x ~ randn [T, C] with
C = 2 * HK * dk + HV * dv (the q, k and v projections side by side), taps
~ randn / sqrt(W) and bias ~ randn * 0.1 (fp32), conv state ~ randn
[N, W-1, C]; norm input o ~ randn and gate z ~ randn [T, HV, dv]; norm
weight ~ 1 + 0.1 * randn [dv] (fp32).
"""
from dataclasses import dataclass
from typing import List, Optional, Sequence

import math
import torch


@dataclass
class GDNInputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor
    beta: torch.Tensor
    cu_seqlens: torch.Tensor
    init_state: Optional[torch.Tensor]
    lengths: List[int]

    @property
    def shape(self):
        T, HK, dk = self.q.shape
        HV, dv = self.v.shape[1], self.v.shape[2]
        return dict(N=len(self.lengths), T=T, HK=HK, HV=HV, dk=dk, dv=dv)

    def cpu(self):
        return self.to("cpu")

    def to(self, device):
        mv = lambda t: None if t is None else t.to(device)  # noqa: E731
        return GDNInputs(mv(self.q), mv(self.k), mv(self.v), mv(self.g), mv(self.beta),
                         mv(self.cu_seqlens), mv(self.init_state), list(self.lengths))


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, gen, device):
    return torch.empty(shape, dtype=torch.float32, device=device).normal_(generator=gen)


def cu_from_lengths(lengths: Sequence[int]) -> torch.Tensor:
    cu = [0]
    for n in lengths:
        cu.append(cu[-1] + int(n))
    return torch.tensor(cu, dtype=torch.int32)


def uniform_lengths(n: int, lo: int, hi: int, seed: int) -> List[int]:
    gen = _gen(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]


def lognormal_lengths(n: int, mean: float, cap: int, seed: int, sigma: float = 1.0) -> List[int]:
    """Lognormal lengths with E[len] = mean before rounding and capping."""
    gen = _gen(seed)
    mu = math.log(mean) - sigma * sigma / 2.0
    z = torch.randn(n, generator=gen, dtype=torch.float64)
    return [int(min(max(round(math.exp(mu + sigma * float(x))), 1), cap)) for x in z]


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def make_inputs(lengths: Sequence[int], HK: int, HV: int, dk: int, dv: int,
                dtype=torch.bfloat16, seed: int = 0, init_scale: Optional[float] = None,
                normalise_qk: bool = True, device="cpu") -> GDNInputs:
    """Packed varlen inputs for ``len(lengths)`` sequences (see module doc).

    ``device`` picks where the seeded generator draws (a CUDA generator is
    much faster for multi-GB workloads); the values for a given seed depend
    on the device type, and both sides of a comparison must use one draw.
    """
    gen = _gen(seed, device)
    T = int(sum(lengths))
    q = _randn((T, HK, dk), gen, device)
    k = _randn((T, HK, dk), gen, device)
    if normalise_qk:
        q, k = _unit_rows(q), _unit_rows(k)
    q, k = q.to(dtype).contiguous(), k.to(dtype).contiguous()
    v = _randn((T, HV, dv), gen, device).to(dtype).contiguous()
    b = _randn((T, HV), gen, device)
    g = -torch.nn.functional.softplus(_randn((T, HV), gen, device))
    beta = torch.sigmoid(b)
    s0 = None
    if init_scale is not None:
        N = len(lengths)
        s0 = (_randn((N, HV, dv, dk), gen, device) * init_scale) if init_scale else \
            torch.zeros(N, HV, dv, dk, device=device)
    return GDNInputs(q, k, v, g.contiguous(), beta.contiguous(), cu_from_lengths(lengths).to(device), s0,
                     list(lengths))


def concat(parts: Sequence[GDNInputs]) -> GDNInputs:
    """Pack several input sets (same head shapes) into one varlen batch, in order."""
    lengths = [n for p in parts for n in p.lengths]
    cat = lambda name: torch.cat([getattr(p, name) for p in parts], 0)  # noqa: E731
    s0 = None
    if any(p.init_state is not None for p in parts):
        s0 = torch.cat([p.init_state if p.init_state is not None else
                        torch.zeros(len(p.lengths), *parts[0].v.shape[1:], parts[0].q.shape[2],
                                    device=parts[0].q.device)
                        for p in parts], 0)
    return GDNInputs(cat("q"), cat("k"), cat("v"), cat("g"), cat("beta"),
                     cu_from_lengths(lengths).to(parts[0].q.device), s0, lengths)


def tiny_config(seed: int = 0) -> GDNInputs:
    """1 sequence, T=64, 2 heads, dk=dv=16, fp32, zero initial state."""
    return make_inputs([64], HK=2, HV=2, dk=16, dv=16, dtype=torch.float32, seed=seed,
                       init_scale=0.0)


def grad_out(T: int, HV: int, dv: int, dtype=torch.bfloat16, seed: int = 6, device="cpu") -> torch.Tensor:
    """Upstream gradient dO ~ randn [T, HV, dv]."""
    return _randn((T, HV, dv), _gen(seed, device), device).to(dtype).contiguous()


def random_states(N: int, HV: int, dv: int, dk: int, seed: int, scale: float = 1.0,
                  device="cpu") -> torch.Tensor:
    """fp32 states ~ randn * scale, layout [N, HV, dv, dk]."""
    return (_randn((N, HV, dv, dk), _gen(seed, device), device) * scale).contiguous()


@dataclass
class LayerInputs:
    a: torch.Tensor            # [T, HV] gate projections (dtype)
    b: torch.Tensor            # [T, HV]
    A_log: torch.Tensor        # [HV] fp32
    dt_bias: torch.Tensor      # [HV] fp32
    x: torch.Tensor            # [T, C] conv input (dtype)
    conv_w: torch.Tensor       # [C, W] fp32
    conv_b: torch.Tensor       # [C] fp32
    conv_state: torch.Tensor   # [N, W-1, C] (dtype)
    o: torch.Tensor            # [T, HV, dv] norm input (dtype)
    z: torch.Tensor            # [T, HV, dv] norm gate (dtype)
    norm_w: torch.Tensor       # [dv] fp32
    cu_seqlens: torch.Tensor
    lengths: List[int]

    def to(self, device):
        kw = {f: (getattr(self, f).to(device) if isinstance(getattr(self, f), torch.Tensor) else getattr(self, f))
              for f in self.__dataclass_fields__}
        return LayerInputs(**kw)


def make_layer_inputs(lengths: Sequence[int], HK: int, HV: int, dk: int, dv: int, W: int = 4,
                      dtype=torch.bfloat16, seed: int = 0, device="cpu", C: Optional[int] = None) -> LayerInputs:
    """Seeded inputs for the gate, conv and norm ops (see module doc)."""
    gen = _gen(seed, device)
    T, N = int(sum(lengths)), len(lengths)
    C = 2 * HK * dk + HV * dv if C is None else int(C)
    a = _randn((T, HV), gen, device).to(dtype).contiguous()
    b = _randn((T, HV), gen, device).to(dtype).contiguous()
    A_log = torch.log(torch.empty(HV, device=device).uniform_(1.0, 16.0, generator=gen))
    dt_bias = _randn((HV,), gen, device) * 0.5 - 2.0
    x = _randn((T, C), gen, device).to(dtype).contiguous()
    conv_w = (_randn((C, W), gen, device) / math.sqrt(W)).contiguous()
    conv_b = _randn((C,), gen, device) * 0.1
    conv_state = _randn((N, W - 1, C), gen, device).to(dtype).contiguous()
    o = _randn((T, HV, dv), gen, device).to(dtype).contiguous()
    z = _randn((T, HV, dv), gen, device).to(dtype).contiguous()
    norm_w = 1.0 + 0.1 * _randn((dv,), gen, device)
    return LayerInputs(a, b, A_log, dt_bias, x, conv_w, conv_b, conv_state, o, z, norm_w,
                       cu_from_lengths(lengths).to(device), list(lengths))
