"""Seeded synthetic inputs for the delta-rule forward and decode workloads.

This module only draws random numbers.  It holds none of the recurrence's
arithmetic, so both the CUDA path and the fp64 oracle consume the same inputs
from it without sharing any computation.  Every tensor is drawn on the CPU
with a ``torch.Generator`` seeded per workload, in a fixed order (q, k, v,
then the gates in the order each workload lists them), and q/k/v are rounded
to the workload's input dtype before either side sees them.

The workloads take the head shapes the pages use (dk = dv = 128, chunk 64,
contexts up to 64K) with these distributions:

* ``kla_fp32_small``   KLA, fp32, B=1 H=2 T=256 d=64 C=64.  q,k,v ~ N(0,1),
  k unnormalised, q L2-normalised at readout.  eta = sigmoid(N(0,1)),
  log alpha = -softplus(N(0,1)+2), eps = 1e-6, S_0 = 0.
* ``gdn_kla_bf16``     GDN and KLA, bf16, B=8 H=8 T=2048 d=128 C=64.
  k = N(0,1) * LogNormal(0,0.5) (one log-normal factor per token, so key
  energy spreads over ~10x), v ~ N(0,1), other gates as above.
* ``pgdn_bf16``        PGDN, bf16, B=4 H=16 T=4096 d=128 C=64.  q,k,v ~ N(0,1)
  with q and k L2-normalised in the kernel; alphaP = sigmoid(N(3,1)),
  betaP = sigmoid(N(0,1)) per (b,t,h); mu = exp(N(0,0.5)) per head; x = 1.5;
  beta = sigmoid(N(0,1)); log alpha as above; floor 1e-12; A_0 = 0.
* ``kdn_bf16``         Diagonal KDN, bf16, B=4 H=16 T=8192 d=128 C=64.  q,k,v
  as for PGDN; per-channel log alpha = -softplus(N(0,1)+2); omega =
  softplus(N(-3,1)) per channel; r = softplus(N(0,1)) per (b,t,h); p_0 = 1;
  information scale 1.
* ``kda_bf16``         KDA (per-channel decay, w = eta k), bf16, B=4 H=16
  T=8192 d=128 C=64; q,k,v as for PGDN; eta = sigmoid(N(0,1)); per-channel
  log alpha = -softplus(N(0,1)+2).
* ``pkda_bf16``        PKDA (the PGDN write key with per-channel decay), bf16,
  B=4 H=16 T=4096 d=128 C=64; the PGDN gates, then per-channel log alpha as
  for KDA.
* ``ikdn_bf16``        isotropic KDN, bf16, B=4 H=16 T=8192 d=128 C=64; q,k,v
  as for PGDN; per-channel log alpha as for Diagonal KDN; omega =
  softplus(N(-3,1)) and r = softplus(N(0,1)) per (b,t,h); b_0 = 1;
  information scale 1.
* ``ekdn_bf16``        exact Kalman memory (dense key covariance), bf16, B=4
  H=16 T=2048 d=128; gates as for Diagonal KDN (per-channel log alpha and
  omega, r per (b,t,h)); P_0 = I.
* ``kla_prefill_bf16`` KLA, bf16, B=1 H=16 T=65536 d=128, inputs as
  ``gdn_kla_bf16``.
* ``kla_decode_bf16``  KLA decode steps at batch 256, H=16, d=128; fresh
  per-step inputs with the ``gdn_kla_bf16`` distributions.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

__all__ = ["Workload", "WORKLOADS", "generate", "generate_decode_step", "small"]


@dataclass(frozen=True)
class Workload:
    name: str
    variants: tuple            # which write rules run on these inputs
    B: int
    T: int
    H: int
    dk: int
    dv: int
    chunk: int
    dtype: str                 # "fp32" or "bf16" for q/k/v/out
    key_dist: str = "normal"   # "normal" or "lognormal_scaled"
    q_l2norm: bool = True
    k_l2norm: bool = False
    eps: float = 1e-6
    x: float = 1.5
    log_floor: float = 1e-12
    info_scale: float = 1.0
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    "kla_fp32_small": Workload("kla_fp32_small", ("kla",), 1, 256, 2, 64, 64, 64, "fp32",
                               seed=1000),
    "gdn_kla_bf16": Workload("gdn_kla_bf16", ("gdn", "kla"), 8, 2048, 8, 128, 128, 64, "bf16",
                             key_dist="lognormal_scaled", seed=1001),
    "pgdn_bf16": Workload("pgdn_bf16", ("pgdn",), 4, 4096, 16, 128, 128, 64, "bf16",
                          k_l2norm=True, seed=1002),
    "kdn_bf16": Workload("kdn_bf16", ("kdn",), 4, 8192, 16, 128, 128, 64, "bf16",
                         k_l2norm=True, seed=1003),
    "kda_bf16": Workload("kda_bf16", ("kda",), 4, 8192, 16, 128, 128, 64, "bf16",
                         k_l2norm=True, seed=1005),
    "pkda_bf16": Workload("pkda_bf16", ("pkda",), 4, 4096, 16, 128, 128, 64, "bf16",
                          k_l2norm=True, seed=1006),
    "ikdn_bf16": Workload("ikdn_bf16", ("ikdn",), 4, 8192, 16, 128, 128, 64, "bf16",
                          k_l2norm=True, seed=1007),
    "ekdn_bf16": Workload("ekdn_bf16", ("ekdn",), 4, 2048, 16, 128, 128, 64, "bf16",
                          k_l2norm=True, seed=1008),
    "kla_prefill_bf16": Workload("kla_prefill_bf16", ("kla",), 1, 65536, 16, 128, 128, 64,
                                 "bf16", key_dist="lognormal_scaled", seed=1004),
    "kla_decode_bf16": Workload("kla_decode_bf16", ("kla",), 256, 1, 16, 128, 128, 64, "bf16",
                                key_dist="lognormal_scaled", seed=2000),
}


def small(base: str, **sizes) -> Workload:
    """A workload with ``base``'s distributions and flags but other sizes/seed."""
    return replace(WORKLOADS[base], **sizes)


def _torch_dtype(name: str):
    return {"fp32": torch.float32, "bf16": torch.bfloat16}[name]


def _softplus(x):
    return torch.nn.functional.softplus(x)


def _draw_qkv(gen, wl: Workload, B, T):
    H, dk, dv = wl.H, wl.dk, wl.dv
    q = torch.randn(B, T, H, dk, generator=gen)
    k = torch.randn(B, T, H, dk, generator=gen)
    if wl.key_dist == "lognormal_scaled":
        scale = torch.exp(0.5 * torch.randn(B, T, H, 1, generator=gen))
        k = k * scale
    v = torch.randn(B, T, H, dv, generator=gen)
    dt = _torch_dtype(wl.dtype)
    return q.to(dt), k.to(dt), v.to(dt)


def _draw_gates(gen, wl: Workload, variant: str, B, T):
    H, dk = wl.H, wl.dk
    g = {}
    if variant in ("gdn", "kla"):
        g["eta"] = torch.sigmoid(torch.randn(B, T, H, generator=gen))
        g["log_alpha"] = -_softplus(torch.randn(B, T, H, generator=gen) + 2.0)
    elif variant == "pgdn":
        g["alphaP"] = torch.sigmoid(torch.randn(B, T, H, generator=gen) + 3.0)
        g["betaP"] = torch.sigmoid(torch.randn(B, T, H, generator=gen))
        g["mu"] = torch.exp(0.5 * torch.randn(H, generator=gen))
        g["eta"] = torch.sigmoid(torch.randn(B, T, H, generator=gen))
        g["log_alpha"] = -_softplus(torch.randn(B, T, H, generator=gen) + 2.0)
    elif variant in ("kdn", "ekdn"):
        g["log_alpha"] = -_softplus(torch.randn(B, T, H, dk, generator=gen) + 2.0)
        g["omega"] = _softplus(torch.randn(B, T, H, dk, generator=gen) - 3.0)
        g["r"] = _softplus(torch.randn(B, T, H, generator=gen))
    elif variant == "ikdn":
        g["log_alpha"] = -_softplus(torch.randn(B, T, H, dk, generator=gen) + 2.0)
        g["omega"] = _softplus(torch.randn(B, T, H, generator=gen) - 3.0)
        g["r"] = _softplus(torch.randn(B, T, H, generator=gen))
    elif variant == "kda":
        g["eta"] = torch.sigmoid(torch.randn(B, T, H, generator=gen))
        g["log_alpha"] = -_softplus(torch.randn(B, T, H, dk, generator=gen) + 2.0)
    elif variant == "pkda":
        g["alphaP"] = torch.sigmoid(torch.randn(B, T, H, generator=gen) + 3.0)
        g["betaP"] = torch.sigmoid(torch.randn(B, T, H, generator=gen))
        g["mu"] = torch.exp(0.5 * torch.randn(H, generator=gen))
        g["eta"] = torch.sigmoid(torch.randn(B, T, H, generator=gen))
        g["log_alpha"] = -_softplus(torch.randn(B, T, H, dk, generator=gen) + 2.0)
    else:
        raise ValueError(variant)
    return g


def generate(wl: Workload, variant: str | None = None, seed: int | None = None):
    """Draw one workload's inputs on the CPU.

    Returns a dict with q, k, v (in the workload dtype) and the variant's
    gates (float32), plus ``variant`` and the flags.  For a workload that
    lists several variants, the q/k/v draw is shared and each variant's gates
    are drawn after it, in the listed order.
    """
    variant = variant or wl.variants[0]
    gen = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    q, k, v = _draw_qkv(gen, wl, wl.B, wl.T)
    gates = None
    for vname in wl.variants if variant in wl.variants else (variant,):
        drawn = _draw_gates(gen, wl, vname, wl.B, wl.T)
        if vname == variant:
            gates = drawn
    out = dict(q=q, k=k, v=v, variant=variant, chunk=wl.chunk, q_l2norm=wl.q_l2norm,
               k_l2norm=wl.k_l2norm, eps=wl.eps, x=wl.x, log_floor=wl.log_floor,
               info_scale=wl.info_scale)
    out.update(gates)
    return out


def generate_decode_step(wl: Workload, step: int, variant: str | None = None):
    """Per-step decode inputs ([B, H, d] tensors) for decode step ``step``.

    Each step has its own generator seeded with ``wl.seed + step``.
    """
    variant = variant or wl.variants[0]
    gen = torch.Generator().manual_seed(wl.seed + step)
    q, k, v = _draw_qkv(gen, wl, wl.B, 1)
    gates = _draw_gates(gen, wl, variant, wl.B, 1)
    out = dict(q=q[:, 0], k=k[:, 0], v=v[:, 0], variant=variant, q_l2norm=wl.q_l2norm,
               k_l2norm=wl.k_l2norm, eps=wl.eps, x=wl.x, log_floor=wl.log_floor,
               info_scale=wl.info_scale)
    for name, t in gates.items():
        out[name] = t if name == "mu" else t[:, 0]
    return out
