"""Seeded synthetic inputs for log-linear attention (forward and decode).

This module only draws random numbers and fixes shapes; it holds none of the method's
arithmetic.  It is the one module both the CPU oracle's callers and the CUDA path's
callers (tests, bench, smoke) use, so that both sides see the same inputs.

Recipes (shapes, distributions) are the five workloads the method is measured on:

* ``linear_T64``      fp32, B1 H1 T64 dk=dv=16 C16 L7, no decay (M^S all ones),
                      q,k ~ N(0,1)/sqrt(dk), v ~ N(0,1), lambda ~ U(0,1), seed 0.
* ``mamba2_T1024``    fp32, B2 H4 T1024 dk=dv=64 C64 L11, Mamba-2 distributions:
                      q,k ~ N(0,1)/sqrt(dk), v ~ N(0,1), log a = -0.1 softplus(N(0,1)),
                      lambda = softplus(N(0,1)).
* ``mamba2_T4096``    bf16 q/k/v, B4 H16 T4096 dk=dv=128 C64 L13, Mamba-2 distributions.
* ``mamba2_T16384``   bf16 q/k/v, B1 H16 T16384 dk=dv=128 C64 L15, Mamba-2 distributions
                      (the pages' pretraining length; the headline forward workload).
* ``decode_B128``     decode step at t=12345, B128 H16 dk=dv=128 L15, fp32 states, bf16
                      tokens, Mamba-2 distributions.
* ``mva_B2H48_T16384`` the pages' kernel-benchmark shape: bf16, B2, 48 heads, head dim
                      (d_v) 64, state dim (d_k) 128, C64, one q/k shared by all heads
                      (Mamba-2's multi-value form), T16384 L15, Mamba-2 distributions.

Draw order for a forward input: q, k, v, log-a noise, lambda noise, all fp32 from one
CPU ``torch.Generator`` seeded with ``seed``; bf16 workloads cast after drawing.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch
import torch.nn.functional as F


@dataclass(frozen=True)
class FwdConfig:
    name: str
    B: int
    H: int
    T: int
    dk: int
    dv: int
    C: int
    L: int
    dtype: str          # "f32" or "bf16" for q, k, v (and out)
    decay: bool         # Mamba-2 decay (True) or M^S all ones (False)
    lam: str            # "uniform" (U(0,1)) or "softplus" (softplus(N(0,1)))
    seed: int = 0
    Hqk: int = 0        # q/k heads shared by the H value heads (0: one q/k per head)

    @property
    def qk_heads(self) -> int:
        return self.Hqk or self.H

    def with_(self, **kw) -> "FwdConfig":
        return replace(self, **kw)


@dataclass(frozen=True)
class DecodeConfig:
    name: str
    B: int
    H: int
    dk: int
    dv: int
    L: int
    t: int
    dtype: str = "bf16"
    decay: bool = True
    seed: int = 0


FWD_CONFIGS = {
    "linear_T64": FwdConfig("linear_T64", 1, 1, 64, 16, 16, 16, 7, "f32", False, "uniform"),
    "mamba2_T1024": FwdConfig("mamba2_T1024", 2, 4, 1024, 64, 64, 64, 11, "f32", True, "softplus"),
    "mamba2_T4096": FwdConfig("mamba2_T4096", 4, 16, 4096, 128, 128, 64, 13, "bf16", True, "softplus"),
    "mamba2_T16384": FwdConfig("mamba2_T16384", 1, 16, 16384, 128, 128, 64, 15, "bf16", True, "softplus"),
    "mva_B2H48_T16384": FwdConfig("mva_B2H48_T16384", 2, 48, 16384, 128, 64, 64, 15, "bf16", True,
                                  "softplus", Hqk=1),
}
DECODE_CONFIG = DecodeConfig("decode_B128", 128, 16, 128, 128, 15, 12345)
HEADLINE_FWD = "mamba2_T16384"


def torch_dtype(name: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def make_fwd_inputs(cfg: FwdConfig):
    """Returns dict(q, k, v, log_a, lam) of CPU tensors in the product's layout:
    q, k [B,T,Hqk,dk]; v [B,T,H,dv]; log_a [B,T,H] fp32 or None; lam [B,T,H,L] fp32."""
    g = _gen(cfg.seed)
    B, T, H, G = cfg.B, cfg.T, cfg.H, cfg.qk_heads
    q = torch.randn(B, T, G, cfg.dk, generator=g) / math.sqrt(cfg.dk)
    k = torch.randn(B, T, G, cfg.dk, generator=g) / math.sqrt(cfg.dk)
    v = torch.randn(B, T, H, cfg.dv, generator=g)
    a_noise = torch.randn(B, T, H, generator=g)
    l_noise = torch.randn(B, T, H, cfg.L, generator=g)
    log_a = -0.1 * F.softplus(a_noise) if cfg.decay else None
    if cfg.lam == "uniform":
        lam = torch.rand(B, T, H, cfg.L, generator=g)
    else:
        lam = F.softplus(l_noise)
    dt = torch_dtype(cfg.dtype)
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
                log_a=None if log_a is None else log_a.contiguous(), lam=lam.contiguous())


def make_int_inputs(B, T, H, dk, dv, L, onehot_level: int, seed: int = 0, dtype="f32"):
    """Small-integer q, k, v in [-2, 2], no decay, one-hot lambda selecting one level.

    Every product and partial sum is an integer far below 2^24, so any correct fp32
    evaluation order returns the same result exactly."""
    g = _gen(seed)
    q = torch.randint(-2, 3, (B, T, H, dk), generator=g).float()
    k = torch.randint(-2, 3, (B, T, H, dk), generator=g).float()
    v = torch.randint(-2, 3, (B, T, H, dv), generator=g).float()
    lam = torch.zeros(B, T, H, L)
    lam[..., onehot_level] = 1.0
    dt = torch_dtype(dtype)
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), log_a=None, lam=lam)


def make_sparse_int_inputs(B, T, H, d, L, onehot_level: int, seed: int = 0, dv=None):
    """bf16 inputs whose every intermediate stays an exactly representable integer even
    through bf16 storage of the chunk states: q, v in {-1, 0, 1}, each k a signed one-hot
    vector (so q.k is in {-1, 0, 1} and a state entry counts the tokens of a block whose k
    hits that feature), no decay, one-hot lambda.  d is d_k; d_v defaults to d."""
    g = _gen(seed)
    q = torch.randint(-1, 2, (B, T, H, d), generator=g).float()
    v = torch.randint(-1, 2, (B, T, H, d if dv is None else dv), generator=g).float()
    hot = torch.randint(0, d, (B, T, H), generator=g)
    sign = torch.randint(0, 2, (B, T, H), generator=g).float() * 2 - 1
    k = torch.zeros(B, T, H, d)
    k.scatter_(3, hot[..., None], sign[..., None])
    lam = torch.zeros(B, T, H, L)
    lam[..., onehot_level] = 1.0
    bf = torch.bfloat16
    return dict(q=q.to(bf), k=k.to(bf), v=v.to(bf), log_a=None, lam=lam)


def make_gdn_inputs(cfg: FwdConfig):
    """Log-Linear Gated DeltaNet inputs: the forward recipe of ``cfg`` (q, v, log a, lambda),
    with each k scaled to unit length (the gated delta rule's keys are L2-normalised, which
    keeps I - beta k k^T a contraction) and a write strength beta = sigmoid(N(0,1)) per
    (b, t, h), drawn after the others.  Returns dict(q, k, v, log_a, beta, lam)."""
    x = make_fwd_inputs(cfg)
    g = _gen(cfg.seed + 7001)
    k = x["k"].float()
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-6)
    beta = torch.sigmoid(torch.randn(cfg.B, cfg.T, cfg.H, generator=g))
    return dict(q=x["q"], k=k.to(x["k"].dtype).contiguous(), v=x["v"], log_a=x["log_a"],
                beta=beta.contiguous(), lam=x["lam"])


def make_gdn_decode_step_inputs(cfg: DecodeConfig):
    """The new token of a Gated DeltaNet decode step at position cfg.t: the decode recipe
    with unit-length k and beta = sigmoid(N(0,1)) [B, H]."""
    x = make_decode_step_inputs(cfg)
    g = _gen(cfg.seed + 7002)
    k = x["k"].float()
    k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-6)
    beta = torch.sigmoid(torch.randn(cfg.B, cfg.H, generator=g))
    return dict(q=x["q"], k=k.to(x["k"].dtype).contiguous(), v=x["v"], log_a=x["log_a"],
                beta=beta.contiguous(), lam=x["lam"])


def make_decode_tokens(cfg: DecodeConfig, b: int, h: int, T: int):
    """Prefill stream of one (b, h): k [T,dk], v [T,dv] (cfg dtype), log_a [T] fp32.

    Seeded by (seed, b, h) so any (b, h) can be regenerated alone."""
    g = _gen(cfg.seed * 1_000_003 + 7919 * b + h + 1)
    k = torch.randn(T, cfg.dk, generator=g) / math.sqrt(cfg.dk)
    v = torch.randn(T, cfg.dv, generator=g)
    a_noise = torch.randn(T, generator=g)
    log_a = -0.1 * F.softplus(a_noise) if cfg.decay else None
    dt = torch_dtype(cfg.dtype)
    return k.to(dt), v.to(dt), log_a


def make_decode_step_inputs(cfg: DecodeConfig):
    """The new token at position cfg.t for every (b, h):
    q, k [B,H,dk]; v [B,H,dv] (cfg dtype); log_a [B,H] fp32 or None; lam [B,H,L]."""
    g = _gen(cfg.seed + 101)
    B, H = cfg.B, cfg.H
    q = torch.randn(B, H, cfg.dk, generator=g) / math.sqrt(cfg.dk)
    k = torch.randn(B, H, cfg.dk, generator=g) / math.sqrt(cfg.dk)
    v = torch.randn(B, H, cfg.dv, generator=g)
    a_noise = torch.randn(B, H, generator=g)
    lam = F.softplus(torch.randn(B, H, cfg.L, generator=g))
    log_a = -0.1 * F.softplus(a_noise) if cfg.decay else None
    dt = torch_dtype(cfg.dtype)
    return dict(q=q.to(dt), k=k.to(dt), v=v.to(dt), log_a=log_a, lam=lam)


def nonempty_levels_before(t: int, L: int):
    """Levels that hold data after position t-1 has been absorbed: level 0 and every
    level l >= 1 with bit l-1 of t-1 set (the bucket sizes of t-1)."""
    if t == 0:
        return []
    prev = t - 1
    return [0] + [l for l in range(1, L) if (prev >> (l - 1)) & 1]


def make_random_state(cfg: DecodeConfig, t: int, seed: int = 7, scale: float = 1.0):
    """A random fp32 state [B,H,L,dk,dv] for a decode step at position t: the levels that
    are non-empty after t-1 hold N(0, scale^2) entries, the others are zero."""
    g = _gen(seed)
    S = torch.zeros(cfg.B, cfg.H, cfg.L, cfg.dk, cfg.dv)
    for l in nonempty_levels_before(t, cfg.L):
        S[:, :, l] = torch.randn(cfg.B, cfg.H, cfg.dk, cfg.dv, generator=g) * scale
    return S
