"""Shared helpers of the parity tests (comparison metrics and tolerances)."""
import numpy as np
import torch

# Tolerances: rel-L2 <= 1e-5 for fp32 inputs; <= 2e-2 for bf16 inputs with fp32
# accumulation (max-abs reported next to it); level indexing exact.
TOL_F32 = 1e-5
TOL_BF16 = 2e-2


def to64(x):
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def rel_l2(got, want):
    got, want = to64(got), to64(want)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def max_abs(got, want):
    return float(np.max(np.abs(to64(got) - to64(want)))) if to64(want).size else 0.0


def cuda(d):
    return {k: (None if v is None else v.cuda()) for k, v in d.items()}


def tol_for(dtype):
    return TOL_F32 if dtype in ("f32", torch.float32) else TOL_BF16


def per_head_qk(x):
    """The same inputs with q and k given per value head: q/k head g serves the value heads
    g * (H / Hqk) .. (g + 1) * (H / Hqk) - 1, so each is repeated H / Hqk times in place.
    Input marshalling for the oracle, whose definition is per head."""
    H, G = x["v"].shape[2], x["q"].shape[2]
    if G == H:
        return x
    y = dict(x)
    for n in ("q", "k"):
        y[n] = x[n].repeat_interleave(H // G, dim=2).contiguous()
    return y


def one_head(x, b, h):
    """The inputs of value head h of batch b alone (B = H = 1), with the q/k of its group:
    input marshalling for the oracle, one head at a time."""
    hq = h // (x["v"].shape[2] // x["q"].shape[2])
    sl = lambda t, j: None if t is None else t[b:b + 1, :, j:j + 1].contiguous()
    return {"q": sl(x["q"], hq), "k": sl(x["k"], hq), "v": sl(x["v"], h),
            "log_a": sl(x["log_a"], h), "lam": sl(x["lam"], h)}
