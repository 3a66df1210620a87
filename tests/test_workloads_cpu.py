"""The seeded input recipe (CPU): shapes, dtypes and value distributions of the synthetic
workloads, their determinism, and the exactness properties the integer generators
promise."""
import math

import numpy as np
import pytest
import torch

import workloads as W


def _inv_softplus(y):
    return np.log(np.expm1(y))


def test_fwd_inputs_shapes_and_dtypes():
    cfg = W.FWD_CONFIGS["mva_B2H48_T16384"].with_(T=256)
    x = W.make_fwd_inputs(cfg)
    assert x["q"].shape == (2, 256, 1, 128) and x["k"].shape == (2, 256, 1, 128)
    assert x["v"].shape == (2, 256, 48, 64)
    assert x["log_a"].shape == (2, 256, 48) and x["lam"].shape == (2, 256, 48, 15)
    assert x["q"].dtype == torch.bfloat16 and x["v"].dtype == torch.bfloat16
    assert x["log_a"].dtype == torch.float32 and x["lam"].dtype == torch.float32
    assert all(t.is_contiguous() for t in x.values())


def test_fwd_inputs_distributions():
    """q, k ~ N(0,1)/sqrt(d_k), v ~ N(0,1), log a = -0.1 softplus(N(0,1)) and
    lambda = softplus(N(0,1)): undoing each transform gives standard normal samples."""
    cfg = W.FwdConfig("dist", 1, 4, 4096, 64, 32, 64, 13, "f32", True, "softplus", seed=3)
    x = W.make_fwd_inputs(cfg)
    n = {"q": x["q"].numpy() * math.sqrt(64), "k": x["k"].numpy() * math.sqrt(64),
         "v": x["v"].numpy()}
    la = x["log_a"].numpy()
    assert (la < 0).all()
    n["log_a"] = _inv_softplus(-10.0 * la.astype(np.float64))
    n["lam"] = _inv_softplus(x["lam"].numpy().astype(np.float64))
    for name, z in n.items():
        assert abs(z.mean()) < 0.02, name
        assert abs(z.std() - 1.0) < 0.02, name
    # the mean decay per step the documentation quotes: -0.1 * E[softplus(Z)] ~ -0.081
    assert abs(la.mean() + 0.0806) < 0.002


def test_uniform_lambda_and_no_decay():
    cfg = W.FWD_CONFIGS["linear_T64"]
    x = W.make_fwd_inputs(cfg)
    assert x["log_a"] is None
    lam = x["lam"].numpy()
    assert (lam >= 0).all() and (lam < 1).all()
    assert x["q"].dtype == torch.float32


def test_fwd_inputs_deterministic_per_seed():
    cfg = W.FWD_CONFIGS["mamba2_T1024"].with_(T=128)
    a, b = W.make_fwd_inputs(cfg), W.make_fwd_inputs(cfg)
    c = W.make_fwd_inputs(cfg.with_(seed=1))
    for name in a:
        assert torch.equal(a[name], b[name]), name
        assert not torch.equal(a[name], c[name]), name


def test_bf16_inputs_are_rounded_draws():
    """A bf16 workload holds the same draws as its fp32 twin, rounded once."""
    cfg = W.FwdConfig("r", 1, 2, 128, 16, 16, 64, 8, "bf16", True, "softplus", seed=5)
    a, b = W.make_fwd_inputs(cfg), W.make_fwd_inputs(cfg.with_(dtype="f32"))
    for name in ("q", "k", "v"):
        assert torch.equal(a[name], b[name].to(torch.bfloat16)), name
    assert torch.equal(a["lam"], b["lam"]) and torch.equal(a["log_a"], b["log_a"])


@pytest.mark.parametrize("level", [0, 3])
def test_int_inputs_are_small_integers_with_one_hot_lambda(level):
    x = W.make_int_inputs(1, 64, 2, 6, 4, 7, level, seed=level)
    for name in ("q", "k", "v"):
        t = x[name]
        assert torch.equal(t, t.round()) and t.abs().max() <= 2, name
    lam = x["lam"]
    assert torch.equal(lam.sum(-1), torch.ones(1, 64, 2)) and torch.all(lam[..., level] == 1)


def test_sparse_int_inputs_keep_dots_in_minus_one_to_one():
    x = W.make_sparse_int_inputs(1, 200, 2, 16, 9, 2, seed=4, dv=8)
    k = x["k"].float()
    assert torch.equal((k != 0).sum(-1), torch.ones(1, 200, 2, dtype=torch.long))
    dots = torch.einsum("bthd,bshd->bhts", x["q"].float(), k)
    assert dots.abs().max() <= 1 and x["v"].shape[-1] == 8


def test_nonempty_levels_follow_the_bits_of_t_minus_one():
    assert W.nonempty_levels_before(0, 15) == []
    assert W.nonempty_levels_before(1, 15) == [0]
    # t = 12345: t - 1 = 0b11000000111000, bits 3, 4, 5, 12, 13
    assert W.nonempty_levels_before(12345, 15) == [0, 4, 5, 6, 13, 14]
