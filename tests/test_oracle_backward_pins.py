"""Pins of the oracle's backward (oracle.backward_direct) to facts outside itself (CPU).

* Brute force: central finite differences of the oracle's own forward (itself pinned in
  test_oracle_pins.py) for every input element on tiny problems.
* Homogeneity: O is linear in each of q, k, v and lambda, so for each of them
  sum(dX ⊙ X) = sum(dO ⊙ O) (Euler's theorem for degree-1 functions).
* Shift invariance: M^S depends on log a only through differences of its prefix sums
  that never include position 0, so d log a_0 = 0.
* Special case: with no decay and lambda = 1 at every level the method is causal linear
  attention, O = (Q K^T ⊙ tril) V; torch's autograd of that plain expression gives the
  q, k, v gradients independently of the oracle's formulas.
"""
import numpy as np
import pytest
import torch

import oracle


def _inputs(B, T, H, dk, dv, L, seed, decay=True):
    r = np.random.default_rng(seed)
    x = dict(q=r.standard_normal((B, T, H, dk)) / np.sqrt(dk),
             k=r.standard_normal((B, T, H, dk)) / np.sqrt(dk),
             v=r.standard_normal((B, T, H, dv)),
             log_a=-0.1 * np.log1p(np.exp(r.standard_normal((B, T, H)))) if decay else None,
             lam=np.log1p(np.exp(r.standard_normal((B, T, H, L)))))
    dout = r.standard_normal((B, T, H, dv))
    return x, dout


def _loss(x, dout):
    return float(np.sum(dout * oracle.forward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"])))


@pytest.mark.parametrize("decay", [True, False])
def test_backward_matches_finite_differences(decay):
    x, dout = _inputs(1, 19, 2, 3, 2, 6, seed=3 if decay else 4, decay=decay)
    g = oracle.backward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout)
    eps = 1e-6
    for name in ("q", "k", "v", "lam", "log_a"):
        if x[name] is None:
            assert g[name] is None
            continue
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(x[name].shape):
            xp = {n: (None if t is None else t.copy()) for n, t in x.items()}
            xp[name][idx] += eps
            lp = _loss(xp, dout)
            xp[name][idx] -= 2 * eps
            lm = _loss(xp, dout)
            fd[idx] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(g[name] - fd) / max(np.linalg.norm(fd), 1e-300)
        assert err < 1e-7, (name, err)


def test_backward_homogeneity_identities():
    x, dout = _inputs(2, 300, 2, 8, 4, 10, seed=7)
    o = oracle.forward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"])
    g = oracle.backward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout)
    ref = float(np.sum(dout * o))
    for name in ("q", "k", "v", "lam"):
        val = float(np.sum(g[name] * x[name]))
        assert abs(val - ref) <= 1e-10 * max(abs(ref), 1.0), name
    # row by row for lambda: sum_l dlam[t, l] lam[t, l] = dO_t . O_t
    np.testing.assert_allclose(np.sum(g["lam"] * x["lam"], axis=-1), np.sum(dout * o, axis=-1),
                               rtol=1e-10, atol=1e-12)


def test_backward_dlog_a_first_position_is_zero():
    x, dout = _inputs(2, 257, 3, 8, 4, 10, seed=9)
    g = oracle.backward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout)
    scale = np.abs(g["log_a"]).max()
    assert scale > 0
    assert np.abs(g["log_a"][:, 0, :]).max() <= 1e-12 * scale


def test_backward_linear_attention_special_case():
    B, T, H, dk, dv, L = 1, 70, 2, 5, 3, 8
    x, dout = _inputs(B, T, H, dk, dv, L, seed=11, decay=False)
    x["lam"] = np.ones((B, T, H, L))
    g = oracle.backward_direct(x["q"], x["k"], x["v"], None, x["lam"], dout)
    q, k, v = (torch.tensor(x[n], requires_grad=True) for n in ("q", "k", "v"))
    tril = torch.tril(torch.ones(T, T, dtype=torch.float64))
    o = torch.einsum("bthd,bshd->bhts", q, k) * tril
    o = torch.einsum("bhts,bshe->bthe", o, v)
    o.backward(torch.tensor(dout))
    for name, t in (("q", q), ("k", k), ("v", v)):
        np.testing.assert_allclose(g[name], t.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_backward_sampled_equals_direct():
    """The row / column evaluation of the sampled backward equals the dense one."""
    x, dout = _inputs(2, 150, 3, 8, 4, 9, seed=13)
    g = oracle.backward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout)
    rows = [0, 1, 7, 64, 127, 149]
    cols = [0, 5, 63, 64, 100, 149]
    heads = [(0, 1), (1, 2)]
    gs = oracle.backward_sampled(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout, rows, cols,
                                 heads)
    for i, (b, h) in enumerate(heads):
        np.testing.assert_allclose(gs["q"][i], g["q"][b, rows, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(gs["lam"][i], g["lam"][b, rows, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(gs["k"][i], g["k"][b, cols, h], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(gs["v"][i], g["v"][b, cols, h], rtol=1e-12, atol=1e-13)
