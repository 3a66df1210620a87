"""Pins of the Log-Linear Gated DeltaNet oracle (CPU).

Each function of ``oracle.gdn_oracle`` is checked against something other than itself:
* the plain Gated DeltaNet recurrence (one state, the published gated delta rule) when
  lambda is the same at every level;
* the already pinned log-linear Mamba-2 oracle when the delta term is dropped;
* the delta rule's defining behaviour (writing a key again replaces what it stored), and
  a hand-worked two-token example;
* the bucket definition of the per-level states, and the direct form at a decode row.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import gdn_oracle
import workloads as W


def _inputs(T, H=2, dk=5, dv=3, L=None, decay=True, seed=0):
    L = L or max((T - 1).bit_length() + 1, 1)
    cfg = W.FwdConfig("gdn_pin", 2, H, T, dk, dv, 4, L, "f32", decay, "softplus", seed=seed)
    return W.make_gdn_inputs(cfg)


def _rel(a, b):
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


@pytest.mark.parametrize("T,decay", [(1, True), (2, False), (7, True), (8, True), (23, True),
                                     (33, False)])
def test_direct_equals_lssb_recurrence(T, decay):
    x = _inputs(T, decay=decay, seed=T)
    d = oracle.gdn_direct(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"])
    r, _ = oracle.gdn_recurrence(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"])
    assert _rel(r, d) <= 1e-12


@pytest.mark.parametrize("decay", [True, False])
def test_constant_lambda_is_plain_gated_deltanet(decay):
    """lambda[t, l] = c_t at every level: the log-linear model is c_t times Gated DeltaNet
    (the published recurrence, written independently with a single state)."""
    x = _inputs(29, decay=decay, seed=3)
    c = x["lam"][..., 0].clone()
    lam = c[..., None].expand_as(x["lam"]).contiguous()
    d = oracle.gdn_direct(x["q"], x["k"], x["v"], x["log_a"], x["beta"], lam)
    g = oracle.gated_deltanet_recurrent(x["q"], x["k"], x["v"], x["log_a"], x["beta"], c=c)
    assert _rel(d, g) <= 1e-12


@pytest.mark.parametrize("decay", [True, False])
def test_without_delta_term_is_loglinear_mamba2(decay):
    """Dropping beta k k^T from the transition leaves alpha_t I: the log-linear Mamba-2 form
    (the pinned oracle's forward_direct) with v scaled by beta."""
    x = _inputs(26, decay=decay, seed=5)
    d = oracle.gdn_direct(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"], delta=False)
    r, _ = oracle.gdn_recurrence(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"],
                                 delta=False)
    vb = x["v"].double() * x["beta"].double()[..., None]   # the product in fp64
    m = oracle.forward_direct(x["q"], x["k"], vb, x["log_a"], x["lam"])
    assert _rel(d, m) <= 1e-12 and _rel(r, m) <= 1e-12


def test_delta_rule_overwrites_a_key():
    """With alpha = beta = 1 and a unit key written twice, the second write replaces the
    first: (I - k k^T)(k v1^T) + k v2^T = k v2^T.  Reading that key at t = 1 gives v2, the
    level-1 bucket (the first token) contributes exactly nothing, and level 0 gives v2."""
    k = torch.tensor([1.0, 0.0]).expand(1, 2, 1, 2).contiguous()
    q = k.clone()
    v = torch.tensor([[1.0, 2.0], [3.0, -1.0]]).reshape(1, 2, 1, 2)
    beta = torch.ones(1, 2, 1)
    for lam_row, want in (([1.0, 1.0], [3.0, -1.0]), ([0.0, 1.0], [0.0, 0.0]),
                          ([1.0, 0.0], [3.0, -1.0])):
        lam = torch.tensor([[1.0, 1.0], lam_row]).reshape(1, 2, 1, 2)
        d = oracle.gdn_direct(q, k, v, None, beta, lam)
        r, S = oracle.gdn_recurrence(q, k, v, None, beta, lam)
        assert np.allclose(d[0, 1, 0], want, atol=1e-15) and np.allclose(r[0, 1, 0], want, atol=1e-15)
        assert np.allclose(d[0, 0, 0], [1.0, 2.0])
    # the state after both writes: level 0 holds k v2^T, level 1 holds the erased first write
    assert np.allclose(S[0, 0, 0], [[3.0, -1.0], [0.0, 0.0]], atol=1e-15)
    assert np.allclose(S[0, 0, 1], 0.0, atol=1e-15)


def test_hand_worked_two_tokens():
    """d_k = 2, one head, decay and beta != 1, worked out by hand:
    o_0 = l0[0] b0 (q0.k0) v0;  o_1 = l1[0] b1 (q1.k1) v1 + l1[1] b0 q1^T A_1 k0 v0 with
    A_1 = a1 (I - b1 k1 k1^T)."""
    k0, k1 = np.array([0.6, 0.8]), np.array([1.0, 0.0])
    q0, q1 = np.array([1.0, -1.0]), np.array([0.5, 2.0])
    v0, v1 = np.array([2.0]), np.array([-1.0])
    b0, b1, a1 = 0.5, 0.25, 0.9
    lam = np.array([[0.3, 0.7], [1.5, 2.5]])
    A1 = a1 * (np.eye(2) - b1 * np.outer(k1, k1))
    want0 = lam[0, 0] * b0 * (q0 @ k0) * v0
    want1 = lam[1, 0] * b1 * (q1 @ k1) * v1 + lam[1, 1] * b0 * (q1 @ A1 @ k0) * v0
    T = lambda a: torch.tensor(np.asarray(a), dtype=torch.float64)
    q = T([q0, q1]).reshape(1, 2, 1, 2)
    k = T([k0, k1]).reshape(1, 2, 1, 2)
    v = T([v0, v1]).reshape(1, 2, 1, 1)
    log_a = T([[np.log(0.7)], [np.log(a1)]]).reshape(1, 2, 1)   # a_0 is never used
    beta = T([[b0], [b1]]).reshape(1, 2, 1)
    lm = T(lam).reshape(1, 2, 1, 2)
    for o in (oracle.gdn_direct(q, k, v, log_a, beta, lm),
              oracle.gdn_recurrence(q, k, v, log_a, beta, lm)[0]):
        assert np.allclose(o[0, 0, 0], want0, rtol=1e-14) and np.allclose(o[0, 1, 0], want1, rtol=1e-14)


@pytest.mark.parametrize("T", [1, 6, 8, 13, 32])
def test_recurrence_state_is_the_bucket_definition(T):
    x = _inputs(T, seed=T + 40)
    L = x["lam"].shape[-1]
    _, S = oracle.gdn_recurrence(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"])
    for b in range(2):
        for h in range(2):
            want = oracle.gdn_states_from_buckets(x["k"][b, :, h], x["v"][b, :, h],
                                                  x["log_a"][b, :, h], x["beta"][b, :, h], T - 1, L)
            assert _rel(S[b, h], want) <= 1e-12


@pytest.mark.parametrize("t", [1, 2, 7, 12, 16, 21])
def test_decode_row_equals_direct(t):
    """The state after t-1 (bucket definition), one decode step, and the direct form's row t
    agree, as do the state after the step and the bucket definition at t."""
    x = _inputs(t + 1, seed=t + 70)
    L = x["lam"].shape[-1]
    S_prev = np.stack([np.stack([oracle.gdn_states_from_buckets(
        x["k"][b, :, h], x["v"][b, :, h], x["log_a"][b, :, h], x["beta"][b, :, h], t - 1, L)
        for h in range(2)]) for b in range(2)])
    S_new, o = oracle.gdn_decode_step(S_prev, x["q"][:, t], x["k"][:, t], x["v"][:, t],
                                      x["log_a"][:, t], x["beta"][:, t], x["lam"][:, t], t)
    d = oracle.gdn_direct(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"], rows=[t])
    assert _rel(o, d[:, t]) <= 1e-12
    for b in range(2):
        for h in range(2):
            want = oracle.gdn_states_from_buckets(x["k"][b, :, h], x["v"][b, :, h],
                                                  x["log_a"][b, :, h], x["beta"][b, :, h], t, L)
            assert _rel(S_new[b, h], want) <= 1e-12


def test_planted_mistakes_fail_the_pins(monkeypatch):
    """A transition with the delta term's sign flipped, or without the gate, must break
    the pin against plain Gated DeltaNet (both planted in the oracle, on the CPU)."""
    x = _inputs(17, seed=9)
    c = x["lam"][..., 0].clone()
    lam = c[..., None].expand_as(x["lam"]).contiguous()
    g = oracle.gated_deltanet_recurrent(x["q"], x["k"], x["v"], x["log_a"], x["beta"], c=c)
    good = gdn_oracle._carry
    bad = [lambda x_, k_, a_, b_, d_: a_ * (x_ + b_ * np.multiply.outer(k_, k_ @ x_)),
           lambda x_, k_, a_, b_, d_: good(x_, k_, 1.0, b_, d_)]
    for fn in bad:
        monkeypatch.setattr(gdn_oracle, "_carry", fn)
        d = gdn_oracle.gdn_direct(x["q"], x["k"], x["v"], x["log_a"], x["beta"], lam)
        assert _rel(d, g) > 1e-3
    monkeypatch.setattr(gdn_oracle, "_carry", good)
