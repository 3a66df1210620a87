"""Plain CPU oracle for Log-Linear Gated DeltaNet: direct form, lssb recurrence, decode step.

TEST INFRASTRUCTURE ONLY, like ``loglinear_oracle``: nothing on the product path imports,
calls or links this module.  It shares no code with the CUDA library.

What the pages fix, and what is read from elsewhere:

* The pages build the log-linear variant of a model by keeping that model's transition
  and composing its attention mask with the hierarchical Fenwick mask M^H (news article,
  section 对Mamba-2和门控DeltaNet的对数线性推广; reading post, section 与已有模型的组合;
  slide deck, slides 35-36).  They name Gated DeltaNet as the second model but print no
  formula for its transition.
* The transition is taken from the published gated delta rule (Yang, Kautz and
  Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta Rule", 2024), in this
  repository's state layout S [d_k, d_v] (o_t = S_t^T q_t):

      S_t = A_t S_{t-1} + beta_t k_t v_t^T,     A_t = alpha_t (I - beta_t k_t k_t^T),

  with alpha_t = exp(log_a_t) the gate and beta_t the write strength.
* Unrolled, o_t = sum_{s<=t} beta_s (q_t^T P_{t,s} k_s) v_s with P_{t,s} = A_t ... A_{s+1}
  (P_{t,t} = I): the model's own structured "attention" matrix.  Composed with M^H:

      o_t = sum_{s<=t} lam[t, level(t, s)] beta_s (q_t^T P_{t,s} k_s) v_s.

* Recurrently: one state per Fenwick bucket, S_t^(l) = sum over the level-l bucket of t of
  P_{t,s} beta_s k_s v_s^T; every old state is carried by A_t, the lssb rule merges,
  promotes and clears exactly as for Mamba-2 (reading post, section 解码：基于 lssb 的状态
  更新), and the new token enters level 0.  Because A_t is linear, carrying each level
  separately equals carrying their sum, so lambda constant across levels gives plain
  Gated DeltaNet.

Shapes: q, k [B, T, H, dk]; v [B, T, H, dv]; log_a [B, T, H] or None (alpha = 1);
beta [B, T, H]; lam [B, T, H, L].  delta=False drops the k k^T term (A_t = alpha_t I),
which is the pages' Mamba-2 form with v scaled by beta.
"""
from __future__ import annotations

import numpy as np

from .loglinear_oracle import _f64, fenwick_partition, level_row, lssb


def _carry(x, k_r, alpha_r, beta_r, delta):
    """A_r x for x [dk] or [dk, dv]: alpha_r (x - beta_r k_r (k_r^T x)); alpha_r x without
    the delta term."""
    if not delta:
        return alpha_r * x
    return alpha_r * (x - beta_r * np.multiply.outer(k_r, k_r @ x))


def gdn_direct(q, k, v, log_a, beta, lam, rows=None, heads=None, delta=True):
    """o_t = sum_{s<=t} lam[t, level(t,s)] beta_s (q_t^T P_{t,s} k_s) v_s, fp64, evaluated
    literally: for each query row t, x = P_{t,s}^T q_t is carried from s = t down to s = 0
    (x <- A_s x, A symmetric), and the score of source s is beta_s k_s . x.

    rows: optional query positions (all if None); heads: optional (b, h) pairs.
    Returns [B, T, H, dv] (rows / heads not evaluated left at zero)."""
    q, k, v, lam, beta = _f64(q), _f64(k), _f64(v), _f64(lam), _f64(beta)
    log_a = _f64(log_a)
    B, T, H, _ = q.shape
    dv = v.shape[-1]
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    out = np.zeros((B, T, H, dv))
    for b, h in heads:
        K, V, bt = k[b, :, h], v[b, :, h], beta[b, :, h]
        alpha = np.ones(T) if log_a is None else np.exp(log_a[b, :, h])
        for t in rows:
            t = int(t)
            lv = level_row(t)
            x = q[b, t, h].copy()
            score = np.zeros(t + 1)
            for s in range(t, -1, -1):
                score[s] = bt[s] * (K[s] @ x)
                if s > 0:
                    x = _carry(x, K[s], alpha[s], bt[s], delta)
            out[b, t, h] = (lam[b, t, h, lv] * score) @ V[: t + 1]
    return out


def gdn_states_from_buckets(k_bh, v_bh, log_a_bh, beta_bh, t: int, L: int, delta=True):
    """Per-level states at position t from their definition: S^(l) = sum over the level-l
    bucket of t of P_{t,s} beta_s k_s v_s^T, each term carried from s to t one transition at
    a time.  k_bh [T, dk], v_bh [T, dv], log_a_bh [T] or None, beta_bh [T]."""
    k_bh, v_bh, beta_bh = _f64(k_bh), _f64(v_bh), _f64(beta_bh)
    log_a_bh = _f64(log_a_bh)
    dk, dv = k_bh.shape[1], v_bh.shape[1]
    alpha = np.ones(t + 1) if log_a_bh is None else np.exp(log_a_bh[: t + 1])
    S = np.zeros((L, dk, dv))
    for lvl, lo, hi in fenwick_partition(t):
        if lvl >= L:
            raise ValueError(f"level {lvl} needs L > {lvl}")
        for s in range(lo, hi):
            term = beta_bh[s] * np.multiply.outer(k_bh[s], v_bh[s])
            for r in range(s + 1, t + 1):
                term = _carry(term, k_bh[r], alpha[r], beta_bh[r], delta)
            S[lvl] += term
    return S


def gdn_decode_step(state, q, k, v, log_a, beta, lam, t: int, delta=True):
    """One decode step of Log-Linear Gated DeltaNet, batched over leading dims.

    Every state held after t-1 is carried by A_t; then the lssb rule: levels 0..lssb(t)
    merge into level lssb(t)+1, levels 1..lssb(t) are cleared (reading post, 解码 section;
    slide deck, slide 21); level 0 receives beta_t k_t v_t^T.  At t = 0 the state starts
    empty.  The output is sum_l lam_l S^(l)^T q_t.

    state [..., L, dk, dv]; q, k [..., dk]; v [..., dv]; log_a, beta [...]; lam [..., L].
    Returns (new_state, o [..., dv]).  Inputs are not modified."""
    S = _f64(state).copy()
    q, k, v, lam, beta = _f64(q), _f64(k), _f64(v), _f64(lam), _f64(beta)
    alpha = np.ones(S.shape[:-3]) if log_a is None else np.exp(_f64(log_a))
    L = S.shape[-3]
    if t == 0:
        S[...] = 0.0
    else:
        l = lssb(t)
        if l + 1 >= L:
            raise ValueError(f"t={t} needs L > {l + 1}")
        a4 = alpha[..., None, None, None]
        if delta:
            # A_t S = alpha (S - beta k (k^T S)) for every level at once
            kS = np.einsum("...d,...lde->...le", k, S)
            S = a4 * (S - beta[..., None, None, None] * k[..., None, :, None] * kS[..., :, None, :])
        else:
            S = a4 * S
        merged = S[..., : l + 1, :, :].sum(axis=-3)
        S[..., l + 1, :, :] = merged
        S[..., 1 : l + 1, :, :] = 0.0
    S[..., 0, :, :] = beta[..., None, None] * k[..., :, None] * v[..., None, :]
    o = np.einsum("...l,...d,...lde->...e", lam, q, S)
    return S, o


def gdn_recurrence(q, k, v, log_a, beta, lam, delta=True):
    """Run gdn_decode_step over t = 0..T-1 for every (b, h).
    Returns (out [B, T, H, dv], final state [B, H, L, dk, dv])."""
    q, k, v, lam, beta = _f64(q), _f64(k), _f64(v), _f64(lam), _f64(beta)
    log_a = _f64(log_a)
    B, T, H, dk = q.shape
    dv, L = v.shape[-1], lam.shape[-1]
    S = np.zeros((B, H, L, dk, dv))
    out = np.zeros((B, T, H, dv))
    for t in range(T):
        la = None if log_a is None else log_a[:, t, :]
        S, out[:, t] = gdn_decode_step(S, q[:, t], k[:, t], v[:, t], la, beta[:, t], lam[:, t],
                                       t, delta=delta)
    return out, S


def gated_deltanet_recurrent(q, k, v, log_a, beta, c=None):
    """Plain Gated DeltaNet by its published recurrence, one state, no levels:
    S_t = alpha_t (S_{t-1} - beta_t k_t (k_t^T S_{t-1})) + beta_t k_t v_t^T,
    o_t = c_t S_t^T q_t (c [B, T, H] or None = 1).  What the log-linear form reduces to
    when lambda is the same at every level."""
    q, k, v, beta = _f64(q), _f64(k), _f64(v), _f64(beta)
    log_a = _f64(log_a)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    S = np.zeros((B, H, dk, dv))
    out = np.zeros((B, T, H, dv))
    for t in range(T):
        kt, vt, bt = k[:, t], v[:, t], beta[:, t]
        alpha = np.ones((B, H)) if log_a is None else np.exp(log_a[:, t])
        kS = np.einsum("bhd,bhde->bhe", kt, S)                       # k_t^T S_{t-1}
        S = alpha[..., None, None] * (S - bt[..., None, None] * kt[..., :, None] * kS[..., None, :])
        S = S + bt[..., None, None] * kt[..., :, None] * vt[..., None, :]
        o = np.einsum("bhd,bhde->bhe", q[:, t], S)
        if c is not None:
            o = o * _f64(c)[:, t, :, None]
        out[:, t] = o
    return out
