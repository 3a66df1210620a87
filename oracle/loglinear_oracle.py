"""Plain CPU oracle for log-linear attention: forward and lssb decode, fp64 NumPy.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports, calls or links this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it. It shares no code, table or helper
with the CUDA library; the two meet only at the seeded inputs of ``workloads``.

Sources (titles of the pages the method is described on):

* "论文阅读：Log-Linear Attention — 基于 Fenwick 树与层次矩阵的对数线性复杂度注意力机制"
  (paper-reading post, below "the reading post"), sections 前缀的层次化分解 (Fenwick
  partition of the prefix), 层级判定算法 (the level walk), 循环形式与输出计算 (per-level
  states and the lambda-weighted readout), 并行形式 (the 8x8 M^H table), 解码：基于 lssb
  的状态更新 (the lssb decode rule), 矩阵分解 / 两阶段计算 (chunked two-stage algorithm),
  与已有模型的组合 (M = M^S ⊙ M^H).
* "算力终结者来了！…AI狂飙进对数时代" (news article, below "the news article"), sections
  结构矩阵 (O = (A ⊙ M) V), 特殊结构：Fenwick树划分, 高效训练算法.
* "【人工知能・深層学習】論文紹介：Log Linear Attention" (slide deck), slides 9, 16,
  19-21, 33-34.

Readings of the pages where the text is silent or garbled (each one is listed in the
repository's design notes too):

1. Decay: M^S[t, s] = prod_{r=s+1..t} a_r (the Mamba-2 semiseparable mask; diagonal 1),
   evaluated as exp(cum_t - cum_s) over fp64 prefix sums of log a.
2. lambda is indexed by the query position and the level: M^H[t, s] = lam[t, level(t, s)].
3. lssb(t) is the 0-based index of the lowest set bit of t; levels 0..lssb(t) merge into
   level lssb(t)+1, levels 1..lssb(t) are cleared, higher levels are kept (times a_t).
4. t = 0: the state starts empty; only level 0 receives k_0 v_0^T.

Shapes follow the product's layout: q, k [B, T, H, dk]; v [B, T, H, dv];
log_a [B, T, H] (None = no decay, M^S all ones); lam [B, T, H, L]; out [B, T, H, dv].
"""
from __future__ import annotations

import numpy as np

# --------------------------------------------------------------------------------------
# L0: the Fenwick partition of the prefix and the level of a source position
# --------------------------------------------------------------------------------------


def fenwick_partition(t: int):
    """Buckets of the prefix [0, t] seen from query position t.

    Reading post, section 前缀的层次化分解: the prefix before t is cut into disjoint
    buckets by starting from t and repeatedly removing the lowest set bit of the running
    boundary; each removal cuts one bucket whose size is that bit.  The bucket cut by a
    bit of value 2^(l-1) is level l.  The query itself forms the size-1 sentinel bucket,
    level 0.  Returns a list of (level, lo, hi) half-open intervals, nearest first.
    """
    if t < 0:
        raise ValueError("t must be >= 0")
    out = [(0, t, t + 1)]
    boundary = t
    while boundary:
        size = boundary & -boundary          # value of the lowest set bit
        out.append((size.bit_length(), boundary - size, boundary))
        boundary -= size
    return out


def level(t: int, s: int) -> int:
    """Level l(t, s) of source s as seen from query t (0 <= s <= t).

    Reading post, section 层级判定算法: the level is the one of the Fenwick bucket of t
    that contains s; s == t is the sentinel bucket, level 0.
    """
    for lvl, lo, hi in fenwick_partition(t):
        if lo <= s < hi:
            return lvl
    raise ValueError(f"source {s} is not in the prefix of query {t}")


def level_row(t: int) -> np.ndarray:
    """Levels l(t, s) for s = 0..t as an int64 array (same walk, one bucket at a time)."""
    row = np.empty(t + 1, dtype=np.int64)
    for lvl, lo, hi in fenwick_partition(t):
        row[lo:hi] = lvl
    return row


def level_matrix(T: int) -> np.ndarray:
    """[T, T] int64 matrix of l(t, s) for s <= t and -1 above the diagonal."""
    m = np.full((T, T), -1, dtype=np.int64)
    for t in range(T):
        m[t, : t + 1] = level_row(t)
    return m


def lssb(t: int) -> int:
    """0-based index of the least significant set bit of t > 0 (reading post, 解码 section)."""
    if t <= 0:
        raise ValueError("lssb is defined for t > 0")
    return (t & -t).bit_length() - 1


# --------------------------------------------------------------------------------------
# L1: masks and the direct parallel form O = (Q K^T ⊙ M^S ⊙ M^H) V
# --------------------------------------------------------------------------------------


def _f64(x):
    """Input upcast to fp64 NumPy.  Torch tensors of 16-bit types (which NumPy lacks) go
    through fp32 exactly; fp32 and fp64 tensors convert directly, so fp64 inputs keep
    their precision."""
    if x is None:
        return None
    if hasattr(x, "detach"):            # torch tensor (any dtype, incl. bfloat16)
        x = x.detach().cpu()
        if x.element_size() < 4:
            x = x.float()
        x = x.numpy()
    return np.asarray(x, dtype=np.float64)


def decay_rows(log_a_bh: np.ndarray | None, rows: np.ndarray, T: int) -> np.ndarray:
    """M^S[t, s] for t in rows and all s < T (zero above the diagonal).

    Reading post, section 与已有模型的组合 and the slide deck, slide 9: M^S is the
    1-semiseparable mask of the Mamba-2 recurrence, prod_{r=s+1..t} a_r for s <= t.
    """
    causal = np.arange(T)[None, :] <= rows[:, None]
    if log_a_bh is None:
        return causal.astype(np.float64)
    cum = np.cumsum(log_a_bh)
    expo = np.where(causal, cum[rows][:, None] - cum[None, :], -np.inf)
    return np.exp(expo)


def hier_rows(lam_bh: np.ndarray, rows: np.ndarray, T: int) -> np.ndarray:
    """M^H[t, s] = lam[t, l(t, s)] for t in rows, zero above the diagonal.

    Reading post, section 并行形式 (the 8x8 table) and the news article, section
    特殊结构：Fenwick树划分: the weight of source s in row t is the query's weight for the
    level that s falls in.
    """
    out = np.zeros((len(rows), T))
    for i, t in enumerate(rows):
        lv = level_row(int(t))
        out[i, : t + 1] = lam_bh[t, lv]
    return out


def forward_direct(q, k, v, log_a, lam, rows=None, heads=None):
    """O = (Q K^T ⊙ M^S ⊙ M^H) V evaluated literally in fp64.

    Reading post, section 并行形式; news article, section 结构矩阵 (O = (A ⊙ M) V with
    A = Q K^T) and section 特殊结构 (M^H from the Fenwick level of s seen from t).

    rows: optional sorted int array of query positions to evaluate (all if None).
    heads: optional list of (b, h) pairs to evaluate (all if None).
    Returns [B, T, H, dv] (rows / heads not evaluated are left at zero).
    """
    q, k, v, lam = _f64(q), _f64(k), _f64(v), _f64(lam)
    log_a = _f64(log_a)
    B, T, H, _ = q.shape
    dv = v.shape[-1]
    rows = np.arange(T) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = [(b, h) for b in range(B) for h in range(H)] if heads is None else heads
    out = np.zeros((B, T, H, dv))
    for b, h in heads:
        Q, K, V = q[b, :, h, :], k[b, :, h, :], v[b, :, h, :]
        la = None if log_a is None else log_a[b, :, h]
        for r0 in range(0, len(rows), 512):
            rr = rows[r0 : r0 + 512]
            A = Q[rr] @ K.T
            M = decay_rows(la, rr, T) * hier_rows(lam[b, :, h, :], rr, T)
            out[b, rr, h, :] = (A * M) @ V
    return out


def backward_direct(q, k, v, log_a, lam, dout):
    """Gradients of sum(dout ⊙ O) for O = (Q K^T ⊙ M^S ⊙ M^H) V, by the chain rule on the
    dense definition, fp64.

    News article, section 讨论与局限性: training needs, besides the gradients of the
    attention terms, those of the level weights lambda; its Figure 4 times the forward and
    backward kernels.  With A = Q K^T, M = M^S ⊙ M^H and dA = dO V^T:
        dV = (A ⊙ M)^T dO,   dQ = (dA ⊙ M) K,   dK = (dA ⊙ M)^T Q,
        dlam[t, l] = sum over s with level(t, s) = l of dA[t, s] A[t, s] M^S[t, s],
    and, since M^S[t, s] = exp(cum_t - cum_s) with cum the prefix sums of log a,
        dcum_t = sum_s G[t, s] - sum_t' G[t', t]   (G = dA ⊙ A ⊙ M),
        dlog_a[i] = sum over t >= i of dcum_t.
    Rows are taken in blocks of 512 (evaluation order only).

    Returns dict(q, k, v, log_a, lam) of fp64 arrays in the input layouts (log_a is None
    when log_a is None).
    """
    q, k, v, lam, do = _f64(q), _f64(k), _f64(v), _f64(lam), _f64(dout)
    log_a = _f64(log_a)
    B, T, H, dk = q.shape
    dv, L = v.shape[-1], lam.shape[-1]
    g = {"q": np.zeros_like(q), "k": np.zeros_like(k), "v": np.zeros_like(v),
         "lam": np.zeros_like(lam), "log_a": None if log_a is None else np.zeros_like(log_a)}
    for b in range(B):
        for h in range(H):
            Q, K, V, dO = q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h]
            la = None if log_a is None else log_a[b, :, h]
            row_sum = np.zeros(T)
            col_sum = np.zeros(T)
            for r0 in range(0, T, 512):
                rr = np.arange(r0, min(T, r0 + 512))
                MS = decay_rows(la, rr, T)
                M = MS * hier_rows(lam[b, :, h, :], rr, T)
                A = Q[rr] @ K.T
                dA = dO[rr] @ V.T
                dAM = dA * M
                g["q"][b, rr, h] = dAM @ K
                g["k"][b, :, h] += dAM.T @ Q[rr]
                g["v"][b, :, h] += (A * M).T @ dO[rr]
                W = dA * A * MS
                for i, t in enumerate(rr):
                    lv = level_row(int(t))
                    np.add.at(g["lam"][b, t, h], lv, W[i, : t + 1])
                G = dAM * A
                row_sum[rr] = G.sum(axis=1)
                col_sum += G.sum(axis=0)
            if la is not None:
                dcum = row_sum - col_sum
                g["log_a"][b, :, h] = np.cumsum(dcum[::-1])[::-1]
    return g


def backward_sampled(q, k, v, log_a, lam, dout, rows, cols, heads):
    """The gradients of backward_direct for chosen positions only, fp64: dq and dlam of the
    query rows `rows`, dk and dv of the source positions `cols`, for the (b, h) pairs in
    `heads`.  Same definition, evaluated one row (for dq, dlam) or one column (for dk, dv)
    at a time, so that long sequences stay cheap:
        dq_t = sum_{s<=t} M[t, s] (dO_t . v_s) k_s,
        dlam[t, l] = sum over the level-l bucket of t of M^S[t, s] (dO_t . v_s)(q_t . k_s),
        dk_s = sum_{t>=s} M[t, s] (dO_t . v_s) q_t,   dv_s = sum_{t>=s} M[t, s] (q_t . k_s) dO_t.
    Returns dict(q [n_heads, len(rows), dk], lam [.., len(rows), L], k [.., len(cols), dk],
    v [.., len(cols), dv]) in the order of `heads`."""
    q, k, v, lam, do = _f64(q), _f64(k), _f64(v), _f64(lam), _f64(dout)
    log_a = _f64(log_a)
    T = q.shape[1]
    rows = np.asarray(rows, dtype=np.int64)
    cols = np.asarray(cols, dtype=np.int64)
    out = {"q": [], "lam": [], "k": [], "v": []}
    for b, h in heads:
        Q, K, V, dO, lm = q[b, :, h], k[b, :, h], v[b, :, h], do[b, :, h], lam[b, :, h]
        cum = np.zeros(T) if log_a is None else np.cumsum(log_a[b, :, h])
        gq = np.zeros((len(rows), Q.shape[1]))
        gl = np.zeros((len(rows), lm.shape[1]))
        for i, t in enumerate(rows):
            lv = level_row(int(t))
            ms = np.exp(cum[t] - cum[: t + 1])
            dov = V[: t + 1] @ dO[t]
            qk = K[: t + 1] @ Q[t]
            gq[i] = (ms * lm[t, lv] * dov) @ K[: t + 1]
            np.add.at(gl[i], lv, ms * dov * qk)
        gk = np.zeros((len(cols), K.shape[1]))
        gv = np.zeros((len(cols), V.shape[1]))
        for i, s0 in enumerate(cols):
            ts = np.arange(s0, T)
            # level(t, s0) for every t >= s0 by its closed form bit_length(t XOR s0), which the
            # pins check against the Fenwick walk; exact integer shifts
            x = ts ^ s0
            lv = np.zeros(len(ts), dtype=np.int64)
            while x.any():
                lv += x > 0
                x = x >> 1
            m = np.exp(cum[ts] - cum[s0]) * lm[ts, lv]
            dov = dO[ts] @ V[s0]
            qk = Q[ts] @ K[s0]
            gk[i] = (m * dov) @ Q[ts]
            gv[i] = (m * qk) @ dO[ts]
        out["q"].append(gq)
        out["lam"].append(gl)
        out["k"].append(gk)
        out["v"].append(gv)
    return {n: np.stack(a) for n, a in out.items()}


# --------------------------------------------------------------------------------------
# L2a: per-level states and the lssb decode recurrence
# --------------------------------------------------------------------------------------


def states_from_buckets(k_bh, v_bh, log_a_bh, t: int, L: int) -> np.ndarray:
    """Per-level states at position t from their definition.

    Reading post, section 循环形式与输出计算 (one state per bucket) and the Dynamic Linear
    Attention page's restatement: S_t^(l) = sum_{s in B_t^(l)} M^S[t, s] k_s v_s^T.
    k_bh [T, dk], v_bh [T, dv], log_a_bh [T] or None.  Returns [L, dk, dv].
    """
    k_bh, v_bh, log_a_bh = _f64(k_bh), _f64(v_bh), _f64(log_a_bh)
    dk, dv = k_bh.shape[1], v_bh.shape[1]
    S = np.zeros((L, dk, dv))
    cum = None if log_a_bh is None else np.cumsum(log_a_bh[: t + 1])
    for lvl, lo, hi in fenwick_partition(t):
        if lvl >= L:
            raise ValueError(f"level {lvl} needs L > {lvl}")
        w = np.ones(hi - lo) if cum is None else np.exp(cum[t] - cum[lo:hi])
        S[lvl] = (k_bh[lo:hi] * w[:, None]).T @ v_bh[lo:hi]
    return S


def decode_step(state, q, k, v, log_a, lam, t: int):
    """One decode step with the lssb rule, batched over leading dims.

    Reading post, section 解码：基于 lssb 的状态更新, and the slide deck, slide 21:
    level 0 receives the new outer product; the levels below and at lssb(t) are merged
    and promoted one level up; the levels in between are cleared; the higher levels are
    kept.  Under the decay mask every state older than t is multiplied by a_t.  The
    output is the lambda-weighted readout of the updated states (循环形式与输出计算).

    state [..., L, dk, dv]; q, k [..., dk]; v [..., dv]; log_a [...] or None;
    lam [..., L].  Returns (new_state, o [..., dv]).  Inputs are not modified.
    """
    S = _f64(state).copy()
    q, k, v, lam = _f64(q), _f64(k), _f64(v), _f64(lam)
    a = np.ones(S.shape[:-3]) if log_a is None else np.exp(_f64(log_a))
    a4 = a[..., None, None, None]
    L = S.shape[-3]
    if t == 0:
        S[...] = 0.0
    else:
        l = lssb(t)
        if l + 1 >= L:
            raise ValueError(f"t={t} needs L > {l + 1}")
        merged = S[..., : l + 1, :, :].sum(axis=-3)
        S[..., l + 2 :, :, :] *= a4
        S[..., l + 1, :, :] = a[..., None, None] * merged
        S[..., 1 : l + 1, :, :] = 0.0
    S[..., 0, :, :] = k[..., :, None] * v[..., None, :]
    # o[e] = sum_l lam_l sum_d q[d] S_l[d, e]
    o = np.einsum("...l,...d,...lde->...e", lam, q, S)
    return S, o


def recurrence(q, k, v, log_a, lam, T_stop=None):
    """Run the lssb recurrence over t = 0..T-1 for every (b, h).

    Returns (out [B, T, H, dv], final state [B, H, L, dk, dv]).
    """
    q, k, v, lam = _f64(q), _f64(k), _f64(v), _f64(lam)
    log_a = _f64(log_a)
    B, T, H, dk = q.shape
    dv, L = v.shape[-1], lam.shape[-1]
    T_stop = T if T_stop is None else T_stop
    S = np.zeros((B, H, L, dk, dv))
    out = np.zeros((B, T, H, dv))
    for t in range(T_stop):
        la = None if log_a is None else log_a[:, t, :]
        S, o = decode_step(S, q[:, t], k[:, t], v[:, t], la, lam[:, t], t)
        out[:, t] = o
    return out, S


# --------------------------------------------------------------------------------------
# L2b: the pages' chunked two-stage algorithm, restated plainly (no shared states)
# --------------------------------------------------------------------------------------


def forward_chunked(q, k, v, log_a, lam, C: int):
    """Two-stage chunked evaluation, fp64.

    Reading post, sections 矩阵分解 and 两阶段计算; news article, section 高效训练算法;
    slide deck, slides 33-34.  M^H splits into a block-diagonal part D (C x C causal
    blocks holding the levels <= log2 C) plus one inter-chunk part per higher level.
    Intra stage: dense masked attention inside each chunk.  Inter stage: at chunk level
    m (token level log2 C + m), chunks are grouped in aligned blocks of 2^(m-1); the
    decayed state of every even block is passed to the tokens of its odd sibling block
    and read out with that level's lambda.  The last chunk may be partial.
    """
    q, k, v, lam = _f64(q), _f64(k), _f64(v), _f64(lam)
    log_a = _f64(log_a)
    if C < 1 or C & (C - 1):
        raise ValueError("C must be a power of two")
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    lc = C.bit_length() - 1
    N = -(-T // C)
    out = np.zeros((B, T, H, dv))
    for b in range(B):
        for h in range(H):
            Q, K, V, lm = q[b, :, h], k[b, :, h], v[b, :, h], lam[b, :, h]
            cum = np.zeros(T) if log_a is None else np.cumsum(log_a[b, :, h])
            # intra stage: the diagonal blocks D
            for j in range(N):
                lo, hi = j * C, min(T, (j + 1) * C)
                for t in range(lo, hi):
                    for s in range(lo, t + 1):
                        w = np.exp(cum[t] - cum[s]) * lm[t, level(t, s)]
                        out[b, t, h] += w * (Q[t] @ K[s]) * V[s]
            # inter stage: one pass per chunk level m >= 1
            m = 1
            while (1 << (m - 1)) < N:
                span = 1 << (m - 1)
                for e0 in range(0, N, 2 * span):
                    o0 = e0 + span                      # first chunk of the odd block
                    if o0 >= N:
                        continue
                    elo, ehi = e0 * C, o0 * C           # tokens of the even block
                    olo, ohi = o0 * C, min(T, (o0 + span) * C)
                    wS = np.exp(cum[ehi - 1] - cum[elo:ehi])
                    state = (K[elo:ehi] * wS[:, None]).T @ V[elo:ehi]
                    for t in range(olo, ohi):
                        g = np.exp(cum[t] - cum[ehi - 1])
                        out[b, t, h] += lm[t, lc + m] * g * (Q[t] @ state)
                m += 1
    return out


# --------------------------------------------------------------------------------------
# Closed forms used to pin the above (textbook special cases)
# --------------------------------------------------------------------------------------


def linear_attention_recurrent(q, k, v, log_a, c=None):
    """Gated linear attention by its recurrence: S_t = a_t S_{t-1} + k_t v_t^T,
    o_t = c_t S_t^T q_t (the Dynamic Linear Attention page's linear-attention
    background; slide deck slides 4-9).  This is what log-linear attention reduces to
    when lambda is the same at every level (reading post, 循环形式与输出计算, the
    degeneration condition).  c [B, T, H] or None (= 1)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    log_a = _f64(log_a)
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    S = np.zeros((B, H, dk, dv))
    out = np.zeros((B, T, H, dv))
    for t in range(T):
        if log_a is not None:
            S *= np.exp(log_a[:, t, :])[..., None, None]
        S += k[:, t, :, :, None] * v[:, t, :, None, :]
        o = np.einsum("bhd,bhde->bhe", q[:, t], S)
        if c is not None:
            o = o * _f64(c)[:, t, :, None]
        out[:, t] = o
    return out
