"""Pins of the CPU oracle to facts outside itself (no GPU).

Each pin comes from the pages (the printed 8x8 level table, the t = 7 / t = 8 bucket
decompositions, the popcount rule), from mathematics (a closed form of the level, the
textbook linear-attention recurrence the method degenerates to, brute force on tiny
inputs) or from the agreement of independently written evaluation orders (direct
masked product, lssb recurrence, chunked two-stage form).  The planted-mistake tests at
the end show that plausible slips in the oracle fail at least one pin.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import loglinear_oracle as ref
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel_l2(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _read_table():
    rows = []
    with open(os.path.join(GOLDEN, "mh_levels_8x8.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append([(-1 if x == "." else int(x)) for x in line.split(":")[1].split()])
    return np.array(rows)


def _read_buckets():
    out = {}
    with open(os.path.join(GOLDEN, "fenwick_buckets.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            head, srcs = line.split(":")
            t, lvl = map(int, head.split())
            out.setdefault(t, {})[lvl] = sorted(int(x) for x in srcs.split())
    return out


# ---------------------------------------------------------------- level / partition


def test_level_matches_printed_8x8_table():
    table = _read_table()
    assert table.shape == (8, 8)
    for t in range(8):
        for s in range(8):
            want = table[t, s]
            if want < 0:
                with pytest.raises(ValueError):
                    oracle.level(t, s)
            else:
                assert oracle.level(t, s) == want, (t, s)
    assert np.array_equal(oracle.level_matrix(8), table)


def test_buckets_t7_t8_match_pages():
    gold = _read_buckets()
    for t, want in gold.items():
        got = {lvl: list(range(lo, hi)) for lvl, lo, hi in oracle.fenwick_partition(t)}
        assert got == want, t


def test_partition_invariants_and_popcount_rule():
    # covers [0, t] disjointly; level-l bucket (l>=1) has size 2^(l-1); the number of
    # non-empty buckets besides the sentinel is popcount(t); at most ceil(log2(t+1))+1
    # buckets in all (the Dynamic Linear Attention page's restatement of the count).
    for t in range(1 << 12):
        parts = oracle.fenwick_partition(t)
        cover = np.zeros(t + 1, np.int64)
        lvls = []
        for lvl, lo, hi in parts:
            cover[lo:hi] += 1
            lvls.append(lvl)
            assert hi - lo == (1 if lvl == 0 else 1 << (lvl - 1))
        assert np.all(cover == 1)
        assert len(lvls) == len(set(lvls))
        assert len(parts) - 1 == bin(t).count("1")
        assert len(parts) <= int(np.ceil(np.log2(t + 1))) + 1


def test_level_closed_form_bruteforce():
    # derived: s lies in the bucket cut by the highest bit where s and t differ
    for t in range(1 << 10):
        row = oracle.level_row(t)
        for s in range(t + 1):
            assert row[s] == (t ^ s).bit_length()
    for t in [1023, 1024, 4095, 12345, 16383]:
        row = oracle.level_row(t)
        s = np.arange(t + 1)
        assert np.array_equal(row, np.array([(t ^ int(x)).bit_length() for x in s]))


def test_lssb_and_level_occupancy_examples():
    assert [oracle.lssb(t) for t in (1, 2, 3, 4, 8, 12, 12344, 12345, 8192)] == \
        [0, 1, 0, 2, 3, 2, 3, 0, 13]
    # occupancy before/after the decode step at t = 12345
    assert W.nonempty_levels_before(12345, 15) == [0, 4, 5, 6, 13, 14]
    after = sorted({lvl for lvl, _, _ in oracle.fenwick_partition(12345)})
    assert after == [0, 1, 4, 5, 6, 13, 14]
    # powers of two collapse the whole history into one bucket (linear attention)
    assert sorted(l for l, _, _ in oracle.fenwick_partition(8192)) == [0, 14]


# ---------------------------------------------------------------- tiny hand example


def test_tiny_hand_computed_example():
    # T = 3, d = 1, no decay.  Levels: l(1,0)=1, l(2,0)=l(2,1)=2, diagonal 0.
    q = np.array([1.0, 2.0, 3.0]).reshape(1, 3, 1, 1)
    k = np.array([1.0, -1.0, 0.5]).reshape(1, 3, 1, 1)
    v = np.array([1.0, 10.0, 100.0]).reshape(1, 3, 1, 1)
    lam = np.array([[0.5, 0.25, 0.125],      # lambda_0[l]
                    [2.0, 3.0, 5.0],         # lambda_1[l]
                    [7.0, 11.0, 13.0]]).reshape(1, 3, 1, 3)
    want = np.array([
        0.5 * (1 * 1) * 1,                                   # o_0 = l0 q0 k0 v0
        3.0 * (2 * 1) * 1 + 2.0 * (2 * -1) * 10,             # o_1 = l1 q1k0v0 + l0 q1k1v1
        13.0 * ((3 * 1) * 1 + (3 * -1) * 10) + 7.0 * (3 * 0.5) * 100,
    ])
    got = oracle.forward_direct(q, k, v, None, lam)[0, :, 0, 0]
    assert np.allclose(got, want, rtol=0, atol=1e-12)
    rec, _ = oracle.recurrence(q, k, v, None, lam)
    assert np.allclose(rec[0, :, 0, 0], want, rtol=0, atol=1e-12)
    # with decay a = [., 0.5, 0.25]: M^S[1,0] = 0.5, M^S[2,0] = 0.125, M^S[2,1] = 0.25
    la = np.log(np.array([0.9, 0.5, 0.25])).reshape(1, 3, 1)
    want_d = np.array([
        0.5 * 1 * 1,
        3.0 * 0.5 * 2 * 1 + 2.0 * (2 * -1) * 10,
        13.0 * (0.125 * 3 * 1 + 0.25 * (3 * -1) * 10) + 7.0 * (3 * 0.5) * 100,
    ])
    got_d = oracle.forward_direct(q, k, v, la, lam)[0, :, 0, 0]
    assert np.allclose(got_d, want_d, rtol=0, atol=1e-12)


def _brute(q, k, v, log_a, lam):
    """Scalar triple loop over (t, s, feature) with the walk-based level."""
    B, T, H, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, T, H, dv))
    for b in range(B):
        for h in range(H):
            for t in range(T):
                for s in range(t + 1):
                    dec = 1.0
                    if log_a is not None:
                        for r in range(s + 1, t + 1):
                            dec *= np.exp(log_a[b, r, h])
                    w = dec * lam[b, t, h, oracle.level(t, s)] * float(q[b, t, h] @ k[b, s, h])
                    out[b, t, h] += w * v[b, s, h]
    return out


def test_direct_matches_scalar_bruteforce():
    rng = np.random.default_rng(3)
    B, T, H, d, L = 1, 13, 2, 3, 5
    q, k, v = (rng.standard_normal((B, T, H, d)) for _ in range(3))
    la = -0.3 * rng.random((B, T, H))
    lam = rng.random((B, T, H, L))
    for log_a in (None, la):
        assert rel_l2(oracle.forward_direct(q, k, v, log_a, lam), _brute(q, k, v, log_a, lam)) < 1e-13


# ---------------------------------------------------------------- three evaluation orders


@pytest.mark.parametrize("T,C,decay", [(64, 16, False), (96, 16, True), (128, 8, True),
                                       (100, 16, True), (37, 4, True), (33, 32, False)])
def test_direct_recurrence_chunked_agree(T, C, decay):
    cfg = W.FwdConfig("t", 1, 2, T, 8, 6, C, (T - 1).bit_length() + 1, "f32", decay, "softplus", seed=T)
    x = W.make_fwd_inputs(cfg)
    d = oracle.forward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"])
    r, S = oracle.recurrence(x["q"], x["k"], x["v"], x["log_a"], x["lam"])
    c = oracle.forward_chunked(x["q"], x["k"], x["v"], x["log_a"], x["lam"], C)
    assert rel_l2(r, d) < 1e-12
    assert rel_l2(c, d) < 1e-12
    # the recurrence's final state is the bucket definition at T-1
    for h in range(cfg.H):
        Sd = oracle.states_from_buckets(x["k"][0, :, h], x["v"][0, :, h],
                                        None if x["log_a"] is None else x["log_a"][0, :, h],
                                        T - 1, cfg.L)
        assert rel_l2(S[0, h], Sd) < 1e-12


def test_degenerates_to_linear_attention():
    # lambda equal across levels (but varying with t) -> c_t * ((Q K^T ⊙ M^S) V)
    cfg = W.FwdConfig("t", 2, 2, 75, 8, 8, 16, 8, "f32", True, "softplus", seed=5)
    x = W.make_fwd_inputs(cfg)
    c = torch.rand(cfg.B, cfg.T, cfg.H) + 0.5
    lam = c[..., None].expand(-1, -1, -1, cfg.L).contiguous()
    d = oracle.forward_direct(x["q"], x["k"], x["v"], x["log_a"], lam)
    lin = oracle.linear_attention_recurrent(x["q"], x["k"], x["v"], x["log_a"], c)
    assert rel_l2(d, lin) < 1e-12
    # no decay, lambda = 1: plain cumulative linear attention
    ones = torch.ones(cfg.B, cfg.T, cfg.H, cfg.L)
    d1 = oracle.forward_direct(x["q"], x["k"], x["v"], None, ones)
    kv = np.cumsum(np.einsum("bthd,bthe->bthde", x["k"].double().numpy(), x["v"].double().numpy()), axis=1)
    cum = np.einsum("bthd,bthde->bthe", x["q"].double().numpy(), kv)
    assert rel_l2(d1, cum) < 1e-12


def test_onehot_lambda_selects_one_bucket():
    # lambda_t = e_l keeps exactly the sources in bucket l of t
    T, L = 40, 7
    x = W.make_int_inputs(1, T, 1, 4, 3, L, onehot_level=0)
    q, k, v = (x[n][0, :, 0].double().numpy() for n in ("q", "k", "v"))
    for lvl in range(L):
        lam = torch.zeros(1, T, 1, L)
        lam[..., lvl] = 1
        got = oracle.forward_direct(x["q"], x["k"], x["v"], None, lam)[0, :, 0]
        want = np.zeros((T, 3))
        for t in range(T):
            for l2, lo, hi in oracle.fenwick_partition(t):
                if l2 == lvl:
                    want[t] = (q[t] @ k[lo:hi].T) @ v[lo:hi]
        assert np.array_equal(got, want), lvl


def test_decode_step_matches_direct_row():
    # decode from the bucket-definition state at t-1 gives forward row t
    cfg = W.FwdConfig("t", 1, 1, 70, 5, 4, 8, 8, "f32", True, "softplus", seed=11)
    x = W.make_fwd_inputs(cfg)
    d = oracle.forward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"])
    k, v, la = x["k"][0, :, 0], x["v"][0, :, 0], x["log_a"][0, :, 0]
    for t in [1, 2, 8, 12, 31, 64, 69]:
        S_prev = oracle.states_from_buckets(k, v, la, t - 1, cfg.L)
        S_new, o = oracle.decode_step(S_prev, x["q"][0, t, 0], k[t], v[t], la[t], x["lam"][0, t, 0], t)
        assert rel_l2(o, d[0, t, 0]) < 1e-12
        assert rel_l2(S_new, oracle.states_from_buckets(k, v, la, t, cfg.L)) < 1e-12


# ---------------------------------------------------------------- planted mistakes


def _pin_suite(fd):
    """Run the numeric pins against a candidate forward; True if all pass (an exception
    raised by the candidate counts as a failed pin)."""
    try:
        return _pin_suite_inner(fd)
    except (IndexError, ValueError):
        return False


def _pin_suite_inner(fd):
    ok = True
    cfg = W.FwdConfig("t", 1, 2, 37, 4, 3, 8, 7, "f32", True, "softplus", seed=2)
    x = W.make_fwd_inputs(cfg)
    d = fd(x["q"], x["k"], x["v"], x["log_a"], x["lam"])
    r, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["log_a"], x["lam"])
    ok &= rel_l2(d, r) < 1e-12
    c = torch.rand(1, cfg.T, cfg.H) + 0.5
    lam = c[..., None].expand(-1, -1, -1, cfg.L).contiguous()
    lin = oracle.linear_attention_recurrent(x["q"], x["k"], x["v"], x["log_a"], c)
    ok &= rel_l2(fd(x["q"], x["k"], x["v"], x["log_a"], lam), lin) < 1e-12
    table = _read_table()
    ok &= bool(np.array_equal(oracle.level_matrix(8), table))
    return bool(ok)


def test_pins_pass_on_the_oracle():
    assert _pin_suite(oracle.forward_direct)


@pytest.mark.parametrize("mutation", ["level_off_by_one", "decay_sign", "lambda_by_source",
                                      "transposed_qk", "dropped_diagonal"])
def test_planted_mistakes_fail_a_pin(monkeypatch, mutation):
    if mutation == "level_off_by_one":
        orig = ref.level_row
        monkeypatch.setattr(ref, "level_row", lambda t: np.minimum(orig(t) + (np.arange(t + 1) < t), 99))
        # level_matrix is built from level_row, so the table pin must fail as well
        fd = ref.forward_direct
    elif mutation == "decay_sign":
        orig_d = ref.decay_rows

        def bad(la, rows, T):
            return orig_d(None if la is None else -la, rows, T) * (np.arange(T)[None] <= rows[:, None])
        monkeypatch.setattr(ref, "decay_rows", bad)
        fd = ref.forward_direct
    elif mutation == "lambda_by_source":
        def bad_h(lam_bh, rows, T):
            out = np.zeros((len(rows), T))
            for i, t in enumerate(rows):
                lv = ref.level_row(int(t))
                out[i, : t + 1] = lam_bh[np.arange(t + 1), lv]
            return out
        monkeypatch.setattr(ref, "hier_rows", bad_h)
        fd = ref.forward_direct
    elif mutation == "transposed_qk":
        def fd(q, k, v, la, lam):
            return ref.forward_direct(k, q, v, la, lam)
    else:
        def fd(q, k, v, la, lam):
            lam2 = torch.as_tensor(np.asarray(lam, dtype=np.float64)).clone()
            lam2[..., 0] = 0.0
            return ref.forward_direct(q, k, v, la, lam2)
    assert not _pin_suite(fd)
