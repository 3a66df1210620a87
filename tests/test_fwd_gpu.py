"""Parity of the CUDA forward with the CPU oracle, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import TOL_BF16, TOL_F32, cuda, max_abs, one_head, per_head_qk, rel_l2, tol_for

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def LL():
    import log_linear_attention_fwd_gb300 as m
    return m


def run(LL, x, chunk, path="auto", out_dtype=None):
    d = cuda(x)
    out = LL.loglinear_fwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], chunk, path=path,
                           out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.cpu()


def oracle_fwd(x, rows=None, heads=None):
    return oracle.forward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"], rows=rows, heads=heads)


# ------------------------------------------------------------------ the workloads


@pytest.mark.parametrize("name", ["linear_T64", "mamba2_T1024"])
def test_fp32_workloads_full(LL, name):
    cfg = W.FWD_CONFIGS[name]
    x = W.make_fwd_inputs(cfg)
    got = run(LL, x, cfg.C)
    want = oracle_fwd(x)
    err = rel_l2(got, want)
    print(f"{name}: rel_l2={err:.3e} max_abs={max_abs(got, want):.3e}")
    assert err <= TOL_F32


def _sample_rows(T, n, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 63, 64, 127, 128, 129, T // 2, T // 2 - 1, T - 129, T - 128, T - 2, T - 1]
    pw = [(1 << p) for p in range(1, T.bit_length()) if (1 << p) < T]
    rows = set(fixed + pw + [p - 1 for p in pw] + list(rng.integers(0, T, n)))
    return np.array(sorted(r for r in rows if 0 <= r < T))


@pytest.mark.parametrize("name", ["mamba2_T4096", "mamba2_T16384"])
def test_bf16_workloads_sampled(LL, name):
    cfg = W.FWD_CONFIGS[name]
    x = W.make_fwd_inputs(cfg)
    got = run(LL, x, cfg.C)
    assert torch.isfinite(got.float()).all()
    # one whole head, plus sampled rows of every head
    full = [(cfg.B - 1, cfg.H - 1)]
    want = oracle_fwd(x, heads=full)
    b, h = full[0]
    err_full = rel_l2(got[b, :, h], want[b, :, h])
    rows = _sample_rows(cfg.T, 96, 1)
    heads = [(b, h) for b in range(cfg.B) for h in range(cfg.H)]
    want_s = oracle_fwd(x, rows=rows, heads=heads)
    err_s = rel_l2(got[:, rows], want_s[:, rows])
    print(f"{name}: rel_l2(full head)={err_full:.3e} rel_l2(sampled rows)={err_s:.3e} "
          f"max_abs={max_abs(got[:, rows], want_s[:, rows]):.3e}")
    assert err_full <= TOL_BF16 and err_s <= TOL_BF16


# ------------------------------------------------------------------ edge cases


@pytest.mark.parametrize("T,C,decay", [(1, 16, True), (2, 16, False), (15, 16, True), (17, 16, True),
                                       (53, 16, True), (200, 8, True), (333, 64, True),
                                       (64, 1, True), (40, 2, False), (1000, 32, True),
                                       (4096, 16, True), (130, 64, False), (700, 256, True)])
def test_ragged_and_chunk_sizes_simt(LL, T, C, decay):
    L = max((T - 1).bit_length() + 1, 1)
    cfg = W.FwdConfig("e", 2, 3, T, 16, 8, C, L, "f32", decay, "softplus", seed=T * 7 + C)
    x = W.make_fwd_inputs(cfg)
    got = run(LL, x, C, path="simt")
    want = oracle_fwd(x)
    assert rel_l2(got, want) <= TOL_F32, (T, C)


@pytest.mark.parametrize("dk,dv", [(1, 4), (7, 3), (32, 16), (128, 128), (96, 64)])
def test_head_dims_simt(LL, dk, dv):
    cfg = W.FwdConfig("e", 1, 2, 150, dk, dv, 32, 9, "f32", True, "softplus", seed=dk + dv)
    x = W.make_fwd_inputs(cfg)
    got = run(LL, x, 32, path="simt")
    assert rel_l2(got, oracle_fwd(x)) <= TOL_F32


def test_extra_levels_strong_and_zero_decay(LL):
    cfg = W.FwdConfig("e", 1, 2, 300, 16, 16, 16, 20, "f32", True, "softplus", seed=9)
    x = W.make_fwd_inputs(cfg)
    for la in (torch.full_like(x["log_a"], -6.0), torch.zeros_like(x["log_a"]),
               x["log_a"] * 30):
        y = dict(x, log_a=la.contiguous())
        got = run(LL, y, 16, path="simt")
        assert torch.isfinite(got).all()
        assert rel_l2(got, oracle_fwd(y)) <= TOL_F32


def test_dtype_combinations_simt(LL):
    cfg = W.FwdConfig("e", 1, 2, 257, 32, 32, 32, 10, "bf16", True, "softplus", seed=4)
    x = W.make_fwd_inputs(cfg)
    want = oracle_fwd(x)
    got32 = run(LL, x, 32, path="simt", out_dtype=torch.float32)
    assert got32.dtype == torch.float32 and rel_l2(got32, want) <= TOL_F32
    got16 = run(LL, x, 32, path="simt")
    assert got16.dtype == torch.bfloat16 and rel_l2(got16, want) <= TOL_BF16
    xf = dict(x, q=x["q"].float(), k=x["k"].float(), v=x["v"].float())
    gotf = run(LL, xf, 32, path="simt", out_dtype=torch.bfloat16)
    assert rel_l2(gotf, want) <= TOL_BF16


def test_empty_problems(LL):
    q = torch.zeros(1, 0, 2, 16, device="cuda")
    lam = torch.zeros(1, 0, 2, 1, device="cuda")
    out = LL.loglinear_fwd(q, q, torch.zeros(1, 0, 2, 8, device="cuda"), None, lam, 16)
    assert out.shape == (1, 0, 2, 8)


# ------------------------------------------------------------------ exact indexing


@pytest.mark.parametrize("T,C,path", [(64, 16, "simt"), (1000, 64, "simt"), (300, 4, "simt"),
                                      (2048, 1, "simt")])
def test_level_map_bit_exact(LL, T, C, path):
    got = LL.debug_level_map(T, C, path=path).cpu().numpy().astype(np.int64)
    want = oracle.level_matrix(T)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("path,C,T,dtype", [("simt", 16, 200, "f32"), ("simt", 8, 517, "f32"),
                                            ("simt", 64, 1024, "bf16")])
def test_onehot_lambda_bit_exact(LL, path, C, T, dtype):
    """Small-integer q, k, v, no decay, lambda = e_l: every level's contribution is an
    exact integer sum in fp32, so the CUDA result must equal the oracle exactly."""
    L = (T - 1).bit_length() + 1
    for lvl in range(L):
        x = W.make_int_inputs(1, T, 2, 8, 8, L, lvl, seed=lvl, dtype=dtype)
        got = run(LL, x, C, path=path, out_dtype=torch.float32)
        want = oracle_fwd(x)
        assert np.array_equal(got.double().numpy(), want), (path, lvl)


# ------------------------------------------------------------------ tensor-core path


@pytest.mark.parametrize("T,C,decay,dv", [(128, 64, True, 128), (300, 64, True, 128),
                                          (1000, 128, True, 128), (2125, 64, True, 128),
                                          (4096, 64, False, 128), (77, 64, True, 128),
                                          (77, 64, True, 64), (1000, 64, True, 64),
                                          (2125, 64, True, 64), (4096, 64, False, 64)])
def test_tc_path_matches_oracle(LL, T, C, decay, dv):
    L = (T - 1).bit_length() + 1
    cfg = W.FwdConfig("tc", 2, 3, T, 128, dv, C, L, "bf16", decay, "softplus", seed=T + C + dv)
    x = W.make_fwd_inputs(cfg)
    assert LL.resolve_path(128, dv, C, 1) == "tc"
    want = oracle_fwd(x)
    got = run(LL, x, C, path="tc")
    got32 = run(LL, x, C, path="tc", out_dtype=torch.float32)
    assert LL.device_error() == 0
    e16, e32 = rel_l2(got, want), rel_l2(got32, want)
    print(f"tc T={T} C={C} dv={dv}: rel_l2 bf16-out={e16:.3e} f32-out={e32:.3e} "
          f"max_abs={max_abs(got32, want):.3e}")
    assert e16 <= TOL_BF16 and e32 <= TOL_BF16


def test_tc_level_map_bit_exact(LL):
    for T in (128, 1000, 4096):
        got = LL.debug_level_map(T, 64, path="tc").cpu().numpy().astype(np.int64)
        assert np.array_equal(got, oracle.level_matrix(T)), T


@pytest.mark.parametrize("T,dv", [(256, 128), (1151, 128), (1151, 64)])
def test_tc_onehot_lambda_bit_exact(LL, T, dv):
    """Integer inputs that stay exact through bf16 states: the tensor-core result must
    equal the oracle bit for bit at every level, intra-tile and inter-tile."""
    L = (T - 1).bit_length() + 1
    for lvl in range(L):
        x = W.make_sparse_int_inputs(1, T, 2, 128, L, lvl, seed=lvl, dv=dv)
        got = run(LL, x, 64, path="tc", out_dtype=torch.float32)
        want = oracle_fwd(x)
        assert np.array_equal(got.double().numpy(), want), lvl
    assert LL.device_error() == 0


def _top_level_rows(T, seed):
    """Query rows in the tiles that read the highest block states of a long sequence:
    every 128-token tile from tile 64 on (its first and last row and one random row),
    the tiles 64, 127, 128 and the last one in full, and a few rows of the early tiles."""
    rng = np.random.default_rng(seed)
    n = -(-T // 128)
    rows = set(range(0, 300, 37))
    for j in range(64, n):
        lo, hi = j * 128, min(T, (j + 1) * 128)
        rows.update({lo, hi - 1, int(rng.integers(lo, hi))})
    for j in (64, 127, 128, n - 1):
        if j < n:
            rows.update(range(j * 128, min(T, (j + 1) * 128), 3))
    return np.array(sorted(r for r in rows if r < T))


@pytest.mark.parametrize("T,dv", [(16384, 128), (20000, 128), (20000, 64)])
def test_tc_onehot_lambda_top_levels(LL, T, dv):
    """Levels up to the top of a 16K (L = 15) and a ragged 20000-token (L = 16) sequence on
    the tensor-core path: with one-hot lambda, no decay and integer inputs that stay exact
    through bf16 states, every level l = 0..L-1 (the block states of tiles >= 64 included:
    chunk levels 7 and 8 of the tile pairing) must equal the oracle bit for bit on rows
    sampled across those tiles."""
    L = (T - 1).bit_length() + 1
    rows = _top_level_rows(T, T + dv)
    for lvl in range(L):
        x = W.make_sparse_int_inputs(1, T, 2, 128, L, lvl, seed=1000 + lvl, dv=dv)
        got = run(LL, x, 64, path="tc", out_dtype=torch.float32)
        want = oracle_fwd(x, rows=rows)
        g = got[:, rows].double().numpy()
        assert np.array_equal(g, want[:, rows]), (lvl, float(np.abs(g - want[:, rows]).max()))
        if lvl >= 13:  # the top levels carry weight in these rows (not a vacuous zero)
            assert np.abs(want[:, rows]).sum() > 0, lvl
    assert LL.device_error() == 0


def test_tc_no_decay_headline_shape(LL):
    """The headline shape (B1 H16 T16384 d128 bf16) without decay, so that every level up to
    l = 14 carries weight: one whole head and sampled rows of every head against the oracle."""
    cfg = W.FWD_CONFIGS["mamba2_T16384"].with_(name="linear_T16384", decay=False, seed=21)
    x = W.make_fwd_inputs(cfg)
    got = run(LL, x, cfg.C, path="tc", out_dtype=torch.float32)
    assert LL.device_error() == 0
    h = 5
    want = oracle_fwd(x, heads=[(0, h)])
    err_full = rel_l2(got[0, :, h], want[0, :, h])
    rows = _sample_rows(cfg.T, 64, 3)
    want_s = oracle_fwd(x, rows=rows, heads=[(0, hh) for hh in range(cfg.H)])
    err_s = rel_l2(got[:, rows], want_s[:, rows])
    print(f"no-decay T16384: rel_l2(full head)={err_full:.3e} rel_l2(sampled rows)={err_s:.3e} "
          f"max_abs={max_abs(got[:, rows], want_s[:, rows]):.3e}")
    assert err_full <= TOL_BF16 and err_s <= TOL_BF16


def test_tc_level_map_headline_length(LL):
    """The tensor-core path's level indexing at T = 16384 (L = 15), row by row against the
    oracle's Fenwick walk."""
    T = 16384
    got = LL.debug_level_map(T, 64, path="tc").cpu().numpy()
    for t in range(T):
        want = oracle.level_row(t)
        assert np.array_equal(got[t, : t + 1].astype(np.int64), want), t
        assert (got[t, t + 1:] == -1).all(), t


@pytest.mark.parametrize("T,dv", [(40000, 128), (40000, 64)])
def test_tc_many_tiles_sampled(LL, T, dv):
    """A deep block tree (313 tiles, not a power of two): the block states of every level
    are merged across many CTAs; sampled rows of every head against the oracle."""
    L = (T - 1).bit_length() + 1
    cfg = W.FwdConfig("tc_deep", 1, 2, T, 128, dv, 64, L, "bf16", True, "softplus", seed=11)
    x = W.make_fwd_inputs(cfg)
    got = run(LL, x, 64, path="tc", out_dtype=torch.float32)
    assert LL.device_error() == 0
    rows = _sample_rows(T, 48, 2)
    want = oracle_fwd(x, rows=rows, heads=[(0, 0), (0, 1)])
    err = rel_l2(got[:, rows], want[:, rows])
    print(f"tc T={T}: rel_l2(sampled rows)={err:.3e}")
    assert err <= TOL_BF16


def test_tc_repeated_calls_same_workspace(LL):
    """The pair counters of the block tree are reset by every call: two calls on one
    workspace give identical results."""
    cfg = W.FwdConfig("tc_rep", 1, 2, 3000, 128, 128, 64, 13, "bf16", True, "softplus", seed=5)
    x = cuda(W.make_fwd_inputs(cfg))
    ws = torch.empty(LL.fwd_workspace_size(1, cfg.T, cfg.H, 128, 128, 64, 1), device="cuda",
                     dtype=torch.uint8)
    outs = []
    for _ in range(3):
        o = LL.loglinear_fwd(x["q"], x["k"], x["v"], x["log_a"], x["lam"], 64, path="tc",
                             workspace=ws)
        torch.cuda.synchronize()
        outs.append(o.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    assert LL.device_error() == 0


# ------------------------------------------------------------------ shared q/k heads


def test_benchmark_shape_full_size_sampled(LL):
    """The pages' benchmark shape as the bench times it (B2, 48 heads sharing one q/k,
    d_k 128, d_v 64, T 16384, bf16) on the tensor-core path: sampled rows of six heads
    against the oracle's per-head definition."""
    cfg = W.FWD_CONFIGS["mva_B2H48_T16384"]
    x = W.make_fwd_inputs(cfg)
    got = run(LL, x, cfg.C, path="tc")
    assert LL.device_error() == 0
    rows = _sample_rows(cfg.T, 48, 5)
    for b, h in [(0, 0), (0, 17), (0, 47), (1, 5), (1, 30), (1, 47)]:
        want = oracle_fwd(one_head(x, b, h), rows=rows, heads=[(0, 0)])
        err = rel_l2(got[b, rows, h], want[0, rows, 0])
        print(f"benchmark shape b={b} h={h}: rel_l2(sampled rows)={err:.3e}")
        assert err <= TOL_BF16


@pytest.mark.parametrize("path,H,Hqk,dk,dv,T,dtype", [
    ("simt", 6, 1, 32, 16, 300, "f32"), ("simt", 6, 2, 32, 16, 300, "f32"),
    ("simt", 6, 3, 16, 32, 129, "f32"),
    ("tc", 4, 1, 128, 64, 1000, "bf16"), ("tc", 6, 2, 128, 64, 2125, "bf16"),
    ("tc", 4, 2, 128, 128, 1000, "bf16"), ("tc", 48, 1, 128, 64, 300, "bf16")])
def test_shared_qk_heads_match_oracle(LL, path, H, Hqk, dk, dv, T, dtype):
    """q/k shared by groups of H / Hqk value heads (Hqk = 1: one q/k for every head) equal
    the per-head definition with q/k repeated over each group."""
    L = (T - 1).bit_length() + 1
    cfg = W.FwdConfig("mva", 2, H, T, dk, dv, 64, L, dtype, True, "softplus", seed=H + Hqk + T,
                      Hqk=Hqk)
    x = W.make_fwd_inputs(cfg)
    assert x["q"].shape[2] == Hqk and x["v"].shape[2] == H
    got = run(LL, x, 64, path=path, out_dtype=torch.float32)
    assert LL.device_error() == 0
    want = oracle_fwd(per_head_qk(x))
    err = rel_l2(got, want)
    print(f"shared q/k {path} H={H} Hqk={Hqk}: rel_l2={err:.3e}")
    assert err <= tol_for(dtype)


# ------------------------------------------------------------------ strided views


def _fused_views(x, H):
    """q, k, v as slices of one fused [B, T, H, 3d] projection buffer (each a strided view
    with a contiguous last dimension), plus a fresh output laid out [B, H, T, dv] and seen
    as [B, T, H, dv]."""
    B, T, _, d = x["q"].shape
    fused = torch.empty(B, T, H, 3 * d, dtype=x["q"].dtype, device="cuda")
    fused[..., :d] = x["q"].cuda()
    fused[..., d:2 * d] = x["k"].cuda()
    fused[..., 2 * d:] = x["v"].cuda()
    return fused[..., :d], fused[..., d:2 * d], fused[..., 2 * d:]


@pytest.mark.parametrize("path,dtype,d,T", [("tc", "bf16", 128, 700), ("simt", "f32", 32, 333),
                                            ("simt", "bf16", 16, 130)])
def test_strided_fused_qkv_and_permuted_out(LL, path, dtype, d, T):
    """The forward on q/k/v slices of a fused projection and into a [B, H, T, dv] output
    buffer (through loglinear_fwd_strided) equals the oracle on the dense tensors."""
    L = (T - 1).bit_length() + 1
    cfg = W.FwdConfig("strided", 2, 3, T, d, d, 64, L, dtype, True, "softplus", seed=d + T)
    x = W.make_fwd_inputs(cfg)
    q, k, v = _fused_views(x, cfg.H)
    assert not q.is_contiguous() and q.stride(-1) == 1
    out_dt = torch.float32
    out_bhtd = torch.empty(cfg.B, cfg.H, T, d, device="cuda", dtype=out_dt)
    out = out_bhtd.permute(0, 2, 1, 3)
    got = LL.loglinear_fwd(q, k, v, x["log_a"].cuda(), x["lam"].cuda(), 64, out=out, path=path)
    torch.cuda.synchronize()
    assert got.data_ptr() == out_bhtd.data_ptr()
    want = oracle_fwd(x)
    err = rel_l2(out_bhtd.permute(0, 2, 1, 3).cpu(), want)
    print(f"strided {path} {dtype} d={d} T={T}: rel_l2={err:.3e}")
    assert err <= tol_for(dtype)
    dense = run(LL, x, 64, path=path, out_dtype=out_dt)
    assert rel_l2(out_bhtd.permute(0, 2, 1, 3).cpu(), dense) <= 1e-6
    assert LL.device_error() == 0


def test_strided_bf16_output_tc(LL):
    """bf16 output through a strided TMA store: out is a [B, T, H, 2*dv] buffer's first half."""
    T = 300
    cfg = W.FwdConfig("strided_o", 1, 2, T, 128, 64, 64, 10, "bf16", True, "softplus", seed=8)
    x = W.make_fwd_inputs(cfg)
    d = cuda(x)
    big = torch.zeros(1, T, 2, 128, device="cuda", dtype=torch.bfloat16)
    out = big[..., :64]
    LL.loglinear_fwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], 64, out=out, path="tc")
    torch.cuda.synchronize()
    assert (big[..., 64:] == 0).all()  # nothing written outside the view
    assert rel_l2(out.cpu(), oracle_fwd(x)) <= TOL_BF16
