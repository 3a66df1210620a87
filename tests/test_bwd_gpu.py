"""Parity of the CUDA backward with the CPU oracle's backward, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import TOL_BF16, cuda, one_head, per_head_qk, rel_l2

pytestmark = pytest.mark.gpu

# fp32 gradients: every term is accumulated in fp32 (relative rounding ~1e-7 per add over
# at most a few thousand terms); 1e-5 rel-L2 leaves two orders of margin.  d log a is a
# suffix sum of q.dQ - k.dK whose terms cancel (its total is exactly 0), so its error is
# measured against the scale of those terms: 1e-4.
TOL_G32 = 1e-5
TOL_DLA32 = 1e-4


@pytest.fixture(scope="module")
def LL():
    import log_linear_attention_fwd_gb300 as m
    return m


def _dout(cfg, seed):
    g = torch.Generator().manual_seed(seed)
    d = torch.randn(cfg.B, cfg.T, cfg.H, cfg.dv, generator=g)
    return d.to(W.torch_dtype(cfg.dtype))


def _oracle_grads(x, dout):
    """Oracle gradients, with q/k gradients summed over each group of heads sharing a q/k
    head (the oracle's definition is per head), and the scale of the terms q_t . dQ_t
    that cancel in d log a (the norm of that [B, T, H] array)."""
    xp = per_head_qk(x)
    g = oracle.backward_direct(xp["q"], xp["k"], xp["v"], xp["log_a"], xp["lam"], dout)
    qf = xp["q"].double().numpy()
    dla_scale = float(np.linalg.norm(np.sum(qf * g["q"], axis=-1)))
    H, G = x["v"].shape[2], x["q"].shape[2]
    for n in ("q", "k"):
        B, T, _, dk = g[n].shape
        g[n] = g[n].reshape(B, T, G, H // G, dk).sum(axis=3)
    return g, dla_scale


def _check(LL, cfg, tol, tol_dla, seed=0, path="auto"):
    x = W.make_fwd_inputs(cfg)
    dout = _dout(cfg, seed + 100)
    d = cuda(x)
    got = LL.loglinear_bwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], dout.cuda(), path=path)
    torch.cuda.synchronize()
    assert LL.device_error() == 0
    want, dla_scale = _oracle_grads(x, dout)
    errs = {}
    for name, gt in zip(("q", "k", "v", "log_a", "lam"), got):
        if want[name] is None:
            assert gt is None
            continue
        if name == "log_a":  # relative to the terms that cancel in it (its value may be 0)
            diff = gt.cpu().double().numpy() - want[name]
            errs[name] = float(np.linalg.norm(diff)) / max(np.linalg.norm(want[name]), dla_scale,
                                                           1e-300)
        else:
            errs[name] = rel_l2(gt.cpu(), want[name])
    print(f"bwd {path} {cfg.name} T={cfg.T} H={cfg.H}/{cfg.qk_heads} dk={cfg.dk} dv={cfg.dv} "
          + " ".join(f"{k}={v:.2e}" for k, v in errs.items()))
    for name, e in errs.items():
        assert e <= (tol_dla if name == "log_a" else tol), (name, e)


@pytest.mark.parametrize("T,decay", [(1, True), (31, True), (32, True), (33, True), (100, False),
                                     (300, True), (1000, True), (2049, True)])
def test_bwd_f32_matches_oracle(LL, T, decay):
    L = max((T - 1).bit_length() + 1, 1)
    cfg = W.FwdConfig("bwd_f32", 2, 3, T, 16, 8, 64, L, "f32", decay, "softplus", seed=T)
    _check(LL, cfg, TOL_G32, TOL_DLA32, seed=T)


@pytest.mark.parametrize("dk,dv", [(7, 5), (32, 64), (128, 128)])
def test_bwd_f32_head_dims(LL, dk, dv):
    cfg = W.FwdConfig("bwd_dims", 1, 2, 450, dk, dv, 64, 10, "f32", True, "softplus", seed=dk)
    _check(LL, cfg, TOL_G32, TOL_DLA32, seed=dk)


@pytest.mark.parametrize("path", ["tc", "simt"])
@pytest.mark.parametrize("T,dv", [(300, 64), (2049, 64), (1000, 128), (77, 128), (4096, 128)])
def test_bwd_bf16_matches_oracle(LL, T, dv, path):
    L = (T - 1).bit_length() + 1
    cfg = W.FwdConfig("bwd_bf16", 1, 2, T, 128, dv, 64, L, "bf16", True, "softplus", seed=T + dv)
    _check(LL, cfg, TOL_BF16, TOL_BF16, seed=T, path=path)


def test_bwd_tc_one_hot_lambda_exact(LL):
    """Integers that stay exact through bf16 states and P': dlambda of the tensor-core
    path equals the oracle's bit for bit at every level, and dq equals it up to the final
    bf16 rounding."""
    T = 1151
    L = (T - 1).bit_length() + 1
    for lvl in range(L):
        x = W.make_sparse_int_inputs(1, T, 2, 128, L, lvl, seed=lvl, dv=64)
        g = torch.Generator().manual_seed(lvl)
        dout = torch.randint(-1, 2, (1, T, 2, 64), generator=g).to(torch.bfloat16)
        d = cuda(x)
        got = LL.loglinear_bwd(d["q"], d["k"], d["v"], None, d["lam"], dout.cuda(), path="tc")
        want = oracle.backward_direct(x["q"], x["k"], x["v"], None, x["lam"], dout)
        assert LL.device_error() == 0
        # dq is exact in fp32 and then cast to dO's bf16: compare with the exact value
        # rounded the same way
        assert torch.equal(got[0].cpu(), torch.tensor(want["q"]).to(torch.bfloat16)), lvl
        assert np.array_equal(got[4].cpu().double().numpy(), want["lam"]), lvl


@pytest.mark.parametrize("H,Hqk,dtype", [(4, 1, "f32"), (6, 2, "f32"), (4, 1, "bf16")])
def test_bwd_shared_qk_heads(LL, H, Hqk, dtype):
    cfg = W.FwdConfig("bwd_mva", 2, H, 700, 32 if dtype == "f32" else 128, 16 if dtype == "f32" else 64,
                      64, 11, dtype, True, "softplus", seed=H + Hqk, Hqk=Hqk)
    tol = TOL_G32 if dtype == "f32" else TOL_BF16
    _check(LL, cfg, tol, TOL_DLA32 if dtype == "f32" else TOL_BF16, seed=H)


def test_bwd_one_hot_lambda_exact(LL):
    """Small integers, no decay, lambda one-hot at each level in turn: every product and
    sum is an integer far below 2^24, so the fp32 gradients equal the oracle's exactly."""
    T, L = 200, 9
    for lvl in range(L):
        x = W.make_int_inputs(1, T, 2, 6, 4, L, lvl, seed=lvl)
        g = torch.Generator().manual_seed(lvl)
        dout = torch.randint(-2, 3, (1, T, 2, 4), generator=g).float()
        d = cuda(x)
        got = LL.loglinear_bwd(d["q"], d["k"], d["v"], None, d["lam"], dout.cuda())
        want = oracle.backward_direct(x["q"], x["k"], x["v"], None, x["lam"], dout)
        for name, gt in zip(("q", "k", "v"), got[:3]):
            assert np.array_equal(gt.cpu().double().numpy(), want[name]), (lvl, name)
        assert np.array_equal(got[4].cpu().double().numpy(), want["lam"]), lvl


def test_bwd_workspace_reuse_and_empty(LL):
    cfg = W.FwdConfig("bwd_rep", 1, 2, 500, 16, 16, 64, 10, "f32", True, "softplus", seed=3)
    x = cuda(W.make_fwd_inputs(cfg))
    dout = _dout(cfg, 1).cuda()
    ws = torch.empty(LL.bwd_workspace_size(1, 500, 2, 2, 16, 16, 10, 0, 0), device="cuda",
                     dtype=torch.uint8)
    a = LL.loglinear_bwd(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout, workspace=ws)
    a = [t.clone() for t in a]
    b = LL.loglinear_bwd(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout, workspace=ws)
    # the mirrored states are summed with float atomics, whose order varies between calls:
    # the calls agree up to that rounding (measured in norm; d log a_0 is such rounding)
    for u, w in zip(a, b):
        assert rel_l2(u.cpu(), w.cpu().double().numpy()) <= 1e-6
    q = torch.zeros(1, 0, 2, 8, device="cuda")
    lam = torch.zeros(1, 0, 2, 3, device="cuda")
    out = LL.loglinear_bwd(q, q, q, None, lam, q)
    assert out[0].shape == (1, 0, 2, 8)


def _positions(T, n, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 127, 128, T // 2, T - 129, T - 2, T - 1]
    return np.unique(np.concatenate([fixed, rng.integers(0, T, n)]))


def test_bwd_tc_full_size_sampled(LL):
    """The headline workload (B1 H16 T16384 dk=dv=128 bf16) on the tensor-core path, as
    the bench times it: dq and dlambda of sampled query rows, dk and dv of sampled source
    positions, on two heads, against the oracle's row and column evaluation."""
    cfg = W.FWD_CONFIGS["mamba2_T16384"]
    x = W.make_fwd_inputs(cfg)
    dout = _dout(cfg, 99)
    d = cuda(x)
    got = LL.loglinear_bwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], dout.cuda(), path="tc")
    torch.cuda.synchronize()
    assert LL.device_error() == 0
    rows, cols = _positions(cfg.T, 24, 1), _positions(cfg.T, 24, 2)
    heads = [(0, 3), (0, 11)]
    want = oracle.backward_sampled(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout, rows,
                                   cols, heads)
    for i, (b, h) in enumerate(heads):
        errs = {"q": rel_l2(got[0][b, rows, h].cpu(), want["q"][i]),
                "lam": rel_l2(got[4][b, rows, h].cpu(), want["lam"][i]),
                "k": rel_l2(got[1][b, cols, h].cpu(), want["k"][i]),
                "v": rel_l2(got[2][b, cols, h].cpu(), want["v"][i])}
        print(f"bwd tc full size head {h}: " + " ".join(f"{k}={e:.2e}" for k, e in errs.items()))
        assert all(e <= TOL_BF16 for e in errs.values()), errs


@pytest.mark.parametrize("T,dv", [(5125, 64), (8269, 128), (70000, 64)])
def test_bwd_tc_long_mirrored_runs_no_decay(LL, T, dv):
    """Without decay every level carries full weight into dk and dv.  41, 65 and 547 tiles
    of 128 tokens: the top slots (32 with 9 reader tiles, one run, stored; 64 and 512,
    levels whose slots can have more readers than one run takes, added with atomics into
    slots zeroed first; 512 has 35 readers, two runs) at tile counts that are not
    multiples of the zeroing period (the whole mirrored-state buffer is zeroed).  dq,
    dlambda of sampled query rows and dk, dv of sampled source positions against the
    oracle."""
    L = (T - 1).bit_length() + 1
    cfg = W.FwdConfig("bwd_runs", 1, 2, T, 128, dv, 64, L, "bf16", False, "softplus", seed=T)
    x = W.make_fwd_inputs(cfg)
    dout = _dout(cfg, 7)
    d = cuda(x)
    got = LL.loglinear_bwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], dout.cuda(), path="tc")
    torch.cuda.synchronize()
    assert LL.device_error() == 0
    rows, cols = _positions(T, 16, 3), _positions(T, 16, 4)
    heads = [(0, 0), (0, 1)]
    want = oracle.backward_sampled(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout, rows,
                                   cols, heads)
    for i, (b, h) in enumerate(heads):
        errs = {"q": rel_l2(got[0][b, rows, h].cpu(), want["q"][i]),
                "lam": rel_l2(got[4][b, rows, h].cpu(), want["lam"][i]),
                "k": rel_l2(got[1][b, cols, h].cpu(), want["k"][i]),
                "v": rel_l2(got[2][b, cols, h].cpu(), want["v"][i])}
        print(f"bwd tc runs T={T} dv={dv} head {h}: " + " ".join(f"{k}={e:.2e}" for k, e in errs.items()))
        assert all(e <= TOL_BF16 for e in errs.values()), errs


def test_bwd_tc_benchmark_shape_sampled(LL):
    """The pages' benchmark shape as the bench times it (B2, 48 heads sharing one q/k,
    d_k 128, d_v 64, T 16384, bf16) on the tensor-core path.  dq and dk of the shared q/k
    head are sums over the 48 heads: the oracle evaluates each head alone at sampled rows
    and columns of batch 0 and adds them up; dv and dlambda on three of the heads."""
    cfg = W.FWD_CONFIGS["mva_B2H48_T16384"]
    x = W.make_fwd_inputs(cfg)
    dout = _dout(cfg, 11)
    d = cuda(x)
    got = LL.loglinear_bwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], dout.cuda(), path="tc")
    torch.cuda.synchronize()
    assert LL.device_error() == 0
    rows, cols = _positions(cfg.T, 8, 5), _positions(cfg.T, 8, 6)
    dq = np.zeros((len(rows), cfg.dk))
    dk = np.zeros((len(cols), cfg.dk))
    errs = {}
    for h in range(cfg.H):
        one = one_head(x, 0, h)
        w = oracle.backward_sampled(one["q"], one["k"], one["v"], one["log_a"], one["lam"],
                                    dout[0:1, :, h:h + 1].contiguous(), rows, cols, [(0, 0)])
        dq += w["q"][0]
        dk += w["k"][0]
        if h in (0, 23, 47):
            errs[f"v{h}"] = rel_l2(got[2][0, cols, h].cpu(), w["v"][0])
            errs[f"lam{h}"] = rel_l2(got[4][0, rows, h].cpu(), w["lam"][0])
    errs["q"] = rel_l2(got[0][0, rows, 0].cpu(), dq)
    errs["k"] = rel_l2(got[1][0, cols, 0].cpu(), dk)
    print("bwd tc benchmark shape: " + " ".join(f"{k}={e:.2e}" for k, e in errs.items()))
    assert all(e <= TOL_BF16 for e in errs.values()), errs


@pytest.mark.parametrize("dv,Hqk", [(128, 0), (64, 1)])
def test_bwd_reads_forward_workspace(LL, dv, Hqk):
    """The backward given a tensor-core forward's workspace (its block states kept) equals
    the backward that recomputes them: dlambda bit for bit, and dq too when every head has
    its own q/k (its arithmetic then has a fixed order); dk, dv, d log a, and dq of shared
    q/k heads (summed over the group's heads with float atomics) up to the order of those
    atomics (which also moves a few bf16 roundings by one step)."""
    cfg = W.FwdConfig("bwd_fws", 1, 4, 1500, 128, dv, 64, 12, "bf16", True, "softplus", seed=dv,
                      Hqk=Hqk)
    x = cuda(W.make_fwd_inputs(cfg))
    dout = _dout(cfg, 5).cuda()
    fws = torch.empty(LL.fwd_workspace_size(cfg.B, cfg.T, cfg.H, 128, dv, 64, 1, "tc"),
                      device="cuda", dtype=torch.uint8)
    LL.loglinear_fwd(x["q"], x["k"], x["v"], x["log_a"], x["lam"], 64, workspace=fws, path="tc")
    a = LL.loglinear_bwd(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout, path="tc",
                         fwd_workspace=fws)
    b = LL.loglinear_bwd(x["q"], x["k"], x["v"], x["log_a"], x["lam"], dout, path="tc")
    torch.cuda.synchronize()
    assert LL.device_error() == 0
    assert torch.equal(a[4], b[4])
    if not Hqk:
        assert torch.equal(a[0], b[0])
    for u, w in zip(a[:4], b[:4]):
        assert rel_l2(u.cpu(), w.cpu().double().numpy()) <= 1e-3


def test_bwd_flags_a_foreign_forward_workspace(LL):
    """A fwd_workspace that a tensor-core forward of these sizes did not write (here one a
    CUDA-core forward filled, whose layout differs, or one of another length) raises bit 2
    of the device error word; the matching workspace raises nothing."""
    T = 300
    cfg = W.FwdConfig("bwd_tag", 1, 2, T, 128, 64, 64, 10, "bf16", True, "softplus", seed=3)
    x = W.make_fwd_inputs(cfg)
    d = cuda(x)
    dout = _dout(cfg, 5).cuda()
    args = (d["q"], d["k"], d["v"], d["log_a"], d["lam"])
    ws_simt = torch.zeros(LL.fwd_workspace_size(1, T, 2, 128, 64, 64, 1, "simt"), device="cuda",
                          dtype=torch.uint8)
    LL.loglinear_fwd(*args, 64, path="simt", workspace=ws_simt)
    assert LL.device_error() == 0
    LL.loglinear_bwd(*args, dout, path="tc", fwd_workspace=ws_simt)
    torch.cuda.synchronize()
    assert LL.device_error() & 4
    ws_tc = torch.zeros(LL.fwd_workspace_size(1, T, 2, 128, 64, 64, 1, "tc"), device="cuda",
                        dtype=torch.uint8)
    LL.loglinear_fwd(*args, 64, path="tc", workspace=ws_tc)
    want = LL.loglinear_bwd(*args, dout, path="tc")
    got = LL.loglinear_bwd(*args, dout, path="tc", fwd_workspace=ws_tc)
    torch.cuda.synchronize()
    assert LL.device_error() == 0
    for g, w in zip(got, want):  # same values up to the order of the float atomics
        if w is not None:
            assert rel_l2(g.cpu(), w.cpu()) <= 1e-3
    # a tensor-core forward of another length over a large enough workspace
    short = {k: (None if v is None else v[:, :250].contiguous()) for k, v in d.items()}
    LL.loglinear_bwd(short["q"], short["k"], short["v"], short["log_a"], short["lam"],
                     dout[:, :250].contiguous(), path="tc", fwd_workspace=ws_tc)
    torch.cuda.synchronize()
    assert LL.device_error() & 4
