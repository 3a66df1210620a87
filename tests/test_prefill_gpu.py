"""Prefill -> decode handoff on the GPU: the per-level decode state after a prompt,
checked against the oracle's bucket definition, and decode steps that continue from it,
checked against the oracle's direct form over the longer sequence."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import TOL_BF16, TOL_F32, cuda, per_head_qk, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def LL():
    import log_linear_attention_fwd_gb300 as m
    return m


def oracle_state(x, T):
    """[B, H, L, dk, dv] per-level states at position T-1 (bucket definition)."""
    x = per_head_qk(x)
    B, _, H, dk = x["q"].shape
    dv, L = x["v"].shape[-1], x["lam"].shape[-1]
    S = np.zeros((B, H, L, dk, dv))
    for b in range(B):
        for h in range(H):
            la = None if x["log_a"] is None else x["log_a"][b, :T, h]
            S[b, h] = oracle.states_from_buckets(x["k"][b, :T, h], x["v"][b, :T, h], la, T - 1, L)
    return S


def check_state(got, want, tol):
    err = rel_l2(got, want)
    # each non-empty level on its own, relative to its own size
    B, H, L = want.shape[:3]
    for lv in range(L):
        w = want[:, :, lv]
        if np.linalg.norm(w) > 0:
            assert rel_l2(got[:, :, lv], w) <= tol, lv
        else:
            assert float(np.abs(got[:, :, lv].double().numpy()).max()) == 0.0, lv
    return err


@pytest.mark.parametrize("T,C", [(1, 16), (2, 16), (17, 16), (64, 16), (100, 8), (257, 32),
                                 (1000, 64)])
def test_prefill_state_simt(LL, T, C):
    L = max((T - 1).bit_length() + 1, 1)
    cfg = W.FwdConfig("p", 2, 3, T, 16, 8, C, L, "f32", True, "softplus", seed=T + 3)
    x = W.make_fwd_inputs(cfg)
    d = cuda(x)
    out, state = LL.loglinear_prefill(d["q"], d["k"], d["v"], d["log_a"], d["lam"], C, path="simt")
    torch.cuda.synchronize()
    err = check_state(state.cpu(), oracle_state(x, T), TOL_F32)
    assert rel_l2(out.cpu(), oracle.forward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"])) <= TOL_F32
    print(f"simt T={T}: state rel_l2={err:.2e}")


@pytest.mark.parametrize("T,dv,Hqk", [(1, 128, 0), (128, 128, 0), (300, 128, 0), (1000, 128, 0),
                                      (2049, 128, 0), (1, 64, 0), (300, 64, 0), (2049, 64, 0),
                                      (2049, 64, 1)])
def test_prefill_state_tc(LL, T, dv, Hqk):
    L = max((T - 1).bit_length() + 1, 1)
    cfg = W.FwdConfig("p", 2, 3, T, 128, dv, 64, L, "bf16", True, "softplus", seed=T + 5, Hqk=Hqk)
    x = W.make_fwd_inputs(cfg)
    d = cuda(x)
    assert LL.resolve_path(128, dv, 64, 1) == "tc"
    out, state = LL.loglinear_prefill(d["q"], d["k"], d["v"], d["log_a"], d["lam"], 64, path="tc")
    torch.cuda.synchronize()
    assert LL.device_error() == 0
    err = check_state(state.cpu(), oracle_state(x, T), TOL_BF16)
    print(f"tc T={T}: state rel_l2={err:.2e}")


@pytest.mark.parametrize("decay", [True, False])
def test_prefill_state_tc_headline_shape(LL, decay):
    """The headline prompt (B1 H16 T16384 dk=dv=128 bf16) on the tensor-core path: at
    t = 16383 every one of the 15 levels holds a bucket (levels 8-14 are the forward's
    block states decayed to t).  Two heads against the bucket definition, level by level;
    without decay the top levels carry full weight."""
    cfg = W.FWD_CONFIGS["mamba2_T16384"].with_(decay=decay, seed=31)
    x = W.make_fwd_inputs(cfg)
    d = cuda(x)
    out, state = LL.loglinear_prefill(d["q"], d["k"], d["v"], d["log_a"], d["lam"], cfg.C,
                                      path="tc")
    torch.cuda.synchronize()
    assert LL.device_error() == 0
    T = cfg.T
    for h in (0, cfg.H - 1):
        la = None if x["log_a"] is None else x["log_a"][0, :, h]
        want = oracle.states_from_buckets(x["k"][0, :, h], x["v"][0, :, h], la, T - 1, cfg.L)
        got = state[0, h].cpu()
        errs = []
        for lv in range(cfg.L):
            if np.linalg.norm(want[lv]) > 1e-30:
                errs.append(rel_l2(got[lv], want[lv]))
                assert errs[-1] <= TOL_BF16, (h, lv, errs[-1])
            else:  # decayed below fp32's range: the state rounds to zero there too
                assert decay and float(got[lv].abs().max()) <= 1e-30, (h, lv)
        if not decay:
            assert len(errs) == cfg.L
        print(f"tc prefill T={T} decay={decay} head {h}: per-level rel_l2 " +
              " ".join(f"{e:.1e}" for e in errs))


@pytest.mark.parametrize("path,T,dk,dv,dtype,H,Hqk", [("simt", 300, 16, 16, "f32", 2, 2),
                                                      ("tc", 1151, 128, 128, "bf16", 2, 2),
                                                      ("tc", 1151, 128, 64, "bf16", 2, 2),
                                                      ("simt", 300, 16, 16, "f32", 4, 2),
                                                      ("tc", 1151, 128, 64, "bf16", 4, 1)])
def test_decode_continues_from_prefill(LL, path, T, dk, dv, dtype, H, Hqk):
    """Prefill T positions, then decode positions T..T+n-1 from the handed-over state; the
    outputs must match the direct form over the whole T+n sequence (q/k shared by groups of
    H / Hqk heads where Hqk < H)."""
    n = 6
    L = (T + n - 1).bit_length() + 1
    cfg = W.FwdConfig("pd", 2, H, T + n, dk, dv, 64, L, dtype, True, "softplus", seed=11, Hqk=Hqk)
    x = W.make_fwd_inputs(cfg)
    d = cuda(x)
    pre = {k: (None if v is None else v[:, :T].contiguous()) for k, v in d.items()}
    _, state = LL.loglinear_prefill(pre["q"], pre["k"], pre["v"], pre["log_a"], pre["lam"], 64,
                                    path=path)
    outs = []
    for t in range(T, T + n):
        o = LL.loglinear_decode_step(state, d["q"][:, t].contiguous(), d["k"][:, t].contiguous(),
                                     d["v"][:, t].contiguous(), d["log_a"][:, t].contiguous(),
                                     d["lam"][:, t].contiguous(), t, out_dtype=torch.float32)
        outs.append(o)
    torch.cuda.synchronize()
    got = torch.stack(outs, dim=1).cpu()  # [B, n, H, dv]
    rows = np.arange(T, T + n)
    xp = per_head_qk(x)
    want = oracle.forward_direct(xp["q"], xp["k"], xp["v"], xp["log_a"], xp["lam"], rows=rows)[:, rows]
    tol = TOL_F32 if dtype == "f32" else TOL_BF16
    err = rel_l2(got, want)
    print(f"{path}: continuation rel_l2={err:.2e}")
    assert err <= tol


def test_prefill_empty_prompt(LL):
    B, H, L, d = 2, 3, 4, 8
    q = torch.zeros(B, 0, H, d, device="cuda")
    lam = torch.zeros(B, 0, H, L, device="cuda")
    la = torch.zeros(B, 0, H, device="cuda")
    state = torch.full((B, H, L, d, d), 7.0, device="cuda")
    _, state = LL.loglinear_prefill(q, q, q, la, lam, 16, state=state, path="simt")
    torch.cuda.synchronize()
    assert float(state.abs().max()) == 0.0


@pytest.mark.parametrize("path,dtype,dk,dv", [("tc", "bf16", 128, 128), ("simt", "f32", 16, 8)])
def test_prefill_with_events_matches_prefill(LL, path, dtype, dk, dv):
    """The timed prefill launches the forward's kernels and then the state kernel, records
    an event around each, and gives the same output and state as loglinear_prefill."""
    T = 700
    cfg = W.FwdConfig("pre_ev", 1, 2, T, dk, dv, 64, (T - 1).bit_length() + 1, dtype, True,
                      "softplus", seed=17)
    d = cuda(W.make_fwd_inputs(cfg))
    out0, S0 = LL.loglinear_prefill(d["q"], d["k"], d["v"], d["log_a"], d["lam"], 64, path=path)
    ws = torch.empty(LL.fwd_workspace_size(1, T, 2, dk, dv, 64, 1 if dtype == "bf16" else 0, path),
                     device="cuda", dtype=torch.uint8)
    out1, S1 = torch.empty_like(out0), torch.empty_like(S0)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    nk = LL.loglinear_prefill_with_events(d["q"], d["k"], d["v"], d["log_a"], d["lam"], 64, ev,
                                          out1, S1, ws, path=path)
    torch.cuda.synchronize()
    assert nk == (2 if path == "tc" else 4)       # forward kernel(s), then the state kernel
    assert torch.equal(out0, out1) and torch.equal(S0, S1)
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(nk)]
    assert all(t >= 0 for t in times)
