"""Parity of the CUDA lssb decode step with the CPU oracle, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import TOL_BF16, TOL_F32, max_abs, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def LL():
    import log_linear_attention_fwd_gb300 as m
    return m


def step(LL, S, inp, t, out_dtype=torch.float32):
    d = {k: (None if v is None else v.cuda()) for k, v in inp.items()}
    Sd = S.cuda()
    out = LL.loglinear_decode_step(Sd, d["q"], d["k"], d["v"], d["log_a"], d["lam"], t,
                                   out_dtype=out_dtype)
    torch.cuda.synchronize()
    return Sd.cpu(), out.cpu()


@pytest.mark.parametrize("dtype,decay", [("f32", True), ("f32", False), ("bf16", True)])
def test_decode_sequence_matches_forward(LL, dtype, decay):
    """Decoding t = 0..T-1 gives the forward rows and the bucket-definition state."""
    cfg = W.FwdConfig("d", 2, 3, 70, 16, 8, 16, 8, dtype, decay, "softplus", seed=21)
    x = W.make_fwd_inputs(cfg)
    want = oracle.forward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"])
    S = torch.full((cfg.B, cfg.H, cfg.L, cfg.dk, cfg.dv), float("nan")).cuda()  # t=0 must reset
    outs = []
    for t in range(cfg.T):
        la = None if x["log_a"] is None else x["log_a"][:, t].contiguous().cuda()
        o = LL.loglinear_decode_step(S, x["q"][:, t].contiguous().cuda(), x["k"][:, t].contiguous().cuda(),
                                     x["v"][:, t].contiguous().cuda(), la,
                                     x["lam"][:, t].contiguous().cuda(), t, out_dtype=torch.float32)
        outs.append(o.cpu())
    got = torch.stack(outs, 1)
    assert rel_l2(got, want) <= TOL_F32
    for b in range(cfg.B):
        for h in range(cfg.H):
            Sd = oracle.states_from_buckets(x["k"][b, :, h], x["v"][b, :, h],
                                            None if x["log_a"] is None else x["log_a"][b, :, h],
                                            cfg.T - 1, cfg.L)
            assert rel_l2(S[b, h].cpu(), Sd) <= TOL_F32


@pytest.mark.parametrize("t", [1, 2, 3, 7, 8, 12, 255, 256, 8192, 12288, 12344, 12345, 16383])
def test_decode_single_step_random_state(LL, t):
    cfg = W.DecodeConfig("d", 3, 4, 32, 16, 15, t, dtype="f32")
    S0 = W.make_random_state(cfg, t, seed=t)
    inp = W.make_decode_step_inputs(cfg)
    S1, o = step(LL, S0, inp, t)
    S_ref, o_ref = oracle.decode_step(S0.double().numpy(), inp["q"], inp["k"], inp["v"],
                                      inp["log_a"], inp["lam"], t)
    assert rel_l2(o, o_ref) <= TOL_F32
    assert rel_l2(S1, S_ref) <= TOL_F32


def test_decode_leaves_empty_levels_untouched(LL):
    """Levels empty after t-1 (other than the merge target) are neither read nor written."""
    t = 12345
    cfg = W.DecodeConfig("d", 2, 2, 16, 16, 15, t, dtype="f32")
    S0 = W.make_random_state(cfg, t, seed=3)
    nonempty = W.nonempty_levels_before(t, cfg.L)
    l = oracle.lssb(t)
    empty = [lv for lv in range(cfg.L) if lv not in nonempty and lv != l + 1]
    for lv in empty:
        S0[:, :, lv] = 777.0
    inp = W.make_decode_step_inputs(cfg)
    S1, o = step(LL, S0, inp, t)
    for lv in empty:
        assert torch.all(S1[:, :, lv] == 777.0)
    S0z = S0.clone()
    for lv in empty:
        S0z[:, :, lv] = 0
    S_ref, o_ref = oracle.decode_step(S0z.double().numpy(), inp["q"], inp["k"], inp["v"],
                                      inp["log_a"], inp["lam"], t)
    assert rel_l2(o, o_ref) <= TOL_F32
    touched = sorted(set(nonempty) | {l + 1})
    assert rel_l2(S1[:, :, touched], S_ref[:, :, touched]) <= TOL_F32


def test_decode_t0_resets_and_bf16_out(LL):
    cfg = W.DecodeConfig("d", 2, 2, 16, 32, 5, 0, dtype="bf16")
    S0 = torch.randn(cfg.B, cfg.H, cfg.L, cfg.dk, cfg.dv)
    inp = W.make_decode_step_inputs(cfg)
    S1, o = step(LL, S0, inp, 0, out_dtype=torch.bfloat16)
    S_ref, o_ref = oracle.decode_step(np.zeros(S0.shape), inp["q"], inp["k"], inp["v"],
                                      inp["log_a"], inp["lam"], 0)
    assert rel_l2(S1, S_ref) <= TOL_F32
    assert o.dtype == torch.bfloat16 and rel_l2(o, o_ref) <= TOL_BF16


def test_decode_many_levels_generic_path(LL):
    # t = 2^20 - 1 + 1 merges 20 levels: exercises the variant without register arrays
    t = (1 << 20)
    cfg = W.DecodeConfig("d", 1, 2, 8, 8, 22, t, dtype="f32")
    S0 = W.make_random_state(cfg, t, seed=5)
    inp = W.make_decode_step_inputs(cfg)
    S1, o = step(LL, S0, inp, t)
    S_ref, o_ref = oracle.decode_step(S0.double().numpy(), inp["q"], inp["k"], inp["v"],
                                      inp["log_a"], inp["lam"], t)
    assert rel_l2(o, o_ref) <= TOL_F32 and rel_l2(S1, S_ref) <= TOL_F32


def test_decode_full_size_workload(LL):
    """B128 H16 d128 L15 at t = 12345, launched at full size.  Every (b, h) starts from a
    random state with the Fenwick occupancy of t-1; a sample of (b, h) is checked against
    the oracle step, and two (b, h) start from their true prefill (bucket definition over
    12345 seeded bf16 tokens)."""
    cfg = W.DECODE_CONFIG
    t = cfg.t
    S0 = W.make_random_state(cfg, t, seed=11, scale=0.05)
    true_bh = [(0, 0), (127, 15)]
    for b, h in true_bh:
        k, v, la = W.make_decode_tokens(cfg, b, h, t)
        S0[b, h] = torch.from_numpy(oracle.states_from_buckets(k, v, la, t - 1, cfg.L)).float()
    inp = W.make_decode_step_inputs(cfg)
    S1, o = step(LL, S0, inp, t, out_dtype=torch.float32)
    rng = np.random.default_rng(0)
    sample = set(true_bh) | {(int(b), int(h)) for b, h in zip(rng.integers(0, cfg.B, 48),
                                                               rng.integers(0, cfg.H, 48))}
    errs_o, errs_s = [], []
    for b, h in sorted(sample):
        S_ref, o_ref = oracle.decode_step(S0[b, h].double().numpy(), inp["q"][b, h], inp["k"][b, h],
                                          inp["v"][b, h], inp["log_a"][b, h], inp["lam"][b, h], t)
        errs_o.append(rel_l2(o[b, h], o_ref))
        errs_s.append(rel_l2(S1[b, h], S_ref))
    print(f"decode full size: max rel_l2 out={max(errs_o):.3e} state={max(errs_s):.3e}")
    assert max(errs_o) <= TOL_F32 and max(errs_s) <= TOL_F32
