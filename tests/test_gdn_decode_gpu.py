"""Parity of the CUDA Log-Linear Gated DeltaNet decode step with the CPU oracle, through
the C ABI (GPU)."""
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


def _dev(x):
    return {k: (None if v is None else v.cuda()) for k, v in x.items()}


def gdn_step(LL, S, inp, t, out_dtype=torch.float32):
    d = _dev(inp)
    Sd = S.cuda()
    out = LL.loglinear_gdn_decode_step(Sd, d["q"], d["k"], d["v"], d["log_a"], d["beta"],
                                       d["lam"], t, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return Sd.cpu(), out.cpu()


@pytest.mark.parametrize("dtype,decay", [("f32", True), ("f32", False), ("bf16", True)])
def test_gdn_decode_sequence_matches_direct(LL, dtype, decay):
    """Decoding t = 0..T-1 from a state full of NaN (t = 0 must reset it) gives the direct
    form's rows and, at the end, the bucket definition of every level's state."""
    cfg = W.FwdConfig("gdn_seq", 2, 3, 45, 16, 8, 16, 7, dtype, decay, "softplus", seed=31)
    x = W.make_gdn_inputs(cfg)
    want = oracle.gdn_direct(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"])
    S = torch.full((cfg.B, cfg.H, cfg.L, cfg.dk, cfg.dv), float("nan")).cuda()
    outs = []
    for t in range(cfg.T):
        sl = lambda n: None if x[n] is None else x[n][:, t].contiguous().cuda()
        o = LL.loglinear_gdn_decode_step(S, sl("q"), sl("k"), sl("v"), sl("log_a"), sl("beta"),
                                         sl("lam"), t, out_dtype=torch.float32)
        outs.append(o.cpu())
    got = torch.stack(outs, 1)
    err = rel_l2(got, want)
    print(f"gdn decode sequence {dtype} decay={decay}: rel_l2={err:.3e}")
    assert err <= TOL_F32
    for b in range(cfg.B):
        for h in range(cfg.H):
            Sd = oracle.gdn_states_from_buckets(x["k"][b, :, h], x["v"][b, :, h],
                                                None if x["log_a"] is None else x["log_a"][b, :, h],
                                                x["beta"][b, :, h], cfg.T - 1, cfg.L)
            assert rel_l2(S[b, h].cpu(), Sd) <= TOL_F32


@pytest.mark.parametrize("t", [0, 1, 2, 3, 7, 8, 12, 255, 256, 8192, 12288, 12344, 12345, 16383])
@pytest.mark.parametrize("dk,dv", [(32, 16), (128, 128)])
def test_gdn_decode_single_step_random_state(LL, t, dk, dv):
    cfg = W.DecodeConfig("gdn_d", 3, 4, dk, dv, 15, t, dtype="f32")
    S0 = W.make_random_state(cfg, t, seed=t + dk)
    inp = W.make_gdn_decode_step_inputs(cfg)
    S1, o = gdn_step(LL, S0, inp, t)
    S_ref, o_ref = oracle.gdn_decode_step(S0.double().numpy(), inp["q"], inp["k"], inp["v"],
                                          inp["log_a"], inp["beta"], inp["lam"], t)
    assert rel_l2(o, o_ref) <= TOL_F32
    assert rel_l2(S1, S_ref) <= TOL_F32


@pytest.mark.parametrize("dk,dv,H,Hqk,dtype", [(7, 4, 3, 3, "f32"), (96, 64, 4, 2, "bf16"),
                                               (128, 32, 6, 1, "bf16"), (1, 8, 2, 2, "f32")])
def test_gdn_decode_shapes_and_shared_qk(LL, dk, dv, H, Hqk, dtype):
    """Other head dims, q/k heads shared by groups of value heads, bf16 tokens and output."""
    t = 12345
    cfg = W.DecodeConfig("gdn_s", 2, H, dk, dv, 15, t, dtype=dtype)
    S0 = W.make_random_state(cfg, t, seed=dk + dv)
    inp = W.make_gdn_decode_step_inputs(cfg)
    for n in ("q", "k"):  # one q/k per group of H / Hqk value heads
        inp[n] = inp[n][:, ::H // Hqk].contiguous()
    per_head = dict(inp)
    for n in ("q", "k"):
        per_head[n] = inp[n].repeat_interleave(H // Hqk, dim=1)
    out_dtype = torch.float32 if dtype == "f32" else torch.bfloat16
    S1, o = gdn_step(LL, S0, inp, t, out_dtype=out_dtype)
    S_ref, o_ref = oracle.gdn_decode_step(S0.double().numpy(), per_head["q"], per_head["k"],
                                          per_head["v"], per_head["log_a"], per_head["beta"],
                                          per_head["lam"], t)
    assert rel_l2(S1, S_ref) <= TOL_F32
    assert rel_l2(o, o_ref) <= (TOL_F32 if dtype == "f32" else TOL_BF16)


def test_gdn_decode_full_size_sampled(LL):
    """The decode workload's shape (B128 H16 d128 L15 fp32 states, bf16 tokens, t = 12345):
    sampled (b, h) against the oracle's step; every output finite."""
    dcfg = W.DECODE_CONFIG
    t = dcfg.t
    gen = torch.Generator(device="cuda").manual_seed(5)
    S = torch.zeros(dcfg.B, dcfg.H, dcfg.L, dcfg.dk, dcfg.dv, device="cuda")
    for lv in W.nonempty_levels_before(t, dcfg.L):
        S[:, :, lv].normal_(0.0, 0.05, generator=gen)
    pairs = [(0, 0), (17, 5), (64, 15), (127, 9)]
    S0 = {p: S[p].cpu() for p in pairs}
    inp = W.make_gdn_decode_step_inputs(dcfg)
    d = _dev(inp)
    o = LL.loglinear_gdn_decode_step(S, d["q"], d["k"], d["v"], d["log_a"], d["beta"], d["lam"], t,
                                     out_dtype=torch.float32).cpu()
    torch.cuda.synchronize()
    assert torch.isfinite(o).all()
    for (b, h) in pairs:
        S_ref, o_ref = oracle.gdn_decode_step(S0[(b, h)].double().numpy(), inp["q"][b, h],
                                              inp["k"][b, h], inp["v"][b, h], inp["log_a"][b, h],
                                              inp["beta"][b, h], inp["lam"][b, h], t)
        assert rel_l2(o[b, h], o_ref) <= TOL_F32, (b, h)
        assert rel_l2(S[b, h].cpu(), S_ref) <= TOL_F32, (b, h)
