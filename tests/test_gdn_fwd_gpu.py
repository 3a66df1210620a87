"""Parity of the CUDA Log-Linear Gated DeltaNet forward (recurrent form) with the CPU
oracle, through the C ABI (GPU)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.helpers import TOL_BF16, TOL_F32, rel_l2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def LL():
    import log_linear_attention_fwd_gb300 as m
    return m


def _dev(x):
    return {k: (None if v is None else v.cuda()) for k, v in x.items()}


def _run(LL, x, L, out_dtype=torch.float32, with_state=True):
    d = _dev(x)
    B, T, Hqk, dk = d["q"].shape
    H, dv = d["v"].shape[2], d["v"].shape[3]
    state = torch.full((B, H, L, dk, dv), float("nan"), device="cuda") if with_state else None
    out = LL.loglinear_gdn_fwd(d["q"], d["k"], d["v"], d["log_a"], d["beta"], d["lam"],
                               out_dtype=out_dtype, state=state)
    torch.cuda.synchronize()
    return out.cpu(), (None if state is None else state.cpu())


@pytest.mark.parametrize("B,H,Hqk,T,dk,dv,dtype,decay", [
    (1, 1, 1, 1, 16, 8, "f32", True),         # one token: level 0 only
    (2, 3, 0, 37, 32, 16, "f32", True),       # ragged stage (16 tokens), several columns
    (1, 4, 1, 130, 64, 24, "f32", False),     # shared q/k head, d_v not a power of two
    (1, 2, 2, 300, 128, 64, "bf16", True),
    (1, 1, 1, 1000, 128, 128, "f32", True),   # 10 levels, 16 column slices
    (2, 2, 0, 77, 7, 3, "f32", True),         # odd d_k, d_v below the 8-column slice
])
def test_gdn_fwd_matches_recurrence(LL, B, H, Hqk, T, dk, dv, dtype, decay):
    """Every output row and the final per-level state against the oracle's lssb recurrence
    (fp64), which its own pins tie to the direct form and to plain Gated DeltaNet."""
    L = max(1, (T - 1).bit_length() + 1) + 1
    cfg = W.FwdConfig("gdn_fwd", B, H, T, dk, dv, 16, L, dtype, decay, "softplus", seed=T + dk,
                      Hqk=Hqk)
    x = W.make_gdn_inputs(cfg)
    want, S_want = oracle.gdn_recurrence(*_bcast_qk(x, H))
    got, S = _run(LL, x, L)
    err, serr = rel_l2(got, want), rel_l2(S, S_want)
    print(f"gdn fwd B{B} H{H} Hqk{Hqk} T{T} dk{dk} dv{dv} {dtype}: out {err:.2e} state {serr:.2e}")
    assert err <= TOL_F32 and serr <= TOL_F32
    assert torch.isfinite(S).all()


def _bcast_qk(x, H):
    """The oracle takes one q/k per value head: repeat the shared q/k heads."""
    q, k = x["q"], x["k"]
    hg = H // q.shape[2]
    if hg > 1:
        q = q.repeat_interleave(hg, dim=2)
        k = k.repeat_interleave(hg, dim=2)
    return q, k, x["v"], x["log_a"], x["beta"], x["lam"]


def test_gdn_fwd_bf16_out(LL):
    cfg = W.FwdConfig("gdn_fwd_bf16", 1, 2, 200, 128, 64, 16, 9, "bf16", True, "softplus", seed=5)
    x = W.make_gdn_inputs(cfg)
    want, _ = oracle.gdn_recurrence(*_bcast_qk(x, cfg.H))
    got, _ = _run(LL, x, cfg.L, out_dtype=torch.bfloat16, with_state=False)
    err = rel_l2(got.float(), want)
    print(f"gdn fwd bf16 out: rel_l2={err:.2e}")
    assert err <= TOL_BF16


def test_gdn_fwd_constant_lambda_is_gated_deltanet(LL):
    """Lambda equal at every level: the plain Gated DeltaNet recurrence (one state)."""
    cfg = W.FwdConfig("gdn_plain", 1, 2, 150, 32, 16, 16, 9, "f32", True, "softplus", seed=9)
    x = W.make_gdn_inputs(cfg)
    c = x["lam"][..., :1]
    x["lam"] = c.expand_as(x["lam"]).contiguous()
    want = oracle.gated_deltanet_recurrent(x["q"], x["k"], x["v"], x["log_a"], x["beta"],
                                           c[..., 0])
    got, _ = _run(LL, x, cfg.L, with_state=False)
    assert rel_l2(got, want) <= TOL_F32


def test_gdn_fwd_then_decode(LL):
    """The forward's final state is the state the decode step continues from: forward over
    T tokens, then decode steps T..T+5, against the oracle over T+6 tokens."""
    T, extra = 100, 6
    cfg = W.FwdConfig("gdn_handoff", 1, 3, T + extra, 64, 32, 16, 9, "f32", True, "softplus",
                      seed=21)
    x = W.make_gdn_inputs(cfg)
    want, _ = oracle.gdn_recurrence(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"])
    head = {k: (None if v is None else v[:, :T].contiguous()) for k, v in x.items()}
    out_head, S = _run(LL, head, cfg.L)
    S = S.cuda()
    outs = [out_head]
    for t in range(T, T + extra):
        sl = lambda n: None if x[n] is None else x[n][:, t].contiguous().cuda()
        o = LL.loglinear_gdn_decode_step(S, sl("q"), sl("k"), sl("v"), sl("log_a"), sl("beta"),
                                         sl("lam"), t, out_dtype=torch.float32)
        outs.append(o.cpu()[:, None])
    got = torch.cat(outs, 1)
    assert rel_l2(got, want) <= TOL_F32


def test_gdn_fwd_long_sampled_rows(LL):
    """T = 70000 (17 levels: the 32-lanes-per-column layout), small heads; rows sampled
    across the sequence against the direct form."""
    T = 70000
    cfg = W.FwdConfig("gdn_long", 1, 1, T, 8, 8, 16, 18, "f32", False, "softplus", seed=3)
    x = W.make_gdn_inputs(cfg)
    x["log_a"] = (torch.full((1, T, 1), -2e-4))  # slow decay: far levels still weigh
    rows = [0, 1, 2, 1023, 1024, 4095, 32767, 32768, 65535, 65536, T - 2, T - 1]
    want = oracle.gdn_direct(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"], rows=rows)
    got, S = _run(LL, x, cfg.L)
    for r in rows:
        assert rel_l2(got[:, r], want[:, r]) <= 1e-4, r
    assert torch.isfinite(S).all()


def test_gdn_fwd_empty(LL):
    """T = 0 leaves an all-zero state; B = 0 does nothing."""
    q = torch.zeros(1, 0, 2, 16, device="cuda")
    v = torch.zeros(1, 0, 2, 8, device="cuda")
    beta = torch.zeros(1, 0, 2, device="cuda")
    lam = torch.zeros(1, 0, 2, 3, device="cuda")
    state = torch.full((1, 2, 3, 16, 8), float("nan"), device="cuda")
    LL.loglinear_gdn_fwd(q, q, v, None, beta, lam, state=state)
    torch.cuda.synchronize()
    assert (state == 0).all()


# ---------------------------------------------------------------- the chunked form


def _run_chunked(LL, x, out_dtype=torch.float32):
    d = _dev(x)
    out = LL.loglinear_gdn_fwd_chunked(d["q"], d["k"], d["v"], d["log_a"], d["beta"], d["lam"],
                                       out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.parametrize("B,H,Hqk,T,dk,dv,dtype,decay", [
    (1, 1, 1, 1, 16, 8, "f32", True),         # one token
    (2, 3, 0, 37, 32, 16, "f32", True),       # one ragged chunk
    (1, 4, 1, 130, 64, 24, "f32", False),     # three chunks, the last ragged; shared q/k
    (1, 2, 2, 300, 128, 64, "bf16", True),
    (1, 3, 1, 600, 128, 128, "bf16", True),   # bf16 rows of 128: 16-byte loads
    (1, 1, 1, 1000, 128, 128, "f32", True),   # 16 chunks: chunk levels 1..4
    (2, 2, 0, 77, 7, 3, "f32", True),         # odd d_k, d_v
    (1, 2, 0, 2100, 32, 32, "f32", False),    # 33 chunks without decay: every level weighs
])
def test_gdn_fwd_chunked_matches_recurrence(LL, B, H, Hqk, T, dk, dv, dtype, decay):
    """The chunked form (UT transform per 64-token chunk, chunk-level states carried by the
    chunk transitions) against the oracle's lssb recurrence, every output row."""
    L = max(1, (T - 1).bit_length() + 1) + 1
    cfg = W.FwdConfig("gdn_chunk", B, H, T, dk, dv, 64, L, dtype, decay, "softplus",
                      seed=T + dk + 1, Hqk=Hqk)
    x = W.make_gdn_inputs(cfg)
    want, _ = oracle.gdn_recurrence(*_bcast_qk(x, H))
    got = _run_chunked(LL, x)
    err = rel_l2(got, want)
    print(f"gdn chunked B{B} H{H} Hqk{Hqk} T{T} dk{dk} dv{dv} {dtype}: rel_l2={err:.2e}")
    assert err <= TOL_F32


def test_gdn_fwd_chunked_unaligned_inputs(LL):
    """q, k, v whose base addresses are 2 bytes off a 16-byte boundary take the kernel's
    element-wise loads instead of its 16-byte ones; the output is the same."""
    cfg = W.FwdConfig("gdn_chunk_u", 1, 2, 300, 128, 128, 64, 10, "bf16", True, "softplus", seed=9)
    x = W.make_gdn_inputs(cfg)
    want = _run_chunked(LL, x)
    d = _dev(x)
    off = {}
    for n in ("q", "k", "v"):
        buf = torch.empty(d[n].numel() + 1, dtype=d[n].dtype, device="cuda")
        off[n] = buf[1:].view(d[n].shape)
        off[n].copy_(d[n])
        assert off[n].data_ptr() % 16 == 2
    got = LL.loglinear_gdn_fwd_chunked(off["q"], off["k"], off["v"], d["log_a"], d["beta"],
                                       d["lam"], out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(got.cpu(), want)


def test_gdn_fwd_chunked_bf16_out_and_constant_lambda(LL):
    """bf16 output; and lambda equal at every level gives plain Gated DeltaNet."""
    cfg = W.FwdConfig("gdn_chunk_b", 1, 2, 500, 128, 64, 64, 10, "bf16", True, "softplus", seed=4)
    x = W.make_gdn_inputs(cfg)
    want, _ = oracle.gdn_recurrence(*_bcast_qk(x, cfg.H))
    got = _run_chunked(LL, x, out_dtype=torch.bfloat16)
    assert rel_l2(got.float(), want) <= TOL_BF16
    cfg2 = W.FwdConfig("gdn_chunk_c", 1, 2, 400, 32, 16, 64, 10, "f32", True, "softplus", seed=6)
    x2 = W.make_gdn_inputs(cfg2)
    c = x2["lam"][..., :1]
    x2["lam"] = c.expand_as(x2["lam"]).contiguous()
    want2 = oracle.gated_deltanet_recurrent(x2["q"], x2["k"], x2["v"], x2["log_a"], x2["beta"],
                                            c[..., 0])
    assert rel_l2(_run_chunked(LL, x2), want2) <= TOL_F32


def test_gdn_fwd_chunked_long_sampled_rows(LL):
    """T = 70000 (1094 chunks, chunk levels up to 11), small heads, slow decay: rows sampled
    across the sequence against the direct form."""
    T = 70000
    cfg = W.FwdConfig("gdn_chunk_long", 1, 1, T, 8, 8, 64, 18, "f32", False, "softplus", seed=3)
    x = W.make_gdn_inputs(cfg)
    x["log_a"] = torch.full((1, T, 1), -2e-4)
    rows = [0, 63, 64, 1023, 1024, 4095, 32767, 32768, 65535, 65536, T - 2, T - 1]
    want = oracle.gdn_direct(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"], rows=rows)
    got = _run_chunked(LL, x)
    for r in rows:
        assert rel_l2(got[:, r], want[:, r]) <= 1e-4, r


def test_gdn_fwd_chunked_matches_recurrent_full_size(LL):
    """Two heads of the headline shape (T = 16384, d_k = d_v = 128, bf16 inputs): the chunked
    and the recurrent GPU forms agree (the recurrent one is pinned to the oracle above)."""
    cfg = W.FwdConfig("gdn_chunk_full", 1, 2, 16384, 128, 128, 64, 15, "bf16", True, "softplus",
                      seed=11)
    x = _dev(W.make_gdn_inputs(cfg))
    a = LL.loglinear_gdn_fwd(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"],
                             out_dtype=torch.float32)
    b = LL.loglinear_gdn_fwd_chunked(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"],
                                     out_dtype=torch.float32)
    torch.cuda.synchronize()
    err = rel_l2(b.cpu(), a.cpu().double().numpy())
    print(f"gdn chunked vs recurrent, T=16384: rel_l2={err:.2e}")
    assert err <= 1e-4


def test_gdn_fwd_chunked_many_chunk_levels(LL):
    """T = 140000: 2188 chunks, 13 chunk-level slots (the wider register layout of the scan);
    sampled rows against the direct form."""
    T = 140000
    cfg = W.FwdConfig("gdn_chunk_longer", 1, 1, T, 4, 8, 64, 19, "f32", False, "softplus", seed=5)
    x = W.make_gdn_inputs(cfg)
    x["log_a"] = torch.full((1, T, 1), -1e-4)
    rows = [131071, 131072, 139999]
    want = oracle.gdn_direct(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"], rows=rows)
    got = _run_chunked(LL, x)
    for r in rows:
        assert rel_l2(got[:, r], want[:, r]) <= 1e-4, r


@pytest.mark.parametrize("T,dk,dv,dtype,decay", [(37, 32, 16, "f32", True),
                                                  (130, 64, 32, "f32", False),
                                                  (1000, 128, 128, "f32", True),
                                                  (2100, 32, 32, "bf16", True)])
def test_gdn_fwd_chunked_final_state(LL, T, dk, dv, dtype, decay):
    """The chunked form's final state (chunk levels from the scan, the last chunk's levels from
    the lssb steps over its tokens) against the oracle's recurrence, every level; and the
    decode step continuing from it."""
    L = (T - 1).bit_length() + 2
    cfg = W.FwdConfig("gdn_chunk_state", 1, 2, T + 3, dk, dv, 64, L, dtype, decay, "softplus",
                      seed=T + 17)
    x = W.make_gdn_inputs(cfg)
    want, _ = oracle.gdn_recurrence(x["q"], x["k"], x["v"], x["log_a"], x["beta"], x["lam"])
    head = {k: (None if v is None else v[:, :T].contiguous()) for k, v in x.items()}
    _, S_want = oracle.gdn_recurrence(head["q"], head["k"], head["v"], head["log_a"],
                                      head["beta"], head["lam"])
    d = _dev(head)
    S = torch.full((1, 2, L, dk, dv), float("nan"), device="cuda")
    LL.loglinear_gdn_fwd_chunked(d["q"], d["k"], d["v"], d["log_a"], d["beta"], d["lam"],
                                 out_dtype=torch.float32, state=S)
    torch.cuda.synchronize()
    assert rel_l2(S.cpu(), S_want) <= TOL_F32
    outs = []
    for t in range(T, T + 3):
        sl = lambda n: None if x[n] is None else x[n][:, t].contiguous().cuda()
        o = LL.loglinear_gdn_decode_step(S, sl("q"), sl("k"), sl("v"), sl("log_a"), sl("beta"),
                                         sl("lam"), t, out_dtype=torch.float32)
        outs.append(o.cpu())
    assert rel_l2(torch.stack(outs, 1), want[:, T:]) <= TOL_F32
