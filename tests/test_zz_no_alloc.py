"""The forward entry point that allocates nothing (loglinear_fwd_noalloc).

It serves callers that cannot allocate device memory (a plugin whose host application
owns all device memory, a real-time loop that may not call cudaMalloc): its scratch is
the library's fixed device array instead of a caller-provided workspace.  This file is
collected last so that a run stopping at the first failure has run every other test.
"""
import ctypes

import pytest
import torch

import oracle
import workloads as W
from tests.helpers import TOL_BF16, TOL_F32, rel_l2

pytestmark = pytest.mark.gpu

# one problem per kernel path, each well inside the fixed scratch
CASES = [
    ("tc", W.FwdConfig("noalloc_tc", 1, 2, 1000, 128, 128, 64, 11, "bf16", True, "softplus")),
    ("simt", W.FwdConfig("noalloc_simt", 2, 4, 1024, 64, 64, 64, 11, "f32", True, "softplus")),
]


def _dev(x):
    return {k: (None if v is None else v.cuda()) for k, v in x.items()}


def _call_noalloc(LL, d, cfg, path, out):
    return LL.lib().loglinear_fwd_noalloc(
        ctypes.c_void_p(d["q"].data_ptr()), ctypes.c_void_p(d["k"].data_ptr()),
        ctypes.c_void_p(d["v"].data_ptr()),
        None if d["log_a"] is None else ctypes.c_void_p(d["log_a"].data_ptr()),
        ctypes.c_void_p(d["lam"].data_ptr()), ctypes.c_void_p(out.data_ptr()),
        cfg.B, cfg.T, cfg.H, cfg.H, cfg.dk, cfg.dv, cfg.L, cfg.C, LL._binding._dtype_code(d["q"]),
        LL._binding._dtype_code(out), LL._binding.PATHS[path],
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("path,cfg", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_oracle_and_workspace_entry_point(path, cfg):
    """Two calls in a row on different inputs: each result against the CPU oracle (the
    definition) and against loglinear_fwd with a caller workspace (same kernels)."""
    import log_linear_attention_fwd_gb300 as LL
    tol = TOL_F32 if cfg.dtype == "f32" else TOL_BF16
    for call, seed in enumerate((11, 12)):
        x = W.make_fwd_inputs(cfg.with_(seed=seed))
        d = _dev(x)
        want_ws = LL.loglinear_fwd(d["q"], d["k"], d["v"], d["log_a"], d["lam"], cfg.C, path=path)
        got = torch.empty_like(want_ws)
        st = _call_noalloc(LL, d, cfg, path, got)
        assert st == 0, LL.status_string(st)
        torch.cuda.synchronize()
        assert LL.device_error() == 0
        want = oracle.forward_direct(x["q"], x["k"], x["v"], x["log_a"], x["lam"])
        err_oracle, err_ws = rel_l2(got.cpu(), want), rel_l2(got, want_ws)
        print(f"noalloc {path} call {call}: rel_l2 vs oracle = {err_oracle:.3e}, "
              f"vs loglinear_fwd = {err_ws:.3e}")
        assert err_oracle <= tol and err_ws <= tol


@pytest.mark.parametrize("path,cfg", CASES, ids=[c[0] for c in CASES])
def test_noalloc_allocates_no_device_memory(path, cfg):
    """After a first call (which loads the module and with it the fixed array), further
    calls leave the device's free memory exactly where it was."""
    import log_linear_attention_fwd_gb300 as LL
    d = _dev(W.make_fwd_inputs(cfg))
    out = torch.empty(cfg.B, cfg.T, cfg.H, cfg.dv, device="cuda", dtype=d["q"].dtype)
    assert _call_noalloc(LL, d, cfg, path, out) == 0
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(5):
        assert _call_noalloc(LL, d, cfg, path, out) == 0
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert LL.device_error() == 0


def test_noalloc_rejects_oversized_problem():
    import log_linear_attention_fwd_gb300 as LL
    # B1 H16 T16384 d128 needs ~192 MiB of scratch, beyond the fixed array
    big = torch.empty(16, device="cuda")
    st = LL.lib().loglinear_fwd_noalloc(
        ctypes.c_void_p(big.data_ptr()), ctypes.c_void_p(big.data_ptr()),
        ctypes.c_void_p(big.data_ptr()), None, ctypes.c_void_p(big.data_ptr()),
        ctypes.c_void_p(big.data_ptr()), 1, 16384, 16, 16, 128, 128, 15, 64, 1, 1, 0, None)
    assert st == LL._binding.LL_ERR_WORKSPACE
