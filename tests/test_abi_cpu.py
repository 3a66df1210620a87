"""C ABI checks that need no GPU: the library loads, exports every function the header
declares, and rejects bad arguments with the documented status before any launch.

Every call below is built to fail host-side validation (or to be a documented no-op),
so none of them reaches a kernel launch even on a machine with a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "loglinear.h")


@pytest.fixture(scope="module")
def L():
    from log_linear_attention_fwd_gb300 import _binding
    return _binding


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(loglinear_\w+)\s*\(", text)))


def test_header_symbols_exported(L):
    names = header_functions()
    assert len(names) >= 7
    lib = ctypes.CDLL(L.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
        assert n in L.SIGNATURES, f"{n} has no ctypes signature"


def test_version_and_status_strings(L):
    lib = L.lib()
    assert lib.loglinear_version() >= 1
    for st in range(8):
        s = lib.loglinear_status_string(st).decode()
        assert s.startswith("LL_")
    assert lib.loglinear_status_string(99).decode() == "unknown status"


FAKE = ctypes.c_void_p(0x1000)   # never dereferenced: every call here fails validation first


def fwd(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, log_a=None, lam=FAKE, out=FAKE, B=1, T=64, H=2, Hqk=None,
             dk=16, dv=16, Lv=7, chunk=16, ind=L.LL_F32, outd=L.LL_F32, path=L.LL_PATH_SIMT,
             ws=None, wsb=0, stream=None)
    a.update(kw)
    hqk = a["H"] if a["Hqk"] is None else a["Hqk"]
    return L.lib().loglinear_fwd(a["q"], a["k"], a["v"], a["log_a"], a["lam"], a["out"], a["B"],
                                 a["T"], a["H"], hqk, a["dk"], a["dv"], a["Lv"], a["chunk"],
                                 a["ind"], a["outd"], a["path"], a["ws"], a["wsb"], a["stream"])


def test_fwd_validation_codes(L):
    assert fwd(L, chunk=3) == L.LL_ERR_SHAPE
    assert fwd(L, chunk=0) == L.LL_ERR_SHAPE
    assert fwd(L, Lv=6) == L.LL_ERR_SHAPE             # T=64 needs L >= 7
    assert fwd(L, T=65, Lv=7) == L.LL_ERR_SHAPE       # T=65 needs L >= 8
    assert fwd(L, ind=7) == L.LL_ERR_DTYPE
    assert fwd(L, outd=-1) == L.LL_ERR_DTYPE
    assert fwd(L, dk=129) == L.LL_ERR_UNSUPPORTED
    assert fwd(L, dv=0) == L.LL_ERR_INVALID
    assert fwd(L, B=-1) == L.LL_ERR_INVALID
    assert fwd(L, path=9) == L.LL_ERR_INVALID
    assert fwd(L, q=None) == L.LL_ERR_INVALID
    assert fwd(L, lam=None) == L.LL_ERR_INVALID
    assert fwd(L, ws=None, wsb=0) == L.LL_ERR_WORKSPACE
    assert fwd(L, ws=FAKE, wsb=16) == L.LL_ERR_WORKSPACE
    # tensor-core path: misaligned q (after every size check passed) -> LL_ERR_ALIGN
    assert fwd(L, dk=128, dv=128, ind=L.LL_BF16, outd=L.LL_BF16, path=L.LL_PATH_TC,
               q=ctypes.c_void_p(0x1002), ws=FAKE, wsb=1 << 40) == L.LL_ERR_ALIGN
    assert fwd(L, dk=64, dv=64, ind=L.LL_BF16, path=L.LL_PATH_TC) == L.LL_ERR_UNSUPPORTED
    assert fwd(L, dk=128, dv=128, ind=L.LL_F32, path=L.LL_PATH_TC) == L.LL_ERR_UNSUPPORTED
    # q/k heads: 1 <= Hqk <= H, H a multiple of Hqk
    assert fwd(L, H=6, Hqk=4) == L.LL_ERR_SHAPE
    assert fwd(L, H=2, Hqk=4) == L.LL_ERR_SHAPE
    assert fwd(L, H=2, Hqk=0) == L.LL_ERR_SHAPE
    assert fwd(L, H=2, Hqk=-1) == L.LL_ERR_INVALID
    assert fwd(L, H=6, Hqk=3, ws=None, wsb=0) == L.LL_ERR_WORKSPACE   # valid grouping
    assert fwd(L, H=6, Hqk=1, ws=None, wsb=0) == L.LL_ERR_WORKSPACE
    # empty problems are no-ops, even with null pointers
    for kw in (dict(B=0), dict(T=0), dict(H=0), dict(H=0, Hqk=0)):
        assert fwd(L, q=None, k=None, v=None, lam=None, out=None, **kw) == L.LL_OK


def test_prefill_validation_codes(L):
    def pre(state, **kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, log_a=None, lam=FAKE, out=FAKE, B=1, T=64, H=2, Hqk=2,
                 dk=16, dv=16, Lv=7, chunk=16, ind=L.LL_F32, outd=L.LL_F32, path=L.LL_PATH_SIMT,
                 ws=None, wsb=0, stream=None)
        a.update(kw)
        return L.lib().loglinear_prefill(a["q"], a["k"], a["v"], a["log_a"], a["lam"], a["out"],
                                         state, a["B"], a["T"], a["H"], a["Hqk"], a["dk"], a["dv"],
                                         a["Lv"], a["chunk"], a["ind"], a["outd"], a["path"],
                                         a["ws"], a["wsb"], a["stream"])
    assert pre(None) == L.LL_ERR_INVALID
    assert pre(ctypes.c_void_p(0x1002)) == L.LL_ERR_ALIGN
    # the forward's own validation applies unchanged
    assert pre(FAKE, chunk=3) == L.LL_ERR_SHAPE
    assert pre(FAKE, Lv=6) == L.LL_ERR_SHAPE
    assert pre(FAKE, ws=None, wsb=0) == L.LL_ERR_WORKSPACE
    assert pre(FAKE, B=0, q=None, k=None, v=None, lam=None, out=None) == L.LL_OK
    assert pre(FAKE, Hqk=3) == L.LL_ERR_SHAPE
    assert pre(FAKE, T=0, Hqk=3) == L.LL_ERR_SHAPE      # checked before the empty-prompt path


def test_workspace_size_and_paths(L):
    sz = L.fwd_workspace_size(1, 64, 2, 16, 16, 16, L.LL_F32, "simt")
    n_states = 1 * 2 * 4 * 16 * 16
    assert sz >= 2 * n_states * 4
    with pytest.raises(L.LoglinearError):
        L.fwd_workspace_size(1, 64, 2, 16, 16, 24, L.LL_F32, "simt")
    assert L.resolve_path(64, 64, 64, L.LL_F32) == "simt"
    assert L.resolve_path(128, 128, 64, L.LL_F32) == "simt"
    assert L.resolve_path(128, 128, 64, L.LL_BF16) == "tc"
    assert L.resolve_path(128, 128, 128, L.LL_BF16) == "tc"
    assert L.resolve_path(128, 128, 256, L.LL_BF16) == "tc"
    assert L.resolve_path(128, 64, 64, L.LL_BF16) == "tc"      # the d_v = 64 instance
    assert L.resolve_path(128, 96, 64, L.LL_BF16) == "simt"
    assert L.resolve_path(64, 128, 64, L.LL_BF16) == "simt"
    assert L.resolve_path(64, 64, 256, L.LL_F32) == "simt"
    # the fp32 path tiles at min(C, 64): C = 256 needs the workspace of C = 64
    assert L.fwd_workspace_size(1, 1000, 2, 16, 16, 256, L.LL_F32) == \
        L.fwd_workspace_size(1, 1000, 2, 16, 16, 64, L.LL_F32)
    assert L.resolve_path(64, 64, 64, L.LL_BF16) == "simt"
    with pytest.raises(L.LoglinearError):
        L.resolve_path(64, 64, 64, L.LL_BF16, "tc")
    # tensor-core workspace: bf16 chunk states + bf16 block states, 128-token tiles
    tc = L.fwd_workspace_size(1, 16384, 16, 128, 128, 64, L.LL_BF16, "tc")
    assert tc >= 16 * 128 * 128 * 128 * (2 + 2)


def dec(L, **kw):
    a = dict(state=FAKE, q=FAKE, k=FAKE, v=FAKE, log_a=None, lam=FAKE, t=5, out=FAKE, B=2, H=2,
             Hqk=2, dk=16, dv=16, Lv=4, ind=L.LL_F32, outd=L.LL_F32, stream=None)
    a.update(kw)
    return L.lib().loglinear_decode_step(a["state"], a["q"], a["k"], a["v"], a["log_a"], a["lam"],
                                         a["t"], a["out"], a["B"], a["H"], a["Hqk"], a["dk"],
                                         a["dv"], a["Lv"], a["ind"], a["outd"], a["stream"])


def test_decode_validation_codes(L):
    assert dec(L, t=-1) == L.LL_ERR_INVALID
    assert dec(L, t=8, Lv=4) == L.LL_ERR_SHAPE       # t=8 reaches level 4 -> L >= 5
    assert dec(L, dv=12) == L.LL_ERR_UNSUPPORTED     # dv must be a power of two
    assert dec(L, dv=2) == L.LL_ERR_UNSUPPORTED
    assert dec(L, dk=200) == L.LL_ERR_UNSUPPORTED
    assert dec(L, ind=5) == L.LL_ERR_DTYPE
    assert dec(L, state=None) == L.LL_ERR_INVALID
    assert dec(L, out=None) == L.LL_ERR_INVALID
    assert dec(L, state=ctypes.c_void_p(0x1004)) == L.LL_ERR_ALIGN
    assert dec(L, B=0, state=None) == L.LL_OK
    assert dec(L, H=4, Hqk=3) == L.LL_ERR_SHAPE
    assert dec(L, Hqk=0) == L.LL_ERR_SHAPE


def test_gdn_decode_validation_codes(L):
    """The Gated DeltaNet decode step checks its arguments before touching the GPU."""
    f = L.lib().loglinear_gdn_decode_step
    p = ctypes.c_void_p(16)  # never dereferenced: every call below fails validation first
    ok = dict(state=p, q=p, k=p, v=p, log_a=None, beta=p, lam=p, t=5, out=p, B=1, H=2, Hqk=2,
              dk=8, dv=8, L=4, i=0, o=0, s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["state"], a["q"], a["k"], a["v"], a["log_a"], a["beta"], a["lam"], a["t"],
                 a["out"], a["B"], a["H"], a["Hqk"], a["dk"], a["dv"], a["L"], a["i"], a["o"], a["s"])

    assert call(beta=None) == L.LL_ERR_INVALID
    assert call(t=-1) == L.LL_ERR_INVALID
    assert call(L=2, t=5) == L.LL_ERR_SHAPE          # t = 5 needs L >= 4
    assert call(Hqk=3) == L.LL_ERR_SHAPE
    assert call(dv=12) == L.LL_ERR_UNSUPPORTED        # d_v not a power of two
    assert call(dk=129) == L.LL_ERR_UNSUPPORTED
    assert call(i=7) == L.LL_ERR_DTYPE
    assert call(state=ctypes.c_void_p(24)) == L.LL_ERR_ALIGN
    assert call(B=0) == L.LL_OK                       # empty: nothing to do


def test_fwd_strided_validation_codes(L):
    """Bad strides are refused on the host before any launch."""
    f = L.lib().loglinear_fwd_strided
    p = ctypes.c_void_p(256)  # never dereferenced: every call below fails validation first
    ws = ctypes.c_void_p(1 << 20)

    def S(b, t, h):
        return ctypes.byref(L.LLStrides(b, t, h))

    B, T, H, d = 2, 64, 4, 128
    def call(qs=None, os_=None, path=0, out_dtype=1):
        ss = L.fwd_workspace_size(B, T, H, d, d, 64, 1, {0: "auto", 1: "simt", 2: "tc"}[path])
        return f(p, qs, p, None, p, None, None, p, p, os_, B, T, H, H, d, d, 7, 64, 1, out_dtype,
                 path, ws, ss, None)

    assert call(qs=S(-1, d * H, d)) == L.LL_ERR_INVALID                 # negative stride
    assert call(os_=S(T * H * d, H * d, d - 1)) == L.LL_ERR_INVALID     # heads overlap
    assert call(os_=S(T * H * d, d, d)) == L.LL_ERR_INVALID             # positions hit heads
    assert call(qs=S(T * H * 3 * d + 4, H * 3 * d, 3 * d), path=2) == L.LL_ERR_ALIGN
    assert call(qs=S(T * H * 3 * d, H * 3 * d, 0), path=2) == L.LL_ERR_UNSUPPORTED


def test_level_map_validation(L):
    lib = L.lib()
    assert lib.loglinear_debug_level_map(-1, 16, 0, FAKE, None) == L.LL_ERR_INVALID
    assert lib.loglinear_debug_level_map(16, 16, 0, None, None) == L.LL_ERR_INVALID
    assert lib.loglinear_debug_level_map(16, 12, 0, FAKE, None) == L.LL_ERR_SHAPE
    assert lib.loglinear_debug_level_map(0, 16, 0, None, None) == L.LL_OK
    assert lib.loglinear_device_error(None, None) == L.LL_ERR_INVALID


def test_binding_rejects_host_tensors(L):
    import torch
    q = torch.zeros(1, 8, 1, 4)
    with pytest.raises(ValueError):
        L.loglinear_fwd(q, q, q, None, torch.zeros(1, 8, 1, 4), 4)


def test_bwd_validation_codes(L):
    def bwd(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, log_a=None, lam=FAKE, dout=FAKE, dq=FAKE, dk=FAKE,
                 dv=FAKE, dla=None, dlam=FAKE, B=1, T=64, H=2, Hqk=2, dkd=16, dvd=16, Lv=7,
                 ind=L.LL_F32, gd=L.LL_F32, path=L.LL_PATH_AUTO, fws=None, fwsb=0, ws=None,
                 wsb=0, stream=None)
        a.update(kw)
        return L.lib().loglinear_bwd(a["q"], a["k"], a["v"], a["log_a"], a["lam"], a["dout"],
                                     a["dq"], a["dk"], a["dv"], a["dla"], a["dlam"], a["B"],
                                     a["T"], a["H"], a["Hqk"], a["dkd"], a["dvd"], a["Lv"],
                                     a["ind"], a["gd"], a["path"], a["fws"], a["fwsb"],
                                     a["ws"], a["wsb"], a["stream"])
    assert bwd(Lv=6) == L.LL_ERR_SHAPE                  # T=64 needs L >= 7
    assert bwd(H=4, Hqk=3) == L.LL_ERR_SHAPE
    assert bwd(ind=3) == L.LL_ERR_DTYPE
    assert bwd(gd=-1) == L.LL_ERR_DTYPE
    assert bwd(dkd=129) == L.LL_ERR_UNSUPPORTED
    assert bwd(dvd=0) == L.LL_ERR_INVALID
    assert bwd(dq=None) == L.LL_ERR_INVALID
    assert bwd(dlam=None) == L.LL_ERR_INVALID
    assert bwd(log_a=FAKE, dla=None) == L.LL_ERR_INVALID   # d log a wanted with a decay
    assert bwd(path=7) == L.LL_ERR_INVALID
    assert bwd(path=L.LL_PATH_TC) == L.LL_ERR_UNSUPPORTED   # fp32, d 16: no tensor-core dQ
    assert bwd(path=L.LL_PATH_TC, dkd=128, dvd=64, ind=L.LL_BF16, gd=L.LL_F32) == \
        L.LL_ERR_UNSUPPORTED                                 # dO must be bf16 as well
    tc_kw = dict(dkd=128, dvd=64, ind=L.LL_BF16, gd=L.LL_BF16, ws=FAKE, wsb=1 << 40)
    assert bwd(path=L.LL_PATH_TC, q=ctypes.c_void_p(0x1002), **tc_kw) == L.LL_ERR_ALIGN
    assert bwd(path=L.LL_PATH_TC, dv=ctypes.c_void_p(0x1008), **tc_kw) == L.LL_ERR_ALIGN
    # a forward's workspace: tensor-core path only, large enough, 256-byte aligned
    assert bwd(fws=FAKE, fwsb=1 << 40) == L.LL_ERR_UNSUPPORTED
    assert bwd(path=L.LL_PATH_TC, fws=FAKE, fwsb=16, **tc_kw) == L.LL_ERR_WORKSPACE
    assert bwd(path=L.LL_PATH_TC, fws=ctypes.c_void_p(0x1010), fwsb=1 << 40, **tc_kw) == \
        L.LL_ERR_ALIGN
    assert bwd() == L.LL_ERR_WORKSPACE
    assert bwd(ws=ctypes.c_void_p(0x1010), wsb=1 << 40) == L.LL_ERR_ALIGN
    assert bwd(T=0, q=None, k=None, v=None, lam=None, dout=None, dq=None, dk=None, dv=None,
               dlam=None) == L.LL_OK
    # nothing to compute: a forward's workspace given to an empty call is not an error
    assert bwd(T=0, path=L.LL_PATH_TC, fws=FAKE, fwsb=1 << 40, **tc_kw) == L.LL_OK
    sz = L.bwd_workspace_size(1, 64, 2, 2, 16, 16, 7, L.LL_F32, L.LL_F32)
    assert sz >= 2 * (1 * 2 * 2 * 16 * 16 * 4) + 2 * 64 * 2 * 16 * 4   # states + per-head dq, dk
    # the tensor-core path: fp32 mirrored states and a forward's bf16 states on the eight
    # 128-token tiles (its states-only form writes no output, so there is no output
    # scratch), and with shared q/k one fp32 dq and dk per q/k head
    tc = L.bwd_workspace_size(1, 1000, 2, 2, 128, 64, 11, L.LL_BF16, L.LL_BF16, "tc")
    st = 2 * 8 * 128 * 64
    assert st * 4 + 2 * st * 2 <= tc < st * 4 + 2 * st * 2 + 1000 * 2 * 64 * 2
    tc1 = L.bwd_workspace_size(1, 1000, 2, 1, 128, 64, 11, L.LL_BF16, L.LL_BF16, "tc")
    assert tc1 >= tc + 2 * 1000 * 1 * 128 * 4
    assert L.bwd_workspace_size(1, 1000, 2, 2, 128, 64, 11, L.LL_BF16, L.LL_BF16) == tc


def test_gdn_fwd_validation_codes(L):
    """The Gated DeltaNet forward checks its arguments before touching the GPU."""
    f = L.lib().loglinear_gdn_fwd
    p = ctypes.c_void_p(16)  # never dereferenced: every call below fails validation first
    ok = dict(q=p, k=p, v=p, log_a=None, beta=p, lam=p, out=p, state=None, B=1, T=100, H=2,
              Hqk=2, dk=8, dv=8, L=8, i=0, o=0, s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["k"], a["v"], a["log_a"], a["beta"], a["lam"], a["out"], a["state"],
                 a["B"], a["T"], a["H"], a["Hqk"], a["dk"], a["dv"], a["L"], a["i"], a["o"], a["s"])

    assert call(beta=None) == L.LL_ERR_INVALID
    assert call(T=-1) == L.LL_ERR_INVALID
    assert call(L=7) == L.LL_ERR_SHAPE                # T = 100 needs L >= 8
    assert call(Hqk=3) == L.LL_ERR_SHAPE
    assert call(dk=129) == L.LL_ERR_UNSUPPORTED
    assert call(dv=129) == L.LL_ERR_UNSUPPORTED
    assert call(L=65) == L.LL_ERR_UNSUPPORTED
    assert call(dk=7, i=1) == L.LL_ERR_UNSUPPORTED    # bf16 rows of odd length
    assert call(o=5) == L.LL_ERR_DTYPE
    assert call(q=ctypes.c_void_p(18)) == L.LL_ERR_ALIGN
    assert call(state=ctypes.c_void_p(19)) == L.LL_ERR_ALIGN
    assert call(B=0) == L.LL_OK                       # empty: nothing to do
    assert call(H=0, Hqk=0) in (L.LL_OK, L.LL_ERR_SHAPE)


def test_gdn_fwd_chunked_validation_codes(L):
    """The chunked Gated DeltaNet forward checks its arguments before touching the GPU."""
    f = L.lib().loglinear_gdn_fwd_chunked
    p = ctypes.c_void_p(16)  # never dereferenced: every call below fails validation first
    need = L.gdn_fwd_chunked_workspace_size(1, 100, 2, 8, 8)
    ok = dict(q=p, k=p, v=p, log_a=None, beta=p, lam=p, out=p, state=None, B=1, T=100, H=2,
              Hqk=2, dk=8, dv=8, L=8, i=0, o=0, ws=ctypes.c_void_p(256), wsb=need - 1, s=None)

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["k"], a["v"], a["log_a"], a["beta"], a["lam"], a["out"], a["state"],
                 a["B"], a["T"], a["H"], a["Hqk"], a["dk"], a["dv"], a["L"], a["i"], a["o"],
                 a["ws"], a["wsb"], a["s"])

    assert need >= 4 * (100 * 2 * 8 + 2 * 2 * 64 * 8 + 2 * 2 * 8 * 8 + 2 * 2 * 8 * 8)
    assert call(beta=None, wsb=need) == L.LL_ERR_INVALID
    assert call(T=-1) == L.LL_ERR_INVALID
    assert call(L=7) == L.LL_ERR_SHAPE                # T = 100 needs L >= 8
    assert call(Hqk=3) == L.LL_ERR_SHAPE
    assert call(dk=129) == L.LL_ERR_UNSUPPORTED
    assert call(o=5) == L.LL_ERR_DTYPE
    assert call() == L.LL_ERR_WORKSPACE               # one byte short
    assert call(wsb=need, ws=ctypes.c_void_p(272)) == L.LL_ERR_ALIGN
    assert call(wsb=need, state=ctypes.c_void_p(258)) == L.LL_ERR_ALIGN
    assert call(wsb=need, state=p, q=ctypes.c_void_p(18)) == L.LL_ERR_ALIGN
    assert call(wsb=need, state=p, dk=7, i=1) == L.LL_ERR_UNSUPPORTED  # bf16 rows, odd d_k
    assert call(T=0) == L.LL_OK                       # empty: nothing to do
