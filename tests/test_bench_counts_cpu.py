"""The bench's roofline arithmetic on the CPU: the algorithmic bytes and FLOPs it divides
by the measured times, checked against counts built from the oracle's Fenwick level
function by brute force, and the guard that drops a recorded DRAM traffic figure once the
kernel's source has changed."""
import json
import os
import shutil

import pytest

import bench
import oracle
import workloads as W


def _inter_levels_of_chunk(j: int, C: int) -> int:
    """Distinct levels above the intra-chunk ones that the queries of chunk j see in the
    earlier chunks (Log-Linear Attention, the Fenwick partition of the prefix): every
    query of the chunk sees the same set, so the first query is enough."""
    t = j * C
    return len({oracle.level(t, s) for s in range(t)} - set(range(C.bit_length())))


@pytest.mark.parametrize("T,C,dk,dv", [(256, 16, 8, 4), (512, 64, 16, 32), (96, 8, 4, 4)])
def test_forward_counts_match_brute_force(T, C, dk, dv):
    cfg = W.FwdConfig("count", 2, 3, T, dk, dv, C, (T - 1).bit_length() + 1, "bf16", True,
                      "softplus")
    nbytes, flops = bench.fwd_algorithmic(cfg)
    N = T // C
    pairs = sum(1 for j in range(N) for t in range(C) for s in range(t + 1))
    readouts = sum(_inter_levels_of_chunk(j, C) for j in range(N))
    want_flops = cfg.B * cfg.H * (pairs * 2 * (dk + dv) + N * 2 * C * dk * dv
                                  + readouts * 2 * C * dk * dv)
    assert flops == want_flops
    tok = cfg.B * T * cfg.H
    # q, k, v, out in bf16; log a and lambda in fp32
    assert nbytes == tok * (2 * dk + 2 * dv) * 2 + tok * 4 + tok * cfg.L * 4


def test_headline_counts():
    """The headline forward moves 272 MiB (q, k, v, out 64 MiB each in bf16, lambda 15 MiB,
    log a 1 MiB) and does 47.3 GFLOP at C = 64."""
    nbytes, flops = bench.fwd_algorithmic(W.FWD_CONFIGS["mamba2_T16384"])
    assert nbytes == 272 * 2**20
    assert abs(flops / 1e9 - 47.31) < 0.01


def test_shared_qk_bytes_count_qk_once():
    """With one q/k head for 48 value heads, q and k are read once per token, not once
    per value head."""
    cfg = W.FWD_CONFIGS["mva_B2H48_T16384"]
    nbytes, _ = bench.fwd_algorithmic(cfg)
    tok = cfg.B * cfg.T
    assert nbytes == tok * 2 * cfg.dk * 2 + tok * cfg.H * (2 * cfg.dv * 2 + 4 + cfg.L * 4)


@pytest.mark.parametrize("t", [12345, 12344, 12288, 8192, 1, 2, 3])
def test_decode_bytes_match_level_sets(t):
    """Levels read: those holding data after t-1 (a level that some s <= t-1 reaches from
    t-1); levels written: every one of those (each is decayed, merged or cleared) plus the
    one that receives the merge (a level reached from t that was empty before)."""
    L = 15
    cfg = W.DecodeConfig("count", 4, 2, 8, 8, L, t)
    pre = {oracle.level(t - 1, s) for s in range(t)}
    post = {oracle.level(t, s) for s in range(t + 1)}
    written = pre | post
    assert bench.decode_algorithmic(cfg) == cfg.B * cfg.H * 8 * 8 * 4 * (len(pre) + len(written))


def test_decode_headline_bytes():
    """At t = 12345 the step reads 6 levels and writes 7 (64 KiB each, B128 H16)."""
    assert bench.decode_algorithmic(W.DECODE_CONFIG) == 128 * 16 * 65536 * 13


def test_traffic_record_dropped_when_source_changes(tmp_path, monkeypatch):
    rec_path = os.path.join(bench.ROOT, "profiles", "traffic_tc_forward_T16384.json")
    with open(rec_path) as f:
        rec = json.load(f)
    # a copy of the tree the record names, at the recorded state
    os.makedirs(tmp_path / "profiles")
    shutil.copy(rec_path, tmp_path / "profiles")
    for src in rec["source_files"]:
        os.makedirs(tmp_path / os.path.dirname(src), exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, src), tmp_path / src)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    want = rec["dram_bytes_read"] + rec["dram_bytes_write"]
    got = bench.load_traffic("tc_forward_kernel")
    if got is None:
        pytest.skip("the kernel's source changed since the record was taken")
    assert got == want
    with open(tmp_path / rec["source_files"][0], "a") as f:
        f.write("\n// edited\n")
    assert bench.load_traffic("tc_forward_kernel") is None
    assert bench.load_traffic("no_such_kernel") is None


@pytest.mark.parametrize("T,dk,dv", [(512, 8, 4), (1024, 16, 8)])
def test_backward_counts_match_brute_force(T, dk, dv):
    """The backward at C = 64: per causal pair in a chunk q.k, dO.v and the dQ, dK, dV
    updates; per chunk the recomputed state; per (chunk, inter level) the dQ readout with
    its dlambda dot, the mirrored part and the dK, dV readouts.  Bytes: the forward's
    inputs and dO read once, their gradients written once."""
    C = 64
    cfg = W.FwdConfig("count", 1, 2, T, dk, dv, C, (T - 1).bit_length() + 1, "bf16", True,
                      "softplus")
    nbytes, flops = bench.bwd_algorithmic(cfg)
    N = T // C
    pairs = sum(1 for j in range(N) for t in range(C) for s in range(t + 1))
    inter = sum(_inter_levels_of_chunk(j, C) for j in range(N))
    per_pair = 2 * dk + 2 * dv + 2 * dk + 2 * dk + 2 * dv
    per_level = 4 * 2 * C * dk * dv + 2 * C * dk
    assert flops == cfg.B * cfg.H * (pairs * per_pair + N * 2 * C * dk * dv + inter * per_level)
    tok = cfg.B * T * cfg.H
    assert nbytes == 2 * (tok * (2 * dk + 2 * dv) * 2 + tok * 4 + tok * cfg.L * 4)
