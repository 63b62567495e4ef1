"""bench.py's bookkeeping, on the CPU: the algorithmic work the rooflines divide by, and
the e2e leg's piece schedule, and the DRAM-traffic records it reports.

The figures are the ones the measurement notes state for the 27B layer (T = 4096,
Hk = 16, Hv = 48, dk = dv = 128, 10240 conv channels) and the 256-sequence decode step.
"""
import os

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

S = dict(Hk=16, Hv=48, dk=128, dv=128)


def gemm(m, n, k):
    return 2.0 * m * n * k


def test_prefill_flops_match_the_per_chunk_products():
    """Per 64-token chunk: [K;Q]K^T per k-head; per v-head Tinv K', Tinv V' and M Vnew
    (C x C by C x d), W S, Q S and K^T Vnew (C x d by d x d), and the triangular solve."""
    C, d = 64, 128
    per_chunk = (S["Hk"] * 2 * gemm(C, C, d)
                 + S["Hv"] * (3 * gemm(C, d, C) + 3 * gemm(C, d, d))
                 + S["Hv"] * C ** 3 / 3.0)
    assert bench.prefill_flops_per_token(**S) == pytest.approx(per_chunk / C, rel=1e-12)
    assert bench.prefill_flops_per_token(**S) == pytest.approx(7.67e6, rel=2e-3)
    assert bench.prefill_flops_per_token(**S) * 4096 == pytest.approx(31.4e9, rel=2e-3)


def test_bytes_of_each_leg():
    # q, k (bf16, 16 heads), v, o (bf16, 48 heads), g, beta (fp32) and one fp32 state
    T = 4096
    act = T * (2 * 16 * 128 + 2 * 48 * 128) * 2 + T * 48 * 4 * 2
    state = 48 * 128 * 128 * 4
    assert bench.prefill_bytes(T, 1, **S) == act + state
    assert bench.prefill_bytes(T, 1, **S) == pytest.approx(138.9e6, rel=1e-3)
    # conv: x read and y written in bf16 over 10240 channels, plus the weights and tails
    assert bench.conv_bytes(T, 10240, 1) == pytest.approx(167.8e6, rel=1e-3)
    total, st = bench.decode_bytes(256, 16, 48, 128, 128, 10240)
    assert st == 2 * 256 * 48 * 128 * 128 * 4          # the state read once, written once
    assert total == pytest.approx(1.661e9, rel=1e-3)


def test_e2e_pieces_cover_the_sequence_in_chunk_multiples():
    T = 4096
    assert sum(bench.E2E_SIXTEENTHS) == 16
    pieces = [T * k // 16 for k in bench.E2E_SIXTEENTHS]
    assert sum(pieces) == T
    assert all(p % 64 == 0 and p > 0 for p in pieces)
    # the last piece is the shortest, and after the largest the pieces only shrink
    top = pieces.index(max(pieces))
    assert pieces[-1] == min(pieces)
    assert pieces[top:] == sorted(pieces[top:], reverse=True)


def test_traffic_records_match_their_sources():
    """Each DRAM-traffic record in profiles/ncu_traffic.json lists the files its kernel's
    device code comes from and their sha1; the bench reports a record only while they
    match, so a committed record must match the committed sources."""
    import hashlib
    import json
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    recs = json.load(open(path))
    assert set(recs) >= {"chunk_tc.cu", "conv1d.cu", "decode.cu"}
    for name, rec in recs.items():
        h = hashlib.sha1()
        for src in rec.get("sources", [name]):
            h.update(open(os.path.join(ROOT, "gated_deltanet_linear_11_gb300", "csrc", src),
                          "rb").read())
        assert rec["sha1"] == h.hexdigest(), name
        assert rec["dram_bytes_per_launch"] > 0
        assert bench.kernel_traffic(name) == rec["dram_bytes_per_launch"]
