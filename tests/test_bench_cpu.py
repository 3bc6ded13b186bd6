"""The benchmark's algorithmic byte and flop model (host logic, no GPU)."""
import importlib.util
import os
import sys

import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    sys.argv = ["bench.py"]
    try:
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


def test_flops_bytes_with_and_without_the_fused_gather():
    """With the row gather fused into GEMM1, the permute moves index tables
    only (no T·H·s read, no P·H·s write) and GEMM1 reads the T token rows once
    instead of the P permuted rows; flops and every other step are unchanged."""
    b = _bench()
    s = wl.CONFIGS["prism_subexpert_T8192"]
    T, H, I, E, k = s.T, s.H, s.I, s.E, s.k_max
    P, active = 147456, E
    plain = b._flops_bytes(s, P, active)
    fused = b._flops_bytes(s, P, active, True)
    assert plain["permute"]["bytes"] - fused["permute"]["bytes"] == T * H * 2 + P * H * 2
    assert plain["grouped_ffn"]["bytes"] - fused["grouped_ffn"]["bytes"] == (P - T) * H * 2
    assert plain["grouped_ffn"]["flops"] == fused["grouped_ffn"]["flops"] == 6 * H * I * P
    for step in ("route", "shared_ffn", "combine"):
        assert plain[step] == fused[step]
    # the FFN's bytes: weights of the active experts, rows in, h out and back, y out
    assert fused["grouped_ffn"]["bytes"] == active * 3 * H * I * 2 + T * H * 2 + 2 * P * I * 2 + P * H * 2
