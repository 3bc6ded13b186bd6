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


def test_route_executed_flops_and_stage_net_fractions():
    """An fp32 router weight on bf16 activations executes three bf16 GEMMs (its
    exact split); a bf16 one executes one.  With the event-pair overhead given,
    each stage also reports its time and fractions less it."""
    b = _bench()
    prism, qwen = wl.CONFIGS["prism_subexpert_T8192"], wl.CONFIGS["qwen3_30b_a3b_T16384"]
    fp = b._flops_bytes(prism, 147456, prism.E)["route"]
    fq = b._flops_bytes(qwen, qwen.T * qwen.k, qwen.E)["route"]
    assert fp["flops_executed"] == 3 * fp["flops"] == 3 * 2 * prism.T * prism.H * prism.E
    assert fq["flops_executed"] == fq["flops"]
    peaks = {"hbm_gbs": 1000.0, "bf16_tflops": 1000.0, "bf16_tflops_sustained": 900.0, "source": "test"}
    stages = {"route": 0.05, "permute": 0.02, "grouped_ffn": 0.6, "combine": 0.1}
    _, st = b._roofline_and_stages(prism, 147456, prism.E, True, stages, peaks, event_ms=0.004)
    r = st["route"]
    assert abs(r["ms_net"] - 0.046) < 1e-12
    assert abs(r["frac_hbm_net"] * 0.046 - r["frac_hbm"] * 0.05) < 1e-12
    assert abs(r["frac_tensor_executed"] - 3 * r["frac_tensor"]) < 1e-12
    _, st0 = b._roofline_and_stages(prism, 147456, prism.E, True, stages, peaks)
    assert "ms_net" not in st0["combine"] and "frac_hbm_net" not in st0["combine"]
