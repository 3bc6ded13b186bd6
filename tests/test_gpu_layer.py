"""Whole-layer parity of the CUDA path with the oracle on every workload:
small versions (spanning several tiles with ragged tails) compared element by
element in full, and the full-size layers compared on every integer output
plus a seeded sample of tokens for the float outputs."""
import pytest

import workloads as wl
from parity_utils import check_layer_full, check_layer_sampled, run_gpu

pytestmark = pytest.mark.gpu

SMALL = [
    ("tiny_fp32_T256_E8", {}),
    ("tiny_fp32_T256_E8", dict(T=1)),
    ("tiny_fp32_T256_E8", dict(T=77, k=8)),                                    # k = E: dense mixture
    ("tiny_fp32_T256_E8", dict(T=50, E=1, k=1, R=1)),                          # plain SwiGLU MLP
    ("dsv2lite_prefill_T4096", dict(T=300, H=256, I=160, I_shared=320, V=3000)),
    ("dsv2lite_decode_T64", dict(H=256, I=160, I_shared=320, V=3000)),
    ("qwen3_30b_a3b_T16384", dict(T=515, H=256, I=96, V=3000)),
    ("prism_subexpert_T8192", dict(T=512, H=256, I=40, V=3000, tokens_per_request=64)),
]


@pytest.mark.parametrize("fused_gather", [True, False], ids=["gather", "x_perm"])
@pytest.mark.parametrize("name,over", SMALL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(SMALL)])
def test_layer_small(name, over, fused_gather):
    """Both ways into the expert GEMM: GEMM1 gathering x rows, and the permute
    writing x_perm (compared with the oracle's permuted rows)."""
    d = wl.make_inputs(wl.scaled(name, **over))
    res, P = run_gpu(d, fused_gather=fused_gather)
    assert (res.x_perm is None) == fused_gather
    check_layer_full(d, res, P)


FULL = ["tiny_fp32_T256_E8", "dsv2lite_decode_T64", "dsv2lite_decode_T256", "dsv2lite_decode_T512",
        "dsv2lite_prefill_T4096", "qwen3_30b_a3b_T16384", "prism_subexpert_T8192"]


@pytest.mark.parametrize("seed", range(8))
def test_layer_random_small(seed):
    """Seeded random small layers on the four model shapes (token count, hidden
    and intermediate sizes drawn at random, rows gathered in GEMM1 or copied by
    the permute), compared with the oracle element by element."""
    import numpy as np
    rng = np.random.default_rng(700 + seed)
    name = ["dsv2lite_prefill_T4096", "qwen3_30b_a3b_T16384", "prism_subexpert_T8192",
            "dsv2lite_decode_T64"][seed % 4]
    h_lo = max(2, (wl.CONFIGS[name].E + 7) // 8)  # biased routing builds E orthonormal router rows: H >= E
    over = dict(T=int(rng.integers(1, 700)), H=int(rng.integers(h_lo, 65)) * 8, I=int(rng.integers(1, 65)) * 8,
                V=3000)
    if wl.CONFIGS[name].I_shared:
        over["I_shared"] = int(rng.integers(1, 65)) * 8
    if wl.CONFIGS[name].k_choices:
        over["tokens_per_request"] = int(rng.integers(1, 80))
    d = wl.make_inputs(wl.scaled(name, **over))
    res, P = run_gpu(d, fused_gather=bool(seed % 2))
    check_layer_full(d, res, P)


@pytest.mark.parametrize("name", FULL)
def test_layer_full_size(name):
    d = wl.make_inputs(wl.CONFIGS[name])
    res, P = run_gpu(d)
    check_layer_sampled(d, res, P)


def test_layer_full_size_fused_gather():
    """The MoE-Prism layer at full size through the path its layer takes by
    default (GEMM1 gathering x rows, no x_perm), on the same sampled checks."""
    d = wl.make_inputs(wl.CONFIGS["prism_subexpert_T8192"])
    res, P = run_gpu(d, fused_gather=True)
    assert res.x_perm is None
    check_layer_sampled(d, res, P)


def _layer(d):
    from token_expert_routing_gb300 import MoELayer
    s = d["spec"]
    return MoELayer(d["w_router"], d["w13"], d["w2"], d["expert_rank"], d["lut"], s.R, s.k_max, d["ws13"], d["ws2"])


@pytest.mark.parametrize("name,over,fused", [
    ("prism_subexpert_T8192", dict(T=256, H=256, V=3000, tokens_per_request=64), True),        # I = 352
    ("prism_subexpert_T8192", dict(T=256, H=256, I=384, V=3000, tokens_per_request=64), True),
    ("prism_subexpert_T8192", dict(T=256, H=256, I=392, V=3000, tokens_per_request=64), False),
    ("qwen3_30b_a3b_T16384", dict(T=256, H=256, V=3000), False),                                # I = 768
    ("tiny_fp32_T256_E8", {}, False),                                                           # fp32 experts
])
def test_layer_fused_gather_default(name, over, fused):
    """Left unset, the permute is fused into GEMM1 exactly for bf16 experts with
    I <= 384 (each x row gathered for at most 3 GEMM1 output tiles), and the
    forward then writes no x_perm."""
    import torch
    d = wl.make_inputs(wl.scaled(name, **over))
    layer = _layer(d)
    assert layer.fused_gather == fused
    s = d["spec"]
    kpt = d["k_per_token"].cuda() if s.k_choices else None
    res = layer.forward(d["x"].cuda(), d["token_ids"].cuda(), kpt, None if s.k_choices else s.k,
                        int(d["k_per_token"].sum()))
    torch.cuda.synchronize()
    assert (res.x_perm is None) == fused


@pytest.mark.parametrize("name", ["dsv2lite_decode_T64", "prism_subexpert_T8192"])
def test_captured_graph_matches_eager(name):
    """A CUDA-graph replay of the layer gives the eager forward's bits, also
    after new inputs are written into the static buffers."""
    import torch
    from token_expert_routing_gb300 import CapturedLayer
    spec = wl.CONFIGS[name]
    if name.startswith("prism"):
        spec = wl.scaled(name, T=1024, tokens_per_request=32)
    d = wl.make_inputs(spec)
    layer = _layer(d)
    per_token = bool(spec.k_choices)
    cap = CapturedLayer(layer, spec.T, None if per_token else spec.k,
                        d["k_per_token"] if per_token else None)
    for seed in (0, 1):
        x = d["x"] if seed == 0 else d["x"].flip(0).contiguous()
        ids = d["token_ids"] if seed == 0 else d["token_ids"].flip(0).contiguous()
        cap.x.copy_(x)
        cap.token_ids.copy_(ids)
        got = cap.replay()
        kpt = d["k_per_token"].cuda() if per_token else None
        want = layer.forward(x.cuda(), ids.cuda(), kpt, None if per_token else spec.k,
                             int(d["k_per_token"].sum()))
        torch.cuda.synchronize()
        for key in ("out", "topk_idx", "pair_to_sorted", "counts"):
            assert torch.equal(getattr(got, key), getattr(want, key)), key


def test_host_pipeline_matches_forward():
    """The overlapped host-buffer path returns each call's own output."""
    import torch
    from token_expert_routing_gb300 import HostPipeline
    spec = wl.scaled("dsv2lite_prefill_T4096", T=512, H=256, I=160, I_shared=320, V=3000)
    d = wl.make_inputs(spec)
    layer = _layer(d)
    pipe = HostPipeline(layer)
    xs = [d["x"], d["x"].flip(0).contiguous(), (d["x"] * 0.5).contiguous()]
    outs = [torch.empty(spec.T, spec.H, dtype=d["x"].dtype).pin_memory() for _ in xs]
    ids = d["token_ids"].pin_memory()
    for x, o in zip(xs, outs):
        pipe.submit(x.pin_memory(), ids, o, k=spec.k)
    pipe.synchronize()
    for x, o in zip(xs, outs):
        want = layer.forward(x.cuda(), ids.cuda(), k=spec.k).out.cpu()
        assert torch.equal(o, want)


@pytest.mark.parametrize("name,over", [("dsv2lite_prefill_T4096", dict(T=512, H=256, I=160, I_shared=320, V=3000)),
                                       ("prism_subexpert_T8192", dict(T=512, H=256, I=40, V=3000,
                                                                      tokens_per_request=64))])
def test_graph_pipeline_matches_forward(name, over):
    """Host-buffer calls through the two captured graphs return each call's
    own output (five calls, so both slots are reused), equal to the eager
    forward; per-token budgets included."""
    import torch
    from token_expert_routing_gb300 import GraphPipeline
    spec = wl.scaled(name, **over)
    d = wl.make_inputs(spec)
    layer = _layer(d)
    per_token = bool(spec.k_choices)
    gp = GraphPipeline(layer, spec.T, None if per_token else spec.k, d["k_per_token"] if per_token else None)
    gen = torch.Generator().manual_seed(5)
    xs = [(d["x"].float() * (0.5 + i) + 0.1 * torch.randn(d["x"].shape, generator=gen)).to(d["x"].dtype)
          for i in range(5)]
    idss = [d["token_ids"].roll(i) for i in range(5)]
    outs = [torch.empty(spec.T, spec.H, dtype=d["x"].dtype).pin_memory() for _ in xs]
    for x, ids, o in zip(xs, idss, outs):
        gp.submit(x.pin_memory(), ids.pin_memory(), o)
    gp.synchronize()
    kpt = d["k_per_token"].cuda() if per_token else None
    P = int(d["k_per_token"].sum())
    for x, ids, o in zip(xs, idss, outs):
        want = layer.forward(x.cuda(), ids.cuda(), kpt, None if per_token else spec.k, P).out.cpu()
        assert torch.equal(o, want)


def test_layer_empty_batch():
    """A forward over no tokens returns an empty output and flags nothing."""
    from token_expert_routing_gb300 import MoELayer, _abi
    d = wl.make_inputs(wl.scaled("dsv2lite_prefill_T4096", T=64, H=256, I=160, I_shared=320, V=3000))
    s = d["spec"]
    layer = MoELayer(d["w_router"], d["w13"], d["w2"], d["expert_rank"], d["lut"], s.R, s.k_max, d["ws13"], d["ws2"])
    x = d["x"][:0].cuda()
    res = layer.forward(x, d["token_ids"][:0].cuda(), None, s.k, 0)
    assert _abi.semmoe_check_errors() == 0
    assert tuple(res.out.shape) == (0, s.H)


FOLDED = [s for s in SMALL if not s[0].startswith("tiny_fp32")]   # bf16 experts


@pytest.mark.parametrize("fused_gather", [True, False], ids=["gather", "x_perm"])
@pytest.mark.parametrize("name,over", FOLDED, ids=[f"{n}-{i}" for i, (n, _) in enumerate(FOLDED)])
def test_layer_small_folded_combine(name, over, fused_gather):
    """The layer with GEMM2 adding its gate-weighted rows straight into the
    token order (no y_perm), against the oracle in full: every integer output
    bit-exact, the output within the bf16 tolerance."""
    d = wl.make_inputs(wl.scaled(name, **over))
    res, P = run_gpu(d, fused_gather=fused_gather, fused_combine=True)
    assert res.y_perm is None
    check_layer_full(d, res, P)


@pytest.mark.parametrize("name", ["qwen3_30b_a3b_T16384", "prism_subexpert_T8192", "dsv2lite_prefill_T4096"])
def test_layer_full_size_folded_combine(name):
    """The full-size layers with the combine folded into GEMM2, on the sampled checks."""
    d = wl.make_inputs(wl.CONFIGS[name])
    res, P = run_gpu(d, fused_gather=name.startswith("prism"), fused_combine=True)
    check_layer_sampled(d, res, P)
