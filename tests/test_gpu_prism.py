"""GPU parity of MoE-Prism's hierarchical gating (semmoe_route_hier) and of the
layer that routes with it, against the oracle.  Sub-expert ids bit-exact
(given the GPU's own fp32 parent logits), gates within the gate tolerance,
layer outputs within the bf16 / fp32 tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity_utils import GATE_ATOL, LOGIT_TOL, TOL, max_rel, np_

pytestmark = pytest.mark.gpu

i32 = dict(dtype=torch.int32, device="cuda")


def abi():
    from token_expert_routing_gb300 import _abi
    return _abi


def run_hier_logits(l, logw, N, k, k_max, per_token=True):
    T, Ep = l.shape
    idx = torch.full((T, k_max), -7, **i32)
    w = torch.full((T, k_max), 7.0, dtype=torch.float32, device="cuda")
    kpt = torch.from_numpy(np.asarray(k, dtype=np.int32)).cuda() if per_token else None
    ku = 0 if per_token else int(k[0])
    abi().semmoe_route_hier(None, None, torch.from_numpy(l).cuda(), None,
                            torch.from_numpy(np.asarray(logw, dtype=np.float32)).cuda(), N, kpt, ku, T, 0, Ep,
                            k_max, idx, w)
    assert abi().semmoe_check_errors() == 0
    return idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("Ep,N,k_max", [(8, 1, 3), (16, 2, 7), (64, 4, 24), (32, 8, 40), (3, 2, 6), (64, 4, 256)])
def test_hier_route_from_logits(Ep, N, k_max):
    rng = np.random.default_rng(Ep * 10 + N)
    T = 1500
    l = rng.standard_normal((T, Ep)).astype(np.float32)
    logw = np.log(rng.dirichlet(np.full(N, 2.0), size=Ep).reshape(-1)).astype(np.float32)
    k = rng.integers(1, k_max + 1, size=T)
    idx, w = run_hier_logits(l, logw, N, k, k_max)
    ref_idx, ref_w = oracle.hier_route(l, logw, N, k, k_max)
    np.testing.assert_array_equal(idx, ref_idx)
    np.testing.assert_allclose(w, ref_w, rtol=0, atol=GATE_ATOL)


def test_hier_route_ties_and_uniform_budget():
    """Quantised logits and weights tie often: ties go to the lower sub-expert."""
    rng = np.random.default_rng(11)
    T, Ep, N, k = 2000, 16, 4, 12
    l = (rng.integers(-3, 4, size=(T, Ep)) * 0.5).astype(np.float32)
    l[:, 5] = -0.0
    logw = (rng.integers(-4, 1, size=Ep * N) * 0.25).astype(np.float32)
    idx, w = run_hier_logits(l, logw, N, np.full(T, k), k, per_token=False)
    ref_idx, ref_w = oracle.hier_route(l, logw, N, np.full(T, k), k)
    np.testing.assert_array_equal(idx, ref_idx)
    np.testing.assert_allclose(w, ref_w, rtol=0, atol=GATE_ATOL)


def test_hier_uniform_weights_match_parent_router():
    """Equal co-activation weights and budgets of m*N: the GPU's hierarchical
    picks are the GPU's own parent top-m, sub-experts in order."""
    rng = np.random.default_rng(12)
    T, Ep, N = 1000, 64, 4
    l = rng.standard_normal((T, Ep)).astype(np.float32)
    m = rng.integers(1, 7, size=T)
    idx, w = run_hier_logits(l, np.full(Ep * N, -np.log(N), dtype=np.float32), N, m * N, 24)
    pidx = torch.empty(T, 6, **i32)
    pw = torch.empty(T, 6, dtype=torch.float32, device="cuda")
    abi().semmoe_route(None, None, torch.from_numpy(l).cuda(), None, torch.from_numpy(m.astype(np.int32)).cuda(), 0,
                       T, 0, Ep, 6, pidx, pw)
    pidx, pw = pidx.cpu().numpy(), pw.cpu().numpy()
    for t in range(T):
        want = [int(e) * N + i for e in pidx[t, :m[t]] for i in range(N)]
        assert idx[t, :m[t] * N].tolist() == want
        np.testing.assert_allclose(w[t, :m[t] * N], np.repeat(pw[t, :m[t]], N), rtol=0, atol=GATE_ATOL)


@pytest.mark.parametrize("xd,wd", [("bf16", "f32"), ("bf16", "bf16"), ("f32", "f32")])
def test_hier_route_with_router_gemm(xd, wd):
    """The parent router GEMM feeding the hierarchical top-k, on the tensor
    cores (bf16 activations) and on the CUDA cores (fp32 activations)."""
    rng = np.random.default_rng(13)
    T, H, Ep, N, k_max = 777, 256, 32, 4, 20
    td = {"bf16": torch.bfloat16, "f32": torch.float32}
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32) / 16).to(td[xd])
    wp = torch.from_numpy(rng.standard_normal((Ep, H)).astype(np.float32) / 16).to(td[wd])
    logw = np.log(rng.dirichlet(np.full(N, 2.0), size=Ep).reshape(-1)).astype(np.float32)
    k = rng.integers(1, k_max + 1, size=T).astype(np.int32)
    idx = torch.empty(T, k_max, **i32)
    w = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
    lg = torch.empty(T, Ep, dtype=torch.float32, device="cuda")
    abi().semmoe_route_hier(x.cuda(), wp.cuda(), None, lg, torch.from_numpy(logw).cuda(), N,
                            torch.from_numpy(k).cuda(), 0, T, H, Ep, k_max, idx, w)
    assert abi().semmoe_check_errors() == 0
    lg = lg.cpu().numpy()
    assert max_rel(lg, oracle.router_logits(x, wp)) < LOGIT_TOL
    ref_idx, ref_w = oracle.hier_route(lg, logw, N, k, k_max)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=0, atol=GATE_ATOL)


def _hier_layer(d, keep_logits=True):
    from token_expert_routing_gb300 import MoELayer
    spec = d["spec"]
    layer = MoELayer(d["w_router_parent"], d["w13"], d["w2"], d["expert_rank"], d["lut"], spec.R, spec.k_max,
                     d["ws13"], d["ws2"], sub_logw=d["sub_logw"])
    kpt = d["k_per_token"].cuda()
    P = int(d["k_per_token"].sum())
    res = layer.forward(d["x"].cuda(), d["token_ids"].cuda(), kpt, None, P, keep_logits=keep_logits)
    assert abi().semmoe_check_errors() == 0
    return res, P


def test_hier_layer_small_full_compare():
    """The whole layer routed hierarchically on a small MoE-Prism-shaped
    layer (256 sub-experts, budgets 12..24), every output against the oracle."""
    spec = workloads.scaled("prism_subexpert_T8192", T=512, H=256, I=64, tokens_per_request=128)
    d = workloads.make_inputs(spec)
    res, P = _hier_layer(d)
    k = d["k_per_token"].numpy()
    lg = np_(res.logits)
    assert max_rel(lg, oracle.router_logits(d["x"], d["w_router_parent"])) < LOGIT_TOL
    idx, w = oracle.hier_route(lg, d["sub_logw"], spec.sub_split, k, spec.k_max)
    np.testing.assert_array_equal(np_(res.topk_idx), idx)
    np.testing.assert_allclose(np_(res.topk_w), w, rtol=0, atol=GATE_ATOL)
    perm = oracle.permute(idx, k, d["expert_rank"], spec.R)
    np.testing.assert_array_equal(np_(res.pair_to_sorted), perm["pair_to_sorted"])
    x_perm = np_(d["x"])[perm["sorted_to_pair"] // spec.k_max]
    y_perm = oracle.grouped_ffn(x_perm, perm["expert_offsets"], perm["phys_to_expert"], d["w13"], d["w2"],
                                spec.dtype)
    # the combine takes the GPU's own gates (compared above) and y rows
    out = oracle.combine(y_perm, perm["pair_to_sorted"], np_(res.topk_w), k, spec.dtype)
    assert max_rel(np_(res.out), out) < TOL[spec.dtype]


def test_hier_layer_full_size_routing():
    """The MoE-Prism workload at full size: routing, bucket tables and the
    local-activation counts from the hierarchical gate, bit-exact."""
    spec = workloads.CONFIGS["prism_subexpert_T8192"]
    d = workloads.make_inputs(spec)
    res, P = _hier_layer(d)
    k = d["k_per_token"].numpy()
    idx, w = oracle.hier_route(np_(res.logits), d["sub_logw"], spec.sub_split, k, spec.k_max)
    np.testing.assert_array_equal(np_(res.topk_idx), idx)
    np.testing.assert_allclose(np_(res.topk_w), w, rtol=0, atol=GATE_ATOL)
    assert int((idx >= 0).sum()) == P
    pred = oracle.affinity_lookup(d["token_ids"], d["lut"])
    counts, remote = oracle.remote_count(idx, k, pred, d["expert_rank"], spec.R)
    np.testing.assert_array_equal(np_(res.counts), counts)
    perm = oracle.permute(idx, k, d["expert_rank"], spec.R)
    for key in ("expert_offsets", "rank_offsets", "sorted_to_pair", "pair_to_sorted"):
        np.testing.assert_array_equal(np_(getattr(res, key)), perm[key], err_msg=key)
