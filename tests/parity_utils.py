"""Helpers for the GPU-vs-oracle parity tests: run the CUDA path through the
C ABI, run the oracle on the same inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle

#: max relative error (normwise, per tensor) for float outputs, by activation type
TOL = {"f32": 1e-4, "bf16": 2e-2}
#: router logits are fp32 sums of H products in both modes
LOGIT_TOL = 2e-5
#: gates: fp32 softmax vs float64 softmax rounded to fp32
GATE_ATOL = 2e-6


def max_rel(got, ref) -> float:
    """max_i |got_i - ref_i| / max_i |ref_i| (normwise infinity error)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    den = np.abs(ref).max()
    return float(np.abs(got - ref).max() / (den if den > 0 else 1.0))


def np_(t) -> np.ndarray:
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        t = t.to(torch.float64)
    return t.numpy()


def run_gpu(d, logits_in=None, fused_gather=False, fused_combine=False):
    """One layer forward of inputs ``d`` (from workloads.make_inputs) on cuda:0;
    fused_gather=True lets GEMM1 gather x rows instead of the permute writing
    x_perm; fused_combine=True lets GEMM2 add its rows into the token order
    instead of writing y_perm."""
    from token_expert_routing_gb300 import MoELayer, _abi
    spec = d["spec"]
    layer = MoELayer(d["w_router"], d["w13"], d["w2"], d["expert_rank"], d["lut"], spec.R, spec.k_max,
                     d["ws13"], d["ws2"], fused_gather=fused_gather, fused_combine=fused_combine)
    x = d["x"].cuda()
    ids = d["token_ids"].cuda()
    P = int(d["k_per_token"].sum())
    kpt = d["k_per_token"].cuda() if spec.k_choices else None
    li = None if logits_in is None else torch.as_tensor(logits_in, dtype=torch.float32).cuda()
    res = layer.forward(x, ids, kpt, None if spec.k_choices else spec.k, P, logits_in=li,
                        keep_logits=li is None)
    bits = _abi.semmoe_check_errors()
    assert bits == 0, f"device error bits {bits:#x}"
    return res, P


def check_routing(d, res, P):
    """Bit-exact checks of everything integer, given the GPU's fp32 logits."""
    spec = d["spec"]
    k = d["k_per_token"].numpy()
    logits = np_(res.logits) if res.logits is not None else None
    if logits is not None:
        ref_logits = oracle.router_logits(d["x"], d["w_router"])
        assert max_rel(logits, ref_logits) < LOGIT_TOL
    idx, w = oracle.topk_route(logits, k, spec.k_max)
    np.testing.assert_array_equal(np_(res.topk_idx), idx)
    np.testing.assert_allclose(np_(res.topk_w), w, rtol=0, atol=GATE_ATOL)
    pred = oracle.affinity_lookup(d["token_ids"], d["lut"])
    np.testing.assert_array_equal(np_(res.pred_rank), pred)
    counts, remote = oracle.remote_count(idx, k, pred, d["expert_rank"], spec.R)
    np.testing.assert_array_equal(np_(res.counts), counts)
    np.testing.assert_array_equal(np_(res.remote), remote)
    perm = oracle.permute(idx, k, d["expert_rank"], spec.R)
    for key in ("expert_offsets", "rank_offsets", "phys_to_expert", "expert_counts", "sorted_to_pair",
                "pair_to_sorted"):
        np.testing.assert_array_equal(np_(getattr(res, key)), perm[key], err_msg=key)
    return idx, w, perm


def check_layer_full(d, res, P):
    """Every output, at sizes the oracle runs in full."""
    spec = d["spec"]
    idx, w, perm = check_routing(d, res, P)
    x_perm = oracle.permute(idx, d["k_per_token"].numpy(), d["expert_rank"], spec.R, d["x"])["x_perm"]
    if res.x_perm is not None:
        np.testing.assert_array_equal(np_(res.x_perm), x_perm)
    y_perm = oracle.grouped_ffn(x_perm, perm["expert_offsets"], perm["phys_to_expert"], d["w13"], d["w2"],
                                spec.dtype)
    if res.y_perm is not None:
        assert max_rel(np_(res.y_perm), y_perm) < TOL[spec.dtype]
    y_shared = None
    if d["ws13"] is not None:
        y_shared = oracle.shared_ffn(d["x"], d["ws13"], d["ws2"], spec.dtype)
        assert max_rel(np_(res.y_shared), y_shared) < TOL[spec.dtype]
    out = oracle.combine(y_perm, perm["pair_to_sorted"], w, d["k_per_token"].numpy(), spec.dtype, y_shared)
    assert max_rel(np_(res.out), out) < TOL[spec.dtype]


def check_layer_sampled(d, res, P, n_tokens=96, seed=0):
    """Full-size check: every integer output in full; the FFN, shared FFN and
    combined output on a seeded sample of tokens (each recomputed by the
    oracle row by row from the GPU-independent routing), and the FFN output
    of the last sorted row of every expert group."""
    spec = d["spec"]
    idx, w, perm = check_routing(d, res, P)
    k = d["k_per_token"].numpy()
    rng = np.random.default_rng(seed)
    toks = np.unique(np.concatenate([rng.choice(spec.T, size=min(n_tokens, spec.T), replace=False),
                                     [0, spec.T - 1]]))
    x = d["x"]
    gpu_out = np_(res.out[torch.as_tensor(toks, device=res.out.device)])
    p2s = perm["pair_to_sorted"]
    pairs = [(n, int(t), j, int(idx[t, j]), int(p2s[t * spec.k_max + j]))
             for n, t in enumerate(toks) for j in range(int(k[t]))]
    qs = torch.as_tensor([q for *_, q in pairs], device=res.out.device)
    if res.x_perm is not None:
        np.testing.assert_array_equal(np_(res.x_perm[qs]), np_(x[torch.as_tensor([t for _, t, *_ in pairs])]))
    ref_y = np.zeros((len(pairs), spec.H))
    for e in sorted({e for *_, e, _ in pairs}):          # one oracle call per expert
        rows = [i for i, pr in enumerate(pairs) if pr[3] == e]
        xs = x[torch.as_tensor([pairs[i][1] for i in rows])]
        _, y = oracle.expert_ffn(xs, d["w13"][e], d["w2"][e], spec.dtype)
        ref_y[rows] = y
    if res.y_perm is not None:       # GEMM2 wrote y_perm (else it added its rows into the output)
        assert max_rel(np_(res.y_perm[qs]), ref_y) < TOL[spec.dtype]
        check_group_tails(d, res, perm)
    acc = np.zeros((len(toks), spec.H))
    if d["ws13"] is not None:
        ys = oracle.shared_ffn(x[torch.as_tensor(toks)], d["ws13"], d["ws2"], spec.dtype)
        gpu_ys = np_(res.y_shared[torch.as_tensor(toks, device=res.y_shared.device)])
        assert max_rel(gpu_ys, ys) < TOL[spec.dtype]
        acc += ys
    for i, (n, t, j, e, q) in enumerate(pairs):            # combine in slot order
        acc[n] += w[t, j] * ref_y[i]
    assert max_rel(gpu_out, oracle.round_to(acc, spec.dtype)) < TOL[spec.dtype]


def check_group_tails(d, res, perm):
    """The FFN output of the last sorted row of every expert group (the ragged
    tail of its last tile), recomputed by the oracle row by row."""
    spec = d["spec"]
    x = d["x"]
    off, pe, s2p = perm["expert_offsets"], perm["phys_to_expert"], perm["sorted_to_pair"]
    tails = [(int(off[b + 1]) - 1, int(pe[b])) for b in range(pe.shape[0]) if off[b + 1] > off[b]]
    gpu_tail = np_(res.y_perm[torch.as_tensor([q for q, _ in tails], device=res.y_perm.device)])
    ref_tail = np.zeros_like(gpu_tail)
    for i, (q, e) in enumerate(tails):
        t = int(s2p[q]) // spec.k_max
        _, ref_tail[i:i + 1] = oracle.expert_ffn(x[t:t + 1], d["w13"][e], d["w2"][e], spec.dtype)
    assert max_rel(gpu_tail, ref_tail) < TOL[spec.dtype]
