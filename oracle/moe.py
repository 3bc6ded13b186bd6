"""Oracle for one affinity-aware MoE layer forward (numpy, float64).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.

Every function takes plain arrays whose values are already the exact values
of the inputs (bf16 or fp32 numbers held in float64 or torch tensors), works
in float64, and rounds to the activation type only where the layer's outputs
are stored: the router logits (fp32), the gates (fp32), the SwiGLU activation
h, the expert output y and the combined output (all in the activation type).

Notation: T tokens, H hidden, E experts, I expert intermediate, R logical
ranks, k_t the per-token budget (its request's k), k_max = max k_t, pair id
p = t * k_max + j for slot j < k_t, P = sum_t k_t.
"""
from __future__ import annotations

import numpy as np
import torch

_F64 = np.float64


def _f64(a) -> np.ndarray:
    """Exact float64 copy of a numpy array or (any-dtype) torch tensor."""
    if isinstance(a, torch.Tensor):
        return a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=_F64)


def _i64(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        return a.detach().to("cpu", torch.int64).numpy()
    return np.asarray(a, dtype=np.int64)


# ---------------------------------------------------------------------------
# rounding
# ---------------------------------------------------------------------------
def bf16_round(a) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 (ties to even), as float64.

    bfloat16 keeps 8 significant bits and fp32's exponent range: the quantum of
    a value m * 2^e (0.5 <= |m| < 1) is 2^(e-8) for normals and 2^-133 below
    2^-126; magnitudes that round to 2^128 or beyond become infinities.
    """
    a = _f64(a)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(a)
        q = np.maximum(e - 8, -133)
        r = np.ldexp(np.rint(np.ldexp(a, -q)), q)
        r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, a), r)
        r = np.where(np.isfinite(a), r, a)
    return r


def round_to(a, dtype: str) -> np.ndarray:
    """Store float64 values in ``dtype``: "f64" (unchanged), "f32" (numpy's
    round-to-nearest-even cast) or "bf16" (``bf16_round``); returned as float64."""
    a = _f64(a)
    if dtype == "f64":
        return a
    if dtype == "f32":
        return a.astype(np.float32).astype(_F64)
    if dtype == "bf16":
        return bf16_round(a)
    raise ValueError(f"unknown dtype {dtype!r}")


def silu(z) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z))."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


# ---------------------------------------------------------------------------
# S1-S2: router
# ---------------------------------------------------------------------------
def router_logits(x, w_router) -> np.ndarray:
    """Gate scores of every token for every expert: logits[t, e] = sum_h x[t,h] Wr[e,h].

    The router (gate) that picks a few experts per token: Semantic Parallelism
    (ko) §1; MoE-Prism (ko) §1.  Accumulated in float64 over the exact input
    values, stored as fp32.
    """
    return round_to(_f64(x) @ _f64(w_router).T, "f32")


def topk_route(logits, k_per_token, k_max: int):
    """Top-k_t experts and their gates for every token.

    The per-request budget k (MoE-Prism (ko) §1, §2 B, §5) makes k a per-token
    value k_t in [1, k_max].  Readings taken (the pages fix none of this):

    * experts are ordered by logit, descending; equal logits keep the lower
      expert index first (a stable sort, so -0.0 and +0.0 tie); slot j holds
      the j-th expert of that order, for j < k_t;
    * the gates are the softmax of the selected logits, renormalised over the
      selection: w_j = exp(l_j - m) / sum_{i<k_t} exp(l_i - m), m = max
      selected logit (fp64, stored as fp32); with k_t = E this is the plain
      softmax;
    * slots j >= k_t are padding: index -1, gate 0.

    Returns topk_idx [T, k_max] int64 and topk_w [T, k_max] float64 (fp32 values).
    """
    l = _f64(logits)
    T, E = l.shape
    k = _i64(k_per_token).reshape(T)
    if k_max > E or (k < 1).any() or (k > k_max).any():
        raise ValueError("need 1 <= k_t <= k_max <= E")
    order = np.argsort(-l, axis=1, kind="stable")[:, :k_max]
    slot = np.arange(k_max)[None, :]
    live = slot < k[:, None]
    topk_idx = np.where(live, order, -1)
    sel = np.take_along_axis(l, order, axis=1)
    m = sel[:, :1]
    ex = np.where(live, np.exp(sel - m), 0.0)
    w = ex / ex.sum(axis=1, keepdims=True)
    return topk_idx, round_to(w, "f32")


# ---------------------------------------------------------------------------
# S3: affinity lookup and the remote-activation counter
# ---------------------------------------------------------------------------
def affinity_lookup(token_ids, lut) -> np.ndarray:
    """Predicted logical rank of each token from its id alone.

    The lightweight token -> expert-group -> device table consulted online
    (Semantic Parallelism (ja) §2.3; built offline from the token-expert
    affinity of (de) §2 A):  pred[t] = lut[token_ids[t]].
    """
    return _i64(lut)[_i64(token_ids)]


def _valid_pairs(topk_idx, k_per_token):
    idx = _i64(topk_idx)
    T, k_max = idx.shape
    k = _i64(k_per_token).reshape(T)
    live = np.arange(k_max)[None, :] < k[:, None]
    p = np.flatnonzero(live.reshape(-1))           # increasing pair ids
    return p, idx.reshape(-1)[p], k_max


def remote_count(topk_idx, k_per_token, pred_rank, expert_rank, R: int):
    """Activations by (predicted source rank, destination rank), and the remote ones.

    A token's activation of expert e is local when e is hosted on the token's
    own rank, remote otherwise; the local activation rate is the local share
    (Semantic Parallelism (ko) §3-§4, (de) §4).  Reading taken: the source of
    pair (t, j) is pred[t], its destination expert_rank[topk_idx[t, j]];
    counts[src][dst] counts pairs, remote[src] = sum over dst != src.

    Returns counts [R, R] and remote [R] (int64).
    """
    p, e, k_max = _valid_pairs(topk_idx, k_per_token)
    src = _i64(pred_rank)[p // k_max]
    dst = _i64(expert_rank)[e]
    counts = np.zeros((R, R), dtype=np.int64)
    np.add.at(counts, (src, dst), 1)
    remote = counts.sum(axis=1) - np.diag(counts)
    return counts, remote


# ---------------------------------------------------------------------------
# S4-S5: the on-device form of the Shuffled-Reduce-Scatter shuffle
# ---------------------------------------------------------------------------
def physical_order(expert_rank):
    """Rank-major expert order: experts sorted by (expert_rank[e], e).

    This is the physical layout that the pages obtain by shuffling the gate
    matrix's columns (Semantic Parallelism (ja) §2.2 A).
    Returns phys_to_expert [E] and phys_of [E] (its inverse).
    """
    er = _i64(expert_rank)
    E = er.shape[0]
    phys_to_expert = np.lexsort((np.arange(E), er))
    phys_of = np.empty(E, dtype=np.int64)
    phys_of[phys_to_expert] = np.arange(E)
    return phys_to_expert, phys_of


def permute(topk_idx, k_per_token, expert_rank, R: int, x=None):
    """Stable sort of the (token, expert) pairs by (destination rank, expert).

    The shuffle that sends each token to the device hosting its target experts
    (Shuffled-Reduce-Scatter: Semantic Parallelism (ko) §2.2, (de) §2 B,
    (ja) §2.2 B) becomes, on one device, a stable permutation of the pairs.
    Reading taken: the key of pair p is phys(topk_idx[p]) (destination rank
    first, expert id second); equal keys keep increasing p.

    Returns a dict with expert_offsets [E+1] (physical order), rank_offsets
    [R+1], phys_to_expert [E], expert_counts [E] (logical order),
    sorted_to_pair [P], pair_to_sorted [T*k_max] (-1 for padding slots) and,
    when x is given, x_perm [P, H] with x_perm[q] = x[sorted_to_pair[q] // k_max].
    """
    idx = _i64(topk_idx)
    T, k_max = idx.shape
    er = _i64(expert_rank)
    E = er.shape[0]
    p, e, _ = _valid_pairs(idx, k_per_token)
    phys_to_expert, phys_of = physical_order(er)
    order = np.argsort(phys_of[e], kind="stable")
    sorted_to_pair = p[order]
    P = p.shape[0]
    pair_to_sorted = np.full(T * k_max, -1, dtype=np.int64)
    pair_to_sorted[sorted_to_pair] = np.arange(P)
    expert_counts = np.bincount(e, minlength=E)
    expert_offsets = np.concatenate([[0], np.cumsum(expert_counts[phys_to_expert])])
    rank_offsets = np.concatenate([[0], np.cumsum(np.bincount(er[e], minlength=R))])
    out = dict(expert_offsets=expert_offsets, rank_offsets=rank_offsets,
               phys_to_expert=phys_to_expert, expert_counts=expert_counts,
               sorted_to_pair=sorted_to_pair, pair_to_sorted=pair_to_sorted)
    if x is not None:
        out["x_perm"] = _f64(x)[sorted_to_pair // k_max]
    return out


# ---------------------------------------------------------------------------
# S6-S7: expert FFN (SwiGLU)
# ---------------------------------------------------------------------------
def expert_ffn(xs, w13_e, w2_e, dtype: str):
    """SwiGLU expert on a block of rows of one expert.

    The expert computation itself is not described on the pages (Semantic
    Parallelism (ko) §1: tokens activate a few experts; MoE-Prism (ko) §2 A:
    experts are made of intermediate neurons).  Reading taken: the SwiGLU FFN
    with w13_e = [W1; W3] of shape [2I, H] (rows 0..I-1 gate, I..2I-1 up) and
    w2_e [H, I]:  h = round(silu(xs W1^T) * (xs W3^T)),  y = round(h W2^T).
    Returns (h, y) as float64 arrays of ``dtype`` values.
    """
    xs = _f64(xs)
    w13_e = _f64(w13_e)
    I = w13_e.shape[0] // 2
    g = xs @ w13_e[:I].T
    u = xs @ w13_e[I:].T
    h = round_to(silu(g) * u, dtype)
    y = round_to(h @ _f64(w2_e).T, dtype)
    return h, y


def grouped_ffn(x_perm, expert_offsets, phys_to_expert, w13, w2, dtype: str):
    """Each physical bucket b's rows [off[b], off[b+1]) go through expert
    phys_to_expert[b].  Returns y_perm [P, H] (``dtype`` values)."""
    x_perm = _f64(x_perm)
    off = _i64(expert_offsets)
    pe = _i64(phys_to_expert)
    y = np.zeros((x_perm.shape[0], w2.shape[1]), dtype=_F64)
    for b in range(pe.shape[0]):
        lo, hi, e = int(off[b]), int(off[b + 1]), int(pe[b])
        if hi > lo:
            _, y[lo:hi] = expert_ffn(x_perm[lo:hi], w13[e], w2[e], dtype)
    return y


def shared_ffn(x, ws13, ws2, dtype: str):
    """Shared experts (concatenated along I) applied to every token, gate 1."""
    return expert_ffn(x, ws13, ws2, dtype)[1]


# ---------------------------------------------------------------------------
# S8: the on-device form of the Shuffled-Allgather (un-permute and combine)
# ---------------------------------------------------------------------------
def combine(y_perm, pair_to_sorted, topk_w, k_per_token, dtype: str, y_shared=None):
    """Restore token order and mix each token's expert outputs by its gates.

    Shuffled-Allgather gathers the expert results and puts them back in the
    original token order (Semantic Parallelism (de) §2 B, (ja) §2.2 B):
    out[t] = y_shared[t] + sum_{j<k_t} w[t,j] * y_perm[pair_to_sorted[t*k_max+j]],
    in float64, stored in ``dtype``.  Reading taken: shared experts enter with
    gate 1; there is no capacity limit and no token is dropped.
    """
    y = _f64(y_perm)
    w = _f64(topk_w)
    T, k_max = w.shape
    k = _i64(k_per_token).reshape(T)
    pts = _i64(pair_to_sorted).reshape(T, k_max)
    H = y.shape[1]
    out = np.zeros((T, H), dtype=_F64) if y_shared is None else _f64(y_shared).copy()
    for j in range(k_max):
        live = k > j
        if live.any():
            out[live] += w[live, j][:, None] * y[pts[live, j]]
    return round_to(out, dtype)


# ---------------------------------------------------------------------------
# the whole layer
# ---------------------------------------------------------------------------
def moe_layer(x, w_router, token_ids, lut, expert_rank, k_per_token, w13, w2, R: int,
              dtype: str, k_max: int | None = None, ws13=None, ws2=None, logits=None):
    """One MoE layer forward: route, look up, count, permute, FFN, combine.

    ``logits`` (fp32 values), when given, replaces the router GEMM so that
    index results can be compared bit for bit with another implementation that
    produced those logits.  Returns a dict of every intermediate.
    """
    x64 = _f64(x)
    lg = router_logits(x64, w_router) if logits is None else _f64(logits)
    k = _i64(k_per_token)
    k_max = int(k.max()) if k_max is None else k_max
    topk_idx, topk_w = topk_route(lg, k, k_max)
    pred = affinity_lookup(token_ids, lut)
    counts, remote = remote_count(topk_idx, k, pred, expert_rank, R)
    perm = permute(topk_idx, k, expert_rank, R, x64)
    y_perm = grouped_ffn(perm["x_perm"], perm["expert_offsets"], perm["phys_to_expert"],
                         w13, w2, dtype)
    y_shared = shared_ffn(x64, ws13, ws2, dtype) if ws13 is not None else None
    out = combine(y_perm, perm["pair_to_sorted"], topk_w, k, dtype, y_shared)
    res = dict(logits=lg, topk_idx=topk_idx, topk_w=topk_w, pred=pred, counts=counts,
               remote=remote, y_perm=y_perm, y_shared=y_shared, out=out)
    res.update(perm)
    return res
