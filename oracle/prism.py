"""Oracle for MoE-Prism's training-free hierarchical gating (numpy).

TEST INFRASTRUCTURE ONLY, like the rest of this package.

MoE-Prism (ko) §2 A splits each monolithic expert into N sub-experts (disjoint
sets of its intermediate neurons) and, for deployment without training,
rebuilds the routing with a hierarchical proxy that scores the sub-experts by
co-activation statistics ("Gating Reconstruction", item 1).  The pages give no
formula; the readings below are the plainest ones the rest of the method
supports, and they reduce to the parent router's own top-k when every
sub-expert of a parent scores alike.
"""
from __future__ import annotations

import numpy as np

from .moe import _f64, _i64, round_to


def sub_scores(parent_logits, sub_logw, N: int) -> np.ndarray:
    """score[t, e*N + i] = l[t, e] + logw[e*N + i], added in fp32.

    Reading taken: the parent router's logit carries the parent level and a
    profiled co-activation weight a[e, i] of each sub-expert (held as its log,
    so the score is a sum) carries the sub-expert level; ordering by the sum
    orders by p_e * a[e, i], p the parent softmax.  fp32 because the scores
    decide the selection, in the kernel's precision.
    """
    l = np.asarray(parent_logits, dtype=np.float32)
    b = np.asarray(sub_logw, dtype=np.float32).reshape(-1)
    T, Ep = l.shape
    if b.shape[0] != Ep * N:
        raise ValueError("sub_logw must hold E_parent * N values")
    return (np.repeat(l, N, axis=1) + b[None, :]).astype(np.float32)


def hier_route(parent_logits, sub_logw, N: int, k_per_token, k_max: int):
    """Top-k_t sub-experts of every token and their gates.

    * sub-experts are ordered by ``sub_scores`` descending, equal scores keep
      the lower sub-expert index e*N + i first; slot j holds the j-th, j < k_t;
    * gate of a selected sub-expert of parent e: p_e renormalised over the
      distinct parents of the selection, w = exp(l_e - m) / sum_{e' in S} exp(l_e' - m),
      m = the largest of those parents' logits (fp64, stored as fp32).  A
      parent's sub-experts all carry its gate: their outputs are parts of the
      parent's output, so selecting every sub-expert of the chosen parents
      gives back the parent router's renormalised top-k;
    * slots j >= k_t are padding: index -1, gate 0.

    Returns topk_idx [T, k_max] int64 (sub-expert ids) and topk_w [T, k_max]
    float64 (fp32 values).
    """
    l = _f64(np.asarray(parent_logits, dtype=np.float32))
    T, Ep = l.shape
    E = Ep * N
    k = _i64(k_per_token).reshape(T)
    if k_max > E or (k < 1).any() or (k > k_max).any():
        raise ValueError("need 1 <= k_t <= k_max <= E_parent * N")
    s = _f64(sub_scores(parent_logits, sub_logw, N))
    order = np.argsort(-s, axis=1, kind="stable")[:, :k_max]
    slot = np.arange(k_max)[None, :]
    live = slot < k[:, None]
    topk_idx = np.where(live, order, -1)
    w = np.zeros((T, k_max))
    for t in range(T):
        par = order[t, :k[t]] // N
        chosen = np.unique(par)
        m = l[t, chosen].max()
        den = np.exp(l[t, chosen] - m).sum()
        w[t, :k[t]] = np.exp(l[t, par] - m) / den
    return topk_idx, round_to(w, "f32")


def split_expert_weights(w13, w2, N: int):
    """Sub-expert weights of parent experts: sub-expert i of parent e holds
    intermediate neurons [i*I/N, (i+1)*I/N) of e (MoE-Prism (ko) §2 A: an
    expert is a set of intermediate neurons), gate rows before up rows.

    w13 [Ep, 2I, H], w2 [Ep, H, I] -> [Ep*N, 2I/N, H], [Ep*N, H, I/N].
    """
    w13 = np.asarray(w13)
    w2 = np.asarray(w2)
    Ep, twoI, H = w13.shape
    I = twoI // 2
    if I % N:
        raise ValueError("I must be a multiple of N")
    Is = I // N
    g = w13[:, :I, :].reshape(Ep, N, Is, H)
    u = w13[:, I:, :].reshape(Ep, N, Is, H)
    s13 = np.concatenate([g, u], axis=2).reshape(Ep * N, 2 * Is, H)
    s2 = w2.reshape(Ep, H, N, Is).transpose(0, 2, 1, 3).reshape(Ep * N, H, Is)
    return s13, s2
