"""Oracle for the table-driven scheduling steps around the layer (numpy).

TEST INFRASTRUCTURE ONLY, like the rest of this package.

* dp_schedule: the online inter-request scheduling of Attention-DP
  (Semantic Parallelism (ko) §2.2 item 2, (de) §2 B, (ja) §2.2 B.1): each
  request's per-token predictions are aggregated and the whole request is
  batched onto the DP rank with the highest affinity.
* transition_lookup: the inter-layer table that maps the experts a token chose
  in one layer to the device it is expected to need in the next (the Markovian
  inter-layer dependency of (ko) §2.1 / (de) §2 A, the "expert sequence -> next
  device" table of (ja) §2.3).
"""
from __future__ import annotations

import numpy as np

from .moe import _i64


def dp_schedule(pred_rank, req_offsets, R: int):
    """Requests placed on DP ranks by their tokens' predicted ranks.

    Readings taken: a request's affinity to rank r is the number of its tokens
    whose predicted rank is r; the request goes to the rank of largest affinity,
    ties (and empty requests) to the lowest rank; requests are then ordered
    stably by their rank, and a rank's batch is its requests' tokens laid end
    to end in that order.  Returns a dict of int64 arrays:
      hist [n_req, R], req_rank [n_req], req_order [n_req] (request ids in
      scheduled order), req_pos [n_req] (its inverse), rank_req_offsets [R+1],
      req_tok_start [n_req] (where request r's first token lands in tok_order),
      tok_order [T] (token ids in scheduled order), tok_rank [T] (the rank of
      the token's request), rank_tok_offsets [R+1].
    """
    pred = _i64(pred_rank)
    off = _i64(req_offsets)
    n = off.shape[0] - 1
    T = pred.shape[0]
    hist = np.zeros((n, R), dtype=np.int64)
    for r in range(n):
        hist[r] = np.bincount(pred[off[r]:off[r + 1]], minlength=R)[:R]
    req_rank = np.argmax(hist, axis=1) if n else np.zeros(0, dtype=np.int64)  # first maximum
    order = np.argsort(req_rank, kind="stable")
    pos = np.empty(n, dtype=np.int64)
    pos[order] = np.arange(n)
    lens = np.diff(off)
    rank_req_offsets = np.concatenate([[0], np.cumsum(np.bincount(req_rank, minlength=R))])
    starts_sched = np.concatenate([[0], np.cumsum(lens[order])])[:-1]
    req_tok_start = np.empty(n, dtype=np.int64)
    req_tok_start[order] = starts_sched
    tok_order = np.concatenate([np.arange(off[r], off[r + 1]) for r in order] or [np.zeros(0)]).astype(np.int64)
    tok_rank = np.repeat(req_rank, lens).astype(np.int64)
    rank_tok = np.zeros(R, dtype=np.int64)
    np.add.at(rank_tok, req_rank, lens)
    return {
        "hist": hist,
        "req_rank": req_rank.astype(np.int64),
        "req_order": order.astype(np.int64),
        "req_pos": pos,
        "rank_req_offsets": rank_req_offsets.astype(np.int64),
        "req_tok_start": req_tok_start,
        "tok_order": tok_order,
        "tok_rank": tok_rank,
        "rank_tok_offsets": np.concatenate([[0], np.cumsum(rank_tok)]).astype(np.int64),
    }


def transition_lookup(topk_idx_prev, k_per_token, trans):
    """Next-layer rank predicted from the experts a token chose in this layer.

    Reading taken: score[r] = sum_{j < k_t} trans[topk_idx_prev[t, j], r], added
    in slot order in fp32 (the same precision as the kernel, since the sum
    decides an argmax); prediction = argmax_r score, ties to the lowest rank.
    trans [E, R] holds the (profiled) transition weights.  Returns int64 [T].
    """
    idx = _i64(topk_idx_prev)
    T, k_max = idx.shape
    k = _i64(k_per_token).reshape(T)
    tr = np.asarray(trans, dtype=np.float32)
    R = tr.shape[1]
    out = np.zeros(T, dtype=np.int64)
    for t in range(T):
        s = np.zeros(R, dtype=np.float32)
        for j in range(int(k[t])):
            e = idx[t, j]
            if e >= 0:
                s = (s + tr[e]).astype(np.float32)
        out[t] = int(np.argmax(s))
    return out
