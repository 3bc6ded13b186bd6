"""Pins of the scheduling oracle (CPU only): brute force, a hand example,
invariants, and special cases that reduce to the layer's own tables."""
import numpy as np

import oracle


def test_dp_schedule_hand_example():
    # 3 requests over R = 3 ranks: [0,0,1] -> rank 0; [2,1,2,1] -> tie 1/2 -> rank 1; [] -> rank 0
    pred = np.array([0, 0, 1, 2, 1, 2, 1])
    off = np.array([0, 3, 7, 7])
    s = oracle.dp_schedule(pred, off, 3)
    np.testing.assert_array_equal(s["hist"], [[2, 1, 0], [0, 2, 2], [0, 0, 0]])
    np.testing.assert_array_equal(s["req_rank"], [0, 1, 0])
    np.testing.assert_array_equal(s["req_order"], [0, 2, 1])
    np.testing.assert_array_equal(s["req_pos"], [0, 2, 1])
    np.testing.assert_array_equal(s["rank_req_offsets"], [0, 2, 3, 3])
    # rank 0 batch: request 0 (tokens 0..2) then the empty request 2; rank 1: request 1
    np.testing.assert_array_equal(s["req_tok_start"], [0, 3, 3])
    np.testing.assert_array_equal(s["tok_order"], [0, 1, 2, 3, 4, 5, 6])
    np.testing.assert_array_equal(s["tok_rank"], [0, 0, 0, 1, 1, 1, 1])
    np.testing.assert_array_equal(s["rank_tok_offsets"], [0, 3, 7, 7])


def test_dp_schedule_hand_example_reordered():
    # requests: [1,1] -> 1, [0] -> 0, [1,0,1] -> 1, [0,0] -> 0  (R = 2)
    pred = np.array([1, 1, 0, 1, 0, 1, 0, 0])
    off = np.array([0, 2, 3, 6, 8])
    s = oracle.dp_schedule(pred, off, 2)
    np.testing.assert_array_equal(s["req_rank"], [1, 0, 1, 0])
    np.testing.assert_array_equal(s["req_order"], [1, 3, 0, 2])
    np.testing.assert_array_equal(s["req_tok_start"], [3, 0, 5, 1])
    np.testing.assert_array_equal(s["tok_order"], [2, 6, 7, 0, 1, 3, 4, 5])
    np.testing.assert_array_equal(s["tok_rank"], [1, 1, 0, 1, 1, 1, 0, 0])
    np.testing.assert_array_equal(s["rank_tok_offsets"], [0, 3, 8])


def test_dp_schedule_brute_force_and_invariants():
    rng = np.random.default_rng(0)
    R = 5
    lens = rng.integers(0, 30, size=60)
    off = np.concatenate([[0], np.cumsum(lens)])
    pred = rng.integers(0, R, size=off[-1])
    s = oracle.dp_schedule(pred, off, R)
    hist, rank, order, pos, ro = s["hist"], s["req_rank"], s["req_order"], s["req_pos"], s["rank_req_offsets"]
    for r in range(60):
        h = [int(np.sum(pred[off[r]:off[r + 1]] == q)) for q in range(R)]
        assert list(hist[r]) == h
        best = max(h)
        assert rank[r] == h.index(best)          # first (lowest) rank among the maxima
    assert sorted(order.tolist()) == list(range(60))
    assert (np.diff(rank[order]) >= 0).all()
    same = np.diff(rank[order]) == 0
    assert (np.diff(order)[same] > 0).all()      # stable
    np.testing.assert_array_equal(pos[order], np.arange(60))
    np.testing.assert_array_equal(np.diff(ro), np.bincount(rank, minlength=R))
    # token side: a permutation of 0..T-1; each rank's slice holds exactly the
    # tokens of its requests, each request contiguous and in order
    T = off[-1]
    tok, rto = s["tok_order"], s["rank_tok_offsets"]
    assert sorted(tok.tolist()) == list(range(T))
    for q in range(R):
        want = [t for r in order if rank[r] == q for t in range(off[r], off[r + 1])]
        assert tok[rto[q]:rto[q + 1]].tolist() == want
    for r in range(60):
        st = s["req_tok_start"][r]
        assert tok[st:st + lens[r]].tolist() == list(range(off[r], off[r + 1]))
        assert (s["tok_rank"][off[r]:off[r + 1]] == rank[r]).all()


def test_transition_lookup_brute_force():
    rng = np.random.default_rng(1)
    E, R, T, k_max = 12, 4, 80, 5
    trans = (rng.integers(0, 4, size=(E, R)) * 0.25).astype(np.float32)   # exact sums, many ties
    idx = np.stack([rng.permutation(E)[:k_max] for _ in range(T)])
    k = rng.integers(1, k_max + 1, size=T)
    idx = np.where(np.arange(k_max)[None, :] < k[:, None], idx, -1)
    got = oracle.transition_lookup(idx, k, trans)
    for t in range(T):
        score = [sum(float(trans[idx[t, j], r]) for j in range(k[t])) for r in range(R)]
        best = max(score)
        assert got[t] == score.index(best)


def test_transition_with_placement_table_is_majority_destination():
    """trans[e][r] = 1 when expert e lives on rank r: the prediction is the
    rank hosting most of the token's experts -- the row of the remote counter's
    destination histogram with the largest count."""
    rng = np.random.default_rng(2)
    E, R, T, k_max = 16, 4, 50, 6
    er = rng.integers(0, R, size=E)
    trans = np.zeros((E, R), dtype=np.float32)
    trans[np.arange(E), er] = 1.0
    l = rng.standard_normal((T, E))
    k = rng.integers(1, k_max + 1, size=T)
    idx, _ = oracle.topk_route(l, k, k_max)
    got = oracle.transition_lookup(idx, k, trans)
    for t in range(T):
        dst = np.bincount(er[idx[t, :k[t]]], minlength=R)
        assert got[t] == int(np.argmax(dst))
