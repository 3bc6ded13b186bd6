"""Pins of the hierarchical-gating oracle (CPU only): special cases that reduce
to the parent router's own top-k, brute force over tiny cases, a hand-worked
example, and the neuron decomposition against the dense mixture of parents."""
import itertools
import math

import numpy as np
import pytest

import oracle


def test_one_sub_expert_per_parent_is_the_plain_router():
    rng = np.random.default_rng(0)
    T, Ep, k_max = 200, 16, 5
    l = rng.standard_normal((T, Ep)).astype(np.float32)
    k = rng.integers(1, k_max + 1, size=T)
    idx, w = oracle.hier_route(l, np.zeros(Ep, dtype=np.float32), 1, k, k_max)
    idx0, w0 = oracle.topk_route(l, k, k_max)
    np.testing.assert_array_equal(idx, idx0)
    np.testing.assert_array_equal(w, w0)


@pytest.mark.parametrize("N", [2, 4])
def test_uniform_weights_select_whole_parents(N):
    """Equal co-activation weights and a budget of m*N sub-experts: the
    selection is every sub-expert of the parent router's top m, parent by
    parent, and each carries its parent's renormalised top-m gate."""
    rng = np.random.default_rng(N)
    T, Ep = 300, 12
    l = rng.standard_normal((T, Ep)).astype(np.float32)
    m = rng.integers(1, 5, size=T)
    logw = np.full(Ep * N, np.log(1.0 / N), dtype=np.float32)
    idx, w = oracle.hier_route(l, logw, N, m * N, 4 * N)
    pidx, pw = oracle.topk_route(l, m, 4)
    for t in range(T):
        want = [int(e) * N + i for e in pidx[t, :m[t]] for i in range(N)]
        assert idx[t, :m[t] * N].tolist() == want
        np.testing.assert_array_equal(w[t, :m[t] * N], np.repeat(pw[t, :m[t]], N))
        assert (idx[t, m[t] * N:] == -1).all() and (w[t, m[t] * N:] == 0).all()


def test_brute_force_tiny():
    """Selection by its rank definition (sub-expert s is taken iff fewer than
    k_t sub-experts beat it, a tie beaten by the lower index; its slot is that
    count) and gates from the parent softmax over the distinct chosen parents,
    all in plain Python loops, with exact ties in logits and weights."""
    rng = np.random.default_rng(7)
    Ep, N = 3, 2
    E = Ep * N
    for trial in range(300):
        l = (rng.integers(-2, 3, size=(1, Ep)) * 0.5).astype(np.float32)
        logw = (rng.integers(-2, 1, size=E) * 0.25).astype(np.float32)
        kt = int(rng.integers(1, E + 1))
        idx, w = oracle.hier_route(l, logw, N, [kt], E)
        score = [np.float32(l[0, s // N]) + np.float32(logw[s]) for s in range(E)]
        want = [-1] * E
        for s in range(E):
            beat = sum(1 for o in range(E) if score[o] > score[s] or (score[o] == score[s] and o < s))
            if beat < kt:
                want[beat] = s
        assert idx[0].tolist() == want
        chosen = sorted({s // N for s in want[:kt]})
        mx = max(float(l[0, e]) for e in chosen)
        den = sum(math.exp(float(l[0, e]) - mx) for e in chosen)
        for j in range(kt):
            g = math.exp(float(l[0, want[j] // N]) - mx) / den
            assert w[0, j] == np.float32(g)


def test_hand_example():
    # parents: logits 1 and 0; co-activation weights 0.7/0.3 and 0.9/0.1.
    # scores: 1+ln .7 = 0.643, 1+ln .3 = -0.204, ln .9 = -0.105, ln .1 = -2.303
    # -> order 0, 2, 1, 3; parent gates e/(e+1) = 0.7310586, 1/(e+1) = 0.2689414
    l = np.array([[1.0, 0.0]], dtype=np.float32)
    logw = np.log(np.array([0.7, 0.3, 0.9, 0.1])).astype(np.float32)
    g0, g1 = math.e / (math.e + 1), 1 / (math.e + 1)
    cases = {1: ([0], [1.0]), 2: ([0, 2], [g0, g1]), 3: ([0, 2, 1], [g0, g1, g0]),
             4: ([0, 2, 1, 3], [g0, g1, g0, g1])}
    for kt, (want_idx, want_w) in cases.items():
        idx, w = oracle.hier_route(l, logw, 2, [kt], 4)
        assert idx[0, :kt].tolist() == want_idx
        np.testing.assert_allclose(w[0, :kt], want_w, rtol=1e-7)


def test_split_weights_partition_the_neurons():
    """Sub-expert i of parent e holds its neurons [i*I/N, (i+1)*I/N): the
    sub-experts' outputs add up to the parent's (float64, no rounding)."""
    rng = np.random.default_rng(3)
    Ep, N, H, I = 3, 4, 16, 24
    w13 = rng.standard_normal((Ep, 2 * I, H))
    w2 = rng.standard_normal((Ep, H, I))
    s13, s2 = oracle.split_expert_weights(w13, w2, N)
    assert s13.shape == (Ep * N, 2 * I // N, H) and s2.shape == (Ep * N, H, I // N)
    x = rng.standard_normal((10, H))
    for e in range(Ep):
        g = x @ w13[e, :I].T
        u = x @ w13[e, I:].T
        parent = (oracle.silu(g) * u) @ w2[e].T
        parts = 0
        for i in range(N):
            s = e * N + i
            Is = I // N
            parts = parts + (oracle.silu(x @ s13[s, :Is].T) * (x @ s13[s, Is:].T)) @ s2[s].T
        np.testing.assert_allclose(parts, parent, rtol=1e-12, atol=1e-12)


def test_every_sub_expert_gives_the_dense_mixture():
    """With every sub-expert selected, the gated sum over sub-experts equals the
    dense softmax mixture of the parent experts."""
    rng = np.random.default_rng(5)
    Ep, N, H, I, T = 4, 2, 8, 12, 6
    w13 = rng.standard_normal((Ep, 2 * I, H)) / np.sqrt(H)
    w2 = rng.standard_normal((Ep, H, I)) / np.sqrt(I)
    s13, s2 = oracle.split_expert_weights(w13, w2, N)
    x = rng.standard_normal((T, H))
    l = rng.standard_normal((T, Ep)).astype(np.float32)
    logw = np.log(rng.dirichlet(np.ones(N), size=Ep).reshape(-1)).astype(np.float32)
    E = Ep * N
    idx, w = oracle.hier_route(l, logw, N, np.full(T, E), E)
    p = np.exp(l.astype(np.float64) - l.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    for t in range(T):
        got = sum(w[t, j] * oracle.expert_ffn(x[t:t + 1], s13[idx[t, j]], s2[idx[t, j]], "f64")[1]
                  for j in range(E))
        want = sum(p[t, e] * oracle.expert_ffn(x[t:t + 1], w13[e], w2[e], "f64")[1] for e in range(Ep))
        np.testing.assert_allclose(got, want, rtol=1e-6, atol=1e-7)


def test_scores_are_fp32_sums():
    l = np.array([[1.0, 2.0 ** -30]], dtype=np.float32)
    logw = np.array([2.0 ** -30, 0.0, 1.0, 0.0], dtype=np.float32)
    s = oracle.sub_scores(l, logw, 2)
    assert s.dtype == np.float32
    # 1 + 2^-30 rounds to 1 in fp32: sub-experts 0 and 1 tie, and 2 (= 1 + 2^-30 -> 1) ties them too
    assert s[0, 0] == s[0, 1] == s[0, 2] == np.float32(1.0)
    idx, _ = oracle.hier_route(l, logw, 2, [3], 3)
    assert idx[0].tolist() == [0, 1, 2]


def test_invalid_budget_rejected():
    with pytest.raises(ValueError):
        oracle.hier_route(np.zeros((1, 2), np.float32), np.zeros(4, np.float32), 2, [5], 5)
    with pytest.raises(ValueError):
        oracle.hier_route(np.zeros((1, 2), np.float32), np.zeros(3, np.float32), 2, [1], 1)
