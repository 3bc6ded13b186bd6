"""Pins of the CPU oracle to facts other than itself (CPU only).

Each test checks the oracle against something it cannot agree with by
construction: a hand-worked example, a brute-force definition, a textbook or
library routine, a closed form, an invariant, or a special case (k = E is a
dense softmax mixture; one expert with gate 1 is a plain SwiGLU MLP).
"""
import itertools
import json
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_hand():
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        d = json.load(f)
    d["logits"] = np.array([[float(v) for v in row] for row in d["logits"]])
    return d


# ---------------------------------------------------------------------------
# rounding and activation
# ---------------------------------------------------------------------------
def test_bf16_round_matches_library_cast():
    rng = np.random.default_rng(1)
    a = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),       # subnormals
        (rng.standard_normal(2000) * 1e38).astype(np.float32),        # near overflow
        np.float32(1.0) + np.arange(-64, 64, dtype=np.float32) * np.float32(2.0 ** -9),  # ties
        np.array([0.0, -0.0, 3.3895313892515355e38, -3.3895313892515355e38], np.float32),
    ])
    ref = torch.from_numpy(a).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_round(a.astype(np.float64))
    np.testing.assert_array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_bf16_round_hand_values():
    u = 2.0 ** -8
    cases = {1.0 + u: 1.0,                       # halfway, even neighbour below
             1.0 + 3 * u: 1.0 + 2 ** -6,          # halfway, even neighbour above
             1.0 + 1.5 * u: 1.0 + 2 ** -7,        # above halfway
             2.0 ** -133: 2.0 ** -133,            # smallest subnormal
             2.0 ** -134: 0.0,                    # halfway to zero -> even (0)
             3.0 * 2.0 ** -134: 2.0 ** -132,      # halfway between 1 and 2 quanta -> 2
             2.0 ** 128: np.inf, -(2.0 ** 128): -np.inf}
    for v, want in cases.items():
        assert oracle.bf16_round(np.array([v]))[0] == want, v


def test_silu_closed_forms():
    z = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(oracle.silu(z), z * scipy.special.expit(z), rtol=1e-14, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    # silu(z) - silu(-z) = z
    np.testing.assert_allclose(oracle.silu(z) - oracle.silu(-z), z, rtol=0, atol=1e-13)


# ---------------------------------------------------------------------------
# router: top-k and gates
# ---------------------------------------------------------------------------
def _brute_topk(l, k):
    """Expert i is chosen iff fewer than k experts beat it, where j beats i when
    l_j > l_i or (l_j == l_i and j < i); its slot is that number."""
    E = len(l)
    idx = [-1] * k
    for i in range(E):
        beat = sum(1 for j in range(E) if l[j] > l[i] or (l[j] == l[i] and j < i))
        if beat < k:
            idx[beat] = i
    return idx


def _tie_logits(rng, T, E):
    l = rng.integers(-3, 4, size=(T, E)).astype(np.float64) * 0.5   # many exact ties
    zero = rng.random((T, E)) < 0.2
    l[zero] = np.where(rng.random(zero.sum()) < 0.5, 0.0, -0.0)
    return l


def test_router_logits_golden():
    """Router logits against values worked by hand (tests/golden/router_logits.json):
    integer inputs (every product and sum exact), a case where the exact sum
    rounded once to fp32 differs from fp32 accumulation, and the fp32 storage
    point itself.  A dropped term, a transposed weight or a sum accumulated in
    fp32 fails one of them."""
    with open(os.path.join(GOLDEN, "router_logits.json")) as f:
        g = json.load(f)
    for name in ("integer_case", "one_rounding_case", "storage_case"):
        c = g[name]
        got = oracle.router_logits(np.array(c["x"], dtype=np.float64), np.array(c["w_router"], dtype=np.float64))
        want = np.array(c["logits"], dtype=np.float64)
        assert got.shape == want.shape, name
        assert np.array_equal(got, want), (name, got, want)
    # the rounding case really separates the two readings
    c = g["one_rounding_case"]
    acc = np.float32(0)
    for a, b in zip(c["x"][0], c["w_router"][0]):
        acc = np.float32(acc + np.float32(a) * np.float32(b))
    assert float(acc) == 1.0 != c["logits"][0][0]
    # not symmetric in x and Wr: transposing the weight gives another result
    c = g["integer_case"]
    wt = np.array(c["w_router"], dtype=np.float64).T
    assert not np.array_equal(oracle.router_logits(np.array(c["x"], dtype=np.float64), wt),
                              np.array(c["logits"], dtype=np.float64))


@pytest.mark.parametrize("E", [1, 2, 3, 8])
def test_topk_brute_force(E):
    rng = np.random.default_rng(E)
    T = 200
    l = _tie_logits(rng, T, E)
    k_max = E
    k = rng.integers(1, E + 1, size=T)
    idx, w = oracle.topk_route(l, k, k_max)
    for t in range(T):
        want = _brute_topk(list(l[t]), int(k[t])) + [-1] * (k_max - int(k[t]))
        assert list(idx[t]) == want


def test_topk_maximises_sum_of_selected_logits():
    rng = np.random.default_rng(7)
    E = 7
    for _ in range(50):
        l = rng.standard_normal(E)
        for k in range(1, E + 1):
            idx, _ = oracle.topk_route(l[None, :], [k], k)
            best = max(sum(l[list(c)]) for c in itertools.combinations(range(E), k))
            assert abs(l[idx[0]].sum() - best) < 1e-12


def test_topk_prefix_property():
    """Cutting a request's budget keeps a prefix of its expert list (MoE-Prism's
    "same model, fewer experts")."""
    rng = np.random.default_rng(3)
    l = _tie_logits(rng, 300, 16)
    full, _ = oracle.topk_route(l, np.full(300, 16), 16)
    for k in range(1, 16):
        idx, _ = oracle.topk_route(l, np.full(300, k), k)
        np.testing.assert_array_equal(idx, full[:, :k])


def test_gates_sum_to_one_and_k_equals_E_is_softmax():
    rng = np.random.default_rng(4)
    l = (rng.standard_normal((500, 12)) * 4).astype(np.float32).astype(np.float64)
    k = rng.integers(1, 13, size=500)
    idx, w = oracle.topk_route(l, k, 12)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, atol=1e-6)
    assert (w[np.arange(12)[None, :] >= k[:, None]] == 0).all()
    # k = E: gates are the plain softmax (library routine), in slot order
    idx, w = oracle.topk_route(l, np.full(500, 12), 12)
    sm = scipy.special.softmax(l, axis=1)
    np.testing.assert_allclose(w, np.take_along_axis(sm, idx, axis=1), rtol=1e-6, atol=1e-12)
    # gates are fp32 values
    assert np.array_equal(w, w.astype(np.float32).astype(np.float64))


def test_topk_input_validation():
    with pytest.raises(ValueError):
        oracle.topk_route(np.zeros((2, 4)), [1, 5], 5)
    with pytest.raises(ValueError):
        oracle.topk_route(np.zeros((2, 4)), [0, 1], 2)


# ---------------------------------------------------------------------------
# the hand-worked example
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["uniform_k2", "per_request_k"])
def test_hand_example(case):
    d = _load_hand()
    c = d[case]
    k = np.array(c["k_per_token"])
    idx, w = oracle.topk_route(d["logits"], k, d["k_max"])
    np.testing.assert_array_equal(idx, c["topk_idx"])
    if "topk_w" in c:
        np.testing.assert_allclose(w, c["topk_w"], rtol=1e-7)
    perm = oracle.permute(idx, k, d["expert_rank"], d["R"])
    for key in ("sorted_to_pair", "pair_to_sorted", "expert_offsets", "rank_offsets"):
        np.testing.assert_array_equal(perm[key], c[key], err_msg=key)
    if "phys_to_expert" in c:
        np.testing.assert_array_equal(perm["phys_to_expert"], c["phys_to_expert"])
        np.testing.assert_array_equal(perm["expert_counts"], c["expert_counts"])
    if "counts" in c:
        counts, remote = oracle.remote_count(idx, k, d["pred_rank"], d["expert_rank"], d["R"])
        np.testing.assert_array_equal(counts, c["counts"])
        np.testing.assert_array_equal(remote, c["remote"])
        assert np.trace(counts) / counts.sum() == c["local_activation_rate"]


# ---------------------------------------------------------------------------
# permutation (the on-device shuffle)
# ---------------------------------------------------------------------------
def _counting_sort(topk_idx, k, expert_rank, R):
    """Textbook stable counting sort, written independently of the oracle:
    bucket order by (rank, expert) found by scanning ranks then experts."""
    T, k_max = topk_idx.shape
    E = len(expert_rank)
    bucket_of = {}
    order = []
    for r in range(R):
        for e in range(E):
            if expert_rank[e] == r:
                bucket_of[e] = len(order)
                order.append(e)
    hist = [0] * E
    for t in range(T):
        for j in range(k[t]):
            hist[bucket_of[topk_idx[t, j]]] += 1
    start = [0] * (E + 1)
    for b in range(E):
        start[b + 1] = start[b] + hist[b]
    nxt = start[:-1].copy()
    s2p = [0] * start[E]
    p2s = [-1] * (T * k_max)
    for t in range(T):
        for j in range(k[t]):
            b = bucket_of[topk_idx[t, j]]
            s2p[nxt[b]] = t * k_max + j
            p2s[t * k_max + j] = nxt[b]
            nxt[b] += 1
    return order, start, s2p, p2s


def _random_routing(rng, T, E, k_max, skew=None, per_token=True):
    l = rng.standard_normal((T, E))
    if skew is not None:
        l[:, skew] += 50.0                     # every token picks expert `skew` first
    k = rng.integers(1, k_max + 1, size=T) if per_token else np.full(T, k_max)
    idx, _ = oracle.topk_route(l, k, k_max)
    return idx, k


@pytest.mark.parametrize("T,E,R,k_max,skew", [
    (1, 1, 1, 1, None), (1, 8, 4, 3, None), (37, 8, 4, 2, None), (64, 16, 4, 5, 3),
    (200, 64, 8, 6, None), (150, 12, 3, 12, None), (90, 10, 5, 4, 9)])
def test_permute_matches_counting_sort(T, E, R, k_max, skew):
    rng = np.random.default_rng(T * 1000 + E)
    idx, k = _random_routing(rng, T, E, k_max, skew)
    er = rng.permutation(np.arange(E) % R)
    perm = oracle.permute(idx, k, er, R)
    order, start, s2p, p2s = _counting_sort(idx, k, er, R)
    np.testing.assert_array_equal(perm["phys_to_expert"], order)
    np.testing.assert_array_equal(perm["expert_offsets"], start)
    np.testing.assert_array_equal(perm["sorted_to_pair"], s2p)
    np.testing.assert_array_equal(perm["pair_to_sorted"], p2s)


def test_permute_invariants():
    rng = np.random.default_rng(11)
    T, E, R, k_max, H = 120, 16, 4, 5, 6
    idx, k = _random_routing(rng, T, E, k_max)
    er = rng.integers(0, R, size=E)            # unbalanced placement, maybe empty ranks
    x = rng.standard_normal((T, H))
    perm = oracle.permute(idx, k, er, R, x)
    P = int(k.sum())
    s2p, p2s = perm["sorted_to_pair"], perm["pair_to_sorted"]
    assert len(s2p) == P
    np.testing.assert_array_equal(p2s[s2p], np.arange(P))
    # un-permute restores every (token, slot) row
    for t in range(T):
        for j in range(k[t]):
            np.testing.assert_array_equal(perm["x_perm"][p2s[t * k_max + j]], x[t])
    # counts are the top-k histogram; offsets its exclusive scan in rank-major order
    live = idx[idx >= 0]
    np.testing.assert_array_equal(perm["expert_counts"], np.bincount(live, minlength=E))
    assert perm["expert_counts"].sum() == P
    np.testing.assert_array_equal(np.diff(perm["expert_offsets"]),
                                  perm["expert_counts"][perm["phys_to_expert"]])
    np.testing.assert_array_equal(np.diff(perm["rank_offsets"]),
                                  np.bincount(er[live], minlength=R))
    # keys are non-decreasing along the sorted order, pair ids increase within a key
    key = np.argsort(perm["phys_to_expert"])[idx.reshape(-1)[s2p]]
    assert (np.diff(key) >= 0).all()
    same = np.diff(key) == 0
    assert (np.diff(s2p)[same] > 0).all()


# ---------------------------------------------------------------------------
# affinity lookup and remote count
# ---------------------------------------------------------------------------
def test_remote_count_brute_force_and_invariants():
    rng = np.random.default_rng(5)
    T, E, R, k_max, V = 80, 12, 3, 4, 50
    idx, k = _random_routing(rng, T, E, k_max)
    er = rng.integers(0, R, size=E)
    lut = rng.integers(0, R, size=V)
    ids = rng.integers(0, V, size=T)
    pred = oracle.affinity_lookup(ids, lut)
    for t in range(T):
        assert pred[t] == lut[ids[t]]
    counts, remote = oracle.remote_count(idx, k, pred, er, R)
    want = np.zeros((R, R), dtype=np.int64)
    for t in range(T):
        for j in range(k[t]):
            want[pred[t], er[idx[t, j]]] += 1
    np.testing.assert_array_equal(counts, want)
    P = int(k.sum())
    assert counts.sum() == P
    assert np.trace(counts) + remote.sum() == P


# ---------------------------------------------------------------------------
# expert FFN and combine
# ---------------------------------------------------------------------------
def test_swiglu_closed_form_rectangular():
    """W1 selects the first I coordinates, W3 = 2 W1, W2 = W1^T:
    y[:, :I] = silu(x[:, :I]) * 2 x[:, :I] and y[:, I:] = 0 (a transposed or
    swapped operand breaks either the shape or the values)."""
    rng = np.random.default_rng(6)
    H, I, n = 12, 5, 9
    x = rng.standard_normal((n, H))
    sel = np.zeros((I, H))
    sel[np.arange(I), np.arange(I)] = 1.0
    w13 = np.concatenate([sel, 2.0 * sel])
    w2 = sel.T.copy()
    h, y = oracle.expert_ffn(x, w13, w2, "f64")
    xi = x[:, :I]
    np.testing.assert_allclose(y[:, :I], xi * scipy.special.expit(xi) * 2 * xi, rtol=1e-14)
    assert (y[:, I:] == 0).all()


def _layer_inputs(rng, T, H, E, I, R, V=40):
    return dict(
        x=rng.standard_normal((T, H)) / np.sqrt(H),
        w_router=rng.standard_normal((E, H)) / np.sqrt(H),
        token_ids=rng.integers(0, V, size=T),
        lut=rng.integers(0, R, size=V),
        expert_rank=np.arange(E) % R,
        w13=rng.standard_normal((E, 2 * I, H)) / np.sqrt(H),
        w2=rng.standard_normal((E, H, I)) / np.sqrt(I),
    )


def test_k_equals_E_is_dense_softmax_mixture():
    """With every expert selected the layer is sum_e softmax_e(x Wr^T) FFN_e(x),
    computed here densely, with no routing, sorting or permutation."""
    rng = np.random.default_rng(8)
    T, H, E, I, R = 23, 16, 6, 10, 3
    d = _layer_inputs(rng, T, H, E, I, R)
    res = oracle.moe_layer(d["x"], d["w_router"], d["token_ids"], d["lut"], d["expert_rank"],
                           np.full(T, E), d["w13"], d["w2"], R, "f64")
    logits = (d["x"] @ d["w_router"].T).astype(np.float32).astype(np.float64)
    gate = scipy.special.softmax(logits, axis=1)
    dense = np.zeros((T, H))
    for e in range(E):
        g = d["x"] @ d["w13"][e, :I].T
        u = d["x"] @ d["w13"][e, I:].T
        dense += gate[:, e:e + 1] * ((g * scipy.special.expit(g) * u) @ d["w2"][e].T)
    # the gates are fp32-rounded, so agreement is to ~1e-7 relative
    np.testing.assert_allclose(res["out"], dense, rtol=2e-6, atol=1e-9)


def test_single_expert_is_plain_swiglu_mlp():
    rng = np.random.default_rng(9)
    T, H, I = 17, 8, 12
    d = _layer_inputs(rng, T, H, 1, I, 1)
    res = oracle.moe_layer(d["x"], d["w_router"], d["token_ids"], d["lut"], d["expert_rank"],
                           np.ones(T, dtype=int), d["w13"], d["w2"], 1, "f64")
    g = d["x"] @ d["w13"][0, :I].T
    u = d["x"] @ d["w13"][0, I:].T
    mlp = (g * scipy.special.expit(g) * u) @ d["w2"][0].T
    np.testing.assert_allclose(res["out"], mlp, rtol=1e-12, atol=1e-15)
    np.testing.assert_array_equal(res["topk_w"], 1.0)


def test_grouped_ffn_routes_each_bucket_to_its_expert():
    """Bucket b's rows [off[b], off[b+1]) go through expert phys_to_expert[b]
    and only those rows: the experts are identical up to a factor e + 1 on W2,
    so each output row names the expert it used (uneven buckets, an empty one,
    a physical order that is not the identity)."""
    rng = np.random.default_rng(12)
    H, I, E = 8, 6, 4
    base13 = rng.standard_normal((2 * I, H))
    base2 = rng.standard_normal((H, I))
    w13 = np.stack([base13] * E)
    w2 = np.stack([(e + 1) * base2 for e in range(E)])
    off = np.array([0, 3, 3, 7, 9])
    pe = np.array([2, 0, 3, 1])
    x = rng.standard_normal((9, H))
    y = oracle.grouped_ffn(x, off, pe, w13, w2, "f64")
    g = x @ base13[:I].T
    u = x @ base13[I:].T
    one = (g * scipy.special.expit(g) * u) @ base2.T  # the factor-1 expert on every row
    for b in range(E):
        for q in range(off[b], off[b + 1]):
            np.testing.assert_allclose(y[q], (pe[b] + 1) * one[q], rtol=1e-12, atol=1e-14)


def test_shared_expert_adds_with_gate_one():
    rng = np.random.default_rng(10)
    T, H, E, I, R, Is = 15, 8, 4, 6, 2, 10
    d = _layer_inputs(rng, T, H, E, I, R)
    ws13 = rng.standard_normal((2 * Is, H))
    ws2 = rng.standard_normal((H, Is))
    k = np.full(T, 2)
    a = oracle.moe_layer(d["x"], d["w_router"], d["token_ids"], d["lut"], d["expert_rank"],
                         k, d["w13"], d["w2"], R, "f64")
    b = oracle.moe_layer(d["x"], d["w_router"], d["token_ids"], d["lut"], d["expert_rank"],
                         k, d["w13"], d["w2"], R, "f64", ws13=ws13, ws2=ws2)
    g = d["x"] @ ws13[:Is].T
    u = d["x"] @ ws13[Is:].T
    np.testing.assert_allclose(b["out"] - a["out"], (g * scipy.special.expit(g) * u) @ ws2.T,
                               rtol=1e-10, atol=1e-12)


def test_combine_hand_values():
    """Two tokens, k_max 2; token 1 has budget 1 (its second slot is padding)."""
    y_perm = np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0]])
    p2s = np.array([2, 0, 1, -1])
    w = np.array([[0.25, 0.75], [1.0, 0.0]])
    out = oracle.combine(y_perm, p2s, w, [2, 1], "f64", y_shared=np.array([[0.5, 0.5], [1.0, 1.0]]))
    np.testing.assert_array_equal(out, [[0.5 + 25 + 0.75, 0.5 + 50 + 1.5], [11.0, 21.0]])


def test_rounding_points_follow_the_storage_type():
    rng = np.random.default_rng(12)
    T, H, E, I, R = 30, 16, 4, 8, 2
    d = _layer_inputs(rng, T, H, E, I, R)
    d["x"] = oracle.bf16_round(d["x"])
    d["w13"] = oracle.bf16_round(d["w13"])
    d["w2"] = oracle.bf16_round(d["w2"])
    for dt in ("f32", "bf16"):
        res = oracle.moe_layer(d["x"], d["w_router"], d["token_ids"], d["lut"],
                               d["expert_rank"], np.full(T, 2), d["w13"], d["w2"], R, dt)
        for key in ("y_perm", "out"):
            np.testing.assert_array_equal(res[key], oracle.round_to(res[key], dt))
        exact = oracle.moe_layer(d["x"], d["w_router"], d["token_ids"], d["lut"],
                                 d["expert_rank"], np.full(T, 2), d["w13"], d["w2"], R, "f64")
        rel = np.abs(res["out"] - exact["out"]).max() / np.abs(exact["out"]).max()
        assert rel < (2 ** -7 if dt == "bf16" else 2 ** -20)
