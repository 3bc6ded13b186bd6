"""Sanity of the seeded synthetic inputs (CPU only)."""
import numpy as np

import workloads as wl


def test_splitmix64_reference_values():
    # first outputs of SplitMix64 seeded with 0 (values published with the generator)
    got = wl.splitmix64(np.array([0], dtype=np.uint64), 3)[0]
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_zipf_ids_follow_the_law():
    rng = np.random.Generator(np.random.PCG64(0))
    V, s = 1000, 1.1
    ids = wl.zipf_ids(rng, 200000, V, s)
    assert ids.min() >= 0 and ids.max() < V
    freq = np.bincount(ids, minlength=V) / len(ids)
    p = wl.zipf_probs(V, s)
    np.testing.assert_allclose(freq[:5], p[:5], rtol=0.05)


def test_preferred_experts_distinct_and_in_range():
    pref = wl.preferred_experts(500, 64, 6, 7)
    assert pref.shape == (500, 6) and pref.min() >= 0 and pref.max() < 64
    assert all(len(set(r)) == 6 for r in pref.tolist())


def test_clustered_placement_is_balanced():
    V, E, R = 2000, 32, 4
    pref = wl.preferred_experts(V, E, 4, 3)
    rank_of = wl.clustered_placement(pref, wl.zipf_probs(V, 1.1), E, R)
    np.testing.assert_array_equal(np.bincount(rank_of, minlength=R), [E // R] * R)
    lut = wl.lut_from_preferences(pref, rank_of, R)
    assert lut.min() >= 0 and lut.max() < R


def test_tiny_layer_inputs():
    d = wl.make_inputs(wl.CONFIGS["tiny_fp32_T256_E8"])
    s = d["spec"]
    assert tuple(d["x"].shape) == (s.T, s.H) and tuple(d["w13"].shape) == (s.E, 2 * s.I, s.H)
    assert tuple(d["w2"].shape) == (s.E, s.H, s.I)
    np.testing.assert_array_equal(d["expert_rank"].numpy(), np.arange(8) % 4)
    assert (d["k_per_token"].numpy() == 2).all()
    d2 = wl.make_inputs(wl.CONFIGS["tiny_fp32_T256_E8"])
    assert bool((d["x"] == d2["x"]).all()) and bool((d["w2"] == d2["w2"]).all())


def test_affinity_bias_reaches_the_logits():
    spec = wl.scaled("dsv2lite_prefill_T4096", T=64, H=256, I=64, V=5000)
    d = wl.make_inputs(spec, with_weights=False)
    logits = d["x"].double() @ d["w_router"].double().T
    pref = wl.preferred_experts(spec.V, spec.E, spec.k_pref, spec.seed)[d["token_ids"].numpy()]
    top = np.argsort(-logits.numpy(), axis=1)[:, :spec.k]
    hit = np.mean([len(set(a) & set(b)) / spec.k for a, b in zip(top.tolist(), pref.tolist())])
    assert hit > 0.6


def test_prism_per_request_budgets():
    spec = wl.scaled("prism_subexpert_T8192", T=1024, H=512, I=32, V=3000)
    d = wl.make_inputs(spec, with_weights=False)
    k = d["k_per_token"].numpy()
    np.testing.assert_array_equal(k[::256], [12, 16, 20, 24])
    er = d["expert_rank"].numpy()
    assert (er.reshape(-1, 4) == er[::4, None]).all()
