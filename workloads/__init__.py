"""Seeded synthetic inputs for the affinity-aware MoE layer.

This module only draws inputs.  It computes none of the layer's arithmetic
(no routing, no sort, no FFN); both the CUDA path's tests/benchmark and the
CPU oracle's tests take their inputs from here, and nothing else is shared
between them.

The pages measure on real models (DeepSeek-V2-Lite, Qwen3-30B-A3B, OLMoE) and
real corpora (ShareGPT, LMSYS-Chat-1M, MMLU); none of those is available, so
every input here is a synthetic stand-in with the shapes of those models'
MoE layers and a token-id distribution with the skew of natural text:

* token ids: a finite Zipf law over V ranks (p(r) proportional to r^-s),
  sampled by inverse CDF; id = rank - 1 (so id 0 is the most frequent);
* token-expert affinity (the pages' observation that a token id alone
  predicts its experts, Semantic Parallelism (ko) §2.1): each id v has
  ``k_pref`` preferred experts drawn from a splitmix64 stream seeded with
  ``seed ^ v``; router logits carry a bias on those experts plus N(0,1) noise;
* expert placement (a stand-in for the pages' offline 0-1 ILP co-clustering,
  Semantic Parallelism (de) §2 B): greedy balanced clustering of experts by
  co-activation mass;
* the token-id -> rank table (Semantic Parallelism (ja) §2.3, lookup table):
  the rank that holds most of an id's preferred experts, ties to the lowest.

Random draws use numpy's PCG64; bf16 casts use torch's (library) conversion.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

__all__ = ["LayerSpec", "CONFIGS", "BENCH_CONFIG", "make_inputs", "splitmix64",
           "zipf_ids", "preferred_experts", "clustered_placement", "lut_from_preferences"]


@dataclass(frozen=True)
class LayerSpec:
    """Shape and input recipe of one MoE layer workload."""
    name: str
    T: int                      # tokens in the batch
    H: int                      # hidden size
    E: int                      # routed experts (sub-experts for the MoE-Prism layer)
    I: int                      # expert intermediate size
    R: int                      # logical ranks
    k: int                      # top-k (uniform), or k_max when k_choices is set
    dtype: str                  # "f32" or "bf16": activations and expert weights
    router_dtype: str           # "f32" or "bf16": router weight
    I_shared: int = 0           # concatenated shared-expert intermediate (0 = none)
    V: int = 1000               # vocabulary size
    zipf_s: Optional[float] = None  # None = uniform token ids
    bias: float = 0.0           # router-logit bias on preferred experts
    k_pref: int = 0             # preferred experts per token id
    placement: str = "modulo"   # "modulo": e % R ; "clustered": greedy co-activation
    lut: str = "uniform"        # "uniform": U[0,R) ; "affinity": rank of most preferred
    sub_split: int = 1          # sub-experts per parent expert (MoE-Prism)
    k_choices: tuple = ()       # per-request top-k budgets, request r gets k_choices[r % len]
    tokens_per_request: int = 1
    req_len_mean: int = 0       # > 0: requests of lognormal length with this mean (prefill batches)
    seed: int = 1000

    @property
    def k_max(self) -> int:
        return max(self.k_choices) if self.k_choices else self.k


def _spec(**kw) -> LayerSpec:
    return LayerSpec(**kw)


CONFIGS = {
    # Tiny correctness layer, fp32 throughout.
    "tiny_fp32_T256_E8": _spec(
        name="tiny_fp32_T256_E8", T=256, H=128, E=8, I=256, R=4, k=2, dtype="f32",
        router_dtype="f32", V=1000, placement="modulo", lut="uniform", seed=1000),
    # DeepSeek-V2-Lite-shaped MoE layer, prefill: 64 routed experts top-6 + 2 shared.
    "dsv2lite_prefill_T4096": _spec(
        name="dsv2lite_prefill_T4096", T=4096, H=2048, E=64, I=1408, R=8, k=6,
        dtype="bf16", router_dtype="f32", I_shared=2816, V=102400, zipf_s=1.1,
        bias=3.0, k_pref=6, placement="clustered", lut="affinity", req_len_mean=512, seed=1001),
    # Decode-shaped variants of the same layer (one token per request).
    "dsv2lite_decode_T64": _spec(
        name="dsv2lite_decode_T64", T=64, H=2048, E=64, I=1408, R=8, k=6,
        dtype="bf16", router_dtype="f32", I_shared=2816, V=102400, zipf_s=1.1,
        bias=3.0, k_pref=6, placement="clustered", lut="affinity", seed=1002),
    "dsv2lite_decode_T256": _spec(
        name="dsv2lite_decode_T256", T=256, H=2048, E=64, I=1408, R=8, k=6,
        dtype="bf16", router_dtype="f32", I_shared=2816, V=102400, zipf_s=1.1,
        bias=3.0, k_pref=6, placement="clustered", lut="affinity", seed=1002),
    "dsv2lite_decode_T512": _spec(
        name="dsv2lite_decode_T512", T=512, H=2048, E=64, I=1408, R=8, k=6,
        dtype="bf16", router_dtype="f32", I_shared=2816, V=102400, zipf_s=1.1,
        bias=3.0, k_pref=6, placement="clustered", lut="affinity", seed=1002),
    # Qwen3-30B-A3B-shaped layer: 128 experts top-8, no shared expert, bf16 router.
    "qwen3_30b_a3b_T16384": _spec(
        name="qwen3_30b_a3b_T16384", T=16384, H=2048, E=128, I=768, R=8, k=8,
        dtype="bf16", router_dtype="bf16", V=151936, zipf_s=1.0, bias=2.5, k_pref=8,
        placement="clustered", lut="affinity", req_len_mean=1024, seed=1003),
    # MoE-Prism elastic layer: 64 experts x 4 sub-experts (I = 1408 / 4 = 352),
    # 32 requests of 256 tokens with budgets {12,16,20,24} in one batch.
    "prism_subexpert_T8192": _spec(
        name="prism_subexpert_T8192", T=8192, H=2048, E=256, I=352, R=8, k=24,
        dtype="bf16", router_dtype="f32", V=102400, zipf_s=1.1, bias=3.0, k_pref=6,
        placement="clustered", lut="affinity", sub_split=4, k_choices=(12, 16, 20, 24),
        tokens_per_request=256, seed=1004),
}

#: the layer the throughput metric is quoted on: the largest workload (by
#: tokens and by FFN flops), on which the grouped FFN's tensor-peak target is set
BENCH_CONFIG = "qwen3_30b_a3b_T16384"


# ---------------------------------------------------------------------------
# random streams
# ---------------------------------------------------------------------------
_MASK64 = np.uint64(0xFFFFFFFFFFFFFFFF)


def splitmix64(seed: np.ndarray, n: int) -> np.ndarray:
    """First ``n`` outputs of Vigna's SplitMix64 generator for each seed.

    ``seed``: uint64 array of shape [S]; returns uint64 [S, n].
    """
    s = np.asarray(seed, dtype=np.uint64).copy()
    out = np.empty((s.shape[0], n), dtype=np.uint64)
    with np.errstate(over="ignore"):
        for i in range(n):
            s = s + np.uint64(0x9E3779B97F4A7C15)
            z = s.copy()
            z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
            z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
            out[:, i] = z ^ (z >> np.uint64(31))
    return out


def zipf_ids(rng: np.random.Generator, T: int, V: int, s: Optional[float]) -> np.ndarray:
    """T token ids in [0, V): uniform when s is None, else finite Zipf(s) by inverse CDF."""
    if s is None:
        return rng.integers(0, V, size=T, dtype=np.int64).astype(np.int32)
    ranks = np.arange(1, V + 1, dtype=np.float64)
    p = ranks ** (-s)
    cdf = np.cumsum(p)
    cdf /= cdf[-1]
    u = rng.random(T)
    ids = np.searchsorted(cdf, u, side="right")
    return np.minimum(ids, V - 1).astype(np.int32)


def zipf_probs(V: int, s: float) -> np.ndarray:
    p = np.arange(1, V + 1, dtype=np.float64) ** (-s)
    return p / p.sum()


def preferred_experts(V: int, n_units: int, k_pref: int, seed: int) -> np.ndarray:
    """[V, k_pref] int32: the first k_pref distinct values (mod n_units) of a
    splitmix64 stream seeded with ``seed ^ v`` for each token id v."""
    draws = 16 * k_pref + 32
    vals = splitmix64(np.uint64(seed) ^ np.arange(V, dtype=np.uint64), draws)
    cand = (vals % np.uint64(n_units)).astype(np.int64)
    taken = np.zeros((V, n_units), dtype=bool)
    pref = np.full((V, k_pref), -1, dtype=np.int64)
    count = np.zeros(V, dtype=np.int64)
    rows = np.arange(V)
    for c in range(draws):
        col = cand[:, c]
        new = (~taken[rows, col]) & (count < k_pref)
        r = rows[new]
        taken[r, col[new]] = True
        pref[r, count[new]] = col[new]
        count[new] += 1
    if (count < k_pref).any():
        raise RuntimeError("preferred-expert stream too short")
    return pref.astype(np.int32)


def clustered_placement(pref: np.ndarray, p_id: np.ndarray, n_units: int, R: int) -> np.ndarray:
    """Greedy balanced co-activation clustering of n_units experts onto R ranks.

    C[e][f] = sum_v p(v) [e in pref(v)][f in pref(v)].  Rank r is seeded with the
    unassigned expert of largest load C[e][e], then grows by the unassigned expert
    with the largest co-activation mass to its members until n_units / R members
    (ties to the lowest id).  Returns rank_of[n_units] int32.
    """
    V, kp = pref.shape
    M = np.zeros((V, n_units), dtype=np.float64)
    M[np.repeat(np.arange(V), kp), pref.reshape(-1)] = 1.0
    C = M.T @ (M * p_id[:, None])
    per = n_units // R
    rank_of = np.full(n_units, -1, dtype=np.int32)
    load = np.diag(C).copy()
    for r in range(R):
        free = np.flatnonzero(rank_of < 0)
        seed_e = free[np.argmax(load[free])]          # argmax returns the first maximum
        rank_of[seed_e] = r
        members = [seed_e]
        while len(members) < per:
            free = np.flatnonzero(rank_of < 0)
            score = C[np.array(members)][:, free].sum(axis=0)
            f = free[np.argmax(score)]
            rank_of[f] = r
            members.append(f)
    return rank_of


def lut_from_preferences(pref: np.ndarray, rank_of_unit: np.ndarray, R: int) -> np.ndarray:
    """lut[v] = the rank holding most of v's preferred units (ties to the lowest rank)."""
    V = pref.shape[0]
    votes = np.zeros((V, R), dtype=np.int64)
    np.add.at(votes, (np.repeat(np.arange(V), pref.shape[1]), rank_of_unit[pref].reshape(-1)), 1)
    return np.argmax(votes, axis=1).astype(np.int32)


_CHUNK = 1 << 24


def _normal_f32(shape, scale: float, seed: int, tag: int) -> np.ndarray:
    """N(0, scale^2) float32 array; fixed 16M-element chunks, each from its own
    PCG64 stream spawned from SeedSequence([seed, tag]), drawn on threads
    (the result does not depend on the thread count)."""
    from concurrent.futures import ThreadPoolExecutor
    n = int(np.prod(shape))
    a = np.empty(n, dtype=np.float32)
    nchunks = (n + _CHUNK - 1) // _CHUNK
    seqs = np.random.SeedSequence([seed, tag]).spawn(nchunks)

    def fill(i):
        g = np.random.Generator(np.random.PCG64(seqs[i]))
        sl = a[i * _CHUNK:min(n, (i + 1) * _CHUNK)]
        g.standard_normal(out=sl, dtype=np.float32)
        sl *= np.float32(scale)

    with ThreadPoolExecutor(max_workers=16) as ex:
        list(ex.map(fill, range(nchunks)))
    return a.reshape(shape)


def request_offsets(T: int, seed: int, mean_len: int = 0, fixed_len: int = 1,
                    empty_every: int = 0) -> np.ndarray:
    """Token offsets [n_req+1] (int32) of the requests in a batch of T tokens.

    mean_len > 0: lengths drawn lognormal (sigma 0.8) with that mean, at least 1,
    the last request cut at T (a prefill batch of prompts); otherwise every
    request has ``fixed_len`` tokens (the last one the remainder).
    empty_every > 0 inserts an empty request after every that many requests.
    """
    if mean_len > 0:
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1001])))
        lens = []
        total = 0
        sigma = 0.8
        mu = np.log(mean_len) - sigma * sigma / 2
        while total < T:
            n = int(max(1, round(rng.lognormal(mu, sigma))))
            n = min(n, T - total)
            lens.append(n)
            total += n
    else:
        full, rest = divmod(T, fixed_len)
        lens = [fixed_len] * full + ([rest] if rest else [])
    if empty_every > 0:
        out = []
        for i, n in enumerate(lens):
            out.append(n)
            if (i + 1) % empty_every == 0:
                out.append(0)
        lens = out
    return np.concatenate([[0], np.cumsum(lens, dtype=np.int64)]).astype(np.int32)


def transition_table(E: int, R: int, seed: int, samples: int = 1000) -> np.ndarray:
    """Expert -> next-layer-rank transition counts [E,R] (float32, integer-valued).

    Row e is ``samples`` draws from a multinomial whose probabilities follow a
    Dirichlet(0.3) law, so each expert leans to a few ranks, as a table profiled
    from a skewed routing trace would.  Integer values keep fp32 sums exact.
    """
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 1002])))
    probs = rng.dirichlet(np.full(R, 0.3), size=E)
    return np.stack([rng.multinomial(samples, p) for p in probs]).astype(np.float32)


def _to(a: np.ndarray, dtype: str) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16) if dtype == "bf16" else t


def make_inputs(spec: LayerSpec, with_weights: bool = True) -> dict:
    """Draw every input of one layer call for ``spec`` (CPU torch tensors).

    Returns x [T,H], w_router [E,H], w13 [E,2I,H] (rows 0..I-1 gate, I..2I-1 up),
    w2 [E,H,I], ws13 [2*I_shared,H] / ws2 [H,I_shared] (or None), token_ids [T],
    lut [V], expert_rank [E], k_per_token [T], req_offsets [n_req+1] (all int32),
    trans [E,R] (float32 next-layer transition counts), for MoE-Prism layers
    w_router_parent [E/N,H] and sub_logw [E] (float32; else None), and the spec.
    """
    rng = np.random.Generator(np.random.PCG64(spec.seed))
    T, H, E, I, R = spec.T, spec.H, spec.E, spec.I, spec.R
    ids = zipf_ids(rng, T, spec.V, spec.zipf_s)
    parents = E // spec.sub_split

    if spec.placement == "modulo":
        expert_rank = (np.arange(E) % R).astype(np.int32)
        pref = None
    else:
        pref = preferred_experts(spec.V, parents, spec.k_pref, spec.seed)
        p_id = zipf_probs(spec.V, spec.zipf_s) if spec.zipf_s else np.full(spec.V, 1.0 / spec.V)
        parent_rank = clustered_placement(pref, p_id, parents, R)
        expert_rank = np.repeat(parent_rank, spec.sub_split).astype(np.int32)

    if spec.lut == "uniform":
        lut = rng.integers(0, R, size=spec.V).astype(np.int32)
    else:
        lut = lut_from_preferences(pref, expert_rank[::spec.sub_split], R)

    if spec.bias == 0.0:
        x = rng.standard_normal((T, H)) / np.sqrt(H)
        w_router = rng.standard_normal((E, H)) / np.sqrt(H)
    else:
        if E > H:
            raise ValueError("affinity-biased routing needs E <= H (orthonormal router rows)")
        # Router with orthonormal rows; x carries the target logits along them
        # plus an orthogonal N(0,1)/sqrt(H) component, so x . Wr^T = target.
        G = rng.standard_normal((H, E))
        Q, _ = np.linalg.qr(G)
        w_router = Q.T.copy()
        target = rng.standard_normal((T, E))
        pt = pref[ids]                                   # [T, k_pref] parent ids
        rows = np.repeat(np.arange(T), pt.shape[1] * spec.sub_split)
        cols = (pt[:, :, None] * spec.sub_split + np.arange(spec.sub_split)).reshape(-1)
        target[rows, cols] += spec.bias
        g = rng.standard_normal((T, H)) / np.sqrt(H)
        g -= (g @ w_router.T) @ w_router
        x = target @ w_router + g

    # MoE-Prism layers: the parent router (row e = the sum of its sub-experts'
    # rows / sqrt(N), so its logits carry the parents' affinity bias) and the
    # sub-experts' co-activation weights a[e, i] ~ Dirichlet(2) over i, as logs.
    N = spec.sub_split
    w_router_parent = sub_logw = None
    if N > 1:
        w_router_parent = w_router.reshape(parents, N, H).sum(axis=1) / np.sqrt(N)
        crng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([spec.seed, 1003])))
        sub_logw = np.log(crng.dirichlet(np.full(N, 2.0), size=parents)).reshape(-1).astype(np.float32)

    if spec.k_choices:
        req = np.arange(T) // spec.tokens_per_request
        kpt = np.asarray(spec.k_choices, dtype=np.int32)[req % len(spec.k_choices)]
    else:
        kpt = np.full(T, spec.k, dtype=np.int32)

    out = dict(
        spec=spec,
        x=_to(x, spec.dtype),
        w_router=_to(w_router, spec.router_dtype),
        token_ids=torch.from_numpy(ids.astype(np.int32)),
        lut=torch.from_numpy(lut),
        expert_rank=torch.from_numpy(expert_rank.astype(np.int32)),
        k_per_token=torch.from_numpy(kpt.astype(np.int32)),
        req_offsets=torch.from_numpy(request_offsets(T, spec.seed, spec.req_len_mean, spec.tokens_per_request)),
        trans=torch.from_numpy(transition_table(E, R, spec.seed)),
        w_router_parent=None if w_router_parent is None else _to(w_router_parent, spec.router_dtype),
        sub_logw=None if sub_logw is None else torch.from_numpy(sub_logw),
        w13=None, w2=None, ws13=None, ws2=None,
    )
    if with_weights:
        tags = iter(range(1, 100))

        def normal(shape, fan_in):
            return _normal_f32(shape, 1.0 / np.sqrt(fan_in), spec.seed, next(tags))
        out["w13"] = _to(normal((E, 2 * I, H), H), spec.dtype)
        out["w2"] = _to(normal((E, H, I), I), spec.dtype)
        if spec.I_shared:
            out["ws13"] = _to(normal((2 * spec.I_shared, H), H), spec.dtype)
            out["ws2"] = _to(normal((H, spec.I_shared), spec.I_shared), spec.dtype)
    return out


def scaled(name: str, **overrides) -> LayerSpec:
    """A copy of a named spec with some fields replaced (smaller parity cases)."""
    return dataclasses.replace(CONFIGS[name], **overrides)
