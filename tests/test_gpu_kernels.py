"""Per-kernel parity of the CUDA path (through the C ABI) with the oracle,
including the degenerate cases: ties and signed zeros, per-token budgets,
E = 1, T = 1, k = E, empty experts, every token on one expert, empty ranks,
and data errors that the kernels must report instead of faulting."""
import numpy as np
import pytest
import torch

import oracle
from parity_utils import GATE_ATOL, LOGIT_TOL, TOL, max_rel, np_

pytestmark = pytest.mark.gpu

i32 = dict(dtype=torch.int32, device="cuda")


def abi():
    from token_expert_routing_gb300 import _abi
    return _abi


def route_logits_in(logits, k, k_max, expect_clean=True):
    T, E = logits.shape
    li = torch.as_tensor(logits, dtype=torch.float32).cuda()
    kpt = torch.as_tensor(k, dtype=torch.int32).cuda()
    idx = torch.empty(T, k_max, **i32)
    w = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
    abi().semmoe_route(None, None, li, None, kpt, 0, T, 0, E, k_max, idx, w)
    if expect_clean:
        assert abi().semmoe_check_errors() == 0
    else:
        torch.cuda.synchronize()
    return np_(idx), np_(w)


@pytest.mark.parametrize("T,E,k_max", [(1, 1, 1), (1, 8, 8), (333, 3, 2), (1000, 8, 8), (517, 64, 6),
                                       (300, 256, 24), (64, 256, 256), (97, 40, 33)])
def test_route_topk_ties_signed_zeros_per_token_k(T, E, k_max):
    rng = np.random.default_rng(T + E)
    logits = (rng.integers(-4, 5, size=(T, E)) * 0.25).astype(np.float32)
    z = rng.random((T, E)) < 0.2
    logits[z] = np.where(rng.random(z.sum()) < 0.5, np.float32(0.0), np.float32(-0.0))
    k = rng.integers(1, k_max + 1, size=T).astype(np.int32)
    idx, w = route_logits_in(logits, k, k_max)
    ref_idx, ref_w = oracle.topk_route(logits, k, k_max)
    np.testing.assert_array_equal(idx, ref_idx)
    np.testing.assert_allclose(w, ref_w, rtol=0, atol=GATE_ATOL)


@pytest.mark.parametrize("xd,wd", [(torch.float32, torch.float32), (torch.bfloat16, torch.float32),
                                   (torch.bfloat16, torch.bfloat16), (torch.float32, torch.bfloat16)])
@pytest.mark.parametrize("T,H,E", [(1, 64, 8), (77, 200, 64), (130, 2048, 256)])
def test_route_gemm(xd, wd, T, H, E):
    rng = np.random.default_rng(H + E)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32) / np.sqrt(H)).to(xd)
    wr = torch.from_numpy(rng.standard_normal((E, H)).astype(np.float32) / np.sqrt(H)).to(wd)
    k_max = min(6, E)
    idx = torch.empty(T, k_max, **i32)
    w = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
    lg = torch.empty(T, E, dtype=torch.float32, device="cuda")
    abi().semmoe_route(x.cuda(), wr.cuda(), None, lg, None, k_max, T, H, E, k_max, idx, w)
    assert abi().semmoe_check_errors() == 0
    assert max_rel(np_(lg), oracle.router_logits(x, wr)) < LOGIT_TOL
    ref_idx, ref_w = oracle.topk_route(np_(lg), np.full(T, k_max), k_max)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_allclose(np_(w), ref_w, rtol=0, atol=GATE_ATOL)


def _route_random(rng, T, E, k_max, skew=None, per_token=True):
    l = rng.standard_normal((T, E)).astype(np.float32)
    if skew is not None:
        l[:, skew] += 50.0
    k = rng.integers(1, k_max + 1, size=T) if per_token else np.full(T, k_max)
    idx, _ = oracle.topk_route(l, k, k_max)
    return idx.astype(np.int32), k.astype(np.int32)


@pytest.mark.parametrize("T,E,R,k_max,skew,H,placement", [
    (1, 1, 1, 1, None, 8, "mod"),
    (1, 8, 4, 3, None, 16, "mod"),
    (5000, 64, 8, 6, None, 64, "mod"),
    (3000, 16, 4, 5, 3, 32, "random"),        # every token picks expert 3 first
    (2049, 10, 5, 4, 9, 8, "unbalanced"),     # ragged chunk, ranks without experts
    (700, 256, 8, 24, None, 16, "mod"),
    (300, 12, 3, 12, None, 16, "mod"),         # k = E
    (300, 256, 256, 4, None, 8, "mod"),        # R = 256: a rank per expert, 257 rank offsets
    (2000, 256, 64, 8, None, 16, "random"),    # R = 64: the remote counter's largest table
])
def test_permute_and_counts(T, E, R, k_max, skew, H, placement):
    rng = np.random.default_rng(T * 7 + E)
    idx, k = _route_random(rng, T, E, k_max, skew)
    if placement == "mod":
        er = (np.arange(E) % R).astype(np.int32)
    elif placement == "random":
        er = rng.permutation(np.arange(E) % R).astype(np.int32)
    else:
        er = np.minimum(rng.integers(0, 2, size=E), R - 1).astype(np.int32) * (R - 1)
    P = int(k.sum())
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16)
    outs = []
    for _ in range(2):  # two runs must be byte-identical (no write races)
        d_idx = torch.from_numpy(idx).cuda()
        eo, ro = torch.empty(E + 1, **i32), torch.empty(R + 1, **i32)
        p2e, ec = torch.empty(E, **i32), torch.empty(E, **i32)
        s2p, p2s = torch.empty(max(P, 1), **i32), torch.empty(T * k_max, **i32)
        xp = torch.empty(P, H, dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(abi().semmoe_permute_workspace_size(T, k_max, E), dtype=torch.uint8, device="cuda")
        abi().semmoe_permute(d_idx, torch.from_numpy(er).cuda(), x.cuda(), T, H, E, R, k_max, P, eo, ro, p2e,
                             ec, s2p, p2s, xp, ws)
        assert abi().semmoe_check_errors() == 0
        outs.append([np_(t) for t in (eo, ro, p2e, ec, s2p[:P], p2s, xp)])
    for a, b in zip(*outs):
        np.testing.assert_array_equal(a, b)
    ref = oracle.permute(idx, k, er, R, x)
    for key, got in zip(("expert_offsets", "rank_offsets", "phys_to_expert", "expert_counts",
                         "sorted_to_pair", "pair_to_sorted", "x_perm"), outs[0]):
        np.testing.assert_array_equal(got, ref[key], err_msg=key)

    # remote counter and lookup on the same routing (the counter takes R <= 64)
    if R > 64:
        return
    V = 500
    lut = rng.integers(0, R, size=V).astype(np.int32)
    ids = rng.integers(0, V, size=T).astype(np.int32)
    pred = torch.empty(T, **i32)
    abi().semmoe_affinity_lookup(torch.from_numpy(ids).cuda(), torch.from_numpy(lut).cuda(), V, R, T, pred)
    counts, remote = torch.empty(R, R, **i32), torch.empty(R, **i32)
    abi().semmoe_remote_count(torch.from_numpy(idx).cuda(), pred, torch.from_numpy(er).cuda(), T, k_max, E, R,
                              counts, remote)
    assert abi().semmoe_check_errors() == 0
    rp = oracle.affinity_lookup(ids, lut)
    np.testing.assert_array_equal(np_(pred), rp)
    rc, rr = oracle.remote_count(idx, k, rp, er, R)
    np.testing.assert_array_equal(np_(counts), rc)
    np.testing.assert_array_equal(np_(remote), rr)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shared", [False, True])
def test_combine(dtype, shared):
    rng = np.random.default_rng(3)
    T, H, E, k_max = 333, 136 if dtype == "bf16" else 132, 16, 5
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    idx, k = _route_random(rng, T, E, k_max)
    _, w = oracle.topk_route(rng.standard_normal((T, E)), k, k_max)
    perm = oracle.permute(idx, k, np.arange(E) % 4, 4)
    P = int(k.sum())
    y = torch.from_numpy(rng.standard_normal((P, H)).astype(np.float32)).to(tdt)
    ys = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(tdt) if shared else None
    out = torch.empty(T, H, dtype=tdt, device="cuda")
    abi().semmoe_combine(y.cuda(), torch.from_numpy(perm["pair_to_sorted"].astype(np.int32)).cuda(),
                         torch.from_numpy(w.astype(np.float32)).cuda(), None if ys is None else ys.cuda(),
                         T, H, k_max, P, out)
    assert abi().semmoe_check_errors() == 0
    ref = oracle.combine(y, perm["pair_to_sorted"], w, k, dtype, ys)
    assert max_rel(np_(out), ref) < (1e-6 if dtype == "f32" else 8e-3)


@pytest.mark.parametrize("dtype,T,H,E,k_max,shared", [
    ("bf16", 1000, 2048, 64, 6, True),      # full 512-element passes, shared row first
    ("bf16", 300, 2056, 64, 8, False),      # a ragged last pass
    ("f32", 257, 1032, 32, 24, True),       # per-token budgets up to 24: padding in most rows
    ("bf16", 129, 520, 64, 32, False),      # every lane holds a slot
    ("bf16", 65, 264, 64, 33, True),        # budgets above 32: the slot read directly
    ("f32", 3, 4, 8, 2, False),             # rows of 16 bytes
    ("bf16", 700, 2048, 256, 24, False),    # the MoE-Prism budget: eight batches of three slots
    ("bf16", 500, 1032, 64, 23, True),      # 23 slots + the shared row, a ragged last pass
    ("f32", 2000, 1024, 64, 8, True),       # fp32 rows, many passes per warp
])
def test_combine_shapes(dtype, T, H, E, k_max, shared):
    """Combine against the oracle on ragged widths and budgets, output
    pre-filled so an unwritten element shows."""
    rng = np.random.default_rng(T + H)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    idx, k = _route_random(rng, T, E, k_max)
    _, w = oracle.topk_route(rng.standard_normal((T, E)), k, k_max)
    perm = oracle.permute(idx, k, np.arange(E) % 4, 4)
    P = int(k.sum())
    y = torch.from_numpy(rng.standard_normal((P, H)).astype(np.float32)).to(tdt).cuda()
    ys = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(tdt).cuda() if shared else None
    p2s = torch.from_numpy(perm["pair_to_sorted"].astype(np.int32)).cuda()
    wd = torch.from_numpy(w.astype(np.float32)).cuda()
    out = torch.full((T, H), 7.0, dtype=tdt, device="cuda")
    abi().semmoe_combine(y, p2s, wd, ys, T, H, k_max, P, out)
    assert abi().semmoe_check_errors() == 0
    ref = oracle.combine(y.cpu(), perm["pair_to_sorted"], w, k, dtype, None if ys is None else ys.cpu())
    assert max_rel(np_(out), ref) < (1e-6 if dtype == "f32" else 8e-3)


def test_data_errors_are_reported_not_faulted():
    """A token id beyond the vocabulary and a table value beyond R are caught
    by the kernels' own bounds checks and reported after a sync."""
    T, V, R = 64, 100, 4
    ids = torch.arange(T, dtype=torch.int32)
    ids[5] = V + 7                       # out of range
    lut = torch.zeros(V, dtype=torch.int32)
    lut[3] = R                           # out of range
    pred = torch.empty(T, **i32)
    abi().semmoe_affinity_lookup(ids.cuda(), lut.cuda(), V, R, T, pred)
    with pytest.raises(abi().SemMoEError) as ei:
        abi().semmoe_check_errors()
    assert ei.value.code == abi().SEMMOE_ERR_DEVICE_CHECK
    assert int(pred[5]) == 0 and int(pred[3]) == 0
    # the error word was cleared by the check
    assert abi().semmoe_check_errors() == 0


def test_bad_budget_is_clamped_and_reported():
    T, E, k_max = 8, 8, 4
    li = torch.randn(T, E, device="cuda")
    kpt = torch.full((T,), 2, **i32)
    kpt[1] = 9
    idx = torch.empty(T, k_max, **i32)
    w = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
    abi().semmoe_route(None, None, li, None, kpt, 0, T, 0, E, k_max, idx, w)
    with pytest.raises(abi().SemMoEError):
        abi().semmoe_check_errors()
    assert (idx[1] >= 0).all()           # clamped to k_max


def test_remote_count_large_pair_list():
    """Pair lists above 2^20 take the multi-CTA counting path."""
    rng = np.random.default_rng(77)
    T, E, R, k_max, V = 140_000, 64, 8, 8, 5000
    idx = np.stack([rng.permutation(E)[:k_max] for _ in range(64)])[rng.integers(0, 64, size=T)]
    k = rng.integers(1, k_max + 1, size=T)
    idx = np.where(np.arange(k_max)[None, :] < k[:, None], idx, -1).astype(np.int32)
    er = (np.arange(E) % R).astype(np.int32)
    lut = rng.integers(0, R, size=V).astype(np.int32)
    ids = rng.integers(0, V, size=T).astype(np.int32)
    pred = torch.empty(T, **i32)
    abi().semmoe_affinity_lookup(torch.from_numpy(ids).cuda(), torch.from_numpy(lut).cuda(), V, R, T, pred)
    counts, remote = torch.empty(R, R, **i32), torch.empty(R, **i32)
    abi().semmoe_remote_count(torch.from_numpy(idx).cuda(), pred, torch.from_numpy(er).cuda(), T, k_max, E, R,
                              counts, remote)
    assert abi().semmoe_check_errors() == 0
    rp = oracle.affinity_lookup(ids, lut)
    rc, rr = oracle.remote_count(idx, k, rp, er, R)
    np.testing.assert_array_equal(np_(counts), rc)
    np.testing.assert_array_equal(np_(remote), rr)


@pytest.mark.parametrize("E,k_max,wd", [(64, 8, torch.float32), (40, 16, torch.float32),
                                        (256, 16, torch.bfloat16), (256, 24, torch.float32),
                                        (128, 8, torch.bfloat16)])
def test_route_tensor_core_per_token_budgets(E, k_max, wd):
    """bf16 activations: the tensor-core router (split over K when the token
    tiles alone leave SMs idle) and the warp-per-token top-k; per-token budgets
    and ties from duplicated router rows."""
    rng = np.random.default_rng(E * 31 + k_max)
    T, H = 515, 256
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32) / np.sqrt(H)).to(torch.bfloat16)
    w = rng.standard_normal((E, H)).astype(np.float32) / np.sqrt(H)
    w[E // 2] = w[3]                      # two experts with identical logits: ties
    wr = torch.from_numpy(w).to(wd)
    kpt = rng.integers(1, k_max + 1, size=T).astype(np.int32)
    idx = torch.empty(T, k_max, **i32)
    gw = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
    lg = torch.empty(T, E, dtype=torch.float32, device="cuda")
    abi().semmoe_route(x.cuda(), wr.cuda(), None, lg, torch.from_numpy(kpt).cuda(), 0, T, H, E, k_max, idx, gw)
    assert abi().semmoe_check_errors() == 0
    assert max_rel(np_(lg), oracle.router_logits(x, wr)) < LOGIT_TOL
    ref_idx, ref_w = oracle.topk_route(np_(lg), kpt, k_max)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_allclose(np_(gw), ref_w, rtol=0, atol=GATE_ATOL)


@pytest.mark.parametrize("seed", range(10))
def test_route_random_shapes_every_router_path(seed):
    """Seeded random router shapes (token counts from one tile to several waves,
    E from 1 to 256, fp32 or bf16 weights, uniform or per-token budgets), so
    that every router form runs -- one CTA per token tile, a cluster of CTAs
    per tile, split-K + top-k: logits within tolerance, picks and gates exact
    given the GPU's logits, and the count table equal to the per-chunk
    histogram of the picks."""
    rng = np.random.default_rng(900 + seed)
    a = abi()
    T = int(rng.choice([1, 37, 128, 129, 700, 3000, 9000, 20000]))
    H = int(rng.integers(1, 49)) * 64 if seed % 2 == 0 else int(rng.integers(1, 257)) * 8
    E = int(rng.choice([1, 6, 16, 64, 100, 128, 256]))
    k_max = int(rng.integers(1, min(E, 32) + 1))
    wd = torch.float32 if seed % 3 else torch.bfloat16
    per_token = seed % 4 == 1
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32) / np.sqrt(H)).to(torch.bfloat16)
    wr = torch.from_numpy(rng.standard_normal((E, H)).astype(np.float32) / np.sqrt(H)).to(wd)
    k = rng.integers(1, k_max + 1, size=T).astype(np.int32) if per_token else np.full(T, k_max, np.int32)
    idx = torch.empty(T, k_max, **i32)
    gw = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
    lg = torch.empty(T, E, dtype=torch.float32, device="cuda")
    stride = a.semmoe_pair_counts_stride(T)
    counts = torch.full((E * stride,), -3, **i32)
    a.semmoe_route(x.cuda(), wr.cuda(), None, lg, torch.from_numpy(k).cuda() if per_token else None,
                   0 if per_token else k_max, T, H, E, k_max, idx, gw, pair_counts=counts)
    assert a.semmoe_check_errors() == 0
    assert max_rel(np_(lg), oracle.router_logits(x, wr)) < LOGIT_TOL, (T, H, E, k_max, wd)
    ref_idx, ref_w = oracle.topk_route(np_(lg), k, k_max)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_allclose(np_(gw), ref_w, rtol=0, atol=GATE_ATOL)
    np.testing.assert_array_equal(np_(counts).reshape(E, stride), _chunk_histogram(ref_idx, k, E, stride))


@pytest.mark.parametrize("wd", [torch.bfloat16, torch.float32])
def test_route_tensor_core_grid_beyond_one_wave(wd):
    """More token tiles than SMs: the router GEMM runs two resident CTAs per SM
    with the smaller operand ring; logits within tolerance, picks bit-exact."""
    rng = np.random.default_rng(77)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T, H, E, k_max = (sms + 3) * 128 + 77, 256, 64, 6
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32) / np.sqrt(H)).to(torch.bfloat16)
    wr = torch.from_numpy(rng.standard_normal((E, H)).astype(np.float32) / np.sqrt(H)).to(wd)
    idx = torch.empty(T, k_max, **i32)
    gw = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
    lg = torch.empty(T, E, dtype=torch.float32, device="cuda")
    abi().semmoe_route(x.cuda(), wr.cuda(), None, lg, None, k_max, T, H, E, k_max, idx, gw)
    assert abi().semmoe_check_errors() == 0
    assert max_rel(np_(lg), oracle.router_logits(x, wr)) < LOGIT_TOL
    ref_idx, ref_w = oracle.topk_route(np_(lg), np.full(T, k_max), k_max)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_allclose(np_(gw), ref_w, rtol=0, atol=GATE_ATOL)


SPLIT_COUNTS = [0, 1, 127, 128, 129, 255, 256, 257, 384, 511, 512, 640, 1000, 3, 900, 2048]


@pytest.mark.parametrize("P,E,H,I", [(1000, 8, 256, 160), (5000, 64, 512, 352), (3000, 16, 512, 640),
                                     (sum(SPLIT_COUNTS), 16, 256, 576), (30000, 64, 512, 704),
                                     (384, 64, 512, 1408), (3072, 64, 256, 200),
                                     (1, 1, 64, 8), (7, 3, 8, 24), (130, 256, 128, 136)])
def test_grouped_ffn_forms_are_bit_identical(P, E, H, I):
    """Every form of the grouped GEMM -- independent CTAs, 2-SM MMA pairs with
    one or two accumulator buffers, both GEMMs in one launch (GEMM2's tiles
    waiting on GEMM1's per m-tile), and the shape-chosen default -- returns
    exactly the same bits, and those bits match the oracle's grouped FFN row by
    row within the bf16 tolerance; one case pins group sizes around the 128-
    and 256-row boundaries (empty groups, 1, 127..129, 255..257 rows), two have
    decode-sized groups (6 and 48 rows on average; I not a multiple of 128), and
    three are tiny (one row; H = 8, smaller than one k-block and one output box;
    256 groups, most of them empty)."""
    rng = np.random.default_rng(P + E)
    if P == sum(SPLIT_COUNTS) and E == len(SPLIT_COUNTS):
        cnt = np.array(SPLIT_COUNTS)
    else:
        cnt = rng.multinomial(P, np.full(E, 1.0 / E))
    off = torch.from_numpy(np.r_[0, np.cumsum(cnt)].astype(np.int32)).cuda()
    pe = torch.from_numpy(rng.permutation(E).astype(np.int32)).cuda()
    x = torch.from_numpy(rng.standard_normal((P, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w13 = torch.from_numpy((rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w2 = torch.from_numpy((rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32)).to(torch.bfloat16).cuda()
    ws = torch.empty(abi().semmoe_grouped_ffn_workspace_size(P, I, 1), dtype=torch.uint8, device="cuda")
    outs = []
    a = abi()
    for form in (a.SEMMOE_FORM_SINGLE, a.SEMMOE_FORM_PAIR1, a.SEMMOE_FORM_PAIR, a.SEMMOE_FORM_FUSED,
                 a.SEMMOE_FORM_DEFAULT):
        y = torch.empty(P, H, dtype=torch.bfloat16, device="cuda")
        a.semmoe_grouped_ffn_form(x, None, 1, 0, off, pe, w13, w2, P, E, H, I, y, ws, form, form)
        assert a.semmoe_check_errors() == 0
        outs.append(y.cpu())
    for o in outs[1:]:
        assert torch.equal(outs[0], o)
    ref = oracle.grouped_ffn(x.cpu(), off.cpu(), pe.cpu(), w13.cpu().to(torch.float64).numpy(),
                             w2.cpu().to(torch.float64).numpy(), "bf16")
    got = outs[0].to(torch.float64).numpy()
    assert max_rel(got, ref) < TOL["bf16"]
    # every group's last row (the ragged tail of its last tile) on its own
    offs = off.cpu().numpy()
    for b in range(E):
        lo, hi = int(offs[b]), int(offs[b + 1])
        if hi > lo:
            assert max_rel(got[hi - 1], ref[hi - 1]) < TOL["bf16"], b


@pytest.mark.parametrize("seed", range(10))
def test_grouped_ffn_one_launch_matches_two_launches_random_groups(seed):
    """Both GEMMs in one launch (GEMM2 tiles waiting on GEMM1's per m-tile)
    against the two single-CTA launches, bit for bit, over seeded random group
    tables: skewed sizes, empty groups, one group holding most rows, one-row
    groups, H and I from 8 up and not multiples of the tile sizes."""
    rng = np.random.default_rng(500 + seed)
    a = abi()
    E = int(rng.choice([1, 3, 17, 64, 200, 256]))
    H = int(rng.integers(1, 65)) * 8
    I = int(rng.integers(1, 97)) * 8
    P = int(rng.integers(1, 3000))
    w = rng.dirichlet(np.full(E, 0.3))
    if seed % 3 == 0:
        w[rng.integers(E)] += 5.0  # one group holds most rows
    cnt = rng.multinomial(P, w / w.sum())
    off = torch.from_numpy(np.r_[0, np.cumsum(cnt)].astype(np.int32)).cuda()
    pe = torch.from_numpy(rng.permutation(E).astype(np.int32)).cuda()
    x = torch.from_numpy(rng.standard_normal((P, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w13 = torch.from_numpy((rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w2 = torch.from_numpy((rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32)).to(torch.bfloat16).cuda()
    ws = torch.empty(a.semmoe_grouped_ffn_workspace_size(P, I, 1), dtype=torch.uint8, device="cuda")
    outs = []
    for form in (a.SEMMOE_FORM_SINGLE, a.SEMMOE_FORM_FUSED, a.SEMMOE_FORM_FUSED):
        y = torch.full((P, H), 3.0, dtype=torch.bfloat16, device="cuda")
        a.semmoe_grouped_ffn_form(x, None, 1, 0, off, pe, w13, w2, P, E, H, I, y, ws, form, form)
        assert a.semmoe_check_errors() == 0
        outs.append(y.cpu())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2]), (P, E, H, I)


@pytest.mark.parametrize("dtype,T,E,k_max,H,I", [("bf16", 1000, 16, 4, 256, 640), ("bf16", 3001, 64, 6, 512, 1408),
                                                 ("bf16", 257, 8, 8, 128, 160), ("bf16", 700, 8, 4, 200, 96),
                                                 ("f32", 300, 8, 3, 64, 96)])
def test_grouped_ffn_gather_matches_permuted(dtype, T, E, k_max, H, I):
    """GEMM1 reading x through sorted_to_pair (row gathers) gives exactly the
    bits of the permute's x_perm followed by the grouped FFN, in every form of
    the grouped GEMM; per-token budgets leave padding slots, so sorted rows map
    to tokens irregularly; H = 200 leaves a partial last k-block (zero-filled
    columns) and a partial last output tile."""
    rng = np.random.default_rng(T + I)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    idx, k = _route_random(rng, T, E, k_max)
    er = (np.arange(E) % 4).astype(np.int32)
    P = int(k.sum())
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(tdt).cuda()
    w13 = torch.from_numpy((rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)).astype(np.float32)).to(tdt).cuda()
    w2 = torch.from_numpy((rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32)).to(tdt).cuda()
    eo, ro = torch.empty(E + 1, **i32), torch.empty(5, **i32)
    p2e, ec = torch.empty(E, **i32), torch.empty(E, **i32)
    s2p, p2s = torch.empty(P, **i32), torch.empty(T * k_max, **i32)
    xp = torch.empty(P, H, dtype=tdt, device="cuda")
    ws = torch.empty(abi().semmoe_permute_workspace_size(T, k_max, E), dtype=torch.uint8, device="cuda")
    abi().semmoe_permute(torch.from_numpy(idx).cuda(), torch.from_numpy(er).cuda(), x, T, H, E, 4, k_max, P, eo, ro,
                         p2e, ec, s2p, p2s, xp, ws)
    fws = torch.empty(abi().semmoe_grouped_ffn_workspace_size(P, I, 1 if dtype == "bf16" else 0), dtype=torch.uint8,
                      device="cuda")
    a = abi()
    # (GEMM1 form of the x_perm call, GEMM1 form of the gathered call, GEMM2 form): single = gathering
    # warps feed the gathered GEMM1; single/TMA gather = the producer's four-row gathers
    forms = [(a.SEMMOE_FORM_SINGLE, a.SEMMOE_FORM_SINGLE, a.SEMMOE_FORM_SINGLE),
             (a.SEMMOE_FORM_SINGLE, a.SEMMOE_FORM_SINGLE_TMA_GATHER, a.SEMMOE_FORM_SINGLE),
             (a.SEMMOE_FORM_PAIR1, a.SEMMOE_FORM_PAIR1, a.SEMMOE_FORM_PAIR1),
             (a.SEMMOE_FORM_PAIR, a.SEMMOE_FORM_PAIR, a.SEMMOE_FORM_PAIR)] if dtype == "bf16" else []
    for f_plain, f_gather, f2 in forms:
        y0 = torch.full((P, H), 3.0, dtype=tdt, device="cuda")
        y1 = torch.full((P, H), 5.0, dtype=tdt, device="cuda")
        a.semmoe_grouped_ffn_form(xp, None, 1, 0, eo, p2e, w13, w2, P, E, H, I, y0, fws, f_plain, f2)
        a.semmoe_grouped_ffn_form(x, s2p, k_max, T, eo, p2e, w13, w2, P, E, H, I, y1, fws, f_gather, f2)
        assert a.semmoe_check_errors() == 0
        assert torch.equal(y0.cpu(), y1.cpu()), (f_plain, f_gather, f2)
    # the production calls, each with its own shape-chosen forms
    y0 = torch.full((P, H), 3.0, dtype=tdt, device="cuda")
    y1 = torch.full((P, H), 5.0, dtype=tdt, device="cuda")
    a.semmoe_grouped_ffn(xp, eo, p2e, w13, w2, P, E, H, I, y0, fws)
    a.semmoe_grouped_ffn_gather(x, s2p, k_max, T, eo, p2e, w13, w2, P, E, H, I, y1, fws)
    assert a.semmoe_check_errors() == 0
    assert torch.equal(y0.cpu(), y1.cpu())
    if dtype == "bf16":  # the CUDA-core path gathers the same way
        cc = a.SEMMOE_FORM_CUDA_CORE
        y0 = torch.empty(P, H, dtype=tdt, device="cuda")
        y1 = torch.empty(P, H, dtype=tdt, device="cuda")
        a.semmoe_grouped_ffn_form(xp, None, 1, 0, eo, p2e, w13, w2, P, E, H, I, y0, fws, cc, cc)
        a.semmoe_grouped_ffn_form(x, s2p, k_max, T, eo, p2e, w13, w2, P, E, H, I, y1, fws, cc, cc)
        assert a.semmoe_check_errors() == 0
        assert torch.equal(y0.cpu(), y1.cpu())


@pytest.mark.parametrize("T,H,E", [(4096, 2048, 64), (300, 512, 256), (77, 200, 7)])
def test_route_with_presplit_weight_is_identical(T, H, E):
    """An fp32 router weight split once (semmoe_route_split_weight) and passed
    as SEMMOE_F32_SPLIT routes exactly as the weight split on every call."""
    rng = np.random.default_rng(T + E)
    x = torch.from_numpy((rng.standard_normal((T, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16).cuda()
    wr = torch.from_numpy((rng.standard_normal((E, H)) / np.sqrt(H)).astype(np.float32)).cuda()
    k_max = min(6, E)
    outs = []
    split = torch.empty(abi().semmoe_route_split_size(H, E), dtype=torch.uint8, device="cuda")
    abi().semmoe_route_split_weight(wr, H, E, split)
    for w, wd in ((wr, None), (split, abi().SEMMOE_F32_SPLIT)):
        idx = torch.empty(T, k_max, **i32)
        gw = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
        lg = torch.empty(T, E, dtype=torch.float32, device="cuda")
        abi().semmoe_route(x, w, None, lg, None, k_max, T, H, E, k_max, idx, gw, w_dtype=wd)
        assert abi().semmoe_check_errors() == 0
        outs.append((lg.cpu(), idx.cpu(), gw.cpu()))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    assert max_rel(np_(outs[0][0]), oracle.router_logits(x, wr)) < LOGIT_TOL


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait that nothing can complete gives up after its bound: the host
    reads SEMMOE_ERR_DEVICE_TIMEOUT with the timeout bit, the error word is
    cleared, and the GPU goes on working."""
    import time
    t0 = time.perf_counter()
    abi().semmoe_selftest_bounded_wait()
    with pytest.raises(abi().SemMoEError) as ei:
        abi().semmoe_check_errors()
    assert ei.value.code == abi().SEMMOE_ERR_DEVICE_TIMEOUT
    assert ei.value.bits & abi().SEMMOE_DEVERR_TIMEOUT
    assert 0.1 < time.perf_counter() - t0 < 60
    assert abi().semmoe_check_errors() == 0
    test_combine("f32", True)  # the context still runs kernels


def test_fused_ffn_ready_wait_runs_out_and_context_survives():
    """The one-launch grouped FFN with GEMM2's readiness waits made unreachable:
    every such wait gives up after its bound, the host reads
    SEMMOE_ERR_DEVICE_TIMEOUT with the timeout bit, and the next one-launch FFN
    on the same workspace (counters zeroed again at launch) is exact."""
    import time
    a = abi()
    rng = np.random.default_rng(2024)
    P, H, I = 300, 256, 200
    x = torch.from_numpy(rng.standard_normal((P, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w13 = torch.from_numpy((rng.standard_normal((1, 2 * I, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w2 = torch.from_numpy((rng.standard_normal((1, H, I)) / np.sqrt(I)).astype(np.float32)).to(torch.bfloat16).cuda()
    ws = torch.empty(a.semmoe_grouped_ffn_workspace_size(P, I, 1), dtype=torch.uint8, device="cuda")
    y = torch.zeros(P, H, dtype=torch.bfloat16, device="cuda")
    t0 = time.perf_counter()
    a.semmoe_selftest_fused_ready_wait(x, w13, w2, P, H, I, y, ws)
    with pytest.raises(a.SemMoEError) as ei:
        a.semmoe_check_errors()
    assert ei.value.code == a.SEMMOE_ERR_DEVICE_TIMEOUT
    assert ei.value.bits & a.SEMMOE_DEVERR_TIMEOUT
    assert 0.1 < time.perf_counter() - t0 < 60
    assert a.semmoe_check_errors() == 0
    off = torch.tensor([0, P], dtype=torch.int32, device="cuda")
    pe = torch.zeros(1, dtype=torch.int32, device="cuda")
    a.semmoe_grouped_ffn_form(x, None, 1, 0, off, pe, w13, w2, P, 1, H, I, y, ws, a.SEMMOE_FORM_FUSED,
                              a.SEMMOE_FORM_FUSED)
    assert a.semmoe_check_errors() == 0
    ref = oracle.grouped_ffn(x.cpu(), off.cpu(), pe.cpu(), w13.cpu().to(torch.float64).numpy(),
                             w2.cpu().to(torch.float64).numpy(), "bf16")
    assert max_rel(y.cpu().to(torch.float64).numpy(), ref) < TOL["bf16"]


def test_empty_batch_through_every_step():
    """T = 0 (and so P = 0) through the router, lookup, remote count, permute,
    grouped FFN and combine: every call succeeds, the tables come out as the
    oracle gives them for an empty batch (physical order, zero offsets and
    counts), and nothing else is written."""
    E, R, k_max, H, I = 8, 4, 3, 64, 96
    er = (np.arange(E) % R).astype(np.int32)
    ref = oracle.permute(np.zeros((0, k_max), np.int32), np.zeros(0, np.int32), er, R)
    e0 = lambda *shape, dt=torch.int32: torch.empty(*shape, dtype=dt, device="cuda")  # noqa: E731
    x = e0(0, H, dt=torch.bfloat16)
    idx, w = e0(0, k_max), e0(0, k_max, dt=torch.float32)
    abi().semmoe_route(x, torch.randn(E, H, device="cuda"), None, None, None, 2, 0, H, E, k_max, idx, w)
    pred = e0(0)
    abi().semmoe_affinity_lookup(e0(0), torch.zeros(10, dtype=torch.int32, device="cuda"), 10, R, 0, pred)
    counts = torch.full((R, R), 7, dtype=torch.int32, device="cuda")
    remote = torch.full((R,), 7, dtype=torch.int32, device="cuda")
    abi().semmoe_remote_count(idx, pred, torch.from_numpy(er).cuda(), 0, k_max, E, R, counts, remote)
    eo, ro = torch.full((E + 1,), -5, **i32), torch.full((R + 1,), -5, **i32)
    p2e, ec = torch.full((E,), -5, **i32), torch.full((E,), -5, **i32)
    ws = torch.empty(abi().semmoe_permute_workspace_size(0, k_max, E), dtype=torch.uint8, device="cuda")
    abi().semmoe_permute(idx, torch.from_numpy(er).cuda(), x, 0, H, E, R, k_max, 0, eo, ro, p2e, ec, e0(1), e0(0),
                         e0(0, H, dt=torch.bfloat16), ws)
    fws = torch.empty(abi().semmoe_grouped_ffn_workspace_size(0, I, 1), dtype=torch.uint8, device="cuda")
    w13 = torch.randn(E, 2 * I, H, device="cuda").to(torch.bfloat16)
    w2 = torch.randn(E, H, I, device="cuda").to(torch.bfloat16)
    y = e0(0, H, dt=torch.bfloat16)
    abi().semmoe_grouped_ffn(e0(0, H, dt=torch.bfloat16), eo, p2e, w13, w2, 0, E, H, I, y, fws)
    out = e0(0, H, dt=torch.bfloat16)
    abi().semmoe_combine(y, e0(0), w, None, 0, H, k_max, 0, out)
    assert abi().semmoe_check_errors() == 0
    for key, got in (("expert_offsets", eo), ("rank_offsets", ro), ("phys_to_expert", p2e), ("expert_counts", ec)):
        np.testing.assert_array_equal(np_(got), ref[key], err_msg=key)
    assert int(counts.sum()) == 0 and int(remote.sum()) == 0


def test_permute_flags_bad_expert_and_pair_count():
    """An expert id past E is skipped (its slot maps to -1) and flagged; a P
    that disagrees with the live pairs is flagged; the other pairs are placed
    exactly as the oracle places them without the bad one."""
    rng = np.random.default_rng(91)
    T, E, R, k_max = 100, 8, 4, 2
    idx, k = _route_random(rng, T, E, k_max)
    er = (np.arange(E) % R).astype(np.int32)
    good = idx.copy()
    good[7, 1] = -1                        # the oracle's view: that slot is padding
    bad = idx.copy()
    bad[7, 1] = E + 3
    k_good = (good >= 0).sum(axis=1)
    P = int(k_good.sum())                  # live pairs without the bad one
    ref = oracle.permute(good, k_good, er, R)
    eo, ro = torch.empty(E + 1, **i32), torch.empty(R + 1, **i32)
    p2e, ec = torch.empty(E, **i32), torch.empty(E, **i32)
    s2p, p2s = torch.empty(P + 1, **i32), torch.empty(T * k_max, **i32)
    ws = torch.empty(abi().semmoe_permute_workspace_size(T, k_max, E), dtype=torch.uint8, device="cuda")
    abi().semmoe_permute(torch.from_numpy(bad).cuda(), torch.from_numpy(er).cuda(), None, T, 0, E, R, k_max, P + 1,
                         eo, ro, p2e, ec, s2p, p2s, None, ws)
    with pytest.raises(abi().SemMoEError) as ei:
        abi().semmoe_check_errors()
    assert ei.value.bits & abi().SEMMOE_DEVERR_EXPERT
    assert ei.value.bits & abi().SEMMOE_DEVERR_PAIRS   # P + 1 passed, P pairs live
    assert int(p2s[7 * k_max + 1]) == -1
    np.testing.assert_array_equal(np_(p2s), ref["pair_to_sorted"])
    np.testing.assert_array_equal(np_(s2p[:P]), ref["sorted_to_pair"])
    np.testing.assert_array_equal(np_(eo), ref["expert_offsets"])


@pytest.mark.parametrize("mode,dtype", [("single", "bf16"), ("pair", "bf16"), ("fused", "bf16"), ("default", "f32")])
def test_grouped_ffn_flags_bad_group_table(mode, dtype):
    """Group offsets that decrease or run past P (SEMMOE_DEVERR_PAIRS) and an
    expert id past E (SEMMOE_DEVERR_EXPERT) are flagged by the kernels' checks
    in every form; those groups are skipped, the valid ones are still computed
    exactly as with a clean table."""
    a = abi()
    form = {"single": a.SEMMOE_FORM_SINGLE, "pair": a.SEMMOE_FORM_PAIR, "fused": a.SEMMOE_FORM_FUSED,
            "default": a.SEMMOE_FORM_DEFAULT}[mode]

    def ffn(xx, off, pe, y):
        a.semmoe_grouped_ffn_form(xx, None, 1, 0, off, pe, w13, w2, P, E, H, I, y, ws, form, form)
    rng = np.random.default_rng(5)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    E, H, I, P = 4, 128, 128, 600
    x = torch.from_numpy(rng.standard_normal((P, H)).astype(np.float32)).to(tdt).cuda()
    w13 = torch.from_numpy((rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)).astype(np.float32)).to(tdt).cuda()
    w2 = torch.from_numpy((rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32)).to(tdt).cuda()
    ws = torch.empty(abi().semmoe_grouped_ffn_workspace_size(P, I, 1 if dtype == "bf16" else 0),
                     dtype=torch.uint8, device="cuda")
    p2e = torch.tensor([0, 1, 2, 3], **i32)
    clean = torch.tensor([0, 300, 300, 450, 600], **i32)
    y0 = torch.zeros(P, H, dtype=tdt, device="cuda")
    ffn(x, clean, p2e, y0)
    assert abi().semmoe_check_errors() == 0
    # group 1 runs backwards (300 -> 200), group 3 past P (450 -> 700)
    bad = torch.tensor([0, 300, 200, 450, 700], **i32)
    y1 = torch.zeros(P, H, dtype=tdt, device="cuda")
    ffn(x, bad, p2e, y1)
    with pytest.raises(abi().SemMoEError) as ei:
        abi().semmoe_check_errors()
    assert ei.value.bits & abi().SEMMOE_DEVERR_PAIRS
    # group 0 is valid, but the valid group 2 (rows 200..449) overlaps it: rows 0..199 are group 0's alone
    assert torch.equal(y1[:200], y0[:200])
    p2e_bad = torch.tensor([0, 1, 9, 3], **i32)        # expert 9 of 4
    y2 = torch.zeros(P, H, dtype=tdt, device="cuda")
    ffn(x, clean, p2e_bad, y2)
    with pytest.raises(abi().SemMoEError) as ei:
        abi().semmoe_check_errors()
    assert ei.value.bits & abi().SEMMOE_DEVERR_EXPERT
    assert torch.equal(y2[:300], y0[:300]) and torch.equal(y2[450:], y0[450:])
    assert not torch.any(y2[300:450] != 0)               # the skipped group wrote nothing


@pytest.mark.parametrize("producer", ["gather-warps", "tma-gather", "pair"])
def test_grouped_ffn_gather_flags_bad_pair_id(producer):
    """A sorted_to_pair entry naming no token (negative, or a token past T)
    sets SEMMOE_DEVERR_PAIRS in every gathering producer; that row reads token
    0 instead, and every other row keeps the bits of the clean call."""
    a = abi()
    f1, f2 = {"gather-warps": (a.SEMMOE_FORM_SINGLE, a.SEMMOE_FORM_SINGLE),
              "tma-gather": (a.SEMMOE_FORM_SINGLE_TMA_GATHER, a.SEMMOE_FORM_SINGLE),
              "pair": (a.SEMMOE_FORM_PAIR, a.SEMMOE_FORM_PAIR)}[producer]
    rng = np.random.default_rng(23)
    E, H, I, T, k_max = 4, 256, 128, 300, 2
    P = T * k_max
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w13 = torch.from_numpy((rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w2 = torch.from_numpy((rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32)).to(torch.bfloat16).cuda()
    ws = torch.empty(abi().semmoe_grouped_ffn_workspace_size(P, I, 1), dtype=torch.uint8, device="cuda")
    eo = torch.tensor([0, 150, 300, 450, 600], **i32)
    p2e = torch.tensor([0, 1, 2, 3], **i32)
    s2p = torch.from_numpy(rng.permutation(P).astype(np.int32)).cuda()
    y0 = torch.zeros(P, H, dtype=torch.bfloat16, device="cuda")
    a.semmoe_grouped_ffn_form(x, s2p, k_max, T, eo, p2e, w13, w2, P, E, H, I, y0, ws, f1, f2)
    assert abi().semmoe_check_errors() == 0
    bad = s2p.clone()
    bad[7], bad[301] = -5, T * k_max + 9               # no token; token T + 4 of T
    y1 = torch.zeros(P, H, dtype=torch.bfloat16, device="cuda")
    a.semmoe_grouped_ffn_form(x, bad, k_max, T, eo, p2e, w13, w2, P, E, H, I, y1, ws, f1, f2)
    with pytest.raises(abi().SemMoEError) as ei:
        abi().semmoe_check_errors()
    assert ei.value.bits & abi().SEMMOE_DEVERR_PAIRS
    keep = torch.ones(P, dtype=torch.bool)
    keep[[7, 301]] = False
    assert torch.equal(y1.cpu()[keep], y0.cpu()[keep])
    # the flagged rows read token 0: the same bits as a clean map sending them to pair 0
    ref_map = s2p.clone()
    ref_map[7], ref_map[301] = 0, 0
    y2 = torch.zeros(P, H, dtype=torch.bfloat16, device="cuda")
    a.semmoe_grouped_ffn_form(x, ref_map, k_max, T, eo, p2e, w13, w2, P, E, H, I, y2, ws, f1, f2)
    assert abi().semmoe_check_errors() == 0
    assert torch.equal(y1.cpu(), y2.cpu())


def test_route_nonfinite_logits_are_skipped_and_flagged():
    """NaN and ±inf logits count as -inf (never picked while finite ones are
    left) and set SEMMOE_DEVERR_NONFINITE; the picks and gates equal the
    oracle's on the logits with those entries set to -inf."""
    rng = np.random.default_rng(17)
    T, E, k_max = 200, 16, 4
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lg[3, 5], lg[10, 0], lg[11, 2], lg[12, 7] = np.nan, np.inf, -np.inf, np.nan
    k = rng.integers(1, k_max + 1, size=T).astype(np.int32)
    idx, w = route_logits_in(lg, k, k_max, expect_clean=False)
    with pytest.raises(abi().SemMoEError) as ei:
        abi().semmoe_check_errors()
    assert ei.value.bits & abi().SEMMOE_DEVERR_NONFINITE
    clean = np.where(np.isfinite(lg), lg, np.float32(-np.inf)).astype(np.float32)
    ref_idx, ref_w = oracle.topk_route(clean, k, k_max)
    np.testing.assert_array_equal(idx, ref_idx)
    np.testing.assert_allclose(w, ref_w, rtol=0, atol=GATE_ATOL)


def test_combine_skips_and_flags_a_slot_past_P():
    """A pair_to_sorted entry >= P is skipped and flagged; the token's sum runs
    over its other slots, exactly as the oracle's with that slot as padding."""
    rng = np.random.default_rng(23)
    T, E, k_max, H = 50, 8, 3, 64
    idx, k = _route_random(rng, T, E, k_max)
    _, w = oracle.topk_route(rng.standard_normal((T, E)), k, k_max)
    perm = oracle.permute(idx, k, np.arange(E) % 4, 4)
    P = int(k.sum())
    y = torch.from_numpy(rng.standard_normal((P, H)).astype(np.float32)).cuda()
    p2s = perm["pair_to_sorted"].astype(np.int32).copy()
    p2s[4] = P + 10                        # token 1, slot 1 (k_max = 3)
    out = torch.full((T, H), 9.0, device="cuda")
    abi().semmoe_combine(y, torch.from_numpy(p2s).cuda(), torch.from_numpy(w.astype(np.float32)).cuda(), None,
                         T, H, k_max, P, out)
    with pytest.raises(abi().SemMoEError) as ei:
        abi().semmoe_check_errors()
    assert ei.value.bits & abi().SEMMOE_DEVERR_PAIRS
    w_ref = w.copy()
    w_ref[1, 1] = 0.0                      # the skipped slot contributes nothing
    ref = oracle.combine(np_(y), perm["pair_to_sorted"], w_ref, k, "f32")
    assert max_rel(np_(out), ref) < 1e-6


@pytest.mark.parametrize("P,E,I", [(5000, 8, 352),    # groups of ~625 rows, I < 512: GEMM1 in pairs, GEMM2 single
                                   (4000, 10, 640)])  # groups of ~400 rows, I >= 512: GEMM1 single, GEMM2 in pairs
def test_grouped_ffn_mixed_default_forms_match_single(P, E, I):
    """The default per-GEMM form choice mixes the 2-SM and single-CTA forms
    within one call; the result is bit-identical to both GEMMs single-CTA."""
    rng = np.random.default_rng(P + I)
    H = 256
    cuts = np.sort(rng.integers(0, P, size=E - 1))
    eo = torch.from_numpy(np.concatenate([[0], cuts, [P]]).astype(np.int32)).cuda()
    p2e = torch.from_numpy(rng.permutation(E).astype(np.int32)).cuda()
    x = torch.from_numpy(rng.standard_normal((P, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w13 = torch.from_numpy((rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w2 = torch.from_numpy((rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32)).to(torch.bfloat16).cuda()
    ws = torch.empty(abi().semmoe_grouped_ffn_workspace_size(P, I, 1), dtype=torch.uint8, device="cuda")
    outs = []
    a = abi()
    for form in (None, a.SEMMOE_FORM_SINGLE):
        y = torch.full((P, H), 7.0, dtype=torch.bfloat16, device="cuda")
        if form is None:
            a.semmoe_grouped_ffn(x, eo, p2e, w13, w2, P, E, H, I, y, ws)
        else:
            a.semmoe_grouped_ffn_form(x, None, 1, 0, eo, p2e, w13, w2, P, E, H, I, y, ws, form, form)
        assert a.semmoe_check_errors() == 0
        outs.append(y.cpu())
    assert torch.equal(outs[0], outs[1])
    ref = oracle.grouped_ffn(x.cpu(), eo.cpu(), p2e.cpu(), w13.cpu().to(torch.float64).numpy(),
                             w2.cpu().to(torch.float64).numpy(), "bf16")
    assert max_rel(outs[0].to(torch.float64).numpy(), ref) < TOL["bf16"]


def _chunk_histogram(idx, k, E, stride):
    """Expected count table: live pairs of expert e among the tokens of 128-token chunk c."""
    T, k_max = idx.shape
    live = np.arange(k_max)[None, :] < np.asarray(k)[:, None]
    tok = np.broadcast_to(np.arange(T)[:, None], (T, k_max))[live]
    cnt = np.zeros((E, stride), dtype=np.int64)
    np.add.at(cnt, (idx[live], tok // 128), 1)
    return cnt


@pytest.mark.parametrize("T,E,R,k_max,per_token,H", [(1, 8, 4, 2, False, 16), (70, 3, 2, 2, True, 8),
                                                    (300, 8, 4, 2, True, 64), (4096, 64, 8, 6, False, 128),
                                                    (5000, 256, 8, 24, True, 16), (16384, 128, 8, 8, False, 32),
                                                    (131200, 4, 2, 2, True, 8)])
def test_route_pair_counts_and_counted_permute(T, E, R, k_max, per_token, H):
    """The router's count table equals the per-chunk histogram of its picks
    (entries past the last chunk are 0), and the permute started from it
    returns exactly the oracle's maps and rows -- as does the permute that counts
    the pairs itself.  T = 131200 has more than 1024 chunks, where the permute
    ignores the table and counts for itself."""
    a = abi()
    rng = np.random.default_rng(T + E)
    logits = (rng.integers(-6, 7, size=(T, E)) * 0.25).astype(np.float32)     # many exact ties
    k = rng.integers(1, k_max + 1, size=T).astype(np.int32) if per_token else np.full(T, k_max, np.int32)
    li = torch.from_numpy(logits).cuda()
    idx = torch.empty(T, k_max, **i32)
    w = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
    stride = a.semmoe_pair_counts_stride(T)
    assert a.semmoe_pair_counts_size(T, E) == E * stride * 4 and stride % 4 == 0
    counts = torch.full((E * stride,), -3, **i32)                               # stale contents are overwritten
    kpt = torch.from_numpy(k).cuda() if per_token else None
    a.semmoe_route(None, None, li, None, kpt, 0 if per_token else k_max, T, 0, E, k_max, idx, w,
                   pair_counts=counts)
    assert a.semmoe_check_errors() == 0
    ref_idx, _ = oracle.topk_route(logits, k, k_max)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_array_equal(np_(counts).reshape(E, stride), _chunk_histogram(ref_idx, k, E, stride))
    er = rng.permutation(np.arange(E) % R).astype(np.int32)
    P = int(k.sum())
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    ref = oracle.permute(ref_idx, k, er, R, x.cpu())
    ws = torch.empty(a.semmoe_permute_workspace_size(T, k_max, E), dtype=torch.uint8, device="cuda")
    for pc in (counts, None):
        outs = dict(expert_offsets=torch.empty(E + 1, **i32), rank_offsets=torch.empty(R + 1, **i32),
                    phys_to_expert=torch.empty(E, **i32), expert_counts=torch.empty(E, **i32),
                    sorted_to_pair=torch.full((P,), -9, **i32), pair_to_sorted=torch.full((T * k_max,), -9, **i32),
                    x_perm=torch.zeros(P, H, dtype=torch.bfloat16, device="cuda"))
        a.semmoe_permute(idx, torch.from_numpy(er).cuda(), x, T, H, E, R, k_max, P, outs["expert_offsets"],
                         outs["rank_offsets"], outs["phys_to_expert"], outs["expert_counts"], outs["sorted_to_pair"],
                         outs["pair_to_sorted"], outs["x_perm"], ws, pair_counts=pc)
        assert a.semmoe_check_errors() == 0
        for key, v in ref.items():
            np.testing.assert_array_equal(np_(outs[key]), v, err_msg=f"{key} (counts {'given' if pc is not None else 'own'})")


def test_hier_route_pair_counts():
    """The hierarchical router counts its sub-expert picks the same way."""
    a = abi()
    rng = np.random.default_rng(77)
    T, Ep, N, k_max = 1000, 16, 4, 12
    l = rng.standard_normal((T, Ep)).astype(np.float32)
    logw = np.log(rng.dirichlet(np.full(N, 2.0), size=Ep)).astype(np.float32).ravel()
    k = rng.integers(1, k_max + 1, size=T).astype(np.int32)
    E = Ep * N
    idx = torch.empty(T, k_max, **i32)
    w = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
    stride = a.semmoe_pair_counts_stride(T)
    counts = torch.full((E * stride,), 5, **i32)
    a.semmoe_route_hier(None, None, torch.from_numpy(l).cuda(), None, torch.from_numpy(logw).cuda(), N,
                        torch.from_numpy(k).cuda(), 0, T, 0, Ep, k_max, idx, w, pair_counts=counts)
    assert a.semmoe_check_errors() == 0
    ref_idx, _ = oracle.hier_route(l, logw, N, k, k_max)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_array_equal(np_(counts).reshape(E, stride), _chunk_histogram(ref_idx, k, E, stride))


@pytest.mark.parametrize("T,H,E,k_max,wd,per_token", [
    (9800, 128, 8, 1, "bf16", False), (9800, 256, 64, 6, "bf16", True), (16384 + 45, 2048, 128, 8, "bf16", False),
    (20485, 256, 256, 24, "bf16", True), (9800, 200, 7, 3, "f32", True), (9800, 512, 64, 16, "f32", False),
    (9800, 128, 64, 32, "bf16", True),
    # fewer than 76 tiles: a cluster of 2, 4 or 8 CTAs per tile, each a slice of H
    (4096, 2048, 64, 6, "f32", False), (300, 200, 7, 3, "f32", True), (64, 2048, 64, 6, "f32", True),
    (3000, 2048, 64, 6, "f32", False), (9000, 1024, 128, 8, "bf16", True), (129, 512, 7, 3, "f32", True),
    # the split-K router and a top-k kernel: an fp32 weight over more than 64 experts (several passes,
    # a partial last one at E = 100), H of two k-blocks, a bf16 weight over 192 experts with few tiles
    (3000, 256, 256, 8, "f32", False), (8192 + 5, 512, 256, 24, "f32", True), (500, 256, 100, 5, "f32", True),
    (300, 128, 7, 3, "f32", True), (700, 256, 256, 24, "bf16", True), (40000, 128, 256, 8, "f32", False)])
def test_router_with_top_k_in_the_gemm_epilogue(T, H, E, k_max, wd, per_token):
    """The one-kernel router (tensor-core GEMM, top-k in the epilogue: one
    thread per token and column range, lists merged in column order), taken
    from 76 tiles of 128 tokens on, and below that its cluster form (each CTA
    of a tile's cluster contracts a slice of H; the partial logits are added in
    slice order through distributed shared memory, CS threads per row select):
    logits within the logit tolerance of the oracle, picks bit-exact against
    the oracle's top-k of the GPU's own logits, gates within the gate
    tolerance, and the count table equal to the per-chunk histogram of the
    picks.  Covers ragged last tiles, per-token budgets, a grid beyond one CTA
    per SM (T = 20485), k_max of 8, 16 and 32, fp32 weights split into bf16
    parts, column groups left empty (E = 7), clusters of 2, 4 and 8 slices of H,
    and six shapes that take the split-K router and a top-k kernel."""
    a = abi()
    rng = np.random.default_rng(T + E + k_max)
    x = torch.from_numpy((rng.standard_normal((T, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16)
    wdt = torch.bfloat16 if wd == "bf16" else torch.float32
    wr = torch.from_numpy(rng.standard_normal((E, H)).astype(np.float32)).to(wdt)
    k = rng.integers(1, k_max + 1, size=T).astype(np.int32) if per_token else np.full(T, k_max, np.int32)
    idx = torch.empty(T, k_max, **i32)
    gw = torch.empty(T, k_max, dtype=torch.float32, device="cuda")
    lg = torch.empty(T, E, dtype=torch.float32, device="cuda")
    stride = a.semmoe_pair_counts_stride(T)
    counts = torch.full((E * stride,), -1, **i32)
    a.semmoe_route(x.cuda(), wr.cuda(), None, lg, torch.from_numpy(k).cuda() if per_token else None,
                   0 if per_token else k_max, T, H, E, k_max, idx, gw, pair_counts=counts)
    assert a.semmoe_check_errors() == 0
    assert max_rel(np_(lg), oracle.router_logits(x, wr)) < LOGIT_TOL
    ref_idx, ref_w = oracle.topk_route(np_(lg), k, k_max)
    np.testing.assert_array_equal(np_(idx), ref_idx)
    np.testing.assert_allclose(np_(gw), ref_w, rtol=0, atol=GATE_ATOL)
    np.testing.assert_array_equal(np_(counts).reshape(E, stride), _chunk_histogram(ref_idx, k, E, stride))


@pytest.mark.parametrize("T,E,k_max,H,fused_copy", [(3000, 64, 6, 2048, True), (16384, 128, 8, 1024, False)])
def test_permute_copy_inside_and_as_its_own_kernel(T, E, k_max, H, fused_copy):
    """The rows are copied inside the ranking kernel below 256 MB of rows and by
    a copy kernel of its own above; both give the oracle's index tables and
    x_perm[q] = x[sorted_to_pair[q] / k_max] exactly (the rows checked on the
    GPU against a plain gather through the oracle-equal map)."""
    a = abi()
    rng = np.random.default_rng(T)
    P = T * k_max
    assert (P * H * 2 >= 256 << 20) == (not fused_copy)
    idx, k = _route_random(rng, T, E, k_max, per_token=False)
    R = 8
    er = rng.permutation(np.arange(E) % R).astype(np.int32)
    x = torch.randn(T, H, device="cuda").to(torch.bfloat16)
    o = dict(expert_offsets=torch.empty(E + 1, **i32), rank_offsets=torch.empty(R + 1, **i32),
             phys_to_expert=torch.empty(E, **i32), expert_counts=torch.empty(E, **i32),
             sorted_to_pair=torch.empty(P, **i32), pair_to_sorted=torch.empty(T * k_max, **i32),
             x_perm=torch.zeros(P, H, dtype=torch.bfloat16, device="cuda"))
    ws = torch.empty(a.semmoe_permute_workspace_size(T, k_max, E), dtype=torch.uint8, device="cuda")
    a.semmoe_permute(torch.from_numpy(idx).cuda(), torch.from_numpy(er).cuda(), x, T, H, E, R, k_max, P,
                     o["expert_offsets"], o["rank_offsets"], o["phys_to_expert"], o["expert_counts"],
                     o["sorted_to_pair"], o["pair_to_sorted"], o["x_perm"], ws)
    assert a.semmoe_check_errors() == 0
    ref = oracle.permute(idx, k, er, R)
    for key, v in ref.items():
        np.testing.assert_array_equal(np_(o[key]), v, err_msg=key)
    want = x.index_select(0, (o["sorted_to_pair"] // k_max).long())
    assert torch.equal(o["x_perm"], want)


@pytest.mark.parametrize("T,E,k_max,H,I,gathered,shared", [
    (500, 16, 4, 256, 640, False, True),      # groups of ~125 rows: GEMM2 in single CTAs
    (8000, 16, 4, 256, 640, True, False),     # groups of ~2000 rows, I >= 512: GEMM2 in 2-SM pairs
    (700, 8, 4, 200, 96, True, True),         # H = 200: a partial last k-block and output tile
    (3000, 64, 6, 512, 352, False, False)])
def test_grouped_ffn_with_folded_combine_matches_oracle(T, E, k_max, H, I, gathered, shared):
    """semmoe_grouped_ffn_combine + semmoe_combine_finish (GEMM2 adding its
    gate-weighted rows into the token order) against the oracle's grouped FFN
    followed by its combine, within the bf16 tolerance; per-token budgets leave
    padding slots; rows from x_perm or gathered from x."""
    a = abi()
    rng = np.random.default_rng(T + I)
    idx, k = _route_random(rng, T, E, k_max)
    _, w = oracle.topk_route(rng.standard_normal((T, E)), k, k_max)   # some gates (values only matter)
    er = (np.arange(E) % 4).astype(np.int32)
    P = int(k.sum())
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w13 = torch.from_numpy((rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w2 = torch.from_numpy((rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32)).to(torch.bfloat16).cuda()
    ys = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).cuda() if shared else None
    eo, ro = torch.empty(E + 1, **i32), torch.empty(5, **i32)
    p2e, ec = torch.empty(E, **i32), torch.empty(E, **i32)
    s2p, p2s = torch.empty(P, **i32), torch.empty(T * k_max, **i32)
    xp = torch.empty(P, H, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(a.semmoe_permute_workspace_size(T, k_max, E), dtype=torch.uint8, device="cuda")
    a.semmoe_permute(torch.from_numpy(idx).cuda(), torch.from_numpy(er).cuda(), x, T, H, E, 4, k_max, P, eo, ro,
                     p2e, ec, s2p, p2s, xp, ws)
    fws = torch.empty(a.semmoe_grouped_ffn_workspace_size(P, I, 1), dtype=torch.uint8, device="cuda")
    acc = torch.full((T, H), 123.0, dtype=torch.float32, device="cuda")       # zeroed by the call
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    tw = torch.from_numpy(w.astype(np.float32)).cuda()
    a.semmoe_grouped_ffn_combine(x if gathered else xp, gathered, s2p, k_max, T, eo, p2e, w13, w2, tw, P, E, H, I,
                                 acc, fws)
    a.semmoe_combine_finish(acc, ys, T, H, out)
    assert a.semmoe_check_errors() == 0
    perm = oracle.permute(idx, k, er, 4, x.cpu())
    y_ref = oracle.grouped_ffn(perm["x_perm"], perm["expert_offsets"], perm["phys_to_expert"],
                               w13.cpu().to(torch.float64).numpy(), w2.cpu().to(torch.float64).numpy(), "bf16")
    ref = oracle.combine(y_ref, perm["pair_to_sorted"], w, k, "bf16", None if ys is None else np_(ys))
    assert max_rel(np_(out), ref) < TOL["bf16"]


def test_folded_combine_flags_a_bad_pair_and_drops_its_row():
    """A sorted_to_pair entry naming no token sets SEMMOE_DEVERR_PAIRS; its row
    is left out of the sums and every token's output is otherwise the oracle's
    with that pair's slot counted as padding."""
    a = abi()
    rng = np.random.default_rng(31)
    T, E, k_max, H, I = 300, 4, 2, 128, 128
    P = T * k_max
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w13 = torch.from_numpy((rng.standard_normal((E, 2 * I, H)) / np.sqrt(H)).astype(np.float32)).to(torch.bfloat16).cuda()
    w2 = torch.from_numpy((rng.standard_normal((E, H, I)) / np.sqrt(I)).astype(np.float32)).to(torch.bfloat16).cuda()
    eo = torch.tensor([0, 150, 300, 450, 600], **i32)
    p2e = torch.tensor([0, 1, 2, 3], **i32)
    s2p_np = rng.permutation(P).astype(np.int32)
    bad_q = 17
    dropped = int(s2p_np[bad_q])
    s2p_np[bad_q] = -3
    w = rng.random((T, k_max)).astype(np.float32)
    fws = torch.empty(a.semmoe_grouped_ffn_workspace_size(P, I, 1), dtype=torch.uint8, device="cuda")
    acc = torch.empty(T, H, dtype=torch.float32, device="cuda")
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    a.semmoe_grouped_ffn_combine(x, True, torch.from_numpy(s2p_np).cuda(), k_max, T, eo, p2e, w13, w2,
                                 torch.from_numpy(w).cuda(), P, E, H, I, acc, fws)
    a.semmoe_combine_finish(acc, None, T, H, out)
    with pytest.raises(a.SemMoEError) as ei:
        a.semmoe_check_errors()
    assert ei.value.bits & a.SEMMOE_DEVERR_PAIRS
    # oracle: the sorted rows' pairs, with the bad row's pair dropped
    x_perm = np_(x)[np.where(s2p_np >= 0, s2p_np, 0) // k_max]
    y_ref = oracle.grouped_ffn(x_perm, eo.cpu(), p2e.cpu(), w13.cpu().to(torch.float64).numpy(),
                               w2.cpu().to(torch.float64).numpy(), "bf16")
    p2s = np.full(T * k_max, -1, dtype=np.int64)
    p2s[s2p_np[s2p_np >= 0]] = np.nonzero(s2p_np >= 0)[0]
    assert p2s[dropped] == -1
    w_ref = w.astype(np.float64)
    w_ref[dropped // k_max, dropped % k_max] = 0.0      # the dropped pair contributes nothing
    ref = oracle.combine(y_ref, p2s, w_ref, np.full(T, k_max), "bf16")
    assert max_rel(np_(out), ref) < TOL["bf16"]
