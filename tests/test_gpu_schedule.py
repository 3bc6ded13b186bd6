"""GPU parity of the scheduling calls around the layer, through the C ABI:
semmoe_dp_schedule (Attention-DP request placement) and
semmoe_transition_lookup (next-layer rank from this layer's experts).
Everything here is integer output: compared bit-exactly with the oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

SCHED_KEYS = ("hist", "req_rank", "req_order", "rank_req_offsets", "req_tok_start", "tok_order", "tok_rank",
              "rank_tok_offsets")


def take_bits():
    """The device error word (0 when clean), cleared by the read."""
    from token_expert_routing_gb300 import _abi
    try:
        return _abi.semmoe_check_errors()
    except _abi.SemMoEError as e:
        assert e.code == _abi.SEMMOE_ERR_DEVICE_CHECK, e
        return e.bits


def gpu_schedule(pred, off, R):
    from token_expert_routing_gb300 import _abi
    pred = torch.as_tensor(np.asarray(pred, dtype=np.int32)).cuda()
    off = torch.as_tensor(np.asarray(off, dtype=np.int32)).cuda()
    T, n = pred.shape[0], off.shape[0] - 1
    i32 = dict(dtype=torch.int32, device="cuda")
    # outputs pre-filled with a sentinel so that an unwritten entry shows
    out = dict(hist=torch.full((max(n, 1), R), -7, **i32), req_rank=torch.full((max(n, 1),), -7, **i32),
               req_order=torch.full((max(n, 1),), -7, **i32), rank_req_offsets=torch.full((R + 1,), -7, **i32),
               req_tok_start=torch.full((max(n, 1),), -7, **i32), tok_order=torch.full((T,), -7, **i32),
               tok_rank=torch.full((T,), -7, **i32), rank_tok_offsets=torch.full((R + 1,), -7, **i32))
    _abi.semmoe_dp_schedule(pred, off, T, n, R, *[out[k] for k in SCHED_KEYS])
    bits = take_bits()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    if n == 0:
        for k in ("hist", "req_rank", "req_order", "req_tok_start"):
            res[k] = res[k][:0]
    return res, bits


def check_schedule(pred, off, R):
    got, bits = gpu_schedule(pred, off, R)
    assert bits == 0, f"device error bits {bits:#x}"
    ref = oracle.dp_schedule(pred, off, R)
    for k in SCHED_KEYS:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    return got


def test_schedule_hand_example():
    got = check_schedule([1, 1, 0, 1, 0, 1, 0, 0], [0, 2, 3, 6, 8], 2)
    assert got["tok_order"].tolist() == [2, 6, 7, 0, 1, 3, 4, 5]


@pytest.mark.parametrize("R", [1, 5, 8, 33, 64])
def test_schedule_mixed_lengths_with_empty_requests(R):
    rng = np.random.default_rng(R)
    off = workloads.request_offsets(6000, seed=R, mean_len=40, empty_every=7)
    pred = rng.integers(0, R, size=6000)
    check_schedule(pred, off, R)


def test_schedule_ties_everywhere():
    # every request holds each of its ranks equally often: ties go to the lowest rank
    R = 6
    lens = np.array([0, 2, 6, 12, 1, 3] * 50)
    off = np.concatenate([[0], np.cumsum(lens)])
    T = off[-1]
    pred = np.zeros(T, dtype=np.int64)
    for r in range(len(lens)):
        n = lens[r]
        pred[off[r]:off[r + 1]] = (np.arange(n) + r) % max(1, min(R, n))
    got = check_schedule(pred, off, R)
    assert got["req_rank"].max() < R


def test_schedule_many_short_requests_several_chunks():
    # one token per request (decode), more requests than one 1024-thread pass
    rng = np.random.default_rng(3)
    T = 5000
    check_schedule(rng.integers(0, 8, size=T), np.arange(T + 1), 8)


def test_schedule_one_long_request_and_wide_path():
    rng = np.random.default_rng(4)
    # a long request dominating a batch (the 4-warp-per-request kernel form)
    check_schedule(rng.integers(0, 8, size=20000), [0, 20000], 8)
    check_schedule(rng.integers(0, 8, size=20000), [0, 7, 19000, 20000], 8)


def test_schedule_empty_batch():
    got, bits = gpu_schedule(np.zeros(0, dtype=np.int32), [0], 4)
    assert bits == 0
    assert got["rank_req_offsets"].tolist() == [0] * 5 and got["rank_tok_offsets"].tolist() == [0] * 5


@pytest.mark.parametrize("name", sorted(workloads.CONFIGS))
def test_schedule_workload_requests(name):
    d = workloads.make_inputs(workloads.CONFIGS[name], with_weights=False)
    pred = oracle.affinity_lookup(d["token_ids"], d["lut"])
    check_schedule(pred, d["req_offsets"].numpy(), d["spec"].R)


def test_schedule_bad_offsets_are_reported():
    """Offsets that run backwards and past T: the kernels clamp every range,
    drop writes past T and set the offsets bit; nothing is read or written out
    of bounds, so the bit is all the caller sees."""
    from token_expert_routing_gb300 import _abi
    pred = np.zeros(16, dtype=np.int32)
    got, bits = gpu_schedule(pred, [0, 10, 4, 16], 2)
    assert bits & _abi.SEMMOE_DEVERR_OFFSETS
    got, bits = gpu_schedule(np.array([0, 1, 9, 0], dtype=np.int32), [0, 2, 4], 2)
    assert bits & _abi.SEMMOE_DEVERR_RANK


def gpu_transition(idx, kpt, ku, trans):
    from token_expert_routing_gb300 import _abi
    T, k_max = idx.shape
    E, R = trans.shape
    out = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    idx_d = torch.as_tensor(np.asarray(idx, dtype=np.int32)).cuda()
    kpt_d = None if kpt is None else torch.as_tensor(np.asarray(kpt, dtype=np.int32)).cuda()
    tr = torch.as_tensor(np.asarray(trans, dtype=np.float32)).cuda()
    _abi.semmoe_transition_lookup(idx_d, kpt_d, ku, tr, T, k_max, E, R, out)
    return out.cpu().numpy(), take_bits()


def padded_topk(rng, T, E, k_max, kpt):
    idx = np.stack([rng.permutation(E)[:k_max] for _ in range(T)]).astype(np.int32)
    return np.where(np.arange(k_max)[None, :] < np.asarray(kpt)[:, None], idx, -1)


@pytest.mark.parametrize("E,R,k_max", [(8, 4, 2), (64, 8, 6), (128, 8, 8), (256, 64, 24), (256, 33, 40),
                                       (16, 1, 3)])
def test_transition_random_tables(E, R, k_max):
    rng = np.random.default_rng(E + R)
    T = 3001
    kpt = rng.integers(1, k_max + 1, size=T)
    idx = padded_topk(rng, T, E, k_max, kpt)
    for trans in (workloads.transition_table(E, R, seed=E),                       # integer counts
                  (rng.integers(0, 3, size=(E, R)) * 0.5).astype(np.float32),     # many exact ties
                  rng.standard_normal((E, R)).astype(np.float32)):               # rounding order matters
        got, bits = gpu_transition(idx, kpt, 0, trans)
        assert bits == 0
        np.testing.assert_array_equal(got, oracle.transition_lookup(idx, kpt, trans))


def test_transition_uniform_k_matches_per_token():
    rng = np.random.default_rng(9)
    T, E, R, k = 4096, 64, 8, 6
    idx = padded_topk(rng, T, E, k, np.full(T, k))
    trans = workloads.transition_table(E, R, seed=1)
    got_u, bits = gpu_transition(idx, None, k, trans)
    assert bits == 0
    np.testing.assert_array_equal(got_u, oracle.transition_lookup(idx, np.full(T, k), trans))


@pytest.mark.parametrize("name", ["dsv2lite_prefill_T4096", "qwen3_30b_a3b_T16384", "prism_subexpert_T8192"])
def test_layer_schedule_and_transition(name):
    """The layer with requests and a transition table: the schedule, the
    source ranks of the remote count and the next-layer prediction against the
    oracle, at the workload's full size (routing from the GPU's own fp32 logits)."""
    from token_expert_routing_gb300 import MoELayer, _abi
    spec = workloads.CONFIGS[name]
    d = workloads.make_inputs(spec, with_weights=True)
    layer = MoELayer(d["w_router"], d["w13"], d["w2"], d["expert_rank"], d["lut"], spec.R, spec.k_max,
                     d["ws13"], d["ws2"], trans=d["trans"])
    kpt = d["k_per_token"].cuda() if spec.k_choices else None
    P = int(d["k_per_token"].sum())
    res = layer.forward(d["x"].cuda(), d["token_ids"].cuda(), kpt, None if spec.k_choices else spec.k, P,
                        keep_logits=True, req_offsets=d["req_offsets"].cuda())
    assert _abi.semmoe_check_errors() == 0
    k = d["k_per_token"].numpy()
    idx, _ = oracle.topk_route(res.logits.cpu().numpy(), k, spec.k_max)
    np.testing.assert_array_equal(res.topk_idx.cpu().numpy(), idx)
    pred = oracle.affinity_lookup(d["token_ids"], d["lut"])
    ref = oracle.dp_schedule(pred, d["req_offsets"].numpy(), spec.R)
    for key in SCHED_KEYS:
        got = res.schedule[key].cpu().numpy()
        if key in ("hist", "req_rank", "req_order", "req_tok_start"):
            got = got[:ref[key].shape[0]]
        np.testing.assert_array_equal(got, ref[key], err_msg=key)
    counts, remote = oracle.remote_count(idx, k, ref["tok_rank"], d["expert_rank"], spec.R)
    np.testing.assert_array_equal(res.counts.cpu().numpy(), counts)
    np.testing.assert_array_equal(res.remote.cpu().numpy(), remote)
    np.testing.assert_array_equal(res.pred_next.cpu().numpy(), oracle.transition_lookup(idx, k, d["trans"]))
