"""Whole-layer parity of the CUDA path with the oracle on every workload:
small versions (spanning several tiles with ragged tails) compared element by
element in full, and the full-size layers compared on every integer output
plus a seeded sample of tokens for the float outputs."""
import pytest

import workloads as wl
from parity_utils import check_layer_full, check_layer_sampled, run_gpu

pytestmark = pytest.mark.gpu

SMALL = [
    ("tiny_fp32_T256_E8", {}),
    ("tiny_fp32_T256_E8", dict(T=1)),
    ("tiny_fp32_T256_E8", dict(T=77, k=8)),                                    # k = E: dense mixture
    ("tiny_fp32_T256_E8", dict(T=50, E=1, k=1, R=1)),                          # plain SwiGLU MLP
    ("dsv2lite_prefill_T4096", dict(T=300, H=256, I=160, I_shared=320, V=3000)),
    ("dsv2lite_decode_T64", dict(H=256, I=160, I_shared=320, V=3000)),
    ("qwen3_30b_a3b_T16384", dict(T=515, H=256, I=96, V=3000)),
    ("prism_subexpert_T8192", dict(T=512, H=256, I=40, V=3000, tokens_per_request=64)),
]


@pytest.mark.parametrize("name,over", SMALL, ids=[f"{n}-{i}" for i, (n, _) in enumerate(SMALL)])
def test_layer_small(name, over):
    d = wl.make_inputs(wl.scaled(name, **over))
    res, P = run_gpu(d)
    check_layer_full(d, res, P)


FULL = ["tiny_fp32_T256_E8", "dsv2lite_decode_T64", "dsv2lite_decode_T256", "dsv2lite_decode_T512",
        "dsv2lite_prefill_T4096", "qwen3_30b_a3b_T16384", "prism_subexpert_T8192"]


@pytest.mark.parametrize("name", FULL)
def test_layer_full_size(name):
    d = wl.make_inputs(wl.CONFIGS[name])
    res, P = run_gpu(d)
    check_layer_sampled(d, res, P)
