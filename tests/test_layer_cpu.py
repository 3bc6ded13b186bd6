"""Host-side logic of the layer object, no GPU needed."""
import torch

from token_expert_routing_gb300.layer import fuse_gather_default


def test_fuse_gather_default_rule():
    """The permute is fused into GEMM1 by default exactly for bf16 experts with
    I <= 384, i.e. at most 3 GEMM1 output tiles of 128 h columns per row."""
    for I in (1, 96, 128, 352, 384):
        assert fuse_gather_default(I, torch.bfloat16)
    for I in (385, 392, 512, 768, 1408):
        assert not fuse_gather_default(I, torch.bfloat16)
    for I in (96, 352, 1408):  # fp32 experts run on the CUDA-core path
        assert not fuse_gather_default(I, torch.float32)
