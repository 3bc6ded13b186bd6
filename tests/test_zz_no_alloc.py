"""The allocation-free permute entry point (semmoe_permute_noalloc).

Some callers cannot allocate device memory -- a plugin running inside a host
engine that owns every byte of device memory, or a serving loop that forbids
cudaMalloc after start-up -- so the library offers a permute whose scratch is
a static device array.  These tests check that it rejects sizes beyond that
array on the host, and that on the GPU it returns exactly what the
workspace-taking semmoe_permute returns, on two calls in a row (the second
with other routing, so stale scratch from the first call would show).

This file is collected last on purpose; it must pass both alone in a fresh
process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch


def test_noalloc_rejects_sizes_beyond_its_static_scratch():
    """The static scratch is sized for E <= 256 experts; larger sizes are refused
    on the host with a clear message, before any device work."""
    from token_expert_routing_gb300 import _abi, build
    build.build()
    lib = _abi.lib()
    p = ctypes.c_void_p(256)
    rc = lib.semmoe_permute_noalloc(p, p, None, 1, 4096, 8, 300, 8, 8, 16, p, p, p, p, p, p, None, None)
    assert rc == _abi.SEMMOE_ERR_INVALID_ARG
    assert "E = 300" in lib.semmoe_last_error().decode()
    rc = lib.semmoe_permute_noalloc(p, p, None, 1, 1 << 28, 16, 256, 8, 8, 16, p, p, p, p, p, p, None, None)
    assert rc == _abi.SEMMOE_ERR_INVALID_ARG
    assert "too large" in lib.semmoe_last_error().decode()


def _routing(rng, T, E, k_max):
    l = rng.standard_normal((T, E))
    order = np.argsort(-l, axis=1, kind="stable")[:, :k_max]
    k = rng.integers(1, k_max + 1, size=T)
    idx = np.where(np.arange(k_max)[None, :] < k[:, None], order, -1)
    return idx.astype(np.int32), k


def _run(fn_name, idx, er, x, T, H, E, R, k_max, P):
    from token_expert_routing_gb300 import _abi
    i32 = dict(dtype=torch.int32, device="cuda")
    outs = dict(expert_offsets=torch.empty(E + 1, **i32), rank_offsets=torch.empty(R + 1, **i32),
                phys_to_expert=torch.empty(E, **i32), expert_counts=torch.empty(E, **i32),
                sorted_to_pair=torch.empty(max(P, 1), **i32), pair_to_sorted=torch.empty(T * k_max, **i32),
                x_perm=torch.empty(P, H, dtype=x.dtype, device="cuda"))
    args = [torch.from_numpy(idx).cuda(), torch.from_numpy(er).cuda(), x, T, H, E, R, k_max, P,
            outs["expert_offsets"], outs["rank_offsets"], outs["phys_to_expert"], outs["expert_counts"],
            outs["sorted_to_pair"], outs["pair_to_sorted"], outs["x_perm"]]
    if fn_name == "semmoe_permute":
        ws = torch.empty(_abi.semmoe_permute_workspace_size(T, k_max, E), dtype=torch.uint8, device="cuda")
        _abi.semmoe_permute(*args, ws)
    else:
        _abi.semmoe_permute_noalloc(*args)
    assert _abi.semmoe_check_errors() == 0
    outs["sorted_to_pair"] = outs["sorted_to_pair"][:P]
    return {k: v.cpu() for k, v in outs.items()}


@pytest.mark.gpu
def test_noalloc_matches_workspace_permute_on_two_calls():
    """Two calls in a row, the second with other routing: each equals the
    workspace-taking permute bit for bit, and the oracle's permutation."""
    import oracle
    rng = np.random.default_rng(2024)
    for T, E, R, k_max, H in ((4096, 64, 8, 6, 256), (3001, 256, 8, 24, 64)):
        idx, k = _routing(rng, T, E, k_max)
        P = int(k.sum())
        er = rng.permutation(np.arange(E) % R).astype(np.int32)
        x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).cuda()
        want = _run("semmoe_permute", idx, er, x, T, H, E, R, k_max, P)
        got = _run("semmoe_permute_noalloc", idx, er, x, T, H, E, R, k_max, P)
        for key in want:
            assert torch.equal(got[key], want[key]), (T, E, key)
        ref = oracle.permute(idx, k, er, R, x.cpu())
        for key in ref:
            g = got[key].to(torch.float64) if key == "x_perm" else got[key]
            assert np.array_equal(g.numpy(), ref[key]), (T, E, key)
