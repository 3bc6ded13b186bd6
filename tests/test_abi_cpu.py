"""The C-ABI library builds, loads and exports every declared entry point;
host-side validation rejects bad arguments before any CUDA call (CPU only)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "semmoe.h")


@pytest.fixture(scope="module")
def lib():
    from token_expert_routing_gb300 import build, _abi
    build.build()
    return _abi.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(semmoe_\w+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    from token_expert_routing_gb300 import _abi
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
        assert n in _abi.SIGNATURES, f"{n} missing from the Python binding"


def test_version(lib):
    assert lib.semmoe_version() >= 100


def test_workspace_sizes(lib):
    assert lib.semmoe_permute_workspace_size(4096, 6, 64) >= 4096 * 6 // 2048 * 64 * 4
    assert lib.semmoe_permute_workspace_size(4096, 6, 64) % 256 == 0
    assert lib.semmoe_grouped_ffn_workspace_size(24576, 1408, 1) >= 24576 * 1408 * 2
    assert lib.semmoe_grouped_ffn_workspace_size(-1, 8, 1) == 0
    assert lib.semmoe_shared_ffn_workspace_size(10, 16, 0) >= 10 * 16 * 4


def _err(lib):
    return lib.semmoe_last_error().decode()


def test_route_validation(lib):
    # E outside [1, 256]
    rc = lib.semmoe_route(None, 1, None, 0, None, None, None, 2, 16, 64, 0, 2, None, None, None, None, 0, None)
    assert rc == 1 and "E" in _err(lib)
    rc = lib.semmoe_route(None, 1, None, 0, None, None, None, 2, 16, 64, 300, 2, None, None, None, None, 0, None)
    assert rc == 1
    # k_max > E
    rc = lib.semmoe_route(None, 1, None, 0, None, None, None, 2, 16, 64, 8, 9, None, None, None, None, 0, None)
    assert rc == 1 and "k_max" in _err(lib)
    # k_uniform outside [1, k_max]
    rc = lib.semmoe_route(None, 1, None, 0, None, None, None, 0, 16, 64, 8, 2, None, None, None, None, 0, None)
    assert rc == 1 and "k_uniform" in _err(lib)
    # null outputs
    rc = lib.semmoe_route(None, 1, None, 0, None, None, None, 2, 16, 64, 8, 2, None, None, None, None, 0, None)
    assert rc == 1 and "null" in _err(lib)
    # T = 0 is a no-op
    assert lib.semmoe_route(None, 1, None, 0, None, None, None, 2, 0, 64, 8, 2, None, None, None, None, 0, None) == 0


def test_permute_validation(lib):
    p = ctypes.c_void_p(256)
    # P larger than T * k_max
    rc = lib.semmoe_permute(p, p, None, 1, 4, 8, 8, 2, 2, 9, p, p, p, p, p, p, None, None, p, 1 << 20, None)
    assert rc == 1 and "P" in _err(lib)
    # undersized workspace
    rc = lib.semmoe_permute(p, p, None, 1, 4, 8, 8, 2, 2, 8, p, p, p, p, p, p, None, None, p, 4, None)
    assert rc == 1 and "workspace" in _err(lib)
    # misaligned workspace
    rc = lib.semmoe_permute(p, p, None, 1, 4, 8, 8, 2, 2, 8, p, p, p, p, p, p, None, None,
                            ctypes.c_void_p(260), 1 << 20, None)
    assert rc == 1
    # x without x_perm
    rc = lib.semmoe_permute(p, p, p, 1, 4, 8, 8, 2, 2, 8, p, p, p, p, p, p, None, None, p, 1 << 20, None)
    assert rc == 1 and "x_perm" in _err(lib)
    # R > E
    rc = lib.semmoe_permute(p, p, None, 1, 4, 8, 4, 5, 2, 8, p, p, p, p, p, p, None, None, p, 1 << 20, None)
    assert rc == 1


def test_ffn_and_combine_validation(lib):
    p = ctypes.c_void_p(1 << 12)
    # I not a multiple of 8
    rc = lib.semmoe_grouped_ffn(p, p, p, p, p, 1, 64, 4, 128, 100, p, p, 1 << 30, None)
    assert rc == 1 and "multiples of 8" in _err(lib)
    # bad dtype
    rc = lib.semmoe_grouped_ffn(p, p, p, p, p, 7, 64, 4, 128, 128, p, p, 1 << 30, None)
    assert rc == 1
    # workspace too small
    rc = lib.semmoe_shared_ffn(p, p, p, 1, 64, 128, 256, p, p, 16, None)
    assert rc == 1 and "workspace" in _err(lib)
    # misaligned y
    rc = lib.semmoe_combine(ctypes.c_void_p(4), p, p, None, 1, 4, 128, 2, 8, p, None)
    assert rc == 1
    # H * 2 bytes not a multiple of 16
    rc = lib.semmoe_combine(p, p, p, None, 1, 4, 12, 2, 8, p, None)
    assert rc == 1
    # no rows: empty activations (null pointers) are fine, nothing is launched
    assert lib.semmoe_grouped_ffn(None, p, p, p, p, 1, 0, 4, 128, 128, None, p, 1 << 30, None) == 0
    assert lib.semmoe_shared_ffn(None, p, p, 1, 0, 128, 256, None, p, 1 << 30, None) == 0
    # rows but no activations
    rc = lib.semmoe_grouped_ffn(None, p, p, p, p, 1, 64, 4, 128, 128, p, p, 1 << 30, None)
    assert rc == 1 and "null" in _err(lib)


def test_remote_count_validation(lib):
    p = ctypes.c_void_p(256)
    rc = lib.semmoe_remote_count(p, p, p, 4, 2, 8, 65, p, p, None)
    assert rc == 1 and "R" in _err(lib)


def test_schedule_validation(lib):
    p = ctypes.c_void_p(256)
    # R outside [1, 64]
    rc = lib.semmoe_dp_schedule(p, p, 8, 2, 65, p, p, p, p, p, p, p, p, None)
    assert rc == 1 and "R = 65" in _err(lib)
    # tokens but no request
    rc = lib.semmoe_dp_schedule(p, p, 8, 0, 4, p, p, p, p, p, p, p, p, None)
    assert rc == 1 and "no request" in _err(lib)
    # null token output
    rc = lib.semmoe_dp_schedule(p, p, 8, 2, 4, p, p, p, p, p, None, p, p, None)
    assert rc == 1 and "null" in _err(lib)
    rc = lib.semmoe_transition_lookup(p, None, 3, p, 8, 2, 16, 4, p, None)
    assert rc == 1 and "k_uniform" in _err(lib)
    rc = lib.semmoe_transition_lookup(p, None, 1, p, 8, 2, 16, 0, p, None)
    assert rc == 1 and "R = 0" in _err(lib)
    rc = lib.semmoe_transition_lookup(p, None, 1, None, 8, 2, 16, 4, p, None)
    assert rc == 1 and "null" in _err(lib)


def test_router_split_validation(lib):
    p = ctypes.c_void_p(256)
    assert lib.semmoe_route_split_size(2048, 64) > 0
    assert lib.semmoe_route_split_size(2047, 64) == 0
    rc = lib.semmoe_route_split_weight(p, 100, 8, p, None)
    assert rc == 1 and "multiple of 8" in _err(lib)
    # a pre-split weight needs bf16 activations
    rc = lib.semmoe_route(p, 0, p, 2, None, None, None, 2, 16, 64, 8, 2, p, p, None, p, 1 << 20, None)
    assert rc == 1 and "dtype" in _err(lib)


def test_product_path_fails_loudly_without_library(monkeypatch):
    from token_expert_routing_gb300 import _abi
    monkeypatch.setattr(_abi, "LIB_PATH", "/nonexistent/libsemmoe.so")
    monkeypatch.setattr(_abi, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        _abi.lib()


def test_ffn_form_validation(lib):
    from token_expert_routing_gb300 import _abi as a
    p = ctypes.c_void_p(1 << 12)

    def call(f1, f2, s2p=None, dtype=1):
        return lib.semmoe_grouped_ffn_form(p, s2p, 2, 64, p, p, p, p, dtype, 64, 4, 128, 128, p, p, 1 << 30, f1, f2,
                                           None)
    # forms outside the enum, or the CUDA-core form in one GEMM only
    assert call(9, 0) == 1 and "form" in _err(lib)
    assert call(a.SEMMOE_FORM_CUDA_CORE, a.SEMMOE_FORM_SINGLE) == 1
    # four-row TMA gathers exist only for a GEMM1 that gathers its rows
    assert call(a.SEMMOE_FORM_SINGLE_TMA_GATHER, a.SEMMOE_FORM_SINGLE) == 1 and "gathered" in _err(lib)
    assert call(a.SEMMOE_FORM_SINGLE, a.SEMMOE_FORM_SINGLE_TMA_GATHER, s2p=p) == 1
    # fp32 runs on CUDA cores only
    assert call(a.SEMMOE_FORM_PAIR, a.SEMMOE_FORM_PAIR, dtype=0) == 1 and "fp32" in _err(lib)
    # the one-launch form covers both GEMMs, from x_perm
    assert call(a.SEMMOE_FORM_FUSED, a.SEMMOE_FORM_SINGLE) == 1 and "form" in _err(lib)
    assert call(a.SEMMOE_FORM_FUSED, a.SEMMOE_FORM_FUSED, s2p=p) == 1 and "FUSED" in _err(lib)
    assert call(a.SEMMOE_FORM_FUSED + 1, a.SEMMOE_FORM_FUSED + 1) == 1
    # no rows: nothing is launched, for any valid form pair
    assert lib.semmoe_grouped_ffn_form(None, None, 1, 0, p, p, p, p, 1, 0, 4, 128, 128, None, p, 1 << 30,
                                       a.SEMMOE_FORM_PAIR, a.SEMMOE_FORM_SINGLE, None) == 0


def test_fused_ready_wait_selftest_validation(lib):
    """The one-launch FFN's failure-path self-test checks its arguments like
    semmoe_grouped_ffn before touching a device."""
    p = ctypes.c_void_p(1 << 12)
    call = lib.semmoe_selftest_fused_ready_wait
    assert call(p, p, p, 0, 128, 128, p, p, 1 << 30, None) == 1 and "P" in _err(lib)
    assert call(p, p, p, 5000, 128, 128, p, p, 1 << 30, None) == 1 and "P" in _err(lib)
    assert call(p, p, p, 64, 100, 128, p, p, 1 << 30, None) == 1 and "multiples of 8" in _err(lib)
    assert call(p, p, p, 64, 128, 128, p, p, 16, None) == 1 and "workspace" in _err(lib)
    assert call(p, None, p, 64, 128, 128, p, p, 1 << 30, None) == 1 and "null" in _err(lib)
