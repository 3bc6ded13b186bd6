"""ctypes binding of libsemmoe.so: the C ABI declared in include/semmoe.h.

Argument marshalling only -- every step runs in the library's CUDA kernels.
Functions carry the C names and take torch tensors (device memory) or None
for pointers; a non-zero status raises SemMoEError with the library's message.
There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsemmoe.so")

SEMMOE_OK, SEMMOE_ERR_INVALID_ARG, SEMMOE_ERR_UNSUPPORTED, SEMMOE_ERR_CUDA, \
    SEMMOE_ERR_DEVICE_CHECK, SEMMOE_ERR_DEVICE_TIMEOUT = range(6)
SEMMOE_F32, SEMMOE_BF16 = 0, 1
SEMMOE_F32_SPLIT = 2   # router weight only: the output of semmoe_route_split_weight
# grouped-FFN kernel forms (semmoe_grouped_ffn_form)
SEMMOE_FORM_DEFAULT, SEMMOE_FORM_SINGLE, SEMMOE_FORM_PAIR1, SEMMOE_FORM_PAIR, SEMMOE_FORM_SINGLE_TMA_GATHER, \
    SEMMOE_FORM_CUDA_CORE, SEMMOE_FORM_FUSED = range(7)
# device error word bits (semmoe_check_errors)
SEMMOE_DEVERR_EXPERT, SEMMOE_DEVERR_TOKEN_ID, SEMMOE_DEVERR_LUT, SEMMOE_DEVERR_K, SEMMOE_DEVERR_PAIRS, \
    SEMMOE_DEVERR_TIMEOUT, SEMMOE_DEVERR_NONFINITE, SEMMOE_DEVERR_OFFSETS, SEMMOE_DEVERR_RANK = \
    (1 << i for i in range(9))

_DTYPE = {torch.float32: SEMMOE_F32, torch.bfloat16: SEMMOE_BF16}

_vp, _i, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t

# name -> (restype, argtypes), in the order of include/semmoe.h
SIGNATURES = {
    "semmoe_last_error": (ctypes.c_char_p, []),
    "semmoe_version": (_i, []),
    "semmoe_kernel_launches": (ctypes.c_ulonglong, []),
    "semmoe_check_errors": (_i, [_vp, ctypes.POINTER(_i)]),
    "semmoe_route_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "semmoe_route": (_i, [_vp, _i, _vp, _i, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _sz, _vp]),
    "semmoe_pair_counts_size": (_sz, [_i, _i]),
    "semmoe_pair_counts_stride": (_i, [_i]),
    "semmoe_route_split_size": (_sz, [_i, _i]),
    "semmoe_route_split_weight": (_i, [_vp, _i, _i, _vp, _vp]),
    "semmoe_route_hier_workspace_size": (_sz, [_i, _i, _i, _i, _i]),
    "semmoe_route_hier": (_i, [_vp, _i, _vp, _i, _vp, _vp, _vp, _i, _vp, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp,
                               _sz, _vp]),
    "semmoe_affinity_lookup": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "semmoe_remote_count": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _vp]),
    "semmoe_permute_workspace_size": (_sz, [_i, _i, _i]),
    "semmoe_permute": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp,
                            _vp, _vp, _vp, _sz, _vp]),
    "semmoe_permute_noalloc": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp,
                                    _vp, _vp, _vp]),
    "semmoe_grouped_ffn_workspace_size": (_sz, [_i, _i, _i]),
    "semmoe_grouped_ffn": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "semmoe_grouped_ffn_gather": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _sz,
                                       _vp]),
    "semmoe_grouped_ffn_form": (_i, [_vp, _vp, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp, _sz,
                                     _i, _i, _vp]),
    "semmoe_grouped_ffn_combine": (_i, [_vp, _i, _vp, _i, _i, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp,
                                        _vp, _sz, _vp]),
    "semmoe_combine_finish": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp]),
    "semmoe_shared_ffn_workspace_size": (_sz, [_i, _i, _i]),
    "semmoe_shared_ffn": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "semmoe_combine": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _vp]),
    "semmoe_selftest_bounded_wait": (_i, [_vp]),
    "semmoe_selftest_fused_ready_wait": (_i, [_vp, _vp, _vp, _i, _i, _i, _vp, _vp, _sz, _vp]),
    "semmoe_dp_schedule": (_i, [_vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "semmoe_transition_lookup": (_i, [_vp, _vp, _i, _vp, _i, _i, _i, _i, _vp, _vp]),
}


class SemMoEError(RuntimeError):
    def __init__(self, code: int, msg: str, bits: int = 0):
        super().__init__(f"[semmoe status {code}] {msg}")
        self.code = code
        self.bits = bits   # device error word bits, for SEMMOE_ERR_DEVICE_CHECK / _TIMEOUT


_lib = None
_lock = threading.Lock()


def lib() -> ctypes.CDLL:
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                       "`python -m token_expert_routing_gb300.build`")
                handle = ctypes.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(handle, name)
                    fn.restype, fn.argtypes = res, args
                _lib = handle
    return _lib


def _check(rc: int) -> None:
    if rc != SEMMOE_OK:
        raise SemMoEError(rc, lib().semmoe_last_error().decode())


def _p(t) -> ctypes.c_void_p | None:
    """Device pointer of a contiguous CUDA tensor (None passes NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return ctypes.c_void_p(t)
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def dtype_code(t: torch.Tensor) -> int:
    try:
        return _DTYPE[t.dtype]
    except KeyError:
        raise ValueError(f"unsupported dtype {t.dtype}") from None


# ---------------------------------------------------------------------------
# one wrapper per C entry point
# ---------------------------------------------------------------------------
def semmoe_version() -> int:
    return lib().semmoe_version()


def semmoe_kernel_launches() -> int:
    return lib().semmoe_kernel_launches()


def semmoe_check_errors(stream=None) -> int:
    """Synchronise the stream and raise if a kernel flagged bad data (the
    error's ``bits`` holds the device error word); returns the bits (0)."""
    bits = ctypes.c_int(0)
    rc = lib().semmoe_check_errors(_stream(stream), ctypes.byref(bits))
    if rc != SEMMOE_OK:
        raise SemMoEError(rc, lib().semmoe_last_error().decode(), bits.value)
    return bits.value


def semmoe_route_workspace_size(T, H, E, x_dtype: int, w_dtype: int) -> int:
    return lib().semmoe_route_workspace_size(T, H, E, x_dtype, w_dtype)


def semmoe_pair_counts_size(T, E) -> int:
    return lib().semmoe_pair_counts_size(T, E)


def semmoe_pair_counts_stride(T) -> int:
    return lib().semmoe_pair_counts_stride(T)


def semmoe_route(x, w_router, logits_in, logits_out, k_per_token, k_uniform, T, H, E, k_max,
                 topk_idx, topk_w, ws=None, stream=None, w_dtype=None, pair_counts=None):
    """Router GEMM + top-k.  ``ws`` defaults to a fresh workspace of the size
    the library asks for (pass one to avoid the allocation); ``w_dtype`` =
    SEMMOE_F32_SPLIT when w_router holds the output of semmoe_route_split_weight;
    ``pair_counts`` (semmoe_pair_counts_size bytes) receives the count table of
    the picks for semmoe_permute."""
    xd = dtype_code(x) if x is not None else SEMMOE_F32
    wd = w_dtype if w_dtype is not None else (dtype_code(w_router) if w_router is not None else SEMMOE_F32)
    if ws is None:
        n = semmoe_route_workspace_size(T, max(H, 1), E, xd, wd)
        ws = torch.empty(n, dtype=torch.uint8, device=topk_idx.device)
    _check(lib().semmoe_route(_p(x), xd, _p(w_router), wd, _p(logits_in), _p(logits_out),
                              _p(k_per_token), k_uniform, T, H, E, k_max, _p(topk_idx), _p(topk_w),
                              _p(pair_counts), _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def semmoe_route_split_size(H, E) -> int:
    return lib().semmoe_route_split_size(H, E)


def semmoe_route_split_weight(w, H, E, split, stream=None):
    _check(lib().semmoe_route_split_weight(_p(w), H, E, _p(split), _stream(stream)))


def semmoe_route_hier_workspace_size(T, H, Ep, x_dtype: int, w_dtype: int) -> int:
    return lib().semmoe_route_hier_workspace_size(T, H, Ep, x_dtype, w_dtype)


def semmoe_route_hier(x, w_parent, logits_in, logits_out, sub_logw, N, k_per_token, k_uniform, T, H, Ep, k_max,
                      topk_idx, topk_w, ws=None, stream=None, w_dtype=None, pair_counts=None):
    """Hierarchical sub-expert routing.  ``ws`` defaults to a fresh workspace
    of the size the library asks for; ``w_dtype`` and ``pair_counts`` as in
    semmoe_route."""
    xd = dtype_code(x) if x is not None else SEMMOE_F32
    wd = w_dtype if w_dtype is not None else (dtype_code(w_parent) if w_parent is not None else SEMMOE_F32)
    if ws is None:
        n = semmoe_route_hier_workspace_size(T, max(H, 1), Ep, xd, wd)
        ws = torch.empty(n, dtype=torch.uint8, device=topk_idx.device)
    _check(lib().semmoe_route_hier(_p(x), xd, _p(w_parent), wd, _p(logits_in), _p(logits_out), _p(sub_logw), N,
                                   _p(k_per_token), k_uniform, T, H, Ep, k_max, _p(topk_idx), _p(topk_w),
                                   _p(pair_counts), _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def semmoe_affinity_lookup(token_ids, lut, V, R, T, pred_rank, stream=None):
    _check(lib().semmoe_affinity_lookup(_p(token_ids), _p(lut), V, R, T, _p(pred_rank), _stream(stream)))


def semmoe_remote_count(topk_idx, pred_rank, expert_rank, T, k_max, E, R, counts, remote, stream=None):
    _check(lib().semmoe_remote_count(_p(topk_idx), _p(pred_rank), _p(expert_rank), T, k_max, E, R,
                                     _p(counts), _p(remote), _stream(stream)))


def semmoe_permute_workspace_size(T, k_max, E) -> int:
    return lib().semmoe_permute_workspace_size(T, k_max, E)


def semmoe_permute(topk_idx, expert_rank, x, T, H, E, R, k_max, P, expert_offsets, rank_offsets,
                   phys_to_expert, expert_counts, sorted_to_pair, pair_to_sorted, x_perm, ws,
                   stream=None, pair_counts=None):
    """``pair_counts``: the router's count table for these topk_idx, or None
    (the permute then counts the pairs itself)."""
    d = dtype_code(x) if x is not None else SEMMOE_F32
    _check(lib().semmoe_permute(_p(topk_idx), _p(expert_rank), _p(x), d, T, H, E, R, k_max, P,
                                _p(expert_offsets), _p(rank_offsets), _p(phys_to_expert),
                                _p(expert_counts), _p(sorted_to_pair), _p(pair_to_sorted), _p(x_perm),
                                _p(pair_counts), _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def semmoe_permute_noalloc(topk_idx, expert_rank, x, T, H, E, R, k_max, P, expert_offsets, rank_offsets,
                           phys_to_expert, expert_counts, sorted_to_pair, pair_to_sorted, x_perm,
                           stream=None):
    """semmoe_permute without a workspace: for callers that cannot allocate
    device memory (the scratch is a static 96 KiB array inside the library)."""
    d = dtype_code(x) if x is not None else SEMMOE_F32
    _check(lib().semmoe_permute_noalloc(_p(topk_idx), _p(expert_rank), _p(x), d, T, H, E, R, k_max, P,
                                        _p(expert_offsets), _p(rank_offsets), _p(phys_to_expert),
                                        _p(expert_counts), _p(sorted_to_pair), _p(pair_to_sorted),
                                        _p(x_perm), _stream(stream)))


def semmoe_grouped_ffn_workspace_size(P, I, dtype: int) -> int:
    return lib().semmoe_grouped_ffn_workspace_size(P, I, dtype)


def semmoe_grouped_ffn(x_perm, expert_offsets, phys_to_expert, w13, w2, P, E, H, I, y_perm, ws,
                       stream=None):
    _check(lib().semmoe_grouped_ffn(_p(x_perm), _p(expert_offsets), _p(phys_to_expert), _p(w13),
                                    _p(w2), dtype_code(w13), P, E, H, I, _p(y_perm), _p(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)))


def semmoe_grouped_ffn_gather(x, sorted_to_pair, k_max, T, expert_offsets, phys_to_expert, w13, w2, P, E, H, I,
                              y_perm, ws, stream=None):
    _check(lib().semmoe_grouped_ffn_gather(_p(x), _p(sorted_to_pair), k_max, T, _p(expert_offsets),
                                           _p(phys_to_expert), _p(w13), _p(w2), dtype_code(w13), P, E, H, I,
                                           _p(y_perm), _p(ws), ws.numel() * ws.element_size(), _stream(stream)))


def semmoe_grouped_ffn_form(x, sorted_to_pair, k_max, T, expert_offsets, phys_to_expert, w13, w2, P, E, H, I,
                            y_perm, ws, form1, form2, stream=None):
    _check(lib().semmoe_grouped_ffn_form(_p(x), _p(sorted_to_pair), k_max, T, _p(expert_offsets),
                                         _p(phys_to_expert), _p(w13), _p(w2), dtype_code(w13), P, E, H, I,
                                         _p(y_perm), _p(ws), ws.numel() * ws.element_size(), form1, form2,
                                         _stream(stream)))


def semmoe_grouped_ffn_combine(x, x_rows_are_tokens, sorted_to_pair, k_max, T, expert_offsets, phys_to_expert, w13,
                               w2, topk_w, P, E, H, I, acc, ws, stream=None):
    _check(lib().semmoe_grouped_ffn_combine(_p(x), int(bool(x_rows_are_tokens)), _p(sorted_to_pair), k_max, T,
                                            _p(expert_offsets), _p(phys_to_expert), _p(w13), _p(w2), _p(topk_w),
                                            dtype_code(w13), P, E, H, I, _p(acc), _p(ws),
                                            ws.numel() * ws.element_size(), _stream(stream)))


def semmoe_combine_finish(acc, y_shared, T, H, out, stream=None):
    _check(lib().semmoe_combine_finish(_p(acc), _p(y_shared), dtype_code(out), T, H, _p(out), _stream(stream)))


def semmoe_shared_ffn_workspace_size(T, I_s, dtype: int) -> int:
    return lib().semmoe_shared_ffn_workspace_size(T, I_s, dtype)


def semmoe_shared_ffn(x, ws13, ws2, T, H, I_s, y_shared, ws, stream=None):
    _check(lib().semmoe_shared_ffn(_p(x), _p(ws13), _p(ws2), dtype_code(ws13), T, H, I_s,
                                   _p(y_shared), _p(ws), ws.numel() * ws.element_size(),
                                   _stream(stream)))


def semmoe_combine(y_perm, pair_to_sorted, topk_w, y_shared, T, H, k_max, P, out, stream=None):
    _check(lib().semmoe_combine(_p(y_perm), _p(pair_to_sorted), _p(topk_w), _p(y_shared),
                                dtype_code(out), T, H, k_max, P, _p(out), _stream(stream)))


def semmoe_dp_schedule(pred_rank, req_offsets, T, n_req, R, hist, req_rank, req_order, rank_req_offsets,
                       req_tok_start, tok_order, tok_rank, rank_tok_offsets, stream=None):
    _check(lib().semmoe_dp_schedule(_p(pred_rank), _p(req_offsets), T, n_req, R, _p(hist), _p(req_rank),
                                    _p(req_order), _p(rank_req_offsets), _p(req_tok_start), _p(tok_order),
                                    _p(tok_rank), _p(rank_tok_offsets), _stream(stream)))


def semmoe_transition_lookup(topk_idx, k_per_token, k_uniform, trans, T, k_max, E, R, pred_next, stream=None):
    _check(lib().semmoe_transition_lookup(_p(topk_idx), _p(k_per_token), k_uniform, _p(trans), T, k_max, E, R,
                                          _p(pred_next), _stream(stream)))


def semmoe_selftest_bounded_wait(stream=None):
    """Launch the wait that can never complete (it gives up after 2 s and sets
    the timeout bit); see include/semmoe.h."""
    _check(lib().semmoe_selftest_bounded_wait(_stream(stream)))


def semmoe_selftest_fused_ready_wait(x_perm, w13, w2, P, H, I, y_perm, ws, stream=None):
    """Run the one-launch grouped FFN with GEMM2's readiness waits made
    unreachable (each gives up after 2 s and sets the timeout bit); see
    include/semmoe.h."""
    _check(lib().semmoe_selftest_fused_ready_wait(_p(x_perm), _p(w13), _p(w2), P, H, I, _p(y_perm), _p(ws),
                                                  ws.numel() * ws.element_size(), _stream(stream)))
