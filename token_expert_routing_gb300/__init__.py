"""Affinity-aware MoE layer forward for GB300 (sm_103a).

A C-ABI library (``libsemmoe.so``, declared in ``include/semmoe.h``) of
hand-written CUDA kernels for one MoE layer forward -- router + top-k,
token-id affinity lookup and remote-activation count, stable permute by
(rank, expert), grouped SwiGLU FFN, combine -- after Sem-MoE's semantic
parallelism and MoE-Prism's per-request routing budgets.  This package holds
the library sources (``csrc/``), its build script, the ctypes binding
(``_abi``) and a thin layer driver (``layer``).
"""
from . import _abi  # noqa: F401
from ._abi import SemMoEError  # noqa: F401
from .layer import CapturedLayer, GraphPipeline, HostPipeline, LayerOutput, MoELayer  # noqa: F401

__all__ = ["MoELayer", "LayerOutput", "HostPipeline", "GraphPipeline", "CapturedLayer", "SemMoEError"]
