"""One affinity-aware MoE layer forward on one GPU, through the C ABI.

``MoELayer.forward`` enqueues the library calls on the current stream:
route -> affinity lookup (-> request scheduling) -> remote count -> permute ->
grouped FFN (+ shared FFN) -> combine, plus the next-layer transition lookup
when the layer holds a transition table.  Torch only provides device memory and the stream; every
step runs in the library's kernels, and nothing synchronises the host.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import _abi as abi


@dataclass
class LayerOutput:
    out: torch.Tensor
    logits: Optional[torch.Tensor]
    topk_idx: torch.Tensor
    topk_w: torch.Tensor
    pred_rank: torch.Tensor
    counts: torch.Tensor
    remote: torch.Tensor
    expert_offsets: torch.Tensor
    rank_offsets: torch.Tensor
    phys_to_expert: torch.Tensor
    expert_counts: torch.Tensor
    sorted_to_pair: torch.Tensor
    pair_to_sorted: torch.Tensor
    x_perm: Optional[torch.Tensor]   # None when GEMM1 gathers x through the permutation
    y_perm: Optional[torch.Tensor]   # None when GEMM2 adds its rows into the token order (fused_combine)
    y_shared: Optional[torch.Tensor]
    schedule: Optional[dict] = None      # semmoe_dp_schedule outputs (when req_offsets is given)
    pred_next: Optional[torch.Tensor] = None  # next-layer rank per token (when trans is held)


def fuse_combine_default(I: int, dtype, shared: bool) -> bool:
    """Whether a layer folds the combine into GEMM2 by default (semmoe_grouped_ffn_combine).

    Off for every shape: the float4 atomic adds in GEMM2's epilogue (about 6 TB/s
    of fp32 payload at best) slow GEMM2 by more than the y_perm round trip and
    the combine kernel cost.  Measured on GB300, whole layer in graph replay,
    unfolded against folded: Qwen3 (I 768) 1044 against 1160 us; MoE-Prism
    (I 352) 821 against 909; DeepSeek prefill 498 against 502; DeepSeek decode
    T = 512 234 against 236."""
    return False


def fuse_gather_default(I: int, dtype) -> bool:
    """Whether a layer fuses the permute's row gather into GEMM1 by default.

    Each x row is gathered once per GEMM1 output tile of 128 h columns, while
    the copy it replaces is written once, so fusing pays off only for narrow
    experts: on for bf16 experts with I <= 384 (at most 3 tiles).  Measured,
    one-stream layer on GB300: MoE-Prism (I 352) 815 against 852 us; Qwen3
    (I 768) 1188 against 1086; DeepSeek (I 1408) 569 against 523.  fp32
    experts take the CUDA-core path, where no tile count applies."""
    return I <= 384 and dtype == torch.bfloat16


class MoELayer:
    """Weights and tables of one MoE layer, resident on a CUDA device.

    w_router [E,H] (fp32 or bf16), w13 [E,2I,H], w2 [E,H,I] (activation type),
    expert_rank [E] and lut [V] int32, R logical ranks, k_max the largest budget;
    ws13 [2*I_s,H] / ws2 [H,I_s] optional shared experts; trans [E,R] fp32 an
    optional expert -> next-layer-rank transition table.  With ``sub_logw``
    [E] fp32 the layer routes by MoE-Prism's hierarchical gating: w_router is
    then the parent router [Ep,H] and each parent owns N = E / Ep sub-experts.
    """

    def __init__(self, w_router, w13, w2, expert_rank, lut, R: int, k_max: int, ws13=None, ws2=None,
                 trans=None, sub_logw=None, fused_gather: Optional[bool] = None,
                 fused_combine: Optional[bool] = None, overlap: bool = True,
                 overlap_shared: bool = True, shared_at: str = "start", device="cuda"):
        dev = torch.device(device)
        c = lambda t: None if t is None else t.to(dev).contiguous()  # noqa: E731
        self.w_router, self.w13, self.w2 = c(w_router), c(w13), c(w2)
        self.expert_rank = c(expert_rank).to(torch.int32)
        self.lut = c(lut).to(torch.int32)
        self.ws13, self.ws2 = c(ws13), c(ws2)
        self.trans = None if trans is None else c(trans).to(torch.float32)
        self.sub_logw = None if sub_logw is None else c(sub_logw).to(torch.float32)
        # overlap: the lookup, scheduling and counting steps (nothing later in
        # the layer reads them) run on a second stream beside the permute and
        # the FFN; overlap_shared: the shared experts' FFN runs there too, from
        # the start of the forward (shared_at="start": it fills the SMs the
        # router and permute leave idle), after the router ("route", measured
        # the same) or after the permute ("permute", 4-7% slower); without
        # overlap_shared it runs at that point in order on the caller's stream
        self.overlap, self.overlap_shared = overlap, overlap_shared
        if shared_at not in ("start", "route", "permute"):
            raise ValueError("shared_at is 'start', 'route' or 'permute'")
        self.shared_at = shared_at  # where the shared experts' FFN forks off: before the router, or after the permute
        self._side = None
        self.E, twoI, self.H = self.w13.shape
        self.I = twoI // 2
        # fused_gather: GEMM1 gathers its rows of x through the permutation and
        # no x_perm is written (bit-identical); None = fuse_gather_default
        if fused_gather is None:
            fused_gather = fuse_gather_default(self.I, self.w13.dtype)
        self.fused_gather = bool(fused_gather)
        # fused_combine: GEMM2 adds its gate-weighted rows into an fp32 token-order
        # accumulator (no y_perm); bf16 experts only; None = fuse_combine_default
        if fused_combine is None:
            fused_combine = fuse_combine_default(self.I, self.w13.dtype, ws13 is not None)
        if fused_combine and self.w13.dtype != torch.bfloat16:
            raise ValueError("fused_combine needs bf16 experts")
        self.fused_combine = bool(fused_combine)
        self.I_s = 0 if ws13 is None else self.ws13.shape[0] // 2
        self.R, self.k_max, self.V = R, k_max, self.lut.shape[0]
        self.Ep = self.w_router.shape[0]          # router rows: experts, or parents (hierarchical)
        if self.sub_logw is not None and (self.E % self.Ep or self.sub_logw.numel() != self.E):
            raise ValueError("hierarchical gating needs E = Ep * N and sub_logw of E values")
        self.dtype = self.w13.dtype
        self.device = dev
        self._ws = {}
        # An fp32 router weight meeting bf16 activations is split into its three
        # bf16 parts once here instead of on every call.
        self.w_route, self.w_route_dtype = self.w_router, abi.dtype_code(self.w_router)
        if self.w_router.dtype == torch.float32 and self.dtype == torch.bfloat16 and self.H % 8 == 0:
            n = abi.semmoe_route_split_size(self.H, self.Ep)
            self.w_route = torch.empty(n, dtype=torch.uint8, device=dev)
            abi.semmoe_route_split_weight(self.w_router, self.H, self.Ep, self.w_route)
            self.w_route_dtype = abi.SEMMOE_F32_SPLIT

    def _router_weight(self, x):
        """The router weight to pass with x, and its type code (the pre-split
        fp32 weight when x is bf16)."""
        if self.w_route_dtype == abi.SEMMOE_F32_SPLIT and x.dtype != torch.bfloat16:
            return self.w_router, abi.dtype_code(self.w_router)
        return self.w_route, self.w_route_dtype

    def _workspace(self, key, nbytes):
        buf = self._ws.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
            self._ws[key] = buf
        return buf

    def _side_stream(self):
        if self._side is None:
            self._side = torch.cuda.Stream(device=self.device)
        return self._side

    def forward(self, x, token_ids, k_per_token=None, k: Optional[int] = None, P: Optional[int] = None,
                logits_in=None, keep_logits: bool = False, stream=None, marks=None,
                req_offsets=None, side_marks=None, mark_external: bool = False) -> LayerOutput:
        """x [T,H] (activation type) and token_ids [T] int32 on the device.

        Budgets: ``k`` for every token, or ``k_per_token`` [T] int32 on the device
        together with ``P`` = its sum (known to the caller, so no host sync).
        ``req_offsets`` [n_req+1] int32 on the device: the batch's requests; when
        given, requests are scheduled onto ranks by affinity and each token's
        source rank for the remote count is its request's rank.
        ``marks``: optional list; a CUDA event is recorded on the stream after
        each step and appended as (step name, event), for per-step timing;
        ``side_marks`` gets (step name, start event, end event) for the steps
        run on the second stream.  ``mark_external``: the marks' events are
        recorded as event nodes when the forward is captured in a CUDA graph
        (so each replay times its steps).  Every step has finished on ``stream``
        when the work enqueued by this call has.
        """
        s = torch.cuda.current_stream() if stream is None else stream
        side = self._side_stream() if (self.overlap or self.overlap_shared) else None

        def mark(name):
            if marks is not None:
                ev = torch.cuda.Event(enable_timing=True, external=True) if mark_external else \
                    torch.cuda.Event(enable_timing=True)
                ev.record(s)
                marks.append((name, ev))

        forked = []

        def fork():
            ev = torch.cuda.Event()
            ev.record(s)
            side.wait_event(ev)
            forked.append(ev)

        def join():
            ev = torch.cuda.Event()
            ev.record(side)
            s.wait_event(ev)

        def side_event():
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(side)
            return ev

        mark("start")
        T = x.shape[0]
        H, E, I, R, k_max = self.H, self.E, self.I, self.R, self.k_max
        dev = self.device
        dcode = abi.dtype_code(self.w13)
        y_shared = None
        shared_side = self.ws13 is not None and self.overlap_shared

        def run_shared():  # the shared experts' FFN: on the second stream, or in order on this one
            nonlocal y_shared
            y_shared = torch.empty(T, H, dtype=x.dtype, device=dev)
            wss = self._workspace("shared", abi.semmoe_shared_ffn_workspace_size(T, self.I_s, dcode))
            if not shared_side:
                abi.semmoe_shared_ffn(x, self.ws13, self.ws2, T, H, self.I_s, y_shared, wss, s)
                mark("shared_ffn")
                return
            fork()
            ev1 = side_event() if side_marks is not None else None
            abi.semmoe_shared_ffn(x, self.ws13, self.ws2, T, H, self.I_s, y_shared, wss, side)
            if side_marks is not None:
                side_marks.append(("shared_ffn", ev1, side_event()))

        has_shared = self.ws13 is not None
        if has_shared and self.shared_at == "start":
            run_shared()
        if k_per_token is None:
            if k is None:
                raise ValueError("give k or k_per_token")
            P = T * k
        elif P is None:
            raise ValueError("k_per_token needs P = sum(k_per_token)")
        i32 = dict(dtype=torch.int32, device=dev)
        Ep = self.Ep
        logits = torch.empty(T, Ep, dtype=torch.float32, device=dev) if keep_logits else None
        topk_idx = torch.empty(T, k_max, **i32)
        topk_w = torch.empty(T, k_max, dtype=torch.float32, device=dev)
        # the router counts its picks per 128-token chunk; the permute starts from that table
        pair_counts = torch.empty(max(abi.semmoe_pair_counts_size(T, E) // 4, 4), **i32)
        if self.sub_logw is None:
            wr, wd = self._router_weight(x)
            ws = self._workspace("route", abi.semmoe_route_workspace_size(T, H, E, abi.dtype_code(x), wd))
            abi.semmoe_route(x, wr, logits_in, logits, k_per_token, k or 0, T, H, E, k_max,
                             topk_idx, topk_w, ws, stream, w_dtype=wd, pair_counts=pair_counts)
        else:
            wr, wd = self._router_weight(x)
            ws = self._workspace("route", abi.semmoe_route_hier_workspace_size(T, H, Ep, abi.dtype_code(x), wd))
            abi.semmoe_route_hier(x, wr, logits_in, logits, self.sub_logw, E // Ep, k_per_token,
                                  k or 0, T, H, Ep, k_max, topk_idx, topk_w, ws, stream, w_dtype=wd,
                                  pair_counts=pair_counts)
        mark("route")
        if has_shared and self.shared_at == "route":
            run_shared()
        ts = s
        if self.overlap:  # lookup .. counts on the second stream
            fork()
            ts = side
            ev0 = side_event() if side_marks is not None else None
        pred = torch.empty(T, **i32)
        abi.semmoe_affinity_lookup(token_ids, self.lut, self.V, R, T, pred, ts)
        src = pred
        sched = None
        if req_offsets is not None:
            n_req = req_offsets.shape[0] - 1
            sched = dict(hist=torch.empty(max(n_req, 1), R, **i32), req_rank=torch.empty(max(n_req, 1), **i32),
                         req_order=torch.empty(max(n_req, 1), **i32), rank_req_offsets=torch.empty(R + 1, **i32),
                         req_tok_start=torch.empty(max(n_req, 1), **i32), tok_order=torch.empty(T, **i32),
                         tok_rank=torch.empty(T, **i32), rank_tok_offsets=torch.empty(R + 1, **i32))
            abi.semmoe_dp_schedule(pred, req_offsets, T, n_req, R, sched["hist"], sched["req_rank"],
                                   sched["req_order"], sched["rank_req_offsets"], sched["req_tok_start"],
                                   sched["tok_order"], sched["tok_rank"], sched["rank_tok_offsets"], ts)
            src = sched["tok_rank"]
        pred_next = None
        if self.trans is not None:
            pred_next = torch.empty(T, **i32)
            abi.semmoe_transition_lookup(topk_idx, k_per_token, k or 0, self.trans, T, k_max, E, R, pred_next,
                                         ts)
        counts = torch.empty(R, R, **i32)
        remote = torch.empty(R, **i32)
        abi.semmoe_remote_count(topk_idx, src, self.expert_rank, T, k_max, E, R, counts, remote, ts)
        if self.overlap:
            if side_marks is not None:
                side_marks.append(("lookup_count", ev0, side_event()))
        else:
            mark("lookup_count")
        expert_offsets = torch.empty(E + 1, **i32)
        rank_offsets = torch.empty(R + 1, **i32)
        phys_to_expert = torch.empty(E, **i32)
        expert_counts = torch.empty(E, **i32)
        sorted_to_pair = torch.empty(max(P, 1), **i32)
        pair_to_sorted = torch.empty(T * k_max, **i32)
        x_perm = None if self.fused_gather else torch.empty(P, H, dtype=x.dtype, device=dev)
        ws = self._workspace("permute", abi.semmoe_permute_workspace_size(T, k_max, E))
        abi.semmoe_permute(topk_idx, self.expert_rank, None if self.fused_gather else x, T, H, E, R, k_max, P,
                           expert_offsets, rank_offsets, phys_to_expert, expert_counts, sorted_to_pair,
                           pair_to_sorted, x_perm, ws, stream, pair_counts=pair_counts)
        mark("permute")
        y_perm = None if self.fused_combine else torch.empty(P, H, dtype=x.dtype, device=dev)
        acc = torch.empty(T, H, dtype=torch.float32, device=dev) if self.fused_combine else None
        if has_shared and self.shared_at == "permute":  # the shared experts beside the routed FFN
            run_shared()
        ws = self._workspace("ffn", abi.semmoe_grouped_ffn_workspace_size(P, I, dcode))
        if self.fused_combine:  # GEMM2 adds its rows into the token order
            abi.semmoe_grouped_ffn_combine(x if self.fused_gather else x_perm, self.fused_gather, sorted_to_pair,
                                           k_max, T, expert_offsets, phys_to_expert, self.w13, self.w2, topk_w,
                                           P, E, H, I, acc, ws, stream)
        elif self.fused_gather:
            abi.semmoe_grouped_ffn_gather(x, sorted_to_pair, k_max, T, expert_offsets, phys_to_expert, self.w13,
                                          self.w2, P, E, H, I, y_perm, ws, stream)
        else:
            abi.semmoe_grouped_ffn(x_perm, expert_offsets, phys_to_expert, self.w13, self.w2, P, E, H, I,
                                   y_perm, ws, stream)
        mark("grouped_ffn")
        if forked:
            join()  # the second stream's steps are done before the combine (and the call's end)
        out = torch.empty(T, H, dtype=x.dtype, device=dev)
        if self.fused_combine:
            abi.semmoe_combine_finish(acc, y_shared, T, H, out, stream)
        else:
            abi.semmoe_combine(y_perm, pair_to_sorted, topk_w, y_shared, T, H, k_max, P, out, stream)
        mark("combine")
        return LayerOutput(out, logits, topk_idx, topk_w, pred, counts, remote, expert_offsets,
                           rank_offsets, phys_to_expert, expert_counts, sorted_to_pair[:P],
                           pair_to_sorted, x_perm, y_perm, y_shared, sched, pred_next)

    def forward_host(self, x_host, ids_host, k_host=None, k: Optional[int] = None, out_host=None,
                     stream=None) -> torch.Tensor:
        """End-to-end call on host tensors (ideally pinned): copy the inputs in,
        run the layer, copy ``out`` back.  Returns the host output tensor."""
        s = torch.cuda.current_stream() if stream is None else stream
        with torch.cuda.stream(s):
            x = x_host.to(self.device, non_blocking=True)
            ids = ids_host.to(self.device, non_blocking=True)
            kpt, P = None, None
            if k_host is not None:
                kpt = k_host.to(self.device, non_blocking=True)
                P = int(k_host.sum())
            res = self.forward(x, ids, kpt, k, P, stream=s)
            if out_host is None:
                out_host = torch.empty(res.out.shape, dtype=res.out.dtype, pin_memory=True)
            out_host.copy_(res.out, non_blocking=True)
        return out_host


class HostPipeline:
    """Host-buffer layer calls with copies overlapped across calls.

    Each ``submit`` copies that call's inputs host→device, runs the layer and
    copies ``out`` back into the given host tensor, like ``MoELayer.forward_host``;
    but uploads and readbacks run on streams of their own (one each, so a
    readback waiting for its call never holds up the next upload),
    double-buffered, so the upload of call i+1 and the readback of call i-1
    overlap the compute of call i.  Host tensors should be pinned.
    ``synchronize()`` waits for all.
    """

    def __init__(self, layer: MoELayer, stream=None):
        self.layer = layer
        self.compute = torch.cuda.current_stream() if stream is None else stream
        self.copy = torch.cuda.Stream(device=layer.device)     # uploads
        self.down = torch.cuda.Stream(device=layer.device)     # readbacks
        self._slot = 0
        self._free = [None, None]      # event: slot's device inputs are no longer read
        self._bufs = [None, None]

    def _buffers(self, slot, x_host, ids_host, k_host):
        b = self._bufs[slot]
        if b is None or b["x"].shape != x_host.shape:
            dev = self.layer.device
            b = dict(x=torch.empty(x_host.shape, dtype=x_host.dtype, device=dev),
                     ids=torch.empty(ids_host.shape, dtype=ids_host.dtype, device=dev),
                     k=None if k_host is None else torch.empty(k_host.shape, dtype=k_host.dtype, device=dev))
            self._bufs[slot] = b
        return b

    def submit(self, x_host, ids_host, out_host, k_host=None, k: Optional[int] = None):
        slot = self._slot
        self._slot ^= 1
        b = self._buffers(slot, x_host, ids_host, k_host)
        P = None if k_host is None else int(k_host.sum())
        with torch.cuda.stream(self.copy):
            if self._free[slot] is not None:
                self.copy.wait_event(self._free[slot])   # the call two back has read these buffers
            b["x"].copy_(x_host, non_blocking=True)
            b["ids"].copy_(ids_host, non_blocking=True)
            if k_host is not None:
                b["k"].copy_(k_host, non_blocking=True)
            uploaded = torch.cuda.Event()
            uploaded.record(self.copy)
        self.compute.wait_event(uploaded)
        with torch.cuda.stream(self.compute):
            res = self.layer.forward(b["x"], b["ids"], b["k"], k, P, stream=self.compute)
            done = torch.cuda.Event()
            done.record(self.compute)
        self._free[slot] = done
        with torch.cuda.stream(self.down):
            self.down.wait_event(done)
            res.out.record_stream(self.down)
            out_host.copy_(res.out, non_blocking=True)
        return out_host

    def synchronize(self):
        self.copy.synchronize()
        self.down.synchronize()
        self.compute.synchronize()


class CapturedLayer:
    """One layer forward captured as a CUDA graph for a fixed batch shape.

    MoE-Prism (ko) §2 B splits the block at the attention/MoE boundary and keeps
    one graph of the MoE segment per routing budget k; this is that segment for
    one (T, k) -- or one per-token budget vector -- with static buffers: write
    the inputs into ``x`` / ``token_ids`` (and ``k_per_token``), ``replay()``,
    read ``result.out``.  Replays launch every kernel of the forward with one
    graph launch.
    """

    def __init__(self, layer: MoELayer, T: int, k: Optional[int] = None, k_per_token_host=None,
                 req_offsets_host=None, warmup: int = 2):
        if (k is None) == (k_per_token_host is None):
            raise ValueError("give exactly one of k and k_per_token_host")
        dev = layer.device
        self.layer = layer
        self.x = torch.zeros(T, layer.H, dtype=layer.dtype, device=dev)
        self.token_ids = torch.zeros(T, dtype=torch.int32, device=dev)
        self.k = k
        self.k_per_token = None
        self.P = None
        if k_per_token_host is not None:
            self.k_per_token = k_per_token_host.to(dev, torch.int32)
            self.P = int(k_per_token_host.sum())
        self.req_offsets = None if req_offsets_host is None else req_offsets_host.to(dev, torch.int32)
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):           # allocate workspaces and set kernel attributes
            for _ in range(warmup):
                layer.forward(self.x, self.token_ids, self.k_per_token, k, self.P, stream=side,
                              req_offsets=self.req_offsets)
        torch.cuda.current_stream(dev).wait_stream(side)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.result = layer.forward(self.x, self.token_ids, self.k_per_token, k, self.P,
                                        stream=torch.cuda.current_stream(dev), req_offsets=self.req_offsets)

    def replay(self) -> LayerOutput:
        self.graph.replay()
        return self.result


class GraphPipeline:
    """Host-buffer calls of one batch shape through captured graphs.

    Like ``HostPipeline`` (pinned inputs uploaded and outputs read back on a
    copy stream, overlapped with the compute of neighbouring calls), but each
    call's compute is one replay of a ``CapturedLayer``: two of them, one per
    double-buffer slot, so call i+1's upload lands in the other graph's static
    inputs while call i runs.  The batch shape and budgets are fixed at
    construction.  ``synchronize()`` waits for all submitted calls.
    """

    def __init__(self, layer: MoELayer, T: int, k: Optional[int] = None, k_per_token_host=None, stream=None):
        self.compute = torch.cuda.current_stream() if stream is None else stream
        self.copy = torch.cuda.Stream(device=layer.device)     # uploads
        self.down = torch.cuda.Stream(device=layer.device)     # readbacks
        self.slots = [CapturedLayer(layer, T, k, k_per_token_host) for _ in range(2)]
        self._done = [None, None]      # event: the slot's last replay has finished
        self._read = [None, None]      # event: the slot's output has been read back
        self._slot = 0

    def submit(self, x_host, ids_host, out_host):
        slot = self._slot
        self._slot ^= 1
        cap = self.slots[slot]
        with torch.cuda.stream(self.copy):
            if self._done[slot] is not None:
                self.copy.wait_event(self._done[slot])  # the call two back no longer reads its inputs
            cap.x.copy_(x_host, non_blocking=True)
            cap.token_ids.copy_(ids_host, non_blocking=True)
            uploaded = torch.cuda.Event()
            uploaded.record(self.copy)
        self.compute.wait_event(uploaded)
        if self._read[slot] is not None:
            self.compute.wait_event(self._read[slot])  # the call two back's output has been read back
        with torch.cuda.stream(self.compute):
            cap.replay()
            done = torch.cuda.Event()
            done.record(self.compute)
        self._done[slot] = done
        with torch.cuda.stream(self.down):
            self.down.wait_event(done)
            out_host.copy_(cap.result.out, non_blocking=True)
            read = torch.cuda.Event()
            read.record(self.down)
        self._read[slot] = read
        return out_host

    def synchronize(self):
        self.copy.synchronize()
        self.down.synchronize()
        self.compute.synchronize()
