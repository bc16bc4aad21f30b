"""Host-side MoE layer: owns the device buffers of one layer pass and calls
the C-ABI entry points in order on one stream.

    forward        route -> dispatch_layout -> permute -> grouped_ffn ->
                   combine
    forward_padded the same on the static-capacity [E, C, D] layout
    forward_train  the forward on the 64-row aligned layout, keeping what
    + backward     the backward pass needs; then combine, expert, permute
                   and router backward
    capture        one step as a CUDA graph
    forward_host_stream  batches from pinned host memory, copies overlapping
                   compute

("Expert Parallelism in LLMs", The Execution Pipeline, steps 1, 2, 4 and 6;
on one GPU the all-to-all steps 3 and 5 are the identity; Backward Pass
Symmetry).  Buffers are sized for the worst case (T*k rows) so no step ever
waits on the host for the dropless row count: expert offsets and kept
counts stay on the device.
"""
from __future__ import annotations

from fractions import Fraction
from typing import Optional

import torch

from . import _lib as L


def expert_capacity(capacity_factor, T, k, E) -> int:
    """C_expert = ceil(CF * k * T / E) from the library's exact integer
    evaluation (moe_expert_capacity), with CF passed as the exact ratio of
    its decimal form; 0 means dropless ("Expert Parallelism in LLMs", Static
    Capacity Factors and Token Dropping)."""
    if capacity_factor is None:
        return 0
    cf = Fraction(str(capacity_factor))
    c = L.moe_expert_capacity(cf.numerator, cf.denominator, T, k, E)
    if c < 0:
        raise ValueError(f"capacity factor {capacity_factor} for T={T} "
                         f"k={k} E={E} is out of range")
    return c


class MoELayer:
    """One MoE layer forward pass on one GPU.

    Weights are device tensors in the layer dtype (bf16 or fp32):
      w_r [E, D], w13 [E, 2F, D] (gate rows then up rows), w2 [E, D, F];
      w13 = w2 = None selects identity experts (Expert_i(h) = h).
    """

    def __init__(self, T, D, E, k, R, w_r, w13=None, w2=None, F=0,
                 score="softmax_topk", sel_bias=None, logit_offset=None,
                 capacity_factor=None, n_groups=1, topk_groups=1,
                 group_score_topk=0, device=None, keep_logits=False,
                 padded=False):
        L.load()
        self._init_args = dict(
            T=T, D=D, E=E, k=k, R=R, F=F, score=score,
            capacity_factor=capacity_factor, n_groups=n_groups,
            topk_groups=topk_groups, group_score_topk=group_score_topk,
            device=device, keep_logits=keep_logits, padded=padded)
        self.ffn_ctas = 0   # CTAs of the grouped FFN; 0 = one per SM
        self.device = torch.device(device or w_r.device)
        self.dtype = w_r.dtype
        self.dcode = L.dtype_code(self.dtype)
        self.T, self.D, self.E, self.k, self.R, self.F = T, D, E, k, R, F
        self.identity = w13 is None
        self.w_r, self.w13, self.w2 = w_r, w13, w2
        self.sel_bias, self.logit_offset = sel_bias, logit_offset
        self.capacity = expert_capacity(capacity_factor, T, k, E)
        self.cfg = L.route_cfg(T, D, E, k, self.dcode, score, n_groups,
                               topk_groups, group_score_topk)
        P = T * k
        dev = self.device
        i32 = dict(dtype=torch.int32, device=dev)
        self.topk_idx = torch.empty((T, k), **i32)
        self.topk_gate = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.logits = (torch.empty((T, E), dtype=torch.float32, device=dev)
                       if keep_logits else None)
        self.route_ws = self._bytes(L.moe_route_workspace_size(self.cfg))
        self.layout_ws = self._bytes(
            L.moe_dispatch_layout_workspace_size(T, k, E))
        self.expert_counts = torch.empty(E, **i32)
        self.expert_offsets = torch.empty(E + 1, **i32)
        self.dst_row = torch.empty(P, **i32)
        self.src_pair = torch.empty(P, **i32)
        self.n_kept = torch.empty(1, **i32)
        self.n_dropped = torch.empty(1, **i32)
        self.rank_send_counts = torch.empty(R, **i32)
        self.rank_send_displs = torch.empty(R, **i32)
        self.xp = torch.empty((max(P, 1), D), dtype=self.dtype, device=dev)
        if self.identity:
            self.yp = self.xp
            self.ffn_ws = None
        else:
            self.yp = torch.empty((max(P, 1), D), dtype=self.dtype,
                                  device=dev)
            self.ffn_ws = self._bytes(L.moe_grouped_ffn_workspace_size(
                E, D, F, P, self.dcode))
        self.y = torch.empty((T, D), dtype=self.dtype, device=dev)
        self.status = torch.zeros(1, **i32)
        # static-capacity [E, C, D] buffers ("Static Capacity Factors and
        # Token Dropping"): every expert owns C rows, padding rows are zero
        self.padded = bool(padded)
        if self.padded:
            if self.capacity <= 0:
                raise ValueError("the padded layout needs a capacity factor")
            rows = E * self.capacity
            self.dst_row_padded = torch.empty(P, **i32)
            self.offsets_padded = torch.empty(E + 1, **i32)
            self.xpad = torch.empty((max(rows, 1), D), dtype=self.dtype,
                                    device=dev)
            self.ypad = self.xpad if self.identity else torch.empty_like(
                self.xpad)
            if not self.identity:
                self.ffn_ws_padded = self._bytes(
                    L.moe_grouped_ffn_workspace_size(E, D, F, rows,
                                                     self.dcode))

    def _bytes(self, n):
        # 256-byte aligned scratch (torch's allocator aligns to >= 512 B)
        return torch.empty(max(int(n), 16), dtype=torch.uint8,
                           device=self.device)

    # ---------------------------------------------------------- steps
    def route(self, x, stream=None):
        L.moe_route(self.cfg, x, self.w_r, self.logit_offset, self.sel_bias,
                    self.topk_idx, self.topk_gate, self.logits,
                    self.route_ws, self.status, stream)

    def dispatch_layout(self, topk_idx=None, stream=None):
        idx = self.topk_idx if topk_idx is None else topk_idx
        L.moe_dispatch_layout(
            self.T, self.k, self.E, self.R, self.capacity, idx,
            self.expert_counts, self.expert_offsets, self.dst_row,
            self.src_pair, self.n_kept, self.n_dropped, self.rank_send_counts,
            self.rank_send_displs, self.layout_ws, self.status, stream)

    def permute(self, x, stream=None):
        L.moe_permute(self.T, self.k, self.D, self.dcode, x, self.dst_row,
                      self.xp, self.status, stream)

    def grouped_ffn(self, stream=None):
        if self.identity:
            return
        L.moe_grouped_ffn(self.E, self.D, self.F, self.T * self.k, self.dcode,
                          self.xp, self.expert_offsets, self.w13, self.w2,
                          self.yp, self.ffn_ws, self.status, stream,
                          max_ctas=self.ffn_ctas)

    def combine(self, topk_gate=None, y=None, stream=None):
        gate = self.topk_gate if topk_gate is None else topk_gate
        out = self.y if y is None else y
        L.moe_combine(self.T, self.k, self.D, self.dcode, self.yp,
                      self.dst_row, gate, out, self.status, stream)
        return out

    # ---------------------------------------------------------- padded
    def padded_layout(self, topk_idx=None, stream=None):
        """Rows of the [E, C, D] buffer for the kept pairs, then zeros in
        the padding rows (moe_padded_layout, moe_pad_fill)."""
        idx = self.topk_idx if topk_idx is None else topk_idx
        L.moe_padded_layout(self.T, self.k, self.E, self.capacity, idx,
                            self.dst_row, self.expert_offsets,
                            self.dst_row_padded, self.offsets_padded,
                            self.status, stream)
        L.moe_pad_fill(self.E, self.capacity, self.D, self.dcode,
                       self.expert_counts, self.xpad, stream)

    def forward_padded(self, x, topk_idx=None, topk_gate=None, y=None,
                       stream=None):
        """The layer on the static-capacity layout: every expert computes
        all of its C rows (padding rows are zero in and zero out)."""
        if topk_idx is None:
            self.route(x, stream)
        self.dispatch_layout(topk_idx, stream)
        self.padded_layout(topk_idx, stream)
        L.moe_permute(self.T, self.k, self.D, self.dcode, x,
                      self.dst_row_padded, self.xpad, self.status, stream)
        if not self.identity:
            L.moe_grouped_ffn(self.E, self.D, self.F,
                              self.E * self.capacity, self.dcode, self.xpad,
                              self.offsets_padded, self.w13, self.w2,
                              self.ypad, self.ffn_ws_padded, self.status,
                              stream)
        gate = self.topk_gate if topk_gate is None else topk_gate
        out = self.y if y is None else y
        L.moe_combine(self.T, self.k, self.D, self.dcode, self.ypad,
                      self.dst_row_padded, gate, out, self.status, stream)
        return out

    # ---------------------------------------------------------- training
    ALIGN = 64

    def _train_buffers(self):
        if getattr(self, "_train", None) is not None:
            return self._train
        T, D, E, k, F = self.T, self.D, self.E, self.k, self.F
        P = T * k
        rows = P + (self.ALIGN - 1) * E
        dev = self.device
        i32 = dict(dtype=torch.int32, device=dev)
        b = dict(rows=rows,
                 dst_a=torch.empty(P, **i32),
                 off_a=torch.empty(E + 1, **i32),
                 xa=torch.empty((rows, D), dtype=self.dtype, device=dev),
                 dga=torch.empty((rows, D), dtype=self.dtype, device=dev),
                 dxa=torch.empty((rows, D), dtype=self.dtype, device=dev),
                 dgate=torch.empty((T, k), dtype=torch.float32, device=dev),
                 dlogits=torch.empty((T, E), dtype=torch.float32, device=dev),
                 dx=torch.empty((T, D), dtype=self.dtype, device=dev),
                 dw_r=torch.empty((E, D), dtype=torch.float32, device=dev),
                 route_bwd_ws=self._bytes(
                     L.moe_route_backward_workspace_size(self.cfg)))
        if self.identity:
            b["ya"] = b["xa"]
        else:
            b["ya"] = torch.empty((rows, D), dtype=self.dtype, device=dev)
            b["ffn_ws"] = self._bytes(L.moe_grouped_ffn_workspace_size(
                E, D, F, rows, self.dcode))
            b["bwd_ws"] = self._bytes(
                L.moe_grouped_ffn_backward_workspace_size(E, D, F, rows,
                                                          self.dcode))
            b["dw13"] = torch.empty((E, 2 * F, D), dtype=torch.float32,
                                    device=dev)
            b["dw2"] = torch.empty((E, D, F), dtype=torch.float32,
                                   device=dev)
        if self.logits is None:
            self.logits = torch.empty((T, E), dtype=torch.float32,
                                      device=dev)
        self._train = b
        return b

    def forward_train(self, x, stream=None):
        """The forward pass on the 64-row aligned training layout, keeping
        what the backward pass needs (x, logits, routing, Xa, Ya)."""
        b = self._train_buffers()
        E, D = self.E, self.D
        self.route(x, stream)
        self.dispatch_layout(None, stream)
        L.moe_aligned_layout(self.T, self.k, E, self.ALIGN, self.topk_idx,
                             self.dst_row, self.expert_offsets, b["dst_a"],
                             b["off_a"], self.status, stream)
        L.moe_aligned_fill(E, D, self.dcode, self.expert_offsets, b["off_a"],
                           b["xa"], stream)
        L.moe_permute(self.T, self.k, D, self.dcode, x, b["dst_a"], b["xa"],
                      self.status, stream)
        if not self.identity:
            L.moe_grouped_ffn(E, D, self.F, b["rows"], self.dcode, b["xa"],
                              b["off_a"], self.w13, self.w2, b["ya"],
                              b["ffn_ws"], self.status, stream)
        L.moe_combine(self.T, self.k, D, self.dcode, b["ya"], b["dst_a"],
                      self.topk_gate, self.y, self.status, stream)
        self._x = x
        return self.y

    def backward(self, dy, stream=None):
        """Gradients of sum(dy * y) for the last forward_train: returns dx
        [T, D] (dtype), dw_r [E, D], dw13 [E, 2F, D], dw2 [E, D, F] (fp32;
        None for identity experts)."""
        b = self._train
        E, D = self.E, self.D
        L.moe_combine_backward(self.T, self.k, D, self.dcode, dy, b["ya"],
                               b["dst_a"], self.topk_gate, b["dga"],
                               b["dgate"], self.status, stream)
        L.moe_aligned_fill(E, D, self.dcode, self.expert_offsets, b["off_a"],
                           b["dga"], stream)
        dxa = b["dga"]
        if not self.identity:
            L.moe_grouped_ffn_backward(E, D, self.F, b["rows"], self.dcode,
                                       b["xa"], b["dga"], b["off_a"],
                                       self.w13, self.w2, b["dxa"],
                                       b["dw13"], b["dw2"], b["bwd_ws"],
                                       self.status, stream)
            dxa = b["dxa"]
        L.moe_permute_backward(self.T, self.k, D, self.dcode, dxa,
                               b["dst_a"], b["dx"], self.status, stream)
        L.moe_route_backward(self.cfg, self._x, self.w_r, self.logits,
                             self.topk_idx, b["dgate"], b["dlogits"],
                             b["dw_r"], b["dx"], b["route_bwd_ws"],
                             self.status, stream)
        return (b["dx"], b["dw_r"], b.get("dw13"), b.get("dw2"))

    # ---------------------------------------------------------- layer
    def forward(self, x, topk_idx=None, topk_gate=None, y=None, stream=None):
        """y = MoE(x) for x [T, D] on the device.  With topk_idx/topk_gate
        given, routing is taken from them (pre-drawn routing) and moe_route
        is skipped.  A layer built with padded=True runs the static-capacity
        layout."""
        if self.padded:
            return self.forward_padded(x, topk_idx, topk_gate, y, stream)
        if topk_idx is None:
            self.route(x, stream)
        self.dispatch_layout(topk_idx, stream)
        self.permute(x, stream)
        self.grouped_ffn(stream)
        return self.combine(topk_gate, y, stream)

    def forward_host(self, x_host, y_host, x_dev, stream=None):
        """End-to-end pass from pinned host memory: copy x in, run the
        layer, copy y out, all on one stream."""
        s = stream or torch.cuda.current_stream()
        with torch.cuda.stream(s):
            x_dev.copy_(x_host, non_blocking=True)
            self.forward(x_dev, stream=s)
            y_host.copy_(self.y, non_blocking=True)
        return y_host

    def forward_host_stream(self, xs_host, ys_host, stream=None,
                            topk_idx=None, topk_gate=None):
        """A stream of batches from pinned host memory through the layer and
        back: batch i+1's host-to-device copy and batch i-1's device-to-host
        copy run on their own streams while batch i computes (two device
        input and output buffers, alternating).  Returns ys_host."""
        s = stream or torch.cuda.current_stream()
        if getattr(self, "_stream_bufs", None) is None:
            self._stream_bufs = dict(
                x=[torch.empty((self.T, self.D), dtype=self.dtype,
                               device=self.device) for _ in range(2)],
                y=[torch.empty((self.T, self.D), dtype=self.dtype,
                               device=self.device) for _ in range(2)],
                h2d=torch.cuda.Stream(device=self.device),
                d2h=torch.cuda.Stream(device=self.device))
        b = self._stream_bufs
        h2d, d2h = b["h2d"], b["d2h"]
        n = len(xs_host)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        x_ready = [ev() for _ in range(n)]
        x_free = [ev() for _ in range(n)]
        y_ready = [ev() for _ in range(n)]
        y_free = [ev() for _ in range(n)]
        h2d.wait_stream(s)
        d2h.wait_stream(s)

        def load(i):
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(x_free[i - 2])
                b["x"][i % 2].copy_(xs_host[i], non_blocking=True)
                x_ready[i].record(h2d)

        load(0)
        for i in range(n):
            if i + 1 < n:
                load(i + 1)
            s.wait_event(x_ready[i])
            if i >= 2:
                s.wait_event(y_free[i - 2])
            self.forward(b["x"][i % 2], topk_idx=topk_idx,
                         topk_gate=topk_gate, y=b["y"][i % 2], stream=s)
            x_free[i].record(s)
            y_ready[i].record(s)
            with torch.cuda.stream(d2h):
                d2h.wait_event(y_ready[i])
                ys_host[i].copy_(b["y"][i % 2], non_blocking=True)
                y_free[i].record(d2h)
        s.wait_stream(d2h)
        return ys_host

    def twin(self):
        """A second layer over the same weights with its own device
        buffers (routing, layout, expert rows, workspaces, output)."""
        a = self._init_args
        return MoELayer(a["T"], a["D"], a["E"], a["k"], a["R"], self.w_r,
                        self.w13, self.w2, F=a["F"], score=a["score"],
                        sel_bias=self.sel_bias,
                        logit_offset=self.logit_offset,
                        capacity_factor=a["capacity_factor"],
                        n_groups=a["n_groups"], topk_groups=a["topk_groups"],
                        group_score_topk=a["group_score_topk"],
                        device=self.device, keep_logits=a["keep_logits"])

    def forward_overlapped(self, xs, ys, stream=None, ffn_ctas=None):
        """Micro-batches xs[i] -> ys[i] (each [T, D] on the device, each its
        own routing decision and capacity), with the routing, layout and
        permute of batch i+1 on a second stream while the grouped FFN and
        combine of batch i run ("Expert Parallelism in LLMs", Overlapping
        All-to-All with Computation: the dispatch of one micro-batch runs
        while another computes).  The grouped FFN runs on ffn_ctas CTAs
        (default: all SMs but 8) so that SMs stay free for the other
        stream.  Two buffer sets alternate (this layer and its twin).
        Returns ys; each ys[i] equals forward(xs[i]) bit for bit."""
        if self.padded:
            raise ValueError("overlap runs the compact layout")
        s = stream or torch.cuda.current_stream()
        if getattr(self, "_overlap", None) is None:
            self._overlap = dict(twin=self.twin(),
                                 side=torch.cuda.Stream(device=self.device))
        o = self._overlap
        layers = [self, o["twin"]]
        side = o["side"]
        if ffn_ctas is None:
            n_sms = torch.cuda.get_device_properties(
                self.device).multi_processor_count
            ffn_ctas = max(2, n_sms - 8)
        n = len(xs)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        front_done = [ev() for _ in range(n)]
        back_done = [ev() for _ in range(n)]
        side.wait_stream(s)

        def front(i):
            lay = layers[i % 2]
            with torch.cuda.stream(side):
                if i >= 2:
                    side.wait_event(back_done[i - 2])
                lay.route(xs[i], side)
                lay.dispatch_layout(None, side)
                lay.permute(xs[i], side)
                front_done[i].record(side)

        saved = [lay.ffn_ctas for lay in layers]
        for lay in layers:
            lay.ffn_ctas = ffn_ctas
        try:
            front(0)
            for i in range(n):
                if i + 1 < n:
                    front(i + 1)
                lay = layers[i % 2]
                s.wait_event(front_done[i])
                lay.grouped_ffn(s)
                lay.combine(None, ys[i], s)
                back_done[i].record(s)
        finally:
            for lay, c in zip(layers, saved):
                lay.ffn_ctas = c
        s.wait_stream(side)
        return ys

    def capture(self, x, topk_idx=None, topk_gate=None, train=False):
        """Captures one forward pass on the device input buffer `x` (its
        storage is reused at every replay) into a CUDA graph and returns a
        function that replays it.  Every call of the pass is asynchronous,
        allocates nothing and never synchronises, so the whole layer is one
        graph launch.  With train=True the training forward and backward
        are captured instead (the replay takes dy, a device buffer whose
        storage is reused).  The first, eager pass sets the kernels'
        shared-memory limits before capture."""
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream())
        dy = torch.zeros_like(self.y) if train else None
        with torch.cuda.stream(s):
            if train:
                self.forward_train(x, s)
                self.backward(dy, s)
            else:
                self.forward(x, topk_idx, topk_gate, stream=s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        if train:
            with torch.cuda.graph(graph, stream=s):
                self.forward_train(x, s)
                self.backward(dy, s)

            def replay(dy_in):
                dy.copy_(dy_in)
                graph.replay()
                return self._train["dx"]
            return replay
        with torch.cuda.graph(graph, stream=s):
            self.forward(x, topk_idx, topk_gate, stream=s)

        def replay():
            graph.replay()
            return self.y
        return replay

    def device_status(self) -> int:
        st = int(self.status.item())
        o = getattr(self, "_overlap", None)
        if st == 0 and o is not None:
            st = int(o["twin"].status.item())
        return st
