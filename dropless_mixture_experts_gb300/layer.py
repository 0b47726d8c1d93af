"""The layer's forward pass and train step, composed from the C-ABI calls.

PyTorch only provides device memory and the current stream here; every step
(routing, permutation, grouped experts, combine, backward) is a call into the
CUDA library.  ``MoELayer`` owns the workspace and the intermediate buffers of
one problem size and reuses them across calls.
"""

from __future__ import annotations

import torch

from . import abi

_DT = {"bf16": (torch.bfloat16, abi.MOE_BF16), "f32": (torch.float32, abi.MOE_F32)}


def _ptr(t):
    return None if t is None else t.data_ptr()


class MoELayer:
    """Buffers and calls for one (tokens, d_model, d_hidden, experts, top_k,
    shared_hidden, dtype) problem on one CUDA device.  capacity > 0 switches
    on capacity routing (each expert keeps its first ``capacity`` pairs).

    shared_sms > 0 (with a shared expert): the shared expert's forward and
    backward run on a second stream beside the routed experts, its
    persistent kernels capped at ``shared_sms`` SMs and the routed ones at
    the rest (``moe_set_sm_limit``); the results are the same as with
    shared_sms = 0, where every call runs on the current stream in turn."""

    def __init__(self, tokens, d_model, d_hidden, experts, top_k, shared_hidden=0, dtype="bf16",
                 device="cuda", train=True, capacity=0, shared_sms=0):
        self.T, self.d, self.h, self.E, self.k, self.hs = (
            int(tokens), int(d_model), int(d_hidden), int(experts), int(top_k), int(shared_hidden))
        self.tdtype, cdt = _DT[dtype]
        self.dtype = dtype
        self.device = torch.device(device)
        self.capacity = int(capacity)
        self.shared_sms = int(shared_sms) if shared_hidden else 0
        self.dims = abi.make_dims(self.T, self.d, self.h, self.E, self.k, self.hs, cdt,
                                  self.capacity)
        self.mode = abi.MOE_SAVE_FOR_BWD if train else abi.MOE_FWD_ONLY
        self.ws_bytes = abi.moe_workspace_bytes(self.dims, self.mode)
        self.PP = abi.moe_padded_rows(self.dims)
        dev, f32, i32, td = self.device, torch.float32, torch.int32, self.tdtype
        T, d, h, E, k, hs, P = self.T, self.d, self.h, self.E, self.k, self.hs, self.T * self.k
        self.ws = torch.empty(self.ws_bytes + 256, dtype=torch.uint8, device=dev)
        off = (-self.ws.data_ptr()) % 256
        self.ws_ptr = self.ws.data_ptr() + off
        self.logits = torch.empty(T, E, dtype=f32, device=dev)
        self.idx = torch.empty(T, k, dtype=i32, device=dev)
        self.gates = torch.empty(T, k, dtype=f32, device=dev)
        self.counts = torch.empty(E, dtype=i32, device=dev)
        self.offsets = torch.empty(E + 1, dtype=i32, device=dev)
        self.perm = torch.empty(P, dtype=i32, device=dev)
        self.inv_perm = torch.empty(P, dtype=i32, device=dev)
        self.h_buf = torch.empty(self.PP, h, dtype=td, device=dev)
        self.a_gate = torch.empty(self.PP, h, dtype=td, device=dev) if train else None
        self.a_up = torch.empty(self.PP, h, dtype=td, device=dev) if train else None
        self.y = torch.empty(T, d, dtype=td, device=dev)
        self.hs_buf = torch.empty(T, hs, dtype=td, device=dev) if hs else None
        self.as_gate = torch.empty(T, hs, dtype=td, device=dev) if (hs and train) else None
        self.as_up = torch.empty(T, hs, dtype=td, device=dev) if (hs and train) else None
        self.loss = torch.zeros(1, dtype=f32, device=dev)
        if train:
            self.dx = torch.empty(T, d, dtype=td, device=dev)
            self.grads = {
                "dw_router": torch.empty(d, E, dtype=f32, device=dev),
                "dw_gate": torch.empty(E, d, h, dtype=f32, device=dev),
                "dw_up": torch.empty(E, d, h, dtype=f32, device=dev),
                "dw_down": torch.empty(E, h, d, dtype=f32, device=dev),
                "dws_gate": torch.empty(d, hs, dtype=f32, device=dev) if hs else None,
                "dws_up": torch.empty(d, hs, dtype=f32, device=dev) if hs else None,
                "dws_down": torch.empty(hs, d, dtype=f32, device=dev) if hs else None,
            }

    # -- the five calls ---------------------------------------------------
    def _stream(self):
        return torch.cuda.current_stream(self.device).cuda_stream

    def route(self, x, w_router, logits_in=None, router_bias=None):
        abi.moe_route(self.dims, _ptr(x), _ptr(w_router), _ptr(logits_in), _ptr(self.logits),
                      _ptr(self.idx), _ptr(self.gates), self.ws_ptr, self.ws_bytes, self._stream(),
                      router_bias=_ptr(router_bias))

    def permute(self):
        abi.moe_permute(self.dims, _ptr(self.idx), _ptr(self.counts), _ptr(self.offsets),
                        _ptr(self.perm), _ptr(self.inv_perm), self.ws_ptr, self.ws_bytes,
                        self._stream())

    def grouped_ffn_fwd(self, x, p, mode):
        abi.moe_grouped_ffn_fwd(self.dims, mode, _ptr(x), _ptr(self.gates), _ptr(p["w_gate"]),
                                _ptr(p["w_up"]), _ptr(p["w_down"]), _ptr(self.h_buf),
                                _ptr(self.a_gate), _ptr(self.a_up), self.ws_ptr, self.ws_bytes,
                                self._stream())

    def combine(self, x, p, mode, upstream=None):
        abi.moe_combine(self.dims, mode, _ptr(x), _ptr(p.get("ws_gate")), _ptr(p.get("ws_up")),
                        _ptr(p.get("ws_down")), _ptr(self.y),
                        _ptr(self.hs_buf), _ptr(self.as_gate if mode else None),
                        _ptr(self.as_up if mode else None), _ptr(upstream),
                        _ptr(self.loss if upstream is not None else None),
                        self.ws_ptr, self.ws_bytes, self._stream())

    def backward(self, x, p, dy):
        g = self.grads
        abi.moe_backward(self.dims, _ptr(dy), _ptr(x), _ptr(p["w_router"]), _ptr(p["w_gate"]),
                         _ptr(p["w_up"]), _ptr(p["w_down"]), _ptr(p.get("ws_gate")),
                         _ptr(p.get("ws_up")), _ptr(p.get("ws_down")), _ptr(self.idx),
                         _ptr(self.gates), _ptr(self.a_gate), _ptr(self.a_up),
                         _ptr(self.h_buf), _ptr(self.as_gate), _ptr(self.as_up),
                         _ptr(self.hs_buf), _ptr(self.dx),
                         _ptr(g["dw_router"]), _ptr(g["dw_gate"]), _ptr(g["dw_up"]),
                         _ptr(g["dw_down"]), _ptr(g["dws_gate"]), _ptr(g["dws_up"]),
                         _ptr(g["dws_down"]), self.ws_ptr, self.ws_bytes, self._stream())

    # -- the shared expert on its own stream ---------------------------------
    def shared_ffn_fwd(self, x, p, mode):
        abi.moe_shared_ffn_fwd(self.dims, mode, _ptr(x), _ptr(p.get("ws_gate")),
                               _ptr(p.get("ws_up")), _ptr(p.get("ws_down")), _ptr(self.hs_buf),
                               _ptr(self.as_gate if mode else None),
                               _ptr(self.as_up if mode else None), self.ws_ptr, self.ws_bytes,
                               self._stream())

    def shared_backward(self, x, p, dy):
        g = self.grads
        abi.moe_shared_backward(self.dims, _ptr(dy), _ptr(x), _ptr(p.get("ws_gate")),
                                _ptr(p.get("ws_up")), _ptr(p.get("ws_down")), _ptr(self.as_gate),
                                _ptr(self.as_up), _ptr(self.hs_buf), _ptr(g["dws_gate"]),
                                _ptr(g["dws_up"]), _ptr(g["dws_down"]), self.ws_ptr,
                                self.ws_bytes, self._stream())

    def backward_routed(self, x, p, dy, shared_done=None):
        g = self.grads
        abi.moe_backward_routed(self.dims, _ptr(dy), _ptr(x), _ptr(p["w_router"]),
                                _ptr(p["w_gate"]), _ptr(p["w_up"]), _ptr(p["w_down"]),
                                _ptr(self.idx), _ptr(self.gates), _ptr(self.a_gate),
                                _ptr(self.a_up), _ptr(self.h_buf), _ptr(self.dx),
                                _ptr(g["dw_router"]), _ptr(g["dw_gate"]), _ptr(g["dw_up"]),
                                _ptr(g["dw_down"]),
                                None if shared_done is None else shared_done.cuda_event,
                                self.ws_ptr, self.ws_bytes, self._stream())

    def _side(self):
        if getattr(self, "sh_stream", None) is None:
            self.sh_stream = torch.cuda.Stream(self.device)
            self.sh_fwd_done = torch.cuda.Event()
            self.sh_bwd_done = torch.cuda.Event()
        return self.sh_stream

    def _overlapped(self, x, p, mode, upstream, dy, logits_in, dy_ready=None):
        """The pass with the shared expert (forward, and backward when dy is
        given) on the side stream beside the routed experts on the current
        stream; the combine waits for the shared forward, the input
        gradient for the shared backward, and the current stream joins the
        side stream at the end."""
        main = torch.cuda.current_stream(self.device)
        side = self._side()
        n = torch.cuda.get_device_properties(self.device).multi_processor_count
        side.wait_stream(main)  # x and the weights are ready
        with torch.cuda.stream(side):
            abi.moe_set_sm_limit(self.shared_sms)
            self.shared_ffn_fwd(x, p, mode)
            self.sh_fwd_done.record(side)
            if dy is not None:
                if dy_ready is not None:
                    side.wait_event(dy_ready)
                self.shared_backward(x, p, dy)
                self.sh_bwd_done.record(side)
        abi.moe_set_sm_limit(max(1, n - self.shared_sms))
        try:
            self.route(x, p["w_router"], logits_in, p.get("router_bias"))
            self.permute()
            self.grouped_ffn_fwd(x, p, mode)
            main.wait_event(self.sh_fwd_done)
            if dy_ready is not None:
                main.wait_event(dy_ready)
            self.combine(x, p, mode | abi.MOE_SHARED_READY, upstream=upstream)
            if dy is not None:
                self.backward_routed(x, p, dy, shared_done=self.sh_bwd_done)
        finally:
            abi.moe_set_sm_limit(0)
        main.wait_stream(side)

    # -- composed passes ---------------------------------------------------
    def forward(self, x, p, logits_in=None):
        """y = layer(x); returns the output buffer (valid until the next call)."""
        if self.shared_sms > 0:
            self._overlapped(x, p, abi.MOE_FWD_ONLY, None, None, logits_in)
            return self.y
        self.route(x, p["w_router"], logits_in, p.get("router_bias"))
        self.permute()
        self.grouped_ffn_fwd(x, p, abi.MOE_FWD_ONLY)
        self.combine(x, p, abi.MOE_FWD_ONLY)
        return self.y

    def train_step(self, x, p, dy, logits_in=None):
        """value_and_grad of L = sum(y * dy): returns (loss [1] device tensor,
        dx, grads dict); all are the layer's buffers."""
        if self.mode != abi.MOE_SAVE_FOR_BWD:
            raise RuntimeError("layer was built with train=False")
        if self.shared_sms > 0:
            self._overlapped(x, p, abi.MOE_SAVE_FOR_BWD, dy, dy, logits_in)
            return self.loss, self.dx, self.grads
        self.route(x, p["w_router"], logits_in, p.get("router_bias"))
        self.permute()
        self.grouped_ffn_fwd(x, p, abi.MOE_SAVE_FOR_BWD)
        self.combine(x, p, abi.MOE_SAVE_FOR_BWD, upstream=dy)
        self.backward(x, p, dy)
        return self.loss, self.dx, self.grads

    def train_step_from_host(self, x_host, p, dy_host, loss_host=None, dx_host=None):
        """The train step on a batch in pinned host memory: x is copied to the
        device on the current stream, the upstream gradient on a side stream
        while the forward pass runs (only the combine needs it), and the value
        and the input gradient are copied back into ``loss_host`` [1] and
        ``dx_host`` [T, d] (pinned, each optional).  Returns the same device
        buffers as ``train_step``; the copies land in the layer's own input
        buffers.  The weight gradients stay on the device, where an optimizer
        step would read them."""
        if self.mode != abi.MOE_SAVE_FOR_BWD:
            raise RuntimeError("layer was built with train=False")
        if getattr(self, "x_dev", None) is None:
            self.x_dev = torch.empty(self.T, self.d, dtype=self.tdtype, device=self.device)
            self.dy_dev = torch.empty(self.T, self.d, dtype=self.tdtype, device=self.device)
            self.side = torch.cuda.Stream(self.device)
            self.dy_ready = torch.cuda.Event()
        main = torch.cuda.current_stream(self.device)
        self.x_dev.copy_(x_host, non_blocking=True)
        self.side.wait_stream(main)  # the previous step has finished with dy_dev
        with torch.cuda.stream(self.side):
            self.dy_dev.copy_(dy_host, non_blocking=True)
            self.dy_ready.record(self.side)
        x = self.x_dev
        if self.shared_sms > 0:
            self._overlapped(x, p, abi.MOE_SAVE_FOR_BWD, self.dy_dev, self.dy_dev, None,
                             dy_ready=self.dy_ready)
        else:
            self.route(x, p["w_router"], None, p.get("router_bias"))
            self.permute()
            self.grouped_ffn_fwd(x, p, abi.MOE_SAVE_FOR_BWD)
            main.wait_event(self.dy_ready)
            self.combine(x, p, abi.MOE_SAVE_FOR_BWD, upstream=self.dy_dev)
            self.backward(x, p, self.dy_dev)
        if loss_host is not None:
            loss_host.copy_(self.loss, non_blocking=True)
        if dx_host is not None:
            dx_host.copy_(self.dx, non_blocking=True)
        return self.loss, self.dx, self.grads

    def train_steps_from_host(self, x_hosts, p, dy_hosts, loss_hosts=None, dx_hosts=None):
        """Train steps on a sequence of batches in pinned host memory,
        pipelined: while step i runs, the inputs of step i + 1 (x and the
        upstream gradient) are copied in on one copy stream and the results
        of step i - 1 (the value and dx, into ``loss_hosts[i - 1]`` [1] and
        ``dx_hosts[i - 1]`` [T, d], each list optional) are copied out on
        another.  Two device slots of the inputs, the value and dx alternate
        between steps; a slot is refilled only after the step that read it
        has finished.  Every step's results equal ``train_step``'s on the same
        batch.  Returns after enqueuing (the current stream joins both copy
        streams at the end): synchronize before reading the host buffers.
        The weight gradients are those of the last step."""
        if self.mode != abi.MOE_SAVE_FOR_BWD:
            raise RuntimeError("layer was built with train=False")
        n = len(x_hosts)
        if n == 0 or len(dy_hosts) != n:
            raise ValueError("one upstream gradient per batch")
        if getattr(self, "slot_x", None) is None:
            mk = lambda: torch.empty(self.T, self.d, dtype=self.tdtype, device=self.device)
            self.slot_x = [mk(), mk()]
            self.slot_dy = [mk(), mk()]
            self.slot_dx = [self.dx, mk()]
            self.slot_loss = [self.loss, torch.zeros_like(self.loss)]
            self.h2d = torch.cuda.Stream(self.device)
            self.d2h = torch.cuda.Stream(self.device)
            self.slot_in = [torch.cuda.Event(), torch.cuda.Event()]
            self.slot_done = [torch.cuda.Event(), torch.cuda.Event()]
            self.slot_out = [torch.cuda.Event(), torch.cuda.Event()]
        main = torch.cuda.current_stream(self.device)
        self.h2d.wait_stream(main)  # earlier work on the slots has finished
        self.d2h.wait_stream(main)

        def load(i):
            s = i % 2
            with torch.cuda.stream(self.h2d):
                if i >= 2:
                    self.h2d.wait_event(self.slot_done[s])  # step i - 2 has read the slot
                self.slot_x[s].copy_(x_hosts[i], non_blocking=True)
                self.slot_dy[s].copy_(dy_hosts[i], non_blocking=True)
                self.slot_in[s].record(self.h2d)

        load(0)
        try:
            for i in range(n):
                s = i % 2
                if i + 1 < n:
                    load(i + 1)
                main.wait_event(self.slot_in[s])
                if i >= 2:
                    # the copies out of step i - 2 have read this slot's value and dx
                    main.wait_event(self.slot_out[s])
                self.dx, self.loss = self.slot_dx[s], self.slot_loss[s]
                self.train_step(self.slot_x[s], p, self.slot_dy[s])
                self.slot_done[s].record(main)
                with torch.cuda.stream(self.d2h):
                    self.d2h.wait_event(self.slot_done[s])
                    if loss_hosts is not None:
                        loss_hosts[i].copy_(self.loss, non_blocking=True)
                    if dx_hosts is not None:
                        dx_hosts[i].copy_(self.dx, non_blocking=True)
                    self.slot_out[s].record(self.d2h)
        finally:
            main.wait_stream(self.h2d)
            main.wait_stream(self.d2h)
        return self.loss, self.dx, self.grads

    def capture(self, fn):
        """Records ``fn()`` -- a composed pass (``train_step``, ``forward``,
        ``train_step_from_host``) on fixed buffers -- into a CUDA graph and
        returns its replay.  The library's calls only launch stream-ordered
        work and allocate nothing, so they record as they are; ``fn`` runs
        once on a side stream first so that one-time setup (kernel
        attributes, the layer's input buffers) happens outside the capture.
        A replay repeats the recorded pass on whatever the buffers hold."""
        main = torch.cuda.current_stream(self.device)
        warm = torch.cuda.Stream(self.device)
        warm.wait_stream(main)
        with torch.cuda.stream(warm):
            fn()
        main.wait_stream(warm)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            fn()
        self._graphs = getattr(self, "_graphs", []) + [graph]  # kept alive with the layer
        return graph.replay

    def device_status(self):
        """(status, detail) recorded by the kernels; synchronises the stream."""
        return abi.moe_read_device_status(self.ws_ptr, self.ws_bytes, self._stream())
