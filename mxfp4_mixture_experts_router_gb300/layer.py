"""A MoE layer on one GPU, assembled from the C ABI calls.

``MoeLayer`` owns the device buffers of one layer (router matrix, expert slab
pool and slot map, shared-expert pool, workspace, per-block outputs) and runs a
block of rows through ``moe_route`` -> ``moe_shared_experts_after_route`` ->
``moe_expert_block`` (routed experts) -> ``moe_combine`` on one stream.  PyTorch only allocates memory and provides the stream; every
step runs in the library's kernels.
"""

from __future__ import annotations

import torch

from . import binding as B


def _device_readable(t, name):
    """The kernels take device memory or pinned host memory (mapped into the device's
    address space); pageable host memory is refused."""
    if not t.is_cuda and not t.is_pinned():
        raise ValueError(f"{name} must be a device tensor or a pinned host tensor")


class MoeLayer:
    def __init__(self, d_model: int, d_ff: int, n_experts: int, top_k: int, n_rows_max: int = 16,
                 n_shared: int = 0, device: str | int = "cuda"):
        self.desc = B.desc(d_model, d_ff, n_experts, top_k)
        self.d, self.f, self.E, self.k = d_model, d_ff, n_experts, top_k
        self.n_rows_max = n_rows_max
        self.n_shared = n_shared
        self.device = torch.device(device)
        self.slab_bytes = B.moe_slab_bytes(self.desc, B.MOE_FMT_MXFP4)
        self.q8_bytes = B.moe_slab_bytes(self.desc, B.MOE_FMT_Q8_0)
        self.slot_bytes = (self.slab_bytes + 255) // 256 * 256
        self.q8_slot_bytes = (self.q8_bytes + 255) // 256 * 256
        ws_bytes = B.moe_workspace_size(self.desc, n_rows_max, n_shared)
        self.ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=self.device)
        self.offsets = B.moe_workspace_offsets(self.desc, n_rows_max, n_shared)
        self.router = None
        self.pool = None
        self.n_slots = 0
        self.expert_slot = torch.zeros(n_experts, dtype=torch.int32, device=self.device)
        self.shared_pool = None
        self.slot_ready = None
        N = n_rows_max
        self.topk_idx = torch.zeros((N, top_k), dtype=torch.int32, device=self.device)
        self.topk_w = torch.zeros((N, top_k), dtype=torch.float32, device=self.device)
        self.logits = torch.zeros((N, n_experts), dtype=torch.float32, device=self.device)
        self.y_part = torch.zeros((N, top_k, d_model), dtype=torch.float32, device=self.device)
        self.out = torch.zeros((N, d_model), dtype=torch.uint16, device=self.device)

    # --- weights -------------------------------------------------------------
    def set_router(self, w_bits: torch.Tensor):
        """bf16 router matrix [E][d] as uint16 bits (host or device)."""
        self.router = w_bits.to(self.device, torch.uint16).contiguous()

    def alloc_pool(self, n_slots: int):
        self.n_slots = n_slots
        self.pool = torch.empty(n_slots * self.slot_bytes, dtype=torch.uint8, device=self.device)

    def attach_pool(self, pool: torch.Tensor, slot_bytes: int, n_slots: int, slot_ready=None):
        """Use an external routed-expert slot pool (a device expert cache) and its
        per-slot ready flags."""
        self.pool = pool
        self.slot_bytes = slot_bytes
        self.n_slots = n_slots
        self.slot_ready = slot_ready

    def put_slab(self, slot: int, slab):
        """Copy one MXFP4 slab (numpy uint8 or tensor) into a pool slot."""
        t = torch.as_tensor(slab, dtype=torch.uint8)
        self.pool[slot * self.slot_bytes: slot * self.slot_bytes + self.slab_bytes].copy_(t, non_blocking=False)

    def set_expert_slots(self, slots):
        self.expert_slot.copy_(torch.as_tensor(slots, dtype=torch.int32))

    def set_shared(self, slabs):
        assert len(slabs) == self.n_shared
        self.shared_pool = torch.empty(max(1, self.n_shared) * self.q8_slot_bytes, dtype=torch.uint8,
                                       device=self.device)
        for i, s in enumerate(slabs):
            self.shared_pool[i * self.q8_slot_bytes: i * self.q8_slot_bytes + self.q8_bytes].copy_(
                torch.as_tensor(s, dtype=torch.uint8))

    def routed_pool(self) -> B.MoePool:
        return B.pool(self.pool, self.slot_bytes, self.n_slots, B.MOE_FMT_MXFP4)

    def shared_pool_desc(self):
        if self.n_shared == 0:
            return None
        return B.pool(self.shared_pool, self.q8_slot_bytes, self.n_shared, B.MOE_FMT_Q8_0)

    # --- views of the workspace ----------------------------------------------
    def ws_view(self, offset: int, count: int, dtype) -> torch.Tensor:
        nbytes = count * torch.empty((), dtype=dtype).element_size()
        return self.ws[offset: offset + nbytes].view(dtype)

    def shared_y(self, n_rows: int) -> torch.Tensor:
        """Shared-expert outputs of the last block, [n_shared][n_rows][d] (the kernels lay
        them out for the block's own row count)."""
        return self.ws_view(self.offsets.shared_y, self.n_shared * n_rows * self.d,
                            torch.float32).view(self.n_shared, n_rows, self.d)

    # --- the layer -------------------------------------------------------------
    def route(self, n_rows: int, x, logits_in=None, stream=None):
        if logits_in is not None and (logits_in.dtype != torch.float32 or not logits_in.is_contiguous()
                                      or logits_in.numel() < n_rows * self.E):
            raise ValueError("logits_in must be a contiguous float32 tensor of n_rows x n_experts")
        if x.element_size() != 2 or not x.is_contiguous():
            raise ValueError("x must be contiguous bf16 rows (2-byte elements)")
        _device_readable(x, "x")
        B.moe_route(self.desc, n_rows, x, self.router if logits_in is None else None, logits_in,
                    self.logits if logits_in is None else None, self.topk_idx, self.topk_w, self.ws,
                    self.n_rows_max, self.n_shared, stream)

    def experts(self, n_rows: int, mode: int = B.MOE_MODE_DECODE, stream=None):
        B.moe_expert_block(self.desc, n_rows, mode, self.routed_pool(), self.expert_slot, self.slot_ready,
                           self.shared_pool_desc(), self.n_shared, self.ws, self.n_rows_max, self.y_part,
                           stream)

    def shared_experts(self, n_rows: int, x, after_route: bool = False, stream=None):
        """The shared experts from x alone (independent of routing); after_route: the
        launch directly follows route() on the same stream and runs beside it."""
        fn = B.moe_shared_experts_after_route if after_route else B.moe_shared_experts
        fn(self.desc, n_rows, x, self.shared_pool_desc(), self.n_shared, self.ws, self.n_rows_max, stream)

    def combine(self, n_rows: int, residual, stream=None, out=None):
        _device_readable(residual, "residual")
        out = self.out if out is None else out
        _device_readable(out, "out")
        if out.dtype != torch.uint16 or not out.is_contiguous() or out.numel() < n_rows * self.d:
            raise ValueError("out must be a contiguous uint16 (bf16 bits) tensor of n_rows x d_model")
        shared_y = self.ws.data_ptr() + self.offsets.shared_y if self.n_shared else None
        B.moe_combine(self.desc, n_rows, residual, self.y_part, self.topk_w, shared_y, self.n_shared,
                      out, stream)

    def forward(self, x, residual, n_rows: int | None = None, logits_in=None, mode=B.MOE_MODE_DECODE,
                stream=None, out=None):
        """Run one block: x, residual bf16 bits [N][d]; returns out bits [N][d].

        One stream: the routing, the shared experts (their kernel starts beside the
        routing: they need x only), the routed experts, the combine; each launch after
        the routing overlaps the tail of the one before it.

        x, residual and out live on the device, or in pinned host memory: the kernels
        then read the rows and write the output in place over the host link (no copy
        launches).  out defaults to ``self.out``."""
        n = x.shape[0] if n_rows is None else n_rows
        self._block(n, x, residual, logits_in, mode, None, out)
        return (self.out if out is None else out)[:n]

    def _side(self):
        if getattr(self, "_side_stream", None) is None:
            self._side_stream = torch.cuda.Stream(device=self.device)
        return self._side_stream

    def _block(self, n, x, residual, logits_in, mode, evs, out=None):
        """route -> shared experts -> routed experts -> combine on the current stream.
        evs, if given: 5 events recorded at the start, once the routing has completed,
        once the shared experts have (and the routing), once the routed experts have,
        and at the end; the middle three on a side branch, so the chained launches of
        the main stream keep overlapping."""
        main = torch.cuda.current_stream()
        chain = self.n_shared > 0 and not (mode & B.MOE_MODE_DEBUG_GU)

        def mark(ev):
            side = self._side()
            side.wait_stream(main)
            ev.record(side)

        if evs:
            evs[0].record(main)
        self.route(n, x, logits_in=logits_in)
        if evs:
            mark(evs[1])
        if chain:
            self.shared_experts(n, x, after_route=True)
            if evs:
                mark(evs[2])
            self.experts(n, mode=mode | B.MOE_MODE_ROUTED_ONLY | B.MOE_MODE_AFTER_SHARED)
        elif evs:
            self.experts(n, mode=mode | B.MOE_MODE_SHARED_ONLY)
            mark(evs[2])
            self.experts(n, mode=mode | B.MOE_MODE_ROUTED_ONLY)
        else:
            self.experts(n, mode=mode)
        if evs:
            mark(evs[3])
        self.combine(n, residual, out=out)
        if evs:
            main.wait_stream(self._side())
            evs[4].record(main)

    def capture(self, x, residual, n_rows: int | None = None, logits_in=None, mode=B.MOE_MODE_DECODE,
                events: bool = False, host_in=None, host_out=None, out=None):
        """Capture one block (route -> experts -> combine) into a CUDA graph.

        The graph reads the block from the given device buffers (x, residual and, if
        given, logits_in): refill them and call ``graph.replay()`` per block; the
        output lands in ``self.out``.  Kernel parameters, including the TMA tensor
        maps, are fixed at capture time.  The graph chains the kernels as forward()
        does.  With events=True five timing events are recorded inside the graph (at
        the start, after the routing, after the shared experts, after the routed
        experts, at the end) and returned; the events are None if the runtime refuses
        them.

        host_in / host_out: pinned host tensors shaped like x[:n] / self.out[:n]; the
        graph then starts by copying host_in into x and ends by copying the output
        into host_out, so one replay takes a block from host memory to host memory.
        Without copies: pass pinned host tensors as x / residual and as out (as for
        forward()); the kernels then read and write them in place."""
        import torch as _torch
        n = x.shape[0] if n_rows is None else n_rows
        side = _torch.cuda.Stream()
        side.wait_stream(_torch.cuda.current_stream())
        with _torch.cuda.stream(side):  # first launches (kernel attributes) outside the capture
            self.forward(x, residual, n_rows=n, logits_in=logits_in, mode=mode, out=out)
        _torch.cuda.current_stream().wait_stream(side)
        _torch.cuda.synchronize()

        for t, name in ((host_in, "host_in"), (host_out, "host_out")):
            if t is not None and (t.is_cuda or not t.is_pinned()):
                raise ValueError(f"{name} must be a pinned host tensor")

        def body(evs):
            if host_in is not None:
                x[:n].copy_(host_in, non_blocking=True)
            self._block(n, x, residual, logits_in, mode, evs, out)
            if host_out is not None:
                host_out.copy_((self.out if out is None else out)[:n], non_blocking=True)

        evs = None
        if events:
            try:  # external events are the ones a graph's event-record nodes can time
                evs = [_torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
            except TypeError:
                evs = None
        g = _torch.cuda.CUDAGraph()
        try:
            with _torch.cuda.graph(g):
                body(evs)
        except RuntimeError:
            if not events:
                raise
            evs = None
            g = _torch.cuda.CUDAGraph()
            with _torch.cuda.graph(g):
                body(None)
        return g, evs

    def error_bits(self, stream=None) -> int:
        return B.moe_get_error(self.ws, stream)
