"""Device expert cache: a slot pool in HBM for (layer, expert) slabs, filled from
pinned host memory on upload streams by the library's cache (``moe_cache_*``).

``DeviceExpertCache`` owns the device pool and the per-slot ready flags;
``prepare(layer, experts, rows, host_ptrs, layer_obj)`` asks the library for slots
(uploading the misses), then points a ``MoeLayer`` at the pool, with its expert ->
slot map and ready flags, so that its expert kernels wait for each slab's chunks
as they land.
"""

from __future__ import annotations

import numpy as np
import torch

from . import binding as B


class DeviceExpertCache:
    def __init__(self, d_model: int, d_ff: int, n_experts: int, top_k: int, n_slots: int, n_streams: int = 8,
                 policy: int = B.MOE_CACHE_LRU, device: str | int = "cuda"):
        self.desc = B.desc(d_model, d_ff, n_experts, top_k)
        self.E = n_experts
        self.device = torch.device(device)
        self.slab_bytes = B.moe_slab_bytes(self.desc, B.MOE_FMT_MXFP4)
        self.slot_bytes = (self.slab_bytes + 255) // 256 * 256
        self.n_slots = n_slots
        self.pool = torch.empty(n_slots * self.slot_bytes, dtype=torch.uint8, device=self.device)
        self.ready = torch.zeros(n_slots, dtype=torch.int32, device=self.device)
        self.handle = B.moe_cache_create(self.desc, self.pool, self.slot_bytes, n_slots, self.ready, n_streams,
                                         policy)
        # pinned staging of the expert -> slot maps, reused only once its copy is done
        self._maps = [torch.full((n_experts,), -1, dtype=torch.int32).pin_memory() for _ in range(8)]
        self._map_done = [None] * len(self._maps)
        self._map_next = 0

    def prepare(self, layer: int, experts, rows, host_ptrs, moe_layer, stream=None):
        """Slots for `experts` of `layer` (misses uploaded from host_ptrs), then the layer
        is pointed at the pool with its expert -> slot map; returns (slots, uploaded)."""
        stream = torch.cuda.current_stream() if stream is None else stream
        slots, uploaded = B.moe_cache_request(self.handle, layer, experts, rows, host_ptrs, stream)
        i = self._map_next
        self._map_next = (i + 1) % len(self._maps)
        if self._map_done[i] is not None:
            self._map_done[i].synchronize()
        m = self._maps[i]
        m.fill_(-1)
        m[torch.as_tensor(np.asarray(experts, dtype=np.int64))] = torch.as_tensor(slots)
        moe_layer.attach_pool(self.pool, self.slot_bytes, self.n_slots, self.ready)
        with torch.cuda.stream(stream):
            moe_layer.expert_slot.copy_(m, non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(stream)
        self._map_done[i] = ev
        return slots, uploaded

    def stats(self) -> dict:
        return B.moe_cache_stats(self.handle)

    def sync(self):
        B.moe_cache_sync(self.handle)

    def close(self):
        if self.handle:
            B.moe_cache_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class CachedLayerRunner:
    """Runs stacked MoE layers whose routed experts live in a ``DeviceExpertCache``,
    in the order a decode engine has to: the routing runs on the GPU, the block's
    selected experts come back to the host, the cache is asked for their slots
    (uploading the misses from the pinned host pool on its upload streams), and the
    expert kernel then runs with the experts already resident first
    (MOE_MODE_ORDERED) while the misses' slabs are still landing.

    After a layer is enqueued, a shallow prefetch asks for up to ``prefetch`` experts
    of the next layer: the ones that layer used on the most rows in the previous
    block (its slabs upload behind the current layer's misses on the same streams).

    body_ptr(layer, experts) -> uint64 numpy array of the experts' pinned host slabs.
    Pages: "Run Kimi 3.1 locally on one GPU", section "Read the experts the router
    needs" (experts scheduled after the router selects them, resident experts first,
    a shallow next-layer prefetch)."""

    def __init__(self, cache: DeviceExpertCache, layer, body_ptr, prefetch: int = 0):
        self.cache = cache
        self.layer = layer
        self.body_ptr = body_ptr
        self.prefetch = prefetch
        o = layer.offsets
        self._o = o
        self._hdr_bytes = o.off + (layer.E + 1) * 4
        self._hdr = torch.empty(self._hdr_bytes, dtype=torch.uint8).pin_memory()
        self._ord = [torch.empty(layer.E, dtype=torch.int32).pin_memory() for _ in range(4)]
        self._ord_done = [None] * 4
        self._ord_next = 0
        self._ev = torch.cuda.Event()
        self.last_used = {}        # layer -> (experts, rows) of the previous block
        self.prefetched = 0
        self.prefetch_uploads = 0

    def run_layer(self, l: int, n: int, x, logits, n_layers: int, stream=None):
        """One layer for a block of n rows (caller logits on the device); returns the
        number of unique experts and of those uploaded."""
        lay = self.layer
        stream = torch.cuda.current_stream() if stream is None else stream
        lay.route(n, x, logits_in=logits)
        self._hdr.copy_(lay.ws[:self._hdr_bytes], non_blocking=True)
        self._ev.record(stream)
        self._ev.synchronize()
        h = self._hdr.numpy()
        U = int(h[self._o.n_unique:self._o.n_unique + 4].view(np.int32)[0])
        uexp = h[self._o.uexp:self._o.uexp + 4 * U].view(np.int32)
        off = h[self._o.off:self._o.off + 4 * (U + 1)].view(np.int32)
        rows = np.diff(off)
        slots, miss = self.cache.prepare(l, uexp, rows, self.body_ptr(l, uexp), lay, stream)
        order = np.argsort(miss, kind="stable").astype(np.int32)  # resident experts first
        i = self._ord_next
        self._ord_next = (i + 1) % len(self._ord)
        if self._ord_done[i] is not None:
            self._ord_done[i].synchronize()
        buf = self._ord[i]
        buf[:U].copy_(torch.from_numpy(order))
        lay.ws_view(self._o.uorder, U, torch.int32).copy_(buf[:U], non_blocking=True)
        ev = torch.cuda.Event()
        ev.record(stream)
        self._ord_done[i] = ev
        from . import binding as B
        lay.experts(n, mode=B.MOE_MODE_DECODE | B.MOE_MODE_ORDERED)
        lay.combine(n, x)
        self.last_used[l] = (uexp.copy(), rows.copy())
        if self.prefetch and l + 1 < n_layers and (l + 1) in self.last_used:
            e1, r1 = self.last_used[l + 1]
            top = e1[np.argsort(-r1, kind="stable")[: self.prefetch]]
            _, up = B.moe_cache_request(self.cache.handle, l + 1, top, np.ones(len(top), np.int32),
                                        self.body_ptr(l + 1, top), stream)
            self.prefetched += len(top)
            self.prefetch_uploads += int(up.sum())
        return U, int(miss.sum())
