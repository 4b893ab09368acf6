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
