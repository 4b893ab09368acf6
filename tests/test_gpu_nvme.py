"""The NVMe expert tier feeding the device expert cache on the GPU: blocks of tiny
layers whose routed experts are read from replicated files into pinned staging
buffers (two chunks each) while the uploads already wait for them on the GPU
(moe_cache_request_staged), then the layer runs; every output equals the layer
with every slab resident, and the first block also matches the CPU oracle.

Page: "Run Kimi 3.1 locally on one GPU", section "Read the experts the router
needs" (experts read from NVMe into pinned memory as the router asks for them,
compute starting as an expert's data lands)."""

import numpy as np
import pytest
import torch

import moe_synth as syn
from gpu_util import assert_close_to_oracle, ensure_built, to_dev_u16
from mxfp4_mixture_experts_router_gb300 import binding as B
from mxfp4_mixture_experts_router_gb300.cache import DeviceExpertCache
from mxfp4_mixture_experts_router_gb300.layer import MoeLayer
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

TINY = syn.TINY
SLAB = TINY.mxfp4_slab_bytes
STRIDE = (SLAB + 4095) // 4096 * 4096
GU = 2 * (TINY.d_ff * TINY.d_model // 2 + TINY.d_ff * TINY.d_model // 32)


def test_layers_from_nvme_through_the_cache(tmp_path):
    ensure_built()
    E, k, d, n = TINY.n_experts, TINY.top_k, TINY.d_model, 2
    n_bodies, n_slots = 24, 10
    bodies = [syn.mxfp4_body_slab(9, b, TINY) for b in range(n_bodies)]
    paths = [str(tmp_path / f"drive{i}.bin") for i in range(2)]
    for p in paths:
        with open(p, "wb") as fh:
            for s in bodies:
                fh.write(s.tobytes() + b"\0" * (STRIDE - SLAB))

    def body_of(layer, e):
        return (layer * 5 + e * 7) % n_bodies

    res = MoeLayer(d, TINY.d_ff, E, k, n_rows_max=n, n_shared=0)  # every body resident: the reference
    res.alloc_pool(n_bodies)
    for b, s in enumerate(bodies):
        res.put_slab(b, s)
    lay = MoeLayer(d, TINY.d_ff, E, k, n_rows_max=n, n_shared=0)
    cache = DeviceExpertCache(d, TINY.d_ff, E, k, n_slots=n_slots, n_streams=2, policy=B.MOE_CACHE_KEEP_MULTI_ROW)
    nv = B.moe_nvme_open(paths, SLAB, STRIDE, n_bodies, depth=2)
    staging = torch.empty((n * k, STRIDE), dtype=torch.uint8).pin_memory()
    flags = torch.zeros(n * k, dtype=torch.int32).pin_memory()
    rng = np.random.default_rng(12)
    bias = 3.0 * rng.normal(size=(2, E))
    reads = 0
    try:
        for blk in range(10):
            layer = blk % 2
            logits = (bias[layer] + rng.normal(size=(n, E))).astype(np.float32)
            x = syn.x_rows(50 + blk, range(n), d)
            xd, ld = to_dev_u16(x), torch.from_numpy(logits).cuda()
            res.set_expert_slots([body_of(layer, e) for e in range(E)])
            ref = res.forward(xd, xd, logits_in=ld).clone()
            idx = orc.select_topk(logits.astype(np.float64), k)
            experts, rows = np.unique(idx, return_counts=True)
            resident = B.moe_cache_lookup(cache.handle, layer, experts)
            src = np.zeros(len(experts), dtype=np.uint64)
            rdy = np.zeros(len(experts), dtype=np.uint64)
            for i, e in enumerate(experts):
                src[i] = staging[i].data_ptr()
                rdy[i] = flags.data_ptr() + 4 * i
                if not resident[i]:  # the miss is read from the drives while the uploads wait for it
                    B.moe_nvme_read(nv, body_of(layer, int(e)), int(src[i]), GU, int(rdy[i]))
                    reads += 1
            slots, miss = B.moe_cache_request_staged(cache.handle, layer, experts, rows, src, rdy)
            assert np.array_equal(miss, 1 - resident)
            m = torch.full((E,), -1, dtype=torch.int32)
            m[torch.from_numpy(experts.astype(np.int64))] = torch.from_numpy(slots)
            lay.attach_pool(cache.pool, cache.slot_bytes, cache.n_slots, cache.ready)
            lay.expert_slot.copy_(m)
            got = lay.forward(xd, xd, logits_in=ld)
            torch.cuda.synchronize()
            cache.sync()
            assert lay.error_bits() == 0
            assert torch.equal(got, ref), blk
            if blk == 0:
                o = orc.moe_layer(x, x, TINY, lambda e, l=layer: bodies[body_of(l, e)], logits=logits)
                assert_close_to_oracle(got.view(torch.int16).cpu().numpy().view(np.uint16), o, "nvme block 0")
        st = cache.stats()
        assert st["misses"] == reads and st["hits"] > 0 and st["evictions"] > 0
        per = [B.moe_nvme_stats(nv, r) for r in range(2)]
        assert sum(p["reads"] for p in per) == reads and all(p["failures"] == 0 for p in per)
    finally:
        B.moe_nvme_close(nv)
        cache.close()
