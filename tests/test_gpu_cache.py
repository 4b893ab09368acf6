"""Device expert cache on the GPU: blocks of several layers run with their routed
experts served from a small cache (fewer slots than the experts they touch, so
slots are evicted and re-uploaded while the kernels run) give bit-for-bit the
outputs of the same layers with every slab resident, and the first and last
blocks also match the CPU oracle on the same expert bodies."""

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


def body_of(layer, expert, n_bodies):
    return (layer * 7 + expert * 3) % n_bodies


def run_case(shape, n_bodies, n_slots, n_rows, n_layers, n_blocks, policy, seed):
    ensure_built()
    E, k, d = shape.n_experts, shape.top_k, shape.d_model
    slabs = [syn.mxfp4_expert_slab(seed, b, shape) for b in range(n_bodies)]
    slab_bytes = slabs[0].size
    host = torch.empty((n_bodies, slab_bytes), dtype=torch.uint8).pin_memory()
    for b, s in enumerate(slabs):
        host[b].copy_(torch.from_numpy(s))
    base = host.data_ptr()

    # every body resident: the reference
    res = MoeLayer(d, shape.d_ff, E, k, n_rows_max=n_rows, n_shared=0)
    res.alloc_pool(n_bodies)
    for b, s in enumerate(slabs):
        res.put_slab(b, s)
    # served from the cache
    lay = MoeLayer(d, shape.d_ff, E, k, n_rows_max=n_rows, n_shared=0)
    cache = DeviceExpertCache(d, shape.d_ff, E, k, n_slots=n_slots, n_streams=2, policy=policy)
    rng = np.random.default_rng(seed)
    bias = 3.0 * rng.normal(size=(n_layers, E))  # per-layer popularity, so that slots get reused
    uploads = 0
    try:
        for blk in range(n_blocks):
            layer = blk % n_layers
            logits = (bias[layer] + rng.normal(size=(n_rows, E))).astype(np.float32)
            x = syn.x_rows(seed + blk, range(n_rows), d)
            xd = to_dev_u16(x)
            ld = torch.from_numpy(logits).cuda()
            # resident reference for this layer
            res.set_expert_slots([body_of(layer, e, n_bodies) for e in range(E)])
            ref = res.forward(xd, xd, logits_in=ld).clone()
            ref_y = res.y_part[:n_rows].clone()
            # the cache: experts of the block (host-side selection on the same logits)
            idx = orc.select_topk(logits.astype(np.float64), k)
            experts, rows = np.unique(idx, return_counts=True)
            ptrs = np.array([base + body_of(layer, int(e), n_bodies) * slab_bytes for e in experts],
                            dtype=np.uint64)
            _, up = cache.prepare(layer, experts, rows, ptrs, lay)
            uploads += int(up.sum())
            got = lay.forward(xd, xd, logits_in=ld)
            torch.cuda.synchronize()
            assert lay.error_bits() == 0
            assert torch.equal(got, ref), blk
            assert torch.equal(lay.y_part[:n_rows], ref_y), blk
            if blk in (0, n_blocks - 1):
                # the cached layer against the oracle on the same bodies and logits
                o = orc.moe_layer(x, x, shape, lambda e, l=layer: slabs[body_of(l, e, n_bodies)], logits=logits)
                assert_close_to_oracle(got.view(torch.int16).cpu().numpy().view(np.uint16), o, f"cached block {blk}")
        cache.sync()
        st = cache.stats()
        assert st["misses"] == uploads and st["evictions"] > 0 and st["hits"] > 0
        return st
    finally:
        cache.close()


@pytest.mark.parametrize("policy", [B.MOE_CACHE_LRU, B.MOE_CACHE_KEEP_MULTI_ROW])
def test_tiny_layers_from_a_small_cache(policy):
    run_case(syn.TINY, n_bodies=40, n_slots=12, n_rows=2, n_layers=3, n_blocks=24, policy=policy, seed=31)


def test_kimi_layers_from_a_small_cache():
    # one layer over 18 slots: its 16 experts per block mostly recur, the boundary churns
    run_case(syn.KIMI, n_bodies=64, n_slots=18, n_rows=1, n_layers=1, n_blocks=8,
             policy=B.MOE_CACHE_KEEP_MULTI_ROW, seed=32)
