"""Parity of the block-scaled tensor-core path (tcgen05) that runs every routed
expert at the Kimi K3.1 layer shape (d=7168, f=1536, 896 experts, top-16),
through the C ABI, against the CPU oracle.

* Exact contraction: with unit E8M0 scales and half-integer activations every
  product and every partial sum of the gate and up projections is exact in fp32,
  so g and u (MOE_MODE_DEBUG_GU) must equal the oracle bit for bit, for blocks of
  1, 5 (the <= 5-row configuration) and 16 rows (the 16-row configuration).
* An expert whose fp32 routing weight underflows to zero contributes nothing:
  replacing its bytes changes no output bit.
* E8M0 scales drawn from a wide exponent range still match the oracle.

Page: "Run Kimi 3.1 locally on one GPU", section "A drafter that leaves the
answer unchanged" (block rows run the same arithmetic as plain steps); the
zero-weight and exact-contraction checks follow from the layer's definition."""

import numpy as np
import pytest
import torch

import moe_synth as syn
from gpu_util import SeededLayer, assert_close_to_oracle
from mxfp4_mixture_experts_router_gb300 import binding as B
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

KIMI = syn.KIMI
E, K_TOP, D, F = KIMI.n_experts, KIMI.top_k, KIMI.d_model, KIMI.d_ff


def logits_over(seed: int, n: int, experts) -> np.ndarray:
    """Router logits that select only among `experts`: N(0,1) on them, -50 elsewhere."""
    rng = np.random.default_rng(seed)
    lg = np.full((n, E), -50.0, dtype=np.float32)
    lg[:, experts] = rng.normal(size=(n, len(experts))).astype(np.float32)
    return lg


def grouping(lay: SeededLayer, n: int):
    off = lay.layer.offsets
    U = int(lay.layer.ws_view(off.n_unique, 1, torch.int32).item())
    uexp = lay.layer.ws_view(off.uexp, U, torch.int32).cpu().numpy()
    offs = lay.layer.ws_view(off.off, U + 1, torch.int32).cpu().numpy()
    pair = lay.layer.ws_view(off.pair, n * K_TOP, torch.int32).cpu().numpy()
    return uexp, offs, pair


@pytest.fixture(scope="module")
def unit_scale_layer():
    experts = list(range(3, 3 + 2 * 20, 2))  # 20 experts, unit scales (E8M0 = 127)
    return SeededLayer(KIMI, seed=21, n_rows_max=16, experts=experts, n_shared=0, scale_range=(127, 127)), experts


@pytest.mark.parametrize("n", [1, 5, 16])
def test_tc_gate_up_integer_exact(unit_scale_layer, n):
    lay, experts = unit_scale_layer
    rng = np.random.default_rng(100 + n)
    vals = rng.integers(-8, 9, size=(n, D)) / 2.0
    x = orc.float_to_bf16_bits(vals)
    lg = logits_over(200 + n, n, experts)
    g = lay.run(x, x, logits=lg, mode=B.MOE_MODE_DECODE | B.MOE_MODE_DEBUG_GU)
    assert np.array_equal(g["idx"], orc.select_topk(lg.astype(np.float64), K_TOP))
    uexp, offs, pair = grouping(lay, n)
    npairs = n * K_TOP
    off = lay.layer.offsets
    dg = lay.layer.ws_view(off.dbg_g, npairs * F, torch.float32).view(npairs, F).cpu().numpy()
    du = lay.layer.ws_view(off.dbg_u, npairs * F, torch.float32).view(npairs, F).cpu().numpy()
    xf = orc.bf16_bits_to_float(x)
    assert np.array_equal(xf, vals)  # half-integers are exact in bf16
    checked = 0
    for u in range(len(uexp)):
        p = orc.mxfp4_planes(lay.get_slab(int(uexp[u])), D, F)
        wg = orc.dequant_mxfp4(*p["gate"])
        wu = orc.dequant_mxfp4(*p["up"])
        prs = pair[offs[u]:offs[u + 1]]
        rows = prs // K_TOP
        want_g = (xf[rows] @ wg.T).astype(np.float32)
        want_u = (xf[rows] @ wu.T).astype(np.float32)
        for i, t in enumerate(range(offs[u], offs[u + 1])):
            assert np.array_equal(dg[t].view(np.uint32), want_g[i].view(np.uint32)), (n, int(uexp[u]), int(prs[i]))
            assert np.array_equal(du[t].view(np.uint32), want_u[i].view(np.uint32)), (n, int(uexp[u]), int(prs[i]))
            checked += 1
    assert checked == npairs
    assert lay.layer.error_bits() == 0


def test_tc_zero_weight_expert_contributes_nothing():
    experts = [int(e) for e in np.random.default_rng(5).choice(E, size=16, replace=False)]
    lay = SeededLayer(KIMI, seed=22, n_rows_max=4, experts=experts, n_shared=0)
    lg = np.full((1, E), -1000.0, dtype=np.float32)
    for i, e in enumerate(experts[:15]):
        lg[0, e] = 200.0 - i
    lg[0, experts[15]] = 40.0                      # exp(40 - 200) underflows fp32: weight 0
    x = syn.x_rows(22, [0], D)
    a = lay.run(x, x, logits=lg)
    assert a["idx"][0, 15] == experts[15] and a["w"][0, 15] == 0.0
    slot = int(lay.layer.expert_slot[experts[15]])
    lay.layer.put_slab(slot, syn.mxfp4_expert_slab(99, 7, KIMI))
    b = lay.run(x, x, logits=lg)
    assert np.array_equal(a["out"], b["out"])
    assert not np.array_equal(a["y"][0, 15].view(np.uint32), b["y"][0, 15].view(np.uint32))
    o = lay.oracle(x, x, logits=lg)
    assert_close_to_oracle(a["out"], o, "zero-weight expert")
    assert lay.layer.error_bits() == 0


def test_tc_wide_scale_range_matches_oracle():
    experts = list(range(100, 100 + 24))
    lay = SeededLayer(KIMI, seed=23, n_rows_max=8, experts=experts, n_shared=0, scale_range=(100, 140))
    n = 3
    lg = logits_over(23, n, experts)
    x = syn.x_rows(23, range(n), D)
    res = syn.x_rows(23, range(n), D, tag=syn.TAG_RESIDUAL)
    g = lay.run(x, res, logits=lg)
    o = lay.oracle(x, res, logits=lg)
    assert np.array_equal(g["idx"], o["idx"])
    assert_close_to_oracle(g["out"], o, "E8M0 in [100, 140]")
    rel_y = np.linalg.norm(g["y"] - o["y"]) / np.linalg.norm(o["y"])
    assert rel_y < 1e-3, rel_y
    assert lay.layer.error_bits() == 0
