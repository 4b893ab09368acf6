"""Blocks of more than 32 rows (the prefill path: three routing launches, the
block-scaled expert kernel with experts split into chunks of at most 16 pairs)
at the Kimi K3.1 layer shape.

A row's arithmetic does not depend on its block, so every sampled row of a
48-row block must equal, bit for bit, the same row run alone through the decode
path; the selection must equal the oracle's on the same logits; ten rows, among
them rows of the experts split into several chunks, are also compared with the
oracle within the layer's tolerance."""

import numpy as np
import pytest

import moe_synth as syn
from gpu_util import SeededLayer, assert_close_to_oracle, topk_gap
from mxfp4_mixture_experts_router_gb300 import binding as B
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

KIMI = syn.KIMI
N = 48
SEED = 41


@pytest.fixture(scope="module")
def prefill():
    rng = np.random.default_rng(SEED)
    E, k = KIMI.n_experts, KIMI.top_k
    hot = rng.choice(E, size=36, replace=False)
    logits = rng.normal(size=(N, E)).astype(np.float32)
    logits[:, hot] += 4.0                                  # most selections fall on 36 experts
    idx = orc.select_topk(logits.astype(np.float64), k)
    experts = sorted(set(idx.ravel().tolist()))
    lay = SeededLayer(KIMI, SEED, n_rows_max=N, experts=experts, n_shared=0)
    x = syn.x_rows(SEED, range(N), KIMI.d_model)
    res = syn.x_rows(SEED, range(N), KIMI.d_model, tag=syn.TAG_RESIDUAL)
    blk = lay.run(x, res, logits=logits, mode=B.MOE_MODE_PREFILL)
    return lay, x, res, logits, idx, blk


def test_prefill_selection_and_weights(prefill):
    lay, _, _, logits, idx, blk = prefill
    assert np.array_equal(blk["idx"], idx)
    w = orc.routing_weights(logits.astype(np.float64), idx)
    np.testing.assert_allclose(blk["w"], w, rtol=2e-6, atol=1e-7)
    counts = np.bincount(idx.ravel(), minlength=KIMI.n_experts)
    assert counts.max() > 16          # some expert is split into several chunks
    assert lay.layer.error_bits() == 0


@pytest.mark.parametrize("row", [0, 7, 19, 33, 47])
def test_prefill_rows_equal_single_rows(prefill, row):
    lay, x, res, logits, _, blk = prefill
    one = lay.run(x[row:row + 1], res[row:row + 1], logits=logits[row:row + 1])
    assert np.array_equal(one["out"][0], blk["out"][row])
    assert np.array_equal(one["y"][0].view(np.uint32), blk["y"][row].view(np.uint32))


def test_prefill_rows_match_oracle(prefill):
    """Ten rows of the 48-row block against the oracle, among them rows routed to the
    experts with the most pairs (split into several chunks of at most 16 pairs)."""
    lay, x, res, logits, idx, blk = prefill
    counts = np.bincount(idx.ravel(), minlength=KIMI.n_experts)
    split = np.flatnonzero(counts > 16)
    on_split = [r for r in range(N) if np.isin(idx[r], split).any()]
    rows = sorted(set([0, 5, 13, 22, 30, 38, 47] + on_split[:3]))
    assert len(rows) >= 8 and any(r in on_split for r in rows)
    o = lay.oracle(x[rows], res[rows], logits=logits[rows])
    assert np.array_equal(blk["idx"][rows], o["idx"])
    for i, r in enumerate(rows):
        one = {"out": o["out"][i:i + 1], "out_bf16": o["out_bf16"][i:i + 1]}
        assert_close_to_oracle(blk["out"][r:r + 1], one, f"prefill row {r}")
        rel_y = np.linalg.norm(blk["y"][r] - o["y"][i]) / np.linalg.norm(o["y"][i])
        assert rel_y < 1e-3, (r, rel_y)


def test_prefill_whole_layer_router_gemm_and_shared_experts():
    """A prefill block of 40 rows as a whole layer: the router GEMM (blocks of more
    than 32 rows), top-16 selection, the routed experts on the block-scaled path and
    the 2 Q8_0 shared experts for every row, against the oracle on sampled rows.  A
    Kimi-shaped layer with 64 routed experts keeps the pool and the oracle small."""
    sh = syn.Shape(d_model=KIMI.d_model, d_ff=KIMI.d_ff, n_experts=64, top_k=16, group=32, n_shared=2)
    n = 40
    lay = SeededLayer(sh, seed=43, n_rows_max=n)
    x = syn.x_rows(43, range(n), sh.d_model)
    res = syn.x_rows(43, range(n), sh.d_model, tag=syn.TAG_RESIDUAL)
    g = lay.run(x, res, mode=B.MOE_MODE_PREFILL)
    assert lay.layer.error_bits() == 0
    rows = [0, 9, 17, 26, 39]
    o = lay.oracle(x[rows], res[rows])
    np.testing.assert_allclose(g["logits"][rows], o["logits"], rtol=0, atol=2e-4)
    for i, r in enumerate(rows):
        if topk_gap(o["logits"][i:i + 1], sh.top_k)[0] > 1e-3:
            assert np.array_equal(g["idx"][r], o["idx"][i]), r
            want = {"out": o["out"][i:i + 1], "out_bf16": o["out_bf16"][i:i + 1]}
        else:  # a near tie at the top-16 boundary: compare on the GPU's own logits
            oo = lay.oracle(x[r:r + 1], res[r:r + 1], logits=g["logits"][r:r + 1])
            want = {"out": oo["out"], "out_bf16": oo["out_bf16"]}
        assert_close_to_oracle(g["out"][r:r + 1], want, f"prefill whole layer row {r}")
    # the shared experts' outputs of every row against the oracle's
    sy = lay.layer.shared_y(n).cpu().numpy()
    xf = orc.bf16_bits_to_float(x[rows])
    for s in range(2):
        wg, wu, wd = orc.q8_0_expert_mats(lay.shared[s], sh.d_model, sh.d_ff)
        want = orc.swiglu_expert(xf, wg, wu, wd)[3]
        err = np.linalg.norm(sy[s][rows] - want) / np.linalg.norm(want)
        assert err < 1e-4, (s, err)
