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
from gpu_util import SeededLayer, assert_close_to_oracle
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
