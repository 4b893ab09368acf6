"""GPU parity at the Kimi K3.1 layer shape (d=7168, f=1536, 896 experts, top-16,
2 Q8_0 shared experts), through the C ABI, against the CPU oracle.

The pool holds every expert the sampled rows and blocks select (plus the
runners-up of the GEMV-routed rows), each streamed once per block."""

import numpy as np
import pytest

import moe_synth as syn
from gpu_util import SeededLayer, assert_close_to_oracle, topk_gap
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

KIMI = syn.KIMI
SEED = 0
DECODE_ROWS = [0, 1, 2]
SIGMAS = (0.1, 0.5, 2.0)


@pytest.fixture(scope="module")
def kimi():
    router = syn.router_weight(SEED, KIMI)
    x = syn.x_rows(SEED, DECODE_ROWS, KIMI.d_model)
    lo = orc.router_logits(x, router)
    experts = set(np.argsort(-lo, axis=1)[:, :24].ravel().tolist())
    blocks = {}
    for i, s in enumerate(SIGMAS):
        lg = syn.block_logits(SEED, 16, KIMI.n_experts, s, block=i)
        blocks[s] = lg
        experts |= set(orc.select_topk(lg.astype(np.float64), KIMI.top_k).ravel().tolist())
    lay = SeededLayer(KIMI, SEED, n_rows_max=16, experts=sorted(experts))
    return lay, x, blocks


def test_decode_rows_match_oracle(kimi):
    lay, x, _ = kimi
    for r in range(len(DECODE_ROWS)):
        xr = x[r:r + 1]
        g = lay.run(xr, xr)
        o = lay.oracle(xr, xr)
        np.testing.assert_allclose(g["logits"], o["logits"], rtol=0, atol=2e-4)
        if topk_gap(o["logits"], KIMI.top_k)[0] > 1e-3:
            assert np.array_equal(g["idx"], o["idx"])
        np.testing.assert_allclose(g["w"], o["w"], rtol=1e-4, atol=1e-6)
        assert_close_to_oracle(g["out"], o, f"kimi decode row {r}")
        rel_y = np.linalg.norm(g["y"] - o["y"]) / np.linalg.norm(o["y"])
        assert rel_y < 1e-3, rel_y


@pytest.mark.parametrize("sigma", SIGMAS)
def test_verification_block_rows_equal_single_rows(kimi, sigma):
    lay, _, blocks = kimi
    logits = blocks[sigma]
    x = syn.x_rows(SEED + 1, range(16), KIMI.d_model)
    res = syn.x_rows(SEED + 1, range(16), KIMI.d_model, tag=syn.TAG_RESIDUAL)
    want_idx = orc.select_topk(logits.astype(np.float64), KIMI.top_k)
    for n in (2, 4, 8, 16):
        blk = lay.run(x[:n], res[:n], logits=logits[:n])
        assert np.array_equal(blk["idx"], want_idx[:n])
        for r in range(n):
            one = lay.run(x[r:r + 1], res[r:r + 1], logits=logits[r:r + 1])
            assert np.array_equal(one["out"][0], blk["out"][r]), (n, r)
            assert np.array_equal(one["y"][0].view(np.uint32), blk["y"][r].view(np.uint32)), (n, r)


def test_verification_block_matches_oracle(kimi):
    lay, _, blocks = kimi
    logits = blocks[0.5]
    x = syn.x_rows(SEED + 2, range(16), KIMI.d_model)
    res = syn.x_rows(SEED + 2, range(16), KIMI.d_model, tag=syn.TAG_RESIDUAL)
    g = lay.run(x, res, logits=logits)
    rows = [0, 15]
    o = lay.oracle(x[rows], res[rows], logits=logits[rows])
    for i, r in enumerate(rows):
        one = {"out": o["out"][i:i + 1], "out_bf16": o["out_bf16"][i:i + 1]}
        assert_close_to_oracle(g["out"][r:r + 1], one, f"kimi block row {r}")
