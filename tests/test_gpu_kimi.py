"""GPU parity at the Kimi K3.1 layer shape (d=7168, f=1536, 896 experts, top-16,
2 Q8_0 shared experts), through the C ABI, against the CPU oracle.

The pool holds every expert the sampled rows and blocks select (plus the
runners-up of the GEMV-routed rows), each streamed once per block."""

import numpy as np
import pytest
import torch

import moe_synth as syn
from gpu_util import SeededLayer, assert_close_to_oracle, topk_gap
from mxfp4_mixture_experts_router_gb300 import binding as B
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


@pytest.mark.parametrize("sigma,rows", [(0.5, [0, 15]), (0.1, list(range(16))), (2.0, list(range(16)))])
def test_verification_block_matches_oracle(kimi, sigma, rows):
    """16-row verification blocks (the 48-column configuration) against the oracle:
    every row at sigma 0.1 (about 24 experts, up to 16 rows each) and 2.0 (about 188
    experts, mostly one row each), two rows at 0.5."""
    lay, _, blocks = kimi
    logits = blocks[sigma]
    x = syn.x_rows(SEED + 2, range(16), KIMI.d_model)
    res = syn.x_rows(SEED + 2, range(16), KIMI.d_model, tag=syn.TAG_RESIDUAL)
    g = lay.run(x, res, logits=logits)
    o = lay.oracle(x[rows], res[rows], logits=logits[rows])
    assert np.array_equal(g["idx"][rows], o["idx"])
    for i, r in enumerate(rows):
        one = {"out": o["out"][i:i + 1], "out_bf16": o["out_bf16"][i:i + 1]}
        assert_close_to_oracle(g["out"][r:r + 1], one, f"kimi block sigma {sigma} row {r}")
        rel_y = np.linalg.norm(g["y"][r] - o["y"][i]) / np.linalg.norm(o["y"][i])
        assert rel_y < 1e-3, (sigma, r, rel_y)


def _route_only(lay, logits):
    """Routing alone through moe_route (caller logits), at the layer's width."""
    n = logits.shape[0]
    x = syn.x_rows(SEED + 7, range(n), KIMI.d_model)
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.uint16)
    ld = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
    lay.layer.route(n, xd, logits_in=ld)
    torch.cuda.synchronize()
    return lay.layer.topk_idx[:n].cpu().numpy(), lay.layer.topk_w[:n].cpu().numpy()


def test_topk_ties_at_full_width(kimi):
    """Ties at the top-16 boundary spread over the whole 896-wide row (so across the
    kernel's float4 blocks and lanes): the lower index wins, as in the oracle."""
    lay, _, _ = kimi
    E, k = KIMI.n_experts, KIMI.top_k
    rng = np.random.default_rng(11)
    lg = np.zeros((7, E), dtype=np.float32)                   # row 0: all equal
    lg[1] = np.round(rng.normal(size=E) * 2) / 4               # few levels: many ties at the boundary
    lg[2] = -1.0
    lg[2, 100:900:37] = 3.0                                    # 22 equal winners for 16 places
    lg[3] = rng.normal(size=E).astype(np.float32)
    lg[3, ::3] = 0.0
    lg[3, 1::3] = -0.0                                         # +0 and -0 tie
    lg[3, rng.permutation(E)[:10]] = 9.0
    lg[4] = 0.5
    lg[4, -40:] = 5.0                                          # 40 tied leaders at the highest indices
    lg[5] = rng.normal(size=E).astype(np.float32)
    lg[5, [3, 400, 895]] = np.nan                              # NaN ranks last
    lg[6] = rng.normal(size=E).astype(np.float32)              # plain
    want = orc.select_topk(lg.astype(np.float64), k)
    ok = ~np.isnan(lg).any(axis=1)
    # blocks of 7 rows (a warp per row), of 2 and of 1 (the whole CTA per row)
    for rows in (7, 2, 1):
        parts = [_route_only(lay, lg[r:r + rows]) for r in range(0, 7, rows)]
        idx = np.concatenate([a for a, _ in parts])
        w = np.concatenate([b for _, b in parts])
        assert np.array_equal(idx, want), rows
        np.testing.assert_allclose(w[ok], orc.routing_weights(lg.astype(np.float64), want)[ok], rtol=2e-6,
                                   atol=1e-7)
        lay.layer.error_bits()  # the NaN row sets the NaN bit; read and clear it


@pytest.mark.parametrize("n", [1, 4])
def test_chained_layer_equals_sequential_calls(kimi, n):
    """forward() chains route -> shared experts (beside the routing) -> routed experts
    (MOE_MODE_AFTER_SHARED: started as the shared experts' CTAs leave) -> combine; the
    same calls made one after another with plain waits give the same bits."""
    lay, _, blocks = kimi
    L = lay.layer
    logits = blocks[2.0][:n]
    x = syn.x_rows(SEED + 5, range(n), KIMI.d_model)
    res = syn.x_rows(SEED + 5, range(n), KIMI.d_model, tag=syn.TAG_RESIDUAL)
    chained = lay.run(x, res, logits=logits)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda().view(torch.uint16)
    rd = torch.from_numpy(np.ascontiguousarray(res).view(np.int16)).cuda().view(torch.uint16)
    ld = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
    L.out.zero_()
    L.route(n, xd, logits_in=ld)
    torch.cuda.synchronize()
    L.experts(n)
    torch.cuda.synchronize()
    L.combine(n, rd)
    torch.cuda.synchronize()
    seq = L.out[:n].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(chained["out"], seq)
    assert L.error_bits() == 0


def _orders(U, seed):
    rng = np.random.default_rng(seed)
    ident = np.arange(U, dtype=np.int32)
    resident_first = np.concatenate([ident[1::3], ident[0::3], ident[2::3]]).astype(np.int32)
    return {"reversed": ident[::-1].copy(), "random": rng.permutation(U).astype(np.int32),
            "resident_first": resident_first}


def test_expert_compute_order_does_not_change_bits(kimi):
    """The routed experts worked in another order (MOE_MODE_ORDERED: reversed, random,
    a third of them first as a device cache would put its resident experts) give every
    output bit of the default order ("Run Kimi 3.1 locally on one GPU", section "What
    is established": outputs match with and without resident-first ordering)."""
    lay, _, blocks = kimi
    L = lay.layer
    n = 8
    logits = blocks[2.0][:n]
    x = syn.x_rows(SEED + 9, range(n), KIMI.d_model)
    base = lay.run(x, x, logits=logits)
    U = int(L.ws_view(L.offsets.n_unique, 1, torch.int32).item())
    assert U > 40
    for name, order in _orders(U, 3).items():
        L.ws_view(L.offsets.uorder, U, torch.int32).copy_(torch.from_numpy(order))
        got = lay.run(x, x, logits=logits, mode=B.MOE_MODE_DECODE | B.MOE_MODE_ORDERED)
        assert np.array_equal(got["out"], base["out"]), name
        assert np.array_equal(got["y"].view(np.uint32), base["y"].view(np.uint32)), name
    assert L.error_bits() == 0
