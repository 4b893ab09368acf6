"""Top-k ties under the router GEMV at the Kimi shape (d = 7168, 896 experts, top 16).

Router rows copied onto other experts give bit-identical logits (each expert's dot
product is reduced in the same fixed order), placed inside one 64-expert group and
across groups, below and above the copied expert's index, at the top-16 boundary and
among the winners.  The selection must be the oracle's on the GPU's own logits (larger
first, ties to the lower index), for blocks of 1 to 4 rows (per-group candidates merged
by rank) and of 5 and 9 rows (a warp per row).

Page: "Run Kimi 3.1 locally on one GPU", section "Read the experts the router needs"
(16 of 896 experts per token)."""

import numpy as np
import pytest
import torch

import moe_synth as syn
from gpu_util import ensure_built
from mxfp4_mixture_experts_router_gb300.layer import MoeLayer
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

KIMI = syn.KIMI


def _router_with_ties(x, seed):
    w = syn.router_weight(seed, KIMI).copy()
    lo = orc.router_logits(x[:1], w)[0]
    rank = np.argsort(-lo, kind="stable")
    rng = np.random.default_rng(seed)
    # the 15th-ranked expert's row onto six others: same group, other groups, lower and higher indices
    b = int(rank[14])
    same = [e for e in range((b // 64) * 64, (b // 64) * 64 + 64) if e != b and e not in rank[:20]][:2]
    others = [int(e) for e in rng.permutation(KIMI.n_experts) if abs(int(e) - b) > 64 and e not in rank[:20]][:4]
    for e in same + others:
        w[e] = w[b]
    # the winner's row onto two more experts (ties among the winners)
    a = int(rank[0])
    for e in [int(e) for e in rng.permutation(KIMI.n_experts) if e not in rank[:20] and e not in same + others][:2]:
        w[e] = w[a]
    return w


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 9])
def test_router_gemv_ties_go_to_the_lower_index(n):
    ensure_built()
    x = syn.x_rows(77, range(n), KIMI.d_model)
    x[1:] = x[0]  # every row of the block sees the same ties
    w = _router_with_ties(x, 5)
    lay = MoeLayer(KIMI.d_model, KIMI.d_ff, KIMI.n_experts, KIMI.top_k, n_rows_max=16, n_shared=0)
    lay.set_router(torch.from_numpy(w.view(np.int16)).view(torch.uint16))
    xd = torch.from_numpy(x.view(np.int16)).cuda().view(torch.uint16)
    lay.route(n, xd)
    torch.cuda.synchronize()
    assert lay.error_bits() == 0
    logits = lay.logits[:n].cpu().numpy()
    idx = lay.topk_idx[:n].cpu().numpy()
    wts = lay.topk_w[:n].cpu().numpy()
    # the constructed ties are there in the GPU's logits
    lo = logits[0]
    vals, counts = np.unique(lo, return_counts=True)
    assert counts.max() >= 3
    want = orc.select_topk(logits.astype(np.float64), KIMI.top_k)
    assert np.array_equal(idx, want)
    np.testing.assert_allclose(wts, orc.routing_weights(logits.astype(np.float64), want), rtol=2e-6, atol=1e-7)
    # and the grouping: every selected expert once, its pairs in row order
    U = int(lay.ws_view(lay.offsets.n_unique, 1, torch.int32).item())
    uexp = lay.ws_view(lay.offsets.uexp, U, torch.int32).cpu().numpy()
    off = lay.ws_view(lay.offsets.off, U + 1, torch.int32).cpu().numpy()
    pair = lay.ws_view(lay.offsets.pair, n * KIMI.top_k, torch.int32).cpu().numpy()
    assert np.array_equal(uexp, np.unique(want))
    for u, e in enumerate(uexp):
        got = pair[off[u]:off[u + 1]]
        exp = [r * KIMI.top_k + int(np.where(want[r] == e)[0][0]) for r in range(n) if e in want[r]]
        assert list(got) == exp
