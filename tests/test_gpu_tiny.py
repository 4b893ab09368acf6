"""GPU parity at the tiny layer shape (d=256, f=64, 32 experts, top-4), through the
C ABI, against the CPU oracle on the same seeded inputs."""

import numpy as np
import pytest
import torch

import moe_synth as syn
from gpu_util import SeededLayer, assert_close_to_oracle, bf16_to_f64, to_dev_u16, topk_gap
from mxfp4_mixture_experts_router_gb300 import binding as B
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

TINY = syn.TINY
TINY_SHARED = syn.Shape(d_model=256, d_ff=64, n_experts=32, top_k=4, group=32, n_shared=2)


@pytest.fixture(scope="module")
def tiny():
    return SeededLayer(TINY, seed=0, n_rows_max=16)


def _check_routing(g, o, k):
    """Logits within fp32 error; selection exact wherever the top-k boundary is not a
    near tie of the fp32 GEMV; weights within fp32 error."""
    np.testing.assert_allclose(g["logits"], o["logits"], rtol=0, atol=1e-5)
    safe = topk_gap(o["logits"], k) > 1e-4
    assert np.array_equal(g["idx"][safe], o["idx"][safe])
    np.testing.assert_allclose(g["w"][safe], o["w"][safe], rtol=2e-6, atol=1e-7)


def test_one_row_matches_oracle(tiny):
    x = syn.x_rows(0, [0], TINY.d_model)
    g = tiny.run(x, x)
    o = tiny.oracle(x, x)
    _check_routing(g, o, TINY.top_k)
    assert_close_to_oracle(g["out"], o, "tiny 1 row")


@pytest.mark.parametrize("n", [1, 2, 4, 16])
def test_blocks_match_oracle(tiny, n):
    x = syn.x_rows(1, range(n), TINY.d_model)
    res = syn.x_rows(1, range(n), TINY.d_model, tag=syn.TAG_RESIDUAL)
    g = tiny.run(x, res)
    o = tiny.oracle(x, res)
    _check_routing(g, o, TINY.top_k)
    assert_close_to_oracle(g["out"], o, f"tiny block of {n}")
    # per (row, slot) expert outputs
    for r in range(n):
        for j in range(TINY.top_k):
            want = o["y"][r, j]
            err = np.linalg.norm(g["y"][r, j] - want) / np.linalg.norm(want)
            assert err < 2e-3, (r, j, err)


def test_block_rows_equal_single_rows_bitwise(tiny):
    n = 16
    x = syn.x_rows(2, range(n), TINY.d_model)
    res = syn.x_rows(2, range(n), TINY.d_model, tag=syn.TAG_RESIDUAL)
    blk = tiny.run(x, res)
    for r in range(n):
        one = tiny.run(x[r:r + 1], res[r:r + 1])
        assert np.array_equal(one["out"][0], blk["out"][r]), r
        assert np.array_equal(one["idx"][0], blk["idx"][r]), r
        assert np.array_equal(one["w"][0].view(np.uint32), blk["w"][r].view(np.uint32)), r
        assert np.array_equal(one["y"][0].view(np.uint32), blk["y"][r].view(np.uint32)), r
        assert np.array_equal(one["logits"][0].view(np.uint32), blk["logits"][r].view(np.uint32)), r


@pytest.mark.parametrize("sigma", [0.1, 0.5, 2.0])
def test_topk_bit_exact_on_given_logits(tiny, sigma):
    n = 16
    logits = syn.block_logits(3, n, TINY.n_experts, sigma)
    x = syn.x_rows(3, range(n), TINY.d_model)
    g = tiny.run(x, x, logits=logits)
    want = orc.select_topk(logits.astype(np.float64), TINY.top_k)
    assert np.array_equal(g["idx"], want)
    w = orc.routing_weights(logits.astype(np.float64), want)
    np.testing.assert_allclose(g["w"], w, rtol=2e-6, atol=1e-7)
    o = tiny.oracle(x, x, logits=logits)
    assert_close_to_oracle(g["out"], o, f"tiny sigma {sigma}")


def test_topk_ties_signed_zero_and_nan(tiny):
    n = 6
    E = TINY.n_experts
    logits = np.zeros((n, E), dtype=np.float32)
    logits[1, ::2] = -0.0                         # -0 equals +0: lower index wins
    logits[2, :] = np.round(np.linspace(-2, 2, E) * 2) / 2  # repeated values
    logits[3, 5] = np.nan                         # NaN ranks last
    logits[3, 7] = -np.inf
    logits[4, :] = -np.inf
    logits[4, 30] = 1.0
    logits[5, :] = 1.0
    x = syn.x_rows(4, range(n), TINY.d_model)
    want = orc.select_topk(logits.astype(np.float64), TINY.top_k)
    g = tiny.run(x, x, logits=logits)
    assert np.array_equal(g["idx"], want)
    assert tiny.layer.error_bits() & B.MOE_EBIT_NAN
    assert tiny.layer.error_bits() == 0  # read-and-clear
    for rows in (2, 1):  # small blocks: the whole CTA selects for each row
        for r in range(0, n, rows):
            g = tiny.run(x[r:r + rows], x[r:r + rows], logits=logits[r:r + rows])
            assert np.array_equal(g["idx"], want[r:r + rows]), (rows, r)
    assert tiny.layer.error_bits() & B.MOE_EBIT_NAN


def test_expert_slot_placement_does_not_change_bits(tiny):
    perm = list(np.random.default_rng(7).permutation(TINY.n_experts))
    other = SeededLayer(TINY, seed=0, n_rows_max=16, slot_perm=perm)
    x = syn.x_rows(5, range(8), TINY.d_model)
    a = tiny.run(x, x)
    b = other.run(x, x)
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["y"].view(np.uint32), b["y"].view(np.uint32))


def test_zero_weight_expert_contributes_nothing():
    lay = SeededLayer(TINY, seed=6, n_rows_max=4)
    logits = np.zeros((1, TINY.n_experts), dtype=np.float32)
    logits[0, [3, 9, 17, 20]] = [200.0, 199.0, 198.0, 40.0]   # exp(-160) underflows fp32
    x = syn.x_rows(6, [0], TINY.d_model)
    a = lay.run(x, x, logits=logits)
    assert a["idx"][0, 3] == 20 and a["w"][0, 3] == 0.0
    lay.layer.put_slab(int(lay.layer.expert_slot[20]), syn.mxfp4_expert_slab(99, 1, TINY))
    b = lay.run(x, x, logits=logits)
    assert np.array_equal(a["out"], b["out"])


def test_gate_up_integer_exact():
    """With unit scales and half-integer activations every product and partial sum is
    exact in fp32, so the gate and up projections must equal the oracle bit for bit."""
    lay = SeededLayer(TINY, seed=8, n_rows_max=4, scale_range=(127, 127))
    n = 3
    vals = np.random.default_rng(8).integers(-8, 9, size=(n, TINY.d_model)) / 2.0
    x = orc.float_to_bf16_bits(vals)
    g = lay.run(x, x, mode=B.MOE_MODE_DECODE | B.MOE_MODE_DEBUG_GU)
    off = lay.layer.offsets
    k = TINY.top_k
    U = int(lay.layer.ws_view(off.n_unique, 1, torch.int32).item())
    uexp = lay.layer.ws_view(off.uexp, U, torch.int32).cpu().numpy()
    offs = lay.layer.ws_view(off.off, U + 1, torch.int32).cpu().numpy()
    pair = lay.layer.ws_view(off.pair, n * k, torch.int32).cpu().numpy()
    npairs = n * k
    dg = lay.layer.ws_view(off.dbg_g, npairs * TINY.d_ff, torch.float32).view(npairs, TINY.d_ff).cpu().numpy()
    du = lay.layer.ws_view(off.dbg_u, npairs * TINY.d_ff, torch.float32).view(npairs, TINY.d_ff).cpu().numpy()
    xf = orc.bf16_bits_to_float(x)
    for u in range(U):
        wg, wu, _ = orc.mxfp4_expert_mats(lay.get_slab(int(uexp[u])), TINY.d_model, TINY.d_ff)
        for t in range(offs[u], offs[u + 1]):
            row = pair[t] // k
            assert np.array_equal(dg[t], (xf[row] @ wg.T).astype(np.float32))
            assert np.array_equal(du[t], (xf[row] @ wu.T).astype(np.float32))
    assert g["idx"].shape == (n, k)


def test_shared_experts_tiny():
    lay = SeededLayer(TINY_SHARED, seed=10, n_rows_max=16)
    for n in (1, 5, 16):
        x = syn.x_rows(10, range(n), TINY.d_model)
        res = syn.x_rows(10, range(n), TINY.d_model, tag=syn.TAG_RESIDUAL)
        g = lay.run(x, res)
        o = lay.oracle(x, res)
        assert_close_to_oracle(g["out"], o, f"tiny shared block {n}")
        sy = lay.layer.shared_y(n).cpu().numpy()
        xf = orc.bf16_bits_to_float(x)
        for s in range(2):
            wg, wu, wd = orc.q8_0_expert_mats(lay.shared[s], TINY.d_model, TINY.d_ff)
            want = orc.swiglu_expert(xf, wg, wu, wd)[3]
            err = np.linalg.norm(sy[s] - want) / np.linalg.norm(want)
            assert err < 1e-4, (n, s, err)


def test_shared_experts_after_routing_match_the_sequential_layer():
    """moe_shared_experts_after_route chained behind moe_route (what forward() does:
    its kernel starts beside the routing and makes its own f16 copy of the rows)
    gives the same bits as one moe_expert_block call after the routing, and so does
    a stand-alone moe_shared_experts call."""
    lay = SeededLayer(TINY_SHARED, seed=11, n_rows_max=16)
    L = lay.layer
    for n in (1, 7, 16):
        x = to_dev_u16(syn.x_rows(11, range(n), TINY.d_model))
        res = to_dev_u16(syn.x_rows(11, range(n), TINY.d_model, tag=syn.TAG_RESIDUAL))
        L.route(n, x)
        L.experts(n)
        L.combine(n, res)
        torch.cuda.synchronize()
        seq_out = L.out[:n].clone()
        seq_shared = L.shared_y(n).clone()
        conc_out = L.forward(x, res).clone()
        torch.cuda.synchronize()
        assert torch.equal(L.shared_y(n), seq_shared), n
        assert torch.equal(conc_out, seq_out), n
        L.shared_y(n).zero_()
        L.shared_experts(n, x)
        torch.cuda.synchronize()
        assert torch.equal(L.shared_y(n), seq_shared), n
        assert L.error_bits() == 0


def test_layer_graph_with_timing_events_matches_forward():
    """The captured layer (chained launches, timing events on a side branch) gives the
    bits of forward(), replay after replay."""
    lay = SeededLayer(TINY_SHARED, seed=13, n_rows_max=16)
    L = lay.layer
    n = 3
    x = to_dev_u16(syn.x_rows(13, range(n), TINY.d_model))
    res = to_dev_u16(syn.x_rows(13, range(n), TINY.d_model, tag=syn.TAG_RESIDUAL))
    want = L.forward(x, res).clone()
    for events in (False, True):
        g, evs = L.capture(x, res, events=events)
        for _ in range(3):
            L.out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(L.out[:n], want)
        if evs:
            t = [evs[0].elapsed_time(evs[i]) for i in range(1, 5)]
            assert all(v >= 0 for v in t) and t[3] >= max(t[:3])
    assert L.error_bits() == 0


def test_layer_graph_from_host_to_host():
    """A graph captured with pinned host buffers copies each block's rows in, runs the
    layer and copies the output back: new rows written into the host buffer between
    replays give the outputs of forward() on those rows."""
    lay = SeededLayer(TINY_SHARED, seed=14, n_rows_max=16)
    L = lay.layer
    n = 2
    rows = [syn.x_rows(14, range(5 * i, 5 * i + n), TINY.d_model) for i in range(3)]
    x = to_dev_u16(rows[0])
    res = to_dev_u16(syn.x_rows(14, range(n), TINY.d_model, tag=syn.TAG_RESIDUAL))
    hin = torch.from_numpy(rows[0].view(np.int16)).view(torch.uint16).pin_memory()
    hout = torch.zeros((n, TINY.d_model), dtype=torch.uint16).pin_memory()
    g, _ = L.capture(x, res, host_in=hin, host_out=hout)
    for r in rows:
        want = L.forward(to_dev_u16(r), res).clone().cpu()
        hin.copy_(torch.from_numpy(r.view(np.int16)).view(torch.uint16))
        hout.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(hout, want)
    with pytest.raises(ValueError):
        L.capture(x, res, host_in=x)
    assert L.error_bits() == 0


def test_layer_reads_and_writes_pinned_host_rows_in_place():
    """Rows and residual in pinned host memory, output to pinned host memory: forward()
    and a captured graph give the bits of the device-resident layer; pageable host
    memory is refused."""
    lay = SeededLayer(TINY_SHARED, seed=15, n_rows_max=16)
    L = lay.layer
    n = 3
    xr = syn.x_rows(15, range(n), TINY.d_model)
    rr = syn.x_rows(15, range(n), TINY.d_model, tag=syn.TAG_RESIDUAL)
    want = L.forward(to_dev_u16(xr), to_dev_u16(rr)).clone().cpu()
    hx = torch.from_numpy(xr.view(np.int16)).view(torch.uint16).pin_memory()
    hr = torch.from_numpy(rr.view(np.int16)).view(torch.uint16).pin_memory()
    ho = torch.zeros((n, TINY.d_model), dtype=torch.uint16).pin_memory()
    got = L.forward(hx, hr, out=ho)
    torch.cuda.synchronize()
    assert got.data_ptr() == ho.data_ptr() and torch.equal(ho, want)
    ho.zero_()
    g, _ = L.capture(hx, hr, out=ho)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(ho, want)
    with pytest.raises(ValueError):
        L.forward(torch.from_numpy(xr.view(np.int16)).view(torch.uint16), hr, out=ho)
    assert L.error_bits() == 0


def test_slot_ready_flag_never_set_times_out_cleanly():
    """A slab whose ready flag nothing sets: the kernel gives up after its bounded
    wait, records MOE_EBIT_TIMEOUT and returns; the context stays usable."""
    lay = SeededLayer(TINY, seed=12, n_rows_max=4)
    x = syn.x_rows(12, [0], TINY.d_model)
    lay.layer.slot_ready = torch.zeros(lay.layer.n_slots, dtype=torch.int32, device="cuda")
    lay.run(x, x)
    assert lay.layer.error_bits() & B.MOE_EBIT_TIMEOUT
    lay.layer.slot_ready.fill_(B.MOE_SLOT_READY)
    ok = lay.run(x, x)
    assert lay.layer.error_bits() == 0
    lay.layer.slot_ready = None
    ref = lay.run(x, x)
    assert np.array_equal(ok["out"], ref["out"])


def test_topk_expert_count_not_a_multiple_of_four():
    """The scalar-load top-k path (30 experts): exact against the oracle, ties included."""
    sh = syn.Shape(d_model=256, d_ff=64, n_experts=30, top_k=4, group=32, n_shared=0)
    lay = SeededLayer(sh, seed=2, n_rows_max=8)
    rng = np.random.default_rng(5)
    lg = rng.normal(size=(5, sh.n_experts)).astype(np.float32)
    lg[1] = 0.0
    lg[2] = np.round(lg[2] * 2) / 2
    lg[3, -6:] = 4.0
    x = syn.x_rows(6, range(5), sh.d_model)
    g = lay.run(x, x, logits=lg)
    want = orc.select_topk(lg.astype(np.float64), sh.top_k)
    assert np.array_equal(g["idx"], want)
    np.testing.assert_allclose(g["w"], orc.routing_weights(lg.astype(np.float64), want), rtol=2e-6, atol=1e-7)
    for r in range(5):  # one row per block: the whole CTA selects
        one = lay.run(x[r:r + 1], x[r:r + 1], logits=lg[r:r + 1])
        assert np.array_equal(one["idx"][0], want[r]), r
        assert np.array_equal(one["w"][0].view(np.uint32), g["w"][r].view(np.uint32)), r
    o = lay.oracle(x, x, logits=lg)
    assert_close_to_oracle(g["out"], o, "30 experts")


def test_expert_compute_order_does_not_change_bits_generic_path(tiny):
    """The same invariance on the engine that serves shapes the block-scaled kernel
    does not (the tiny layer): reversed and random expert orders."""
    L = tiny.layer
    n = 16
    x = syn.x_rows(14, range(n), TINY.d_model)
    base = tiny.run(x, x)
    U = int(L.ws_view(L.offsets.n_unique, 1, torch.int32).item())
    rng = np.random.default_rng(4)
    for order in (np.arange(U)[::-1], rng.permutation(U)):
        L.ws_view(L.offsets.uorder, U, torch.int32).copy_(torch.from_numpy(np.ascontiguousarray(order, np.int32)))
        got = tiny.run(x, x, mode=B.MOE_MODE_DECODE | B.MOE_MODE_ORDERED)
        assert np.array_equal(got["out"], base["out"])
        assert np.array_equal(got["y"].view(np.uint32), base["y"].view(np.uint32))
    assert L.error_bits() == 0
