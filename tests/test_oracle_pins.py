"""Pins of the CPU oracle to facts outside itself (no GPU needed).

Each test checks one oracle function against something the pages or the
mathematics fix: printed byte counts, the bit-field definition of the MX formats,
a library conversion, a closed form, exact rational arithmetic, or a brute force
written independently with scalar loops.
"""

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import moe_synth as syn
from oracle import moe_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "page_figures.json")


def _fig(name):
    with open(GOLDEN) as fh:
        return json.load(fh)[name]["value"]


# ---------------------------------------------------------------------------
# storage layout
# ---------------------------------------------------------------------------

def test_expert_file_size_fixes_group_32():
    """'Each expert is a 17,547,264-byte MXFP4 file' (Run Kimi 3.1 locally on one GPU,
    One GPU, three storage tiers): three 7168x1536 matrices at 4 bits plus one byte per
    g elements fit that count only for g = 32."""
    total = _fig("mxfp4_expert_file_bytes")
    d, f = 7168, 1536
    per_bit = Fraction(total, 3 * d * f) - Fraction(1, 2)
    assert per_bit == Fraction(1, 32)
    assert syn.KIMI.mxfp4_slab_bytes == total
    slab = np.zeros(total, dtype=np.uint8)
    planes = orc.mxfp4_planes(slab, d, f, 32)
    assert sum(c.size + s.size for c, s in planes.values()) == total
    # 82,432 experts of that size are about 1.45 TB
    tb = _fig("experts_all_layers") * total / 1e12
    assert abs(tb - _fig("unique_payload_tb")) < 0.005
    assert _fig("experts_all_layers") == _fig("moe_layers") * _fig("experts_per_layer")


def test_q8_0_slab_size():
    """Q8_0 keeps one int8 per value and one fp16 per 32."""
    assert syn.KIMI.q8_0_slab_bytes == 3 * 7168 * 1536 * (1 + 2 / 32) == 35094528
    slab = np.zeros(syn.KIMI.q8_0_slab_bytes, dtype=np.uint8)
    planes = orc.q8_0_planes(slab, 7168, 1536)
    assert sum(q.size + 2 * d.size for q, d in planes.values()) == slab.size


@pytest.mark.parametrize("lo,hi", [(200, 200), (120, 127)])
def test_mxfp4_plane_positions(lo, hi):
    """The oracle finds the scale planes exactly where the generator drew the restricted
    exponent range; the code planes hold the full byte range."""
    sh = syn.TINY
    slab = syn.mxfp4_expert_slab(3, 5, sh, scale_lo=lo, scale_hi=hi)
    planes = orc.mxfp4_planes(slab, sh.d_model, sh.d_ff)
    for codes, scales in planes.values():
        assert scales.min() >= lo and scales.max() <= hi
        assert codes.max() > 200 and codes.min() < 50
    assert planes["gate"][0].shape == (sh.d_ff, sh.d_model // 2)
    assert planes["down"][1].shape == (sh.d_model, sh.d_ff // 32)


# ---------------------------------------------------------------------------
# element formats
# ---------------------------------------------------------------------------

def _e2m1_from_bits(c):
    """OCP MX v1.0 FP4 E2M1: sign, 2 exponent bits with bias 1, 1 mantissa bit;
    exponent field 0 is subnormal."""
    s, e, m = (c >> 3) & 1, (c >> 1) & 3, c & 1
    mag = 2.0 ** (e - 1) * (1 + m / 2) if e else (m / 2) * 2.0 ** (1 - 1)
    return -mag if s else mag


def test_e2m1_exhaustive():
    got = orc.e2m1_to_float(np.arange(16))
    for c in range(16):
        assert got[c] == _e2m1_from_bits(c)
    assert math.copysign(1.0, got[8]) == -1.0  # code 8 is -0
    assert sorted(set(abs(v) for v in got)) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e8m0_exhaustive_vs_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch without float8_e8m0fnu")
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    got = orc.e8m0_to_float(np.arange(256))
    assert np.isnan(got[255]) and np.isnan(ref[255])
    np.testing.assert_array_equal(got[:255], ref[:255])
    for s in (0, 1, 127, 254):
        assert got[s] == math.ldexp(1.0, s - 127)


def test_mxfp4_dequant_all_codes_all_scales():
    """Every code at every finite scale, with nibble order low = even K."""
    rows = []
    scales = []
    for s in range(255):
        # one group of 32: codes 0..15 then 15..0
        seq = list(range(16)) + list(range(15, -1, -1))
        rows.append(bytes((seq[2 * i] | (seq[2 * i + 1] << 4)) for i in range(16)))
        scales.append([s])
    codes = np.frombuffer(b"".join(rows), dtype=np.uint8).reshape(255, 16)
    w = orc.dequant_mxfp4(codes, np.array(scales, dtype=np.uint8))
    seq = list(range(16)) + list(range(15, -1, -1))
    for s in range(255):
        for kk in range(32):
            assert w[s, kk] == _e2m1_from_bits(seq[kk]) * math.ldexp(1.0, s - 127)


def test_q8_0_dequant_exhaustive():
    q = np.arange(-128, 128, dtype=np.int16).astype(np.int8)
    q = np.tile(q, 1).reshape(8, 32)  # 8 groups of 32 covering all 256 int8 values
    dvals = np.arange(0, 0x7C00, 37, dtype=np.uint16)  # finite positive fp16 sweep
    for db in dvals[::7]:
        dbits = np.full((8, 1), db, dtype=np.uint16)
        w = orc.dequant_q8_0(q, dbits)
        dv = float(np.array([db], dtype=np.uint16).view(np.float16)[0])
        for r in range(8):
            for kk in range(32):
                assert w[r, kk] == int(q[r, kk]) * dv


def _bf16_table():
    allb = np.arange(0x7F81, dtype=np.uint32)  # non-negative finite bf16 patterns and +inf
    vals = (allb << 16).view(np.float32).astype(np.float64)
    vals[0x7F80] = 2.0 ** 128  # IEEE overflow: round as if the next exponent existed, then inf
    return vals, allb


def test_bf16_rounding_bruteforce():
    vals, pats = _bf16_table()
    rng = np.random.default_rng(0)
    xs = list(rng.standard_normal(2000) * 10.0 ** rng.integers(-40, 38, 2000))
    # exact midpoints between neighbours (ties to even), subnormal range, overflow edge
    mids = (vals[1000:1100] + vals[1001:1101]) / 2
    xs += list(mids) + list(-mids) + [1e-40, 3e-39, 2.0 ** -133 * 0.5, 3.4e38, 3.3895e38]
    xs = np.array(xs)
    got = orc.float_to_bf16_bits(xs)
    for x, g in zip(xs, got):
        a = abs(x)
        j = np.searchsorted(vals, a)
        cands = [j - 1, j] if 0 < j < len(vals) else [min(j, len(vals) - 1)]
        best = min(cands, key=lambda c: (abs(vals[c] - a), pats[c] & 1))
        want = int(pats[best]) | (0x8000 if x < 0 else 0)
        assert int(g) == want, (x, hex(int(g)), hex(want))


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def test_router_logits_exact_rational():
    rng = np.random.default_rng(1)
    xb = syn._to_bf16_bits(rng.standard_normal((3, 96)))
    wb = syn._to_bf16_bits(rng.standard_normal((5, 96)) * 0.02)
    got = orc.router_logits(xb, wb)
    xf = orc.bf16_bits_to_float(xb)
    wf = orc.bf16_bits_to_float(wb)
    for n in range(3):
        for e in range(5):
            exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(xf[n], wf[e]))
            bound = 96 * 2.0 ** -52 * float(sum(abs(Fraction(float(a)) * Fraction(float(b)))
                                                 for a, b in zip(xf[n], wf[e])))
            assert abs(Fraction(got[n, e]) - exact) <= Fraction(bound)


def _brute_topk(row, k):
    """Repeatedly take the best remaining expert: larger value first, then lower index;
    NaN after every number."""
    left = list(range(len(row)))
    out = []
    for _ in range(k):
        best = None
        for e in left:
            v = row[e]
            if best is None:
                best = e
                continue
            bv = row[best]
            if math.isnan(bv) and not math.isnan(v):
                best = e
            elif not math.isnan(v) and not math.isnan(bv) and v > bv:
                best = e
        out.append(best)
        left.remove(best)
    return out


@pytest.mark.parametrize("E,k", [(32, 4), (32, 32), (896, 16), (896, 1)])
def test_select_topk_bruteforce(E, k):
    rng = np.random.default_rng(E + k)
    l = np.round(rng.standard_normal((6, E)) * 2) / 2  # many exact ties
    l[0, :] = 0.0
    l[0, ::3] = -0.0                                    # -0 equals +0
    l[1, 5] = np.nan
    l[1, 7] = -np.inf
    l[2, :] = np.nan
    got = orc.select_topk(l, k)
    for r in range(6):
        assert list(got[r]) == _brute_topk(list(l[r]), k)


def test_routing_weights_closed_forms():
    from scipy.special import expit
    rng = np.random.default_rng(2)
    l = rng.standard_normal((50, 896)) * 1.7
    idx = orc.select_topk(l, 16)
    w = orc.routing_weights(l, idx)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(np.diff(w, axis=1) <= 0)
    w1 = orc.routing_weights(l, orc.select_topk(l, 1))
    assert np.all(w1 == 1.0)
    i2 = orc.select_topk(l, 2)
    w2 = orc.routing_weights(l, i2)
    a = np.take_along_axis(l, i2.astype(np.int64), 1)
    np.testing.assert_allclose(w2[:, 0], expit(a[:, 0] - a[:, 1]), rtol=1e-14)


def test_group_pairs_partition():
    rng = np.random.default_rng(3)
    for n, E, k in [(1, 896, 16), (16, 896, 16), (5, 32, 4), (16, 32, 32)]:
        l = rng.standard_normal((n, E))
        idx = orc.select_topk(l, k)
        uexp, off, pair = orc.group_pairs(idx, E)
        assert list(uexp) == sorted(set(idx.reshape(-1).tolist()))
        assert off[0] == 0 and off[-1] == n * k and np.all(np.diff(off) > 0)
        assert sorted(pair.tolist()) == list(range(n * k))
        for u, e in enumerate(uexp):
            pr = pair[off[u]:off[u + 1]]
            assert np.all(np.diff(pr) > 0)
            assert np.all(idx.reshape(-1)[pr] == e)


# ---------------------------------------------------------------------------
# expert MLP and the layer
# ---------------------------------------------------------------------------

def test_silu_closed_form():
    from scipy.special import expit
    g = np.linspace(-60, 60, 2001)
    np.testing.assert_allclose(orc.silu(g), g * expit(g), rtol=1e-14, atol=1e-300)
    assert orc.silu(np.array([0.0]))[0] == 0.0


def _nib(b, k):
    return (b >> 4) if k & 1 else (b & 15)


def _brute_layer(xb, rb, shape, slabs, wrb, shared):
    """Scalar-loop restatement of the layer straight from the slab bytes: no numpy
    matmul, its own offset arithmetic and its own code/scale decoding."""
    d, f, E, k, G = shape.d_model, shape.d_ff, shape.n_experts, shape.top_k, shape.group
    xs = [[float(v) for v in orc.bf16_bits_to_float(row)] for row in xb]
    wr = [[float(v) for v in orc.bf16_bits_to_float(row)] for row in wrb]
    outs = []

    def mx(slab, base, rows, K, r, c):
        code = _nib(int(slab[base + r * (K // 2) + c // 2]), c)
        s = int(slab[base + rows * K // 2 + r * (K // G) + c // G])
        return _e2m1_from_bits(code) * math.ldexp(1.0, s - 127)

    def q8(slab, base, rows, K, r, c):
        q = int(slab[base + r * K + c])
        q = q - 256 if q > 127 else q
        lo = int(slab[base + rows * K + 2 * (r * (K // G) + c // G)])
        hi = int(slab[base + rows * K + 2 * (r * (K // G) + c // G) + 1])
        dv = float(np.array([lo | (hi << 8)], dtype=np.uint16).view(np.float16)[0])
        return q * dv

    def mlp(x, slab, get, per_matrix):
        h = []
        for j in range(f):
            g = sum(x[c] * get(slab, 0, f, d, j, c) for c in range(d))
            u = sum(x[c] * get(slab, per_matrix, f, d, j, c) for c in range(d))
            h.append(g / (1 + math.exp(-g)) * u)
        return [sum(h[j] * get(slab, 2 * per_matrix, d, f, c, j) for j in range(f)) for c in range(d)]

    pm_mx = d * f // 2 + d * f // G
    pm_q8 = d * f + 2 * d * f // G
    for n, x in enumerate(xs):
        lg = [sum(a * b for a, b in zip(x, wr[e])) for e in range(E)]
        sel = _brute_topk([float(np.float32(v)) for v in lg], k)
        ex = [math.exp(lg[e] - lg[sel[0]]) for e in sel]
        w = [v / sum(ex) for v in ex]
        out = [float(v) for v in orc.bf16_bits_to_float(rb[n])]
        for j, e in enumerate(sel):
            y = mlp(x, slabs[e], mx, pm_mx)
            out = [o + w[j] * yy for o, yy in zip(out, y)]
        for s in shared:
            y = mlp(x, s, q8, pm_q8)
            out = [o + yy for o, yy in zip(out, y)]
        outs.append(out)
    return np.array(outs)


@pytest.mark.slow
def test_tiny_layer_against_scalar_brute_force():
    sh = syn.Shape(d_model=64, d_ff=32, n_experts=8, top_k=3, group=32, n_shared=1)
    seed = 11
    xb = syn.x_rows(seed, range(2), sh.d_model)
    rb = syn.x_rows(seed, range(2), sh.d_model, tag=syn.TAG_RESIDUAL)
    wrb = syn.router_weight(seed, sh, sigma=0.3)
    slabs = {e: syn.mxfp4_expert_slab(seed, e, sh) for e in range(sh.n_experts)}
    shared = [syn.q8_0_shared_slab(seed, 0, sh)]
    got = orc.moe_layer(xb, rb, sh, slabs.__getitem__, router_w_bits=wrb, shared_slabs=shared)
    want = _brute_layer(xb, rb, sh, slabs, wrb, shared)
    np.testing.assert_allclose(got["out"], want, rtol=1e-11, atol=1e-9 * np.abs(want).max())


def test_tiny_dense_equivalence():
    """Evaluating every expert on every row and weighting by a vector that is zero off the
    top-k gives the sparse, grouped result."""
    sh = syn.TINY
    seed = 5
    xb = syn.x_rows(seed, range(4), sh.d_model)
    wrb = syn.router_weight(seed, sh)
    slabs = {e: syn.mxfp4_expert_slab(seed, e, sh) for e in range(sh.n_experts)}
    r = orc.moe_layer(xb, xb, sh, slabs.__getitem__, router_w_bits=wrb)
    x = orc.bf16_bits_to_float(xb)
    dense = orc.bf16_bits_to_float(xb).copy()
    wvec = np.zeros((4, sh.n_experts))
    for n in range(4):
        wvec[n, r["idx"][n]] = r["w"][n]
    for e in range(sh.n_experts):
        wg, wu, wd = orc.mxfp4_expert_mats(slabs[e], sh.d_model, sh.d_ff)
        y = orc.swiglu_expert(x, wg, wu, wd)[3]
        dense += wvec[:, e:e + 1] * y
    np.testing.assert_allclose(r["out"], dense, rtol=1e-12, atol=1e-12 * np.abs(dense).max())


def test_zero_weight_expert_contributes_nothing():
    sh = syn.TINY
    seed = 9
    xb = syn.x_rows(seed, range(1), sh.d_model)
    logits = np.zeros((1, sh.n_experts))
    logits[0, :sh.top_k] = [900.0, 899.0, 898.0, 0.0]  # gap > 745: exp underflows to 0.0
    slabs = {e: syn.mxfp4_expert_slab(seed, e, sh) for e in range(sh.n_experts)}
    a = orc.moe_layer(xb, xb, sh, slabs.__getitem__, logits=logits)
    assert a["w"][0, -1] == 0.0 and a["idx"][0, -1] == 3
    slabs2 = dict(slabs)
    slabs2[3] = syn.mxfp4_expert_slab(seed + 1, 77, sh)
    b = orc.moe_layer(xb, xb, sh, slabs2.__getitem__, logits=logits)
    np.testing.assert_array_equal(a["out"], b["out"])


def test_expert_weight_sums_and_selection_in_layer():
    sh = syn.TINY
    seed = 4
    logits = syn.block_logits(seed, 8, sh.n_experts, 0.5)
    xb = syn.x_rows(seed, range(8), sh.d_model)
    slabs = {e: syn.mxfp4_expert_slab(seed, e, sh) for e in range(sh.n_experts)}
    r = orc.moe_layer(xb, xb, sh, slabs.__getitem__, logits=logits)
    np.testing.assert_allclose(r["w"].sum(1), 1.0, atol=1e-14)
    for n in range(8):
        assert list(r["idx"][n]) == _brute_topk(list(logits[n].astype(np.float64)), sh.top_k)
