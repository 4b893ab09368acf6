"""CPU oracle for the block-batched MXFP4 mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only the tests under ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py`` use it.  It shares no
code with the CUDA path; its only common dependency is the seeded input
generator ``moe_synth``, which carries none of the method's arithmetic.

Everything here is plain numpy in float64, written step by step from the pages:

* "Run Kimi 3.1 locally on one GPU" (argonautlabs.ai), sections
  "One GPU, three storage tiers" (MXFP4 experts, one 17,547,264-byte file per
  expert; Q8_0 spine), "Read the experts the router needs" (896 experts per
  layer, 16 selected per token) and "A drafter that leaves the answer unchanged"
  (a block reads each expert once for all its rows; block rows run the same
  arithmetic as plain steps).
* "Run Kimi K3 and K3.1 Pro Locally: Hardware and K3 Speed Tests"
  (computingforgeeks.com), section "Kimi K3 and K3.1 Pro in numbers" (16 of 896
  routed experts plus 2 shared) and "Confirm the checkpoint format and size"
  (MXFP4 expert weights; router and shared experts unquantised BF16 in the
  checkpoint, here carried as a BF16 router and Q8_0 shared experts, since the
  first page quantises the whole non-expert spine to Q8_0).

Readings where the pages are silent (the pages give the formats and counts, not these steps):

* Router function: softmax over the router logits, the k largest kept, their
  probabilities renormalised to sum to 1 (routed scaling 1).  Selection is done
  on the logits; ties go to the lower expert index; NaN ranks below -inf.
* MXFP4 is the OCP Microscaling v1.0 format: E2M1 elements with one E8M0 scale
  per 32 consecutive elements along K.  The group of 32 and the one-byte scale
  are what make three 7168x1536 matrices occupy exactly 17,547,264 bytes.
* Q8_0: int8 values with one fp16 scale per 32 consecutive values along K.
* SwiGLU expert: h = silu(x Wg^T) * (x Wu^T), y = h Wd^T, silu(g) = g/(1+e^-g).
* Shared experts are unweighted and run on every row.
* out = bf16_rne(residual + sum_j w_j y_j + sum_s shared_s).

Parity status of every function is given in its docstring ("pinned by ...").
"""

from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------------------
# element formats
# ---------------------------------------------------------------------------

# E2M1 (OCP MX v1.0): sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
# Magnitudes of the eight non-negative codes.
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def e2m1_to_float(codes) -> np.ndarray:
    """Value of each 4-bit E2M1 code (0..15).  Pinned by an exhaustive test against the
    bit-field definition of the OCP MX FP4 format."""
    c = np.asarray(codes, dtype=np.int64)
    mag = _E2M1_MAG[c & 7]
    return np.where(c & 8, -mag, mag)


def e8m0_to_float(s) -> np.ndarray:
    """Value 2^(s-127) of each E8M0 scale byte; 255 is NaN.  Pinned exhaustively against
    torch's float8_e8m0fnu conversion and exact powers of two."""
    s = np.asarray(s, dtype=np.int64)
    v = np.ldexp(1.0, s - 127)
    return np.where(s == 255, np.nan, v)


def fp16_bits_to_float(bits) -> np.ndarray:
    """IEEE binary16 bit patterns -> float64 (exact)."""
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)


def bf16_bits_to_float(bits) -> np.ndarray:
    """bfloat16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def float_to_bf16_bits(v) -> np.ndarray:
    """Round float64 values to bfloat16, nearest-even, in one rounding (no detour through
    float32).  Pinned against brute-force nearest-even over all bf16 neighbours."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(over="ignore", invalid="ignore"):
        m, e = np.frexp(a)                                   # a = m * 2^e, m in [0.5, 1)
        normal_q = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)  # 8 significant bits, ties to even
        sub_q = np.ldexp(np.rint(np.ldexp(a, 133)), -133)    # bf16 subnormal spacing 2^-133
        q = np.where(a < 2.0 ** -126, sub_q, normal_q)
        q = np.where(q >= 2.0 ** 128, np.inf, q)             # rounds past the largest finite
        q = np.where(np.isnan(v), np.nan, q)
        q = np.copysign(q, v)
    bits = (q.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return np.where(np.isnan(v), np.uint16(0x7FC0), bits)


# ---------------------------------------------------------------------------
# storage: expert slabs
# ---------------------------------------------------------------------------

def mxfp4_planes(slab: np.ndarray, d_model: int, d_ff: int, group: int = 32) -> dict:
    """Split one MXFP4 expert slab into (codes, scales) per matrix.

    Slab layout, in order: gate codes [f][d/2], gate scales [f][d/group], up codes
    [f][d/2], up scales [f][d/group], down codes [d][f/2], down scales [d][f/group];
    codes row-major with the even-K element in the low nibble.  The pages give only
    the total ("each expert is a 17,547,264-byte MXFP4 file"); the plane order is this
    implementation's reading.  Pinned by the byte-count identity and by the scale
    planes holding exactly the drawn exponent range."""
    slab = np.asarray(slab, dtype=np.uint8)
    out = {}
    off = 0
    for name, rows, k in (("gate", d_ff, d_model), ("up", d_ff, d_model), ("down", d_model, d_ff)):
        nc = rows * k // 2
        ns = rows * k // group
        codes = slab[off:off + nc].reshape(rows, k // 2)
        off += nc
        scales = slab[off:off + ns].reshape(rows, k // group)
        off += ns
        out[name] = (codes, scales)
    if off != slab.size:
        raise ValueError(f"slab has {slab.size} bytes, layout needs {off}")
    return out


def q8_0_planes(slab: np.ndarray, d_model: int, d_ff: int, group: int = 32) -> dict:
    """Split one Q8_0 expert slab into (int8 q, fp16 d bits) per matrix, same plane order
    as the MXFP4 slab.  Pinned by the byte-count identity."""
    slab = np.asarray(slab, dtype=np.uint8)
    out = {}
    off = 0
    for name, rows, k in (("gate", d_ff, d_model), ("up", d_ff, d_model), ("down", d_model, d_ff)):
        nq = rows * k
        nd = rows * k // group
        q = slab[off:off + nq].view(np.int8).reshape(rows, k)
        off += nq
        dbits = slab[off:off + 2 * nd].view(np.uint16).reshape(rows, k // group)
        off += 2 * nd
        out[name] = (q, dbits)
    if off != slab.size:
        raise ValueError(f"slab has {slab.size} bytes, layout needs {off}")
    return out


def dequant_mxfp4(codes: np.ndarray, scales: np.ndarray, group: int = 32) -> np.ndarray:
    """W[r][k] = E2M1(code[r][k]) * 2^(scale[r][k // group] - 127), float64 [rows][K].
    Pinned by the exhaustive code x scale test and an encode/decode round trip."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows, half = codes.shape
    lo = e2m1_to_float(codes & 0x0F)
    hi = e2m1_to_float(codes >> 4)
    vals = np.empty((rows, 2 * half), dtype=np.float64)
    vals[:, 0::2] = lo
    vals[:, 1::2] = hi
    sc = e8m0_to_float(scales)
    return (vals.reshape(rows, -1, group) * sc[:, :, None]).reshape(rows, 2 * half)


def dequant_q8_0(q: np.ndarray, dbits: np.ndarray, group: int = 32) -> np.ndarray:
    """W[r][k] = q[r][k] * fp16(d[r][k // group]), float64 [rows][K].  Pinned exhaustively."""
    q = np.asarray(q, dtype=np.int8).astype(np.float64)
    rows, k = q.shape
    d = fp16_bits_to_float(dbits)
    return (q.reshape(rows, -1, group) * d[:, :, None]).reshape(rows, k)


# ---------------------------------------------------------------------------
# routing
# ---------------------------------------------------------------------------

def router_logits(x_bits: np.ndarray, w_bits: np.ndarray) -> np.ndarray:
    """logit[n][e] = sum_c x[n][c] * Wr[e][c] in float64 (bf16 products are exact in
    float64).  Pinned against exact rational arithmetic on small cases."""
    x = bf16_bits_to_float(x_bits)
    w = bf16_bits_to_float(w_bits)
    return x @ w.T


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per row, in rank order: larger logit first, equal
    logits by lower index, NaN after every number (then by index); -0 equals +0.
    Pinned against a brute-force repeated-maximum selection."""
    l = np.asarray(logits, dtype=np.float64)
    n, e = l.shape
    if not 1 <= k <= e:
        raise ValueError("need 1 <= k <= n_experts")
    idx = np.arange(e)
    out = np.empty((n, k), dtype=np.int32)
    for r in range(n):
        row = l[r]
        nan = np.isnan(row)
        key = np.where(nan, 0.0, -row) + 0.0  # +0.0 folds -0 into +0
        order = np.lexsort((idx, key, nan))
        out[r] = order[:k]
    return out


def routing_weights(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """w[n][j] = exp(l_j - l_max) / sum over the selected i of exp(l_i - l_max): the
    softmax restricted to the selected experts, i.e. softmax then renormalise.
    Pinned by sum = 1, k = 1 giving exactly 1, and the logistic closed form at k = 2."""
    l = np.asarray(logits, dtype=np.float64)
    sel = np.take_along_axis(l, np.asarray(idx, dtype=np.int64), axis=1)
    top = sel[:, :1]
    ex = np.exp(sel - top)
    return ex / ex.sum(axis=1, keepdims=True)


def group_pairs(idx: np.ndarray, n_experts: int):
    """Group a block's (row, slot) pairs by selected expert, so each expert is read once
    for all its rows.  Returns (uexp, off, pair): uexp = selected experts ascending
    [U]; pairs of uexp[u] are pair[off[u]:off[u+1]], each pair = row*k + slot,
    ascending.  Pinned by partition invariants."""
    idx = np.asarray(idx, dtype=np.int64)
    n, k = idx.shape
    flat = idx.reshape(-1)
    pid = np.arange(n * k)
    order = np.lexsort((pid, flat))
    uexp, counts = np.unique(flat, return_counts=True)
    off = np.zeros(len(uexp) + 1, dtype=np.int32)
    off[1:] = np.cumsum(counts)
    if len(uexp) and (uexp.min() < 0 or uexp.max() >= n_experts):
        raise ValueError("expert index out of range")
    return uexp.astype(np.int32), off, pid[order].astype(np.int32)


# ---------------------------------------------------------------------------
# experts and the layer
# ---------------------------------------------------------------------------

def silu(g: np.ndarray) -> np.ndarray:
    """silu(g) = g / (1 + exp(-g)).  Pinned against scipy's logistic function."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def swiglu_expert(x: np.ndarray, wg: np.ndarray, wu: np.ndarray, wd: np.ndarray,
                  out_cols=None) -> tuple:
    """One expert on rows x [r][d]: g = x Wg^T, u = x Wu^T, h = silu(g) u, y = h Wd^T.
    Returns (g, u, h, y); with out_cols only those output columns of y are formed.
    Pinned against a scalar-loop brute force on tiny shapes."""
    g = x @ wg.T
    u = x @ wu.T
    h = silu(g) * u
    y = h @ (wd if out_cols is None else wd[out_cols]).T
    return g, u, h, y


def mxfp4_expert_mats(slab: np.ndarray, d_model: int, d_ff: int, group: int = 32) -> tuple:
    p = mxfp4_planes(slab, d_model, d_ff, group)
    return tuple(dequant_mxfp4(*p[m], group=group) for m in ("gate", "up", "down"))


def q8_0_expert_mats(slab: np.ndarray, d_model: int, d_ff: int, group: int = 32) -> tuple:
    p = q8_0_planes(slab, d_model, d_ff, group)
    return tuple(dequant_q8_0(*p[m], group=group) for m in ("gate", "up", "down"))


def moe_layer(x_bits, residual_bits, shape, get_slab, router_w_bits=None, logits=None,
              shared_slabs=(), out_cols=None, select_in_fp32: bool = True):
    """The whole MoE layer for a block of rows, in float64.

    Steps: router logits (or caller-supplied logits) -> top-k selection -> renormalised
    weights -> group rows by expert -> per expert SwiGLU MLP on its rows -> weighted sum
    over the k slots -> plus the unweighted shared experts -> plus the residual -> bf16.

    get_slab(e) returns the MXFP4 slab of expert e.  When the logits come from the
    router GEMV, the selection is taken on the float64 logits rounded to float32
    (``select_in_fp32``), the precision the GPU path selects in; the weights use the
    float64 logits.  out_cols restricts the output columns (sampled checks).

    Returns a dict with logits, idx, w, y (per row and slot, float64 [N][k][cols]),
    shared (float64 [N][cols]), out (float64) and out_bf16 (uint16 bits)."""
    d, f, g, k = shape.d_model, shape.d_ff, shape.group, shape.top_k
    x = bf16_bits_to_float(x_bits)
    n = x.shape[0]
    if logits is None:
        logits = router_logits(x_bits, router_w_bits)
        sel_logits = logits.astype(np.float32).astype(np.float64) if select_in_fp32 else logits
    else:
        logits = np.asarray(logits, dtype=np.float64)
        sel_logits = logits
    idx = select_topk(sel_logits, k)
    w = routing_weights(logits, idx)
    uexp, off, pair = group_pairs(idx, shape.n_experts)
    cols = np.arange(d) if out_cols is None else np.asarray(out_cols)
    y = np.zeros((n, k, len(cols)), dtype=np.float64)
    for u, e in enumerate(uexp):
        pr = pair[off[u]:off[u + 1]]
        rows, slots = pr // k, pr % k
        wg, wu, wd = mxfp4_expert_mats(get_slab(int(e)), d, f, g)
        _, _, _, ye = swiglu_expert(x[rows], wg, wu, wd, out_cols=cols)
        y[rows, slots] = ye
    shared = np.zeros((n, len(cols)), dtype=np.float64)
    for s in shared_slabs:
        wg, wu, wd = q8_0_expert_mats(s, d, f, g)
        shared += swiglu_expert(x, wg, wu, wd, out_cols=cols)[3]
    res = bf16_bits_to_float(residual_bits)[:, cols]
    routed = np.einsum("nk,nkc->nc", w, y)
    out = res + routed + shared
    return dict(logits=logits, idx=idx, w=w, uexp=uexp, off=off, pair=pair, y=y,
                shared=shared, out=out, out_bf16=float_to_bf16_bits(out), cols=cols)
