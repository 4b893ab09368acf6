"""Seeded synthetic inputs for the block-batched MXFP4 mixture-of-experts layer.

This module is the ONLY code shared by the CPU oracle (``oracle/``) and the
CUDA path's tests and benchmark.  It holds no arithmetic of the method: it
draws bytes and Gaussian samples from a counter-based generator and lays them
out in the documented storage formats.  Everything it returns is plain numpy
(bf16 and fp16 values are returned as their uint16 bit patterns).

Generator: the SplitMix64 output function (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", OOPSLA 2014) applied to a
counter, ``out(i) = mix(key + (i + 1) * 0x9E3779B97F4A7C15)``.  Keys are
derived by chaining the same mix over (seed, stream tag, indices), so every
plane of every expert is an independent, position-addressable stream.

Workload shapes follow "Run Kimi 3.1 locally on one GPU" (section "Read the
experts the router needs": 896 experts per layer, 16 selected) and "Run Kimi
K3 and K3.1 Pro locally" (section "Kimi K3 and K3.1 Pro in numbers": 16 of
896 plus 2 shared).  The hidden size 7168 and expert width 1536 are the ones
that reproduce the 17,547,264-byte MXFP4 expert file of the first page
(section "One GPU, three storage tiers").
"""

from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK = (1 << 64) - 1

# stream tags
TAG_X = 1
TAG_ROUTER = 2
TAG_EXPERT = 3
TAG_SHARED = 4
TAG_LOGIT_BASE = 5
TAG_LOGIT_ROW = 6
TAG_BODY = 7
TAG_RESIDUAL = 8


@dataclass(frozen=True)
class Shape:
    """Layer shape: hidden size, expert width, routed experts, top-k, scale group, shared experts."""

    d_model: int
    d_ff: int
    n_experts: int
    top_k: int
    group: int = 32
    n_shared: int = 0

    @property
    def mxfp4_slab_bytes(self) -> int:
        """Bytes of one MXFP4 expert slab: three matrices of d*f 4-bit codes plus one byte per 32."""
        per_matrix = self.d_model * self.d_ff // 2 + self.d_model * self.d_ff // self.group
        return 3 * per_matrix

    @property
    def q8_0_slab_bytes(self) -> int:
        """Bytes of one Q8_0 expert slab: three matrices of d*f int8 plus one fp16 per 32."""
        per_matrix = self.d_model * self.d_ff + 2 * self.d_model * self.d_ff // self.group
        return 3 * per_matrix


# The small layer used for exhaustive checks, and the Kimi-shaped layer.
TINY = Shape(d_model=256, d_ff=64, n_experts=32, top_k=4, group=32, n_shared=0)
KIMI = Shape(d_model=7168, d_ff=1536, n_experts=896, top_k=16, group=32, n_shared=2)

# E8M0 exponents drawn for the synthetic experts (2^-7 .. 2^0).
SCALE_LO, SCALE_HI = 120, 127


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _mix_int(z: int) -> int:
    z &= _MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def stream_key(seed: int, *parts: int) -> int:
    """Key of one independent stream, from the seed and a tuple of small integers."""
    k = _mix_int(seed * 0x9E3779B97F4A7C15 + 0x632BE59BD9B4E019)
    for p in parts:
        k = _mix_int(k + (int(p) + 1) * 0x9E3779B97F4A7C15)
    return k


def u64(key: int, start: int, n: int) -> np.ndarray:
    """Outputs start .. start+n-1 of the stream ``key`` as uint64."""
    with np.errstate(over="ignore"):
        c = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        return _mix64(np.uint64(key) + c * _GOLDEN)


def uniform01(key: int, start: int, n: int) -> np.ndarray:
    """Uniform doubles in [0, 1) with 53 random bits."""
    return (u64(key, start, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(key: int, n: int) -> np.ndarray:
    """n standard normal doubles (Box-Muller on two uniforms per sample)."""
    r = u64(key, 0, 2 * n)
    a = ((r[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    b = (r[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    return np.sqrt(-2.0 * np.log(a)) * np.cos(2.0 * math.pi * b)


def _to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float -> bf16 bit pattern, via float32, rounding to nearest even."""
    b = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_normal(key: int, shape: tuple, sigma: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return _to_bf16_bits(normal(key, n) * sigma).reshape(shape)


# ---------------------------------------------------------------------------
# activations, router, logits
# ---------------------------------------------------------------------------

def x_rows(seed: int, rows, d_model: int, tag: int = TAG_X) -> np.ndarray:
    """bf16 N(0,1) activation rows (uint16 bits) [len(rows)][d]; row r is its own stream."""
    rows = list(rows)
    out = np.empty((len(rows), d_model), dtype=np.uint16)
    for i, r in enumerate(rows):
        out[i] = bf16_normal(stream_key(seed, tag, r), (d_model,))
    return out


def router_weight(seed: int, shape: Shape, sigma: float = 0.02, layer: int = 0) -> np.ndarray:
    """bf16 router matrix W_r [E][d] (uint16 bits), N(0, sigma)."""
    return bf16_normal(stream_key(seed, TAG_ROUTER, layer), (shape.n_experts, shape.d_model), sigma)


def block_logits(seed: int, n_rows: int, n_experts: int, sigma: float, block: int = 0) -> np.ndarray:
    """Router logits of a verification block: a base N(0,1) vector shared by the block
    plus per-row N(0, sigma) noise, as float32 [N][E]."""
    base = normal(stream_key(seed, TAG_LOGIT_BASE, block), n_experts)
    noise = normal(stream_key(seed, TAG_LOGIT_ROW, block), n_rows * n_experts).reshape(n_rows, n_experts)
    return (base[None, :] + sigma * noise).astype(np.float32)


def independent_logits(seed: int, n_rows: int, n_experts: int, block: int = 0) -> np.ndarray:
    """Independent N(0,1) router logits per row (prefill workload), float32 [N][E]."""
    return normal(stream_key(seed, TAG_LOGIT_ROW, 1000 + block), n_rows * n_experts).reshape(
        n_rows, n_experts).astype(np.float32)


# ---------------------------------------------------------------------------
# expert slabs
# ---------------------------------------------------------------------------

def _random_bytes(key: int, nbytes: int) -> np.ndarray:
    n64 = (nbytes + 7) // 8
    return u64(key, 0, n64).view(np.uint8)[:nbytes]


def mxfp4_expert_slab(seed: int, expert: int, shape: Shape, layer: int = 0,
                      scale_lo: int = SCALE_LO, scale_hi: int = SCALE_HI,
                      key: int | None = None) -> np.ndarray:
    """One MXFP4 expert slab (uint8 [slab_bytes]).

    Planes, in order: gate codes [f][d/2], gate scales [f][d/32], up codes [f][d/2],
    up scales [f][d/32], down codes [d][f/2], down scales [d][f/32].  Codes are
    uniform over all 16 E2M1 nibbles (low nibble = even K index); each scale byte is
    an E8M0 exponent uniform in [scale_lo, scale_hi].
    """
    d, f, g = shape.d_model, shape.d_ff, shape.group
    if key is None:
        key = stream_key(seed, TAG_EXPERT, layer, expert)
    slab = _random_bytes(key, shape.mxfp4_slab_bytes).copy()
    span = scale_hi - scale_lo + 1
    sizes = [(f * d // 2, f * d // g), (f * d // 2, f * d // g), (d * f // 2, d * f // g)]
    off = 0
    for codes, scales in sizes:
        off += codes
        sc = slab[off:off + scales]
        if span & (span - 1) == 0:
            sc[:] = scale_lo + (sc & (span - 1))
        else:
            sc[:] = scale_lo + (sc % span)
        off += scales
    assert off == slab.size
    return slab


def body_of(layer: int, expert: int, n_bodies: int = 1024) -> int:
    """Which of the n_bodies distinct expert bodies (layer, expert) maps to."""
    return stream_key(0x5EED, TAG_BODY, layer, expert) % n_bodies


def mxfp4_body_slab(seed: int, body: int, shape: Shape) -> np.ndarray:
    """Expert slab number ``body`` of the pool of distinct bodies used by stacked layers."""
    return mxfp4_expert_slab(seed, 0, shape, key=stream_key(seed, TAG_BODY, body))


def q8_0_shared_slab(seed: int, index: int, shape: Shape, layer: int = 0) -> np.ndarray:
    """One Q8_0 shared-expert slab (uint8 [slab_bytes]).

    Planes, in order: gate q [f][d] int8, gate d [f][d/32] fp16, up q, up d,
    down q [d][f] int8, down d [d][f/32] fp16.  q is uniform over [-127, 127];
    d is uniform in [1e-3, 1e-2] rounded to fp16.
    """
    d, f, g = shape.d_model, shape.d_ff, shape.group
    key = stream_key(seed, TAG_SHARED, layer, index)
    out = np.empty(shape.q8_0_slab_bytes, dtype=np.uint8)
    off = 0
    for plane, (nq, nd) in enumerate([(f * d, f * d // g), (f * d, f * d // g), (d * f, d * f // g)]):
        kq = stream_key(key, 2 * plane)
        kd = stream_key(key, 2 * plane + 1)
        q = (u64(kq, 0, nq) % np.uint64(255)).astype(np.int16) - 127
        out[off:off + nq] = q.astype(np.int8).view(np.uint8)
        off += nq
        dv = (1e-3 + 9e-3 * uniform01(kd, 0, nd)).astype(np.float16)
        out[off:off + 2 * nd] = dv.view(np.uint8)
        off += 2 * nd
    assert off == out.size
    return out


def mxfp4_slabs_parallel(seed: int, experts, shape: Shape, layer: int = 0, threads: int = 8):
    """Generate several expert slabs concurrently (numpy releases the GIL); yields (expert, slab)
    in order, keeping at most 2*threads slabs in flight."""
    experts = list(experts)
    window = 2 * threads
    with ThreadPoolExecutor(max_workers=threads) as ex:
        futs = {}
        for i in range(min(window, len(experts))):
            futs[i] = ex.submit(mxfp4_expert_slab, seed, experts[i], shape, layer)
        for i, e in enumerate(experts):
            slab = futs.pop(i).result()
            j = i + window
            if j < len(experts):
                futs[j] = ex.submit(mxfp4_expert_slab, seed, experts[j], shape, layer)
            yield e, slab
