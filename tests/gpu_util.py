"""Helpers of the GPU parity tests: build seeded layers on the device through the
public layer object, run the oracle on the same inputs, and compare."""

from __future__ import annotations

import numpy as np
import torch

import moe_synth as syn
from mxfp4_mixture_experts_router_gb300 import binding as B
from mxfp4_mixture_experts_router_gb300 import build as build_mod
from mxfp4_mixture_experts_router_gb300.layer import MoeLayer
from oracle import moe_oracle as orc

# Tolerance of the floating-point outputs against the oracle (relative L2 error and
# per-element error relative to the oracle's rms).
REL_L2 = 2e-3
ELEM_RMS = 1e-2


def ensure_built():
    build_mod.build()
    B.lib()


class SeededLayer:
    """A MoeLayer filled with the seeded synthetic weights of one shape, plus the
    host copies the oracle reads."""

    def __init__(self, shape: syn.Shape, seed: int, n_rows_max: int, experts=None, slot_perm=None,
                 router_sigma: float = 0.02, n_shared: int | None = None,
                 scale_range=(syn.SCALE_LO, syn.SCALE_HI)):
        ensure_built()
        self.shape = shape
        self.seed = seed
        self.scale_range = scale_range
        self.n_shared = shape.n_shared if n_shared is None else n_shared
        E = shape.n_experts
        self.experts = list(range(E)) if experts is None else sorted(set(int(e) for e in experts))
        self.layer = MoeLayer(shape.d_model, shape.d_ff, E, shape.top_k, n_rows_max, self.n_shared)
        self.router_bits = syn.router_weight(seed, shape, sigma=router_sigma)
        self.layer.set_router(torch.from_numpy(self.router_bits.view(np.int16)).view(torch.uint16))
        n_slots = len(self.experts)
        order = list(range(n_slots)) if slot_perm is None else list(slot_perm)
        self.layer.alloc_pool(n_slots)
        self.slabs = {}
        slots = np.zeros(E, dtype=np.int32)
        for i, e in enumerate(self.experts):
            slab = syn.mxfp4_expert_slab(seed, e, shape, scale_lo=scale_range[0], scale_hi=scale_range[1])
            self.slabs[e] = slab
            slot = order[i]
            self.layer.put_slab(slot, slab)
            slots[e] = slot
        self.layer.set_expert_slots(slots)
        self.shared = [syn.q8_0_shared_slab(seed, s, shape) for s in range(self.n_shared)]
        if self.n_shared:
            self.layer.set_shared(self.shared)

    def get_slab(self, e):
        if e not in self.slabs:
            self.slabs[e] = syn.mxfp4_expert_slab(self.seed, e, self.shape, scale_lo=self.scale_range[0],
                                                  scale_hi=self.scale_range[1])
        return self.slabs[e]

    def run(self, x_bits: np.ndarray, res_bits: np.ndarray, logits=None, mode=B.MOE_MODE_DECODE):
        x = to_dev_u16(x_bits)
        r = to_dev_u16(res_bits)
        lg = None if logits is None else torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
        out = self.layer.forward(x, r, logits_in=lg, mode=mode)
        torch.cuda.synchronize()
        n = x_bits.shape[0]
        return dict(out=out.view(torch.int16).cpu().numpy().view(np.uint16).copy(),
                    idx=self.layer.topk_idx[:n].cpu().numpy().copy(),
                    w=self.layer.topk_w[:n].cpu().numpy().copy(),
                    logits=self.layer.logits[:n].cpu().numpy().copy(),
                    y=self.layer.y_part[:n].cpu().numpy().copy())

    def oracle(self, x_bits, res_bits, logits=None, out_cols=None):
        return orc.moe_layer(x_bits, res_bits, self.shape, self.get_slab,
                             router_w_bits=self.router_bits if logits is None else None,
                             logits=logits, shared_slabs=self.shared[:self.n_shared], out_cols=out_cols)


def to_dev_u16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.uint16)


def bf16_to_f64(bits):
    return orc.bf16_bits_to_float(bits)


def assert_close_to_oracle(out_bits, oracle, what=""):
    """GPU bf16 output against the oracle (a dict slice with the float64 `out` and its
    bf16 rounding `out_bf16`).  Relative L2 is taken against the rounded oracle.  The
    per-element bar |err| <= 1e-2 * rms applies to the layer's value before the final
    bf16 rounding: through the bf16 output that is |out - exact| <= 1e-2 * rms + half a
    bf16 ulp of the exact value (round-to-nearest adds at most that half ulp, so two
    correct implementations can round the same element to neighbouring bf16 values)."""
    got = bf16_to_f64(out_bits)
    exact = np.asarray(oracle["out"], np.float64)
    want = bf16_to_f64(oracle["out_bf16"])
    assert np.all(np.isfinite(got)), what
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    rms = np.sqrt(np.mean(exact ** 2))
    _, e = np.frexp(exact)
    half_ulp = np.where(exact != 0, np.ldexp(1.0, e - 9), 0.0)
    excess = np.abs(got - exact) - half_ulp
    worst = excess.max() / rms
    assert rel <= REL_L2, f"{what}: relative L2 {rel:.3e} > {REL_L2}"
    assert worst <= ELEM_RMS, f"{what}: max (|err| - ulp/2)/rms {worst:.3e} > {ELEM_RMS}"
    return rel, worst


def topk_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Distance between the k-th and (k+1)-th largest logit of each row."""
    s = -np.sort(-np.asarray(logits, np.float64), axis=1)
    if s.shape[1] <= k:
        return np.full(s.shape[0], np.inf)
    return s[:, k - 1] - s[:, k]
