"""The allocation-free Q8_0 entry point (q8_0_block_matmul_noalloc).

It exists for callers that cannot allocate device memory (a process whose pool
allocator owns all of HBM, or a latency-critical path that cannot afford a
synchronising cudaMalloc).  It takes its scratch from a static device array
inside the library, so its results must match the allocating entry point
q8_0_block_matmul, call after call, even though every call reuses the array.
This file sorts last so that a run stopping at the first failure has run every
other test first.
"""

import numpy as np
import pytest
import torch

import moe_synth as syn
from gpu_util import ensure_built, to_dev_u16
from mxfp4_mixture_experts_router_gb300 import binding as B
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu


def _weights(d_model, d_ff, seed):
    sh = syn.Shape(d_model=d_model, d_ff=d_ff, n_experts=1, top_k=1, n_shared=1)
    pl = orc.q8_0_planes(syn.q8_0_shared_slab(seed, 0, sh), d_model, d_ff)
    dev = {}
    for name, (q, d) in pl.items():
        dev[name] = (torch.from_numpy(np.ascontiguousarray(q)).cuda(),
                     torch.from_numpy(np.ascontiguousarray(d).view(np.int16)).cuda())
    return dev


def _both(n, k_in, n_out, x, x_dtype, q, dq, q2, d2, epi):
    ws = torch.zeros(B.q8_0_workspace_size(n, k_in, n_out), dtype=torch.uint8, device="cuda")
    want = torch.zeros((n, n_out), dtype=torch.float32, device="cuda")
    got = torch.full((n, n_out), float("nan"), dtype=torch.float32, device="cuda")
    B.q8_0_block_matmul(n, k_in, n_out, x, x_dtype, q, dq, q2, d2, epi, want, ws)
    B.q8_0_block_matmul_noalloc(n, k_in, n_out, x, x_dtype, q, dq, q2, d2, epi, got)
    torch.cuda.synchronize()
    return got.cpu().numpy(), want.cpu().numpy()


def _close(got, want):
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert rel <= 1e-5, rel
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))


def test_noalloc_matches_allocating_entry_point_on_consecutive_calls():
    ensure_built()
    d, f = 7168, 1536
    w = _weights(d, f, seed=31)
    # call 1: SwiGLU gate/up of a 5-row block (largest K the array allows)
    x1 = to_dev_u16(syn.x_rows(31, range(5), d))
    got, want = _both(5, d, f, x1, B.MOE_DTYPE_BF16, *w["gate"], *w["up"], B.MOE_EPI_SWIGLU)
    _close(got, want)
    # call 2: a plain 16-row down projection with fp32 input, reusing the array
    h = torch.from_numpy(np.random.default_rng(32).standard_normal((16, f)).astype(np.float32) * 1e4).cuda()
    got, want = _both(16, f, d, h, B.MOE_DTYPE_F32, *w["down"], None, None, B.MOE_EPI_NONE)
    _close(got, want)
    # call 3: a plain 16-row 7168 -> 1536 projection, whose K is split (partial sums
    # and arrival counters in the array)
    x3 = to_dev_u16(syn.x_rows(33, range(16), d))
    qd, dd = w["gate"]
    for _ in range(2):
        got, want = _both(16, d, f, x3, B.MOE_DTYPE_BF16, qd, dd, None, None, B.MOE_EPI_NONE)
        _close(got, want)
    # no device-side error in any call (the error word collects them until read)
    assert B.q8_0_noalloc_get_error() == 0


def test_noalloc_rejects_sizes_beyond_its_array():
    ensure_built()
    L = B.lib()
    # 17 rows or K > 7168: refused on the host, nothing launched
    assert L.q8_0_block_matmul_noalloc(17, 7168, 1536, 256, 0, 256, 256, 256, 256, B.MOE_EPI_SWIGLU, 256,
                                       None) == B.MOE_ERR_UNSUPPORTED
    assert L.q8_0_block_matmul_noalloc(1, 7424, 1536, 256, 0, 256, 256, 256, 256, B.MOE_EPI_SWIGLU, 256,
                                       None) == B.MOE_ERR_UNSUPPORTED
