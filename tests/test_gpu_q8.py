"""GPU parity of the stand-alone Q8_0 block matmul (q8_0_block_matmul) through the C ABI."""

import numpy as np
import pytest
import torch

import moe_synth as syn
from gpu_util import ensure_built, to_dev_u16
from mxfp4_mixture_experts_router_gb300 import binding as B
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu


def _planes(d_model, d_ff, seed):
    sh = syn.Shape(d_model=d_model, d_ff=d_ff, n_experts=1, top_k=1, n_shared=1)
    slab = syn.q8_0_shared_slab(seed, 0, sh)
    return orc.q8_0_planes(slab, d_model, d_ff)


def _dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return t.cuda().view(dtype) if dtype is not None else t.cuda()


def _run(n, k_in, n_out, x, x_dtype, q, dq, q2, d2, epi, y=None):
    ensure_built()
    ws = torch.zeros(B.q8_0_workspace_size(n, k_in, n_out), dtype=torch.uint8, device="cuda")
    if y is None:
        y = torch.zeros((n, n_out), dtype=torch.float32, device="cuda")
    B.q8_0_block_matmul(n, k_in, n_out, x, x_dtype, q, dq, q2, d2, epi, y, ws)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("n", [1, 5, 16])
@pytest.mark.parametrize("k_in,n_out", [(256, 128), (1536, 7168), (7168, 1536)])
def test_plain_matmul_bf16(n, k_in, n_out):
    # the down plane of a (d=n_out, f=k_in) slab is [n_out][k_in]
    pl = _planes(n_out, k_in, seed=n + k_in)["down"]
    q, dq = pl
    x = syn.x_rows(20, range(n), k_in)
    y = _run(n, k_in, n_out, to_dev_u16(x), B.MOE_DTYPE_BF16, _dev(q, None), _dev(dq.view(np.int16), torch.int16),
             None, None, B.MOE_EPI_NONE)
    want = orc.bf16_bits_to_float(x) @ orc.dequant_q8_0(q, dq).T
    rel = np.linalg.norm(y - want) / np.linalg.norm(want)
    assert rel < 1e-5, rel


# 1536 -> 7168 runs unsplit; 7168 -> 1536 has few 64-row items and splits K (the
# ranges' sums are added by the last item of each row block, then accumulated into y)
@pytest.mark.parametrize("k_in,n_out", [(1536, 7168), (7168, 1536)])
@pytest.mark.parametrize("n", [1, 16])
def test_plain_matmul_f32_input_and_accumulate(n, k_in, n_out):
    q, dq = _planes(n_out, k_in, seed=3)["down"]
    rng = np.random.default_rng(n)
    xf = (rng.standard_normal((n, k_in)) * 1e4).astype(np.float32)  # h-like magnitudes
    y0 = rng.standard_normal((n, n_out)).astype(np.float32)
    y = torch.from_numpy(y0.copy()).cuda()
    got = _run(n, k_in, n_out, torch.from_numpy(xf).cuda(), B.MOE_DTYPE_F32, _dev(q, None),
               _dev(dq.view(np.int16), torch.int16), None, None, B.MOE_EPI_ACCUM, y=y)
    want = y0.astype(np.float64) + xf.astype(np.float64) @ orc.dequant_q8_0(q, dq).T
    rel = np.linalg.norm(got - want) / np.linalg.norm(want)
    assert rel < 1e-5, rel


# 7168 -> 128: two 64-row blocks, K split into ranges of one 256-wide chunk each
@pytest.mark.parametrize("k_in,n_out", [(512, 128), (7168, 128)])
def test_plain_matmul_integer_exact(k_in, n_out):
    """Unit scales and integer activations: every product and sum is exact (|partial
    sums| < 127 * 6 * 7168 < 2^24), whatever the split of K."""
    n = 4
    q = np.random.default_rng(1).integers(-127, 128, size=(n_out, k_in)).astype(np.int8)
    dq = np.full((n_out, k_in // 32), 0x3C00, dtype=np.uint16)  # fp16 1.0
    xi = np.random.default_rng(2).integers(-6, 7, size=(n, k_in))
    x = orc.float_to_bf16_bits(xi.astype(np.float64))
    y = _run(n, k_in, n_out, to_dev_u16(x), B.MOE_DTYPE_BF16, _dev(q, None), _dev(dq.view(np.int16), torch.int16),
             None, None, B.MOE_EPI_NONE)
    want = (xi.astype(np.int64) @ q.astype(np.int64).T).astype(np.float32)
    assert np.array_equal(y, want)


@pytest.mark.parametrize("n", [1, 7, 16])
def test_swiglu_matches_oracle(n):
    d, f = 7168, 1536
    pl = _planes(d, f, seed=4)
    (qg, dg), (qu, du) = pl["gate"], pl["up"]
    x = syn.x_rows(21, range(n), d)
    y = _run(n, d, f, to_dev_u16(x), B.MOE_DTYPE_BF16, _dev(qg, None), _dev(dg.view(np.int16), torch.int16),
             _dev(qu, None), _dev(du.view(np.int16), torch.int16), B.MOE_EPI_SWIGLU)
    xf = orc.bf16_bits_to_float(x)
    g = xf @ orc.dequant_q8_0(qg, dg).T
    u = xf @ orc.dequant_q8_0(qu, du).T
    want = orc.silu(g) * u
    rel = np.linalg.norm(y - want) / np.linalg.norm(want)
    assert rel < 1e-5, rel


def test_rows_do_not_depend_on_the_block():
    d, f = 7168, 1536
    pl = _planes(d, f, seed=5)
    (qg, dg), (qu, du) = pl["gate"], pl["up"]
    x = syn.x_rows(22, range(16), d)
    args = (_dev(qg, None), _dev(dg.view(np.int16), torch.int16), _dev(qu, None), _dev(du.view(np.int16), torch.int16))
    blk = _run(16, d, f, to_dev_u16(x), B.MOE_DTYPE_BF16, *args, B.MOE_EPI_SWIGLU)
    for r in (0, 7, 15):
        one = _run(1, d, f, to_dev_u16(x[r:r + 1]), B.MOE_DTYPE_BF16, *args, B.MOE_EPI_SWIGLU)
        assert np.array_equal(one[0].view(np.uint32), blk[r].view(np.uint32)), r


def test_plain_matmul_reuses_its_workspace():
    """Consecutive calls on one workspace with K split (7168 -> 1536) give the result
    of a fresh workspace, bit for bit: every call leaves the arrival counters of its
    split row blocks at zero."""
    ensure_built()
    k_in, n_out, n = 7168, 1536, 8
    q, dq = _planes(n_out, k_in, seed=6)["down"]
    args = (_dev(q, None), _dev(dq.view(np.int16), torch.int16), None, None, B.MOE_EPI_NONE)
    x = to_dev_u16(syn.x_rows(23, range(n), k_in))
    want = _run(n, k_in, n_out, x, B.MOE_DTYPE_BF16, *args)
    ws = torch.zeros(B.q8_0_workspace_size(n, k_in, n_out), dtype=torch.uint8, device="cuda")
    for rep in range(4):
        y = torch.full((n, n_out), float("nan"), dtype=torch.float32, device="cuda")
        B.q8_0_block_matmul(n, k_in, n_out, x, B.MOE_DTYPE_BF16, *args, y, ws)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().view(np.uint32), want.view(np.uint32)), rep
    assert B.moe_get_error(ws) == 0
