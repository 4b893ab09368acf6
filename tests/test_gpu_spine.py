"""Q8_0 spine matmuls at attention-projection shapes (q8_0_block_matmul), through the
C ABI, against the CPU oracle, for blocks of 1, 8 and 16 rows.

Page: "Run Kimi 3.1 locally on one GPU", section "A drafter that leaves the answer
unchanged": the spine's matrix multiplies load each weight once for up to eight
rows, and a block's rows run the same arithmetic as plain steps.  The pages give no
attention dimensions; the shapes are the projections of a 7168-wide MLA attention
block with a 1536-wide query latent, 64 heads of 192 (query) and 128 (value)."""

import numpy as np
import pytest
import torch

import moe_synth as syn
from gpu_util import ensure_built, to_dev_u16
from mxfp4_mixture_experts_router_gb300 import binding as B
from oracle import moe_oracle as orc

pytestmark = pytest.mark.gpu

# (k_in, n_out): query down-projection, query up-projection, output projection
SHAPES = [(7168, 1536), (1536, 12288), (8192, 7168)]


def _weights(k_in, n_out, seed):
    sh = syn.Shape(d_model=n_out, d_ff=k_in, n_experts=1, top_k=1, n_shared=1)
    q, dq = orc.q8_0_planes(syn.q8_0_shared_slab(seed, 0, sh), n_out, k_in)["down"]
    return q, dq


def _run(n, k_in, n_out, x_dev, q_dev, d_dev):
    ws = torch.zeros(B.q8_0_workspace_size(n, k_in, n_out), dtype=torch.uint8, device="cuda")
    y = torch.zeros((n, n_out), dtype=torch.float32, device="cuda")
    B.q8_0_block_matmul(n, k_in, n_out, x_dev, B.MOE_DTYPE_BF16, q_dev, d_dev, None, None, B.MOE_EPI_NONE, y, ws)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("k_in,n_out", SHAPES)
def test_spine_projection_matches_oracle_and_rows_are_block_invariant(k_in, n_out):
    ensure_built()
    q, dq = _weights(k_in, n_out, seed=k_in + n_out)
    q_dev = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    d_dev = torch.from_numpy(np.ascontiguousarray(dq).view(np.int16)).cuda()
    w = orc.dequant_q8_0(q, dq)
    x = syn.x_rows(40 + k_in, range(16), k_in)
    xf = orc.bf16_bits_to_float(x)
    single = [_run(1, k_in, n_out, to_dev_u16(x[r:r + 1]), q_dev, d_dev)[0] for r in range(16)]
    for n in (1, 8, 16):
        y = _run(n, k_in, n_out, to_dev_u16(x[:n]), q_dev, d_dev)
        want = xf[:n] @ w.T
        rel = np.linalg.norm(y - want) / np.linalg.norm(want)
        assert rel < 1e-5, (n, rel)
        assert np.abs(y - want).max() <= 1e-4 * np.sqrt(np.mean(want ** 2)) + 1e-30, n
        for r in range(n):  # a row of the block is the row run alone, bit for bit
            assert np.array_equal(y[r].view(np.uint32), single[r].view(np.uint32)), (n, r)
