"""The GEMM on operands with plain fp32 block scales (the pages' s_B = amax /
qmax): bf16 per-block partials on the tensor cores, rescaled by s_A s_B on
the CUDA cores.  Against the oracle's fp64 product of the dequantized
operands: bit-exact with unit scales (every partial and sum is an exact small
dyadic), relative Frobenius error <= 1e-5 otherwise."""
import numpy as np
import pytest
import torch

import oracle as orc
from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import gpu_quantize, to_dev

pytestmark = pytest.mark.gpu
FP32 = ufp4.SCALE_FP32


def _operand(rng, rows, K, grid, bc, scales="unit"):
    nib = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
    if grid == "int4":
        nib[nib == 8] = 0
    codes = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    if scales == "unit":
        sc = np.ones((rows, K // bc), dtype=np.float32)
    else:
        sc = rng.lognormal(0.0, 2.0, size=(rows, K // bc)).astype(np.float32)
    return codes, sc


def _gemm(ac, asc, bc_, bsc, M, N, K, grid, block):
    desc = ufp4.make_desc(grid=grid, block=block, scale_fmt=FP32)
    A = [torch.from_numpy(ac).cuda(), torch.from_numpy(asc).cuda()]
    B = [torch.from_numpy(bc_).cuda(), torch.from_numpy(bsc).cuda()]
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, ufp4.ufp4_gemm_workspace_size(M, N, K, desc)), dtype=torch.uint8, device="cuda")
    ufp4.ufp4_gemm(ufp4.qtensor(*A, M, K), ufp4.qtensor(*B, N, K), desc, D, ws)
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    return D.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("grid,block", [("e1m2", (1, 16)), ("int4", (1, 32)), ("e2m1", (1, 16)),
                                        ("e2m1r2", (1, 32))])
@pytest.mark.parametrize("shape", [(128, 128, 128), (256, 384, 512), (200, 300, 640)])
def test_fp32_scale_gemm_exact_with_unit_scales(grid, block, shape):
    M, N, K = shape
    rng = np.random.default_rng(M + N + K)
    ac, asc = _operand(rng, M, K, grid, block[1])
    bc_, bsc = _operand(rng, N, K, grid, block[1])
    D = _gemm(ac, asc, bc_, bsc, M, N, K, grid, block)
    ref = orc.gemm_reference(ac, asc, bc_, bsc, grid=grid, block=block, scale_fmt=orc.SCALE_FP32)
    np.testing.assert_array_equal(D, ref)


@pytest.mark.parametrize("grid,block", [("e1m2", (1, 16)), ("int4", (1, 32)), ("e2m1", (1, 16))])
def test_fp32_scale_gemm_random_scales(grid, block):
    M, N, K = 384, 512, 1024
    rng = np.random.default_rng(41)
    ac, asc = _operand(rng, M, K, grid, block[1], scales="random")
    bc_, bsc = _operand(rng, N, K, grid, block[1], scales="random")
    D = _gemm(ac, asc, bc_, bsc, M, N, K, grid, block)
    ref = orc.gemm_reference(ac, asc, bc_, bsc, grid=grid, block=block, scale_fmt=orc.SCALE_FP32)
    assert np.linalg.norm(D - ref) / np.linalg.norm(ref) <= 1e-5


def test_fp32_scale_gemm_on_quantized_fprop():
    """X and W quantized with the pages' fp32 scales (1 x 16, E1M2, RHT n=16),
    then Y = Q(X) Q(W)^T on those scales directly."""
    x, w = inputs.dense_fprop(m=1024, n=768, k=2048)
    kw = dict(grid="e1m2", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=orc.SCALE_FP32)
    qa = gpu_quantize(to_dev(x), out_mask=ufp4.OUT_ROWWISE, **kw)["row"]
    qb = gpu_quantize(to_dev(w), out_mask=ufp4.OUT_ROWWISE, **kw)["row"]
    D = _gemm(qa[0], qa[1], qb[0], qb[1], 1024, 768, 2048, "e1m2", (1, 16))
    ref = orc.gemm_reference(qa[0], qa[1], qb[0], qb[1], grid="e1m2", block=(1, 16), scale_fmt=orc.SCALE_FP32)
    assert np.linalg.norm(D - ref) / np.linalg.norm(ref) <= 1e-5
