"""Diagnostics (single-tensor and GEMM-output error figures): the library's
sums against the oracle's exact fp64 sums, through the C ABI.  The library
adds 16-element fp32 partial sums (fused multiply-adds) in fp64, so the bar
is a relative difference of 1e-5; the two-matrix sums use fp32 products
(exact to 2^-24 relative) and the bar there is 1e-6."""
import numpy as np
import pytest
import torch

import oracle as orc
from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import gpu_quantize, to_dev

pytestmark = pytest.mark.gpu


def _close(a, b, tol=1e-5):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert (np.abs(a - b) <= tol * np.maximum(np.abs(b), 1e-300)).all(), (a, b)


@pytest.mark.parametrize("grid,block,n,fmt,rounding", [
    ("e1m2", (1, 16), 16, orc.SCALE_FP32, orc.RTNE),
    ("int4", (1, 32), 64, orc.SCALE_UE8M0, orc.SR),
    ("e2m1", (1, 16), 128, orc.SCALE_UE8M0, orc.RTNE),
    ("e2m1r2", (1, 16), 16, orc.SCALE_FP32, orc.SR),
    ("e2m1", (32, 32), 32, orc.SCALE_UE8M0, orc.RTNE),
    ("e1m2", (1, 16), 1, orc.SCALE_UE8M0, orc.RTNE),
])
def test_quant_error_stats_match_oracle(grid, block, n, fmt, rounding):
    x = inputs.tiny_check(320, 1024)
    kw = dict(grid=grid, block=block, n=n, sign_seed=inputs.SIGN_SEED, scale_fmt=fmt, rounding=rounding,
              sr_seed=inputs.SR_SEED)
    xd = to_dev(x)
    desc = ufp4.make_desc(out_mask=ufp4.OUT_ROWWISE, **kw)
    codes, scales = ufp4.quantize(xd, desc)["row"]
    stats = torch.zeros(4, dtype=torch.float64, device="cuda")
    ufp4.ufp4_quant_error_stats(xd, desc, ufp4.qtensor(codes, scales, 320, 1024), stats)
    torch.cuda.synchronize()
    ref = orc.quant_error_stats(x, codes.cpu().numpy(), scales.cpu().numpy(), grid=grid, block=block,
                                scale_fmt=fmt, n=n, sign_seed=inputs.SIGN_SEED)
    _close(stats.cpu().numpy(), ref)


def test_error_stats_of_two_matrices():
    rng = np.random.default_rng(3)
    a = rng.standard_normal((300, 700)).astype(np.float32)
    b = (a + 1e-3 * rng.standard_normal((300, 700))).astype(np.float32)
    A = torch.zeros((300, 768), dtype=torch.float32, device="cuda")  # padded leading dimensions
    B = torch.zeros((300, 704), dtype=torch.float32, device="cuda")
    A[:, :700] = torch.from_numpy(a)
    B[:, :700] = torch.from_numpy(b)
    stats = torch.zeros(4, dtype=torch.float64, device="cuda")
    ufp4.ufp4_error_stats(A[:, :700], B[:, :700], stats)
    torch.cuda.synchronize()
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    _close(stats.cpu().numpy(), [(a64 * a64).sum(), ((b64 - a64) ** 2).sum(), (a64 * b64).sum(), (b64 * b64).sum()],
           1e-6)


def test_gemm_output_error_against_the_fp64_reference():
    """The GEMM-output diagnostic: the quantized GEMM's fp32 output against the
    oracle's fp64 product of the dequantized operands, relative error <= 1e-5."""
    x, w = inputs.dense_fprop(m=512, n=384, k=1024)
    kw = dict(grid="e1m2", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=orc.SCALE_UE8M0)
    qa = gpu_quantize(to_dev(x), out_mask=ufp4.OUT_ROWWISE, **kw)["row"]
    qb = gpu_quantize(to_dev(w), out_mask=ufp4.OUT_ROWWISE, **kw)["row"]
    A = [torch.from_numpy(qa[0]).cuda(), torch.from_numpy(qa[1]).cuda()]
    B = [torch.from_numpy(qb[0]).cuda(), torch.from_numpy(qb[1]).cuda()]
    desc = ufp4.make_desc(grid="e1m2", block=(1, 16), scale_fmt=ufp4.SCALE_UE8M0)
    D = torch.empty((512, 384), dtype=torch.float32, device="cuda")
    ws = torch.empty(ufp4.ufp4_gemm_workspace_size(512, 384, 1024, desc), dtype=torch.uint8, device="cuda")
    ufp4.ufp4_gemm(ufp4.qtensor(*A, 512, 1024), ufp4.qtensor(*B, 384, 1024), desc, D, ws)
    ref = orc.gemm_reference(qa[0], qa[1], qb[0], qb[1], grid="e1m2", block=(1, 16))
    R = torch.from_numpy(ref.astype(np.float32)).cuda()
    stats = torch.zeros(4, dtype=torch.float64, device="cuda")
    ufp4.ufp4_error_stats(R, D, stats)
    torch.cuda.synchronize()
    s = stats.cpu().numpy()
    assert np.sqrt(s[1] / s[0]) <= 1e-5
