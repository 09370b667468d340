"""MXFP8 (the format the 2D-block page keeps for the Query and Key
projections, read as OCP MX: E4M3 elements, one E8M0 scale per 32) through
the C ABI: the row kernel's codes and scales bit-exact against the oracle,
dequantize bit-exact, and the FP8 tensor-core GEMM on the codes in place
within 1e-5 relative Frobenius of the oracle's fp64 product."""
import numpy as np
import pytest
import torch

import oracle as orc
from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import assert_bitwise, gpu_quantize, to_dev

pytestmark = pytest.mark.gpu
TOL = 1e-5


def _kw(n):
    return dict(grid="mxfp8", block=(1, 32), n=n, sign_seed=inputs.SIGN_SEED, scale_fmt=ufp4.SCALE_UE8M0,
                out_mask=ufp4.OUT_ROWWISE)


def _outliers(rows, cols, seed):
    return inputs.with_element_outliers(inputs.normal_bf16(rows, cols, seed), 0.001, 50.0, seed + 1)


@pytest.mark.parametrize("n", [1, 16, 32, 64, 128])
@pytest.mark.parametrize("shape", [(256, 1024), (200, 96), (130, 4096)])
def test_mxfp8_quantize_matches_oracle(n, shape):
    """Full and ragged 128 x 128 tiles (200 rows, 96 columns), n from none to 128."""
    r, c = shape
    if c % n:
        pytest.skip("n must divide the row")
    x = _outliers(r, c, 31 + r)
    got = gpu_quantize(to_dev(x), **_kw(n))["row"]
    codes, scales = orc.quantize_mxfp8(x, n=n, sign_seed=inputs.SIGN_SEED)
    assert_bitwise(got[0], codes, f"mxfp8 codes n={n} {r}x{c}")
    assert_bitwise(got[1], scales, f"mxfp8 scales n={n} {r}x{c}")


def test_mxfp8_dense_operand_and_extremes():
    """The dense FPROP X (channel outliers x30), plus rows of zeros, tiny
    values and large values (up to 1e37, so that n = 16 cannot overflow)."""
    x, _ = inputs.dense_fprop(m=1024, n=256, k=2048)
    x = x.copy()
    x[0] = 0
    x[1] = inputs.f32_to_bf16_bits(np.full(2048, -1e-30, dtype=np.float32))
    x[2] = inputs.f32_to_bf16_bits(np.linspace(-1e37, 1e37, 2048, dtype=np.float32))  # no overflow through n = 16
    got = gpu_quantize(to_dev(x), **_kw(16))["row"]
    codes, scales = orc.quantize_mxfp8(x, n=16, sign_seed=inputs.SIGN_SEED)
    assert_bitwise(got[0], codes, "mxfp8 codes")
    assert_bitwise(got[1], scales, "mxfp8 scales")


def test_mxfp8_batch_equals_single_calls():
    shapes = [(300, 576), (0, 64), (128, 1024)]
    xs = [_outliers(r, c, 41 + r) if r else np.zeros((0, c), np.uint16) for r, c in shapes]
    desc = ufp4.make_desc(**_kw(16))
    devs = [to_dev(x) for x in xs]
    bufs = [ufp4.alloc_quantized(r, c, desc, "cuda") for r, c in shapes]
    ufp4.ufp4_rht_quantize_batch(devs, desc, [ufp4.qtensor(cb, sb, r, c) for (cb, sb), (r, c) in zip(bufs, shapes)])
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    for x, (cb, sb), (r, c) in zip(xs, bufs, shapes):
        if r == 0:
            continue
        codes, scales = orc.quantize_mxfp8(x, n=16, sign_seed=inputs.SIGN_SEED)
        assert_bitwise(cb.cpu().numpy(), codes, f"batch codes {r}x{c}")
        assert_bitwise(sb.cpu().numpy(), scales, f"batch scales {r}x{c}")


def test_mxfp8_dequantize_is_exact():
    x = _outliers(128, 512, 51)
    codes, scales = orc.quantize_mxfp8(x)
    desc = ufp4.make_desc(**_kw(1))
    cb, sb = torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda()
    out = torch.empty((128, 512), dtype=torch.float32, device="cuda")
    ufp4.ufp4_dequantize(ufp4.qtensor(cb, sb, 128, 512), desc, False, out)
    torch.cuda.synchronize()
    ref = orc.dequantize_mxfp8(codes, scales)
    assert np.array_equal(out.cpu().numpy().astype(np.float64), ref)


def _gemm(ac, asc, bc, bsc, M, N, K):
    desc = ufp4.make_desc(**_kw(1))
    A = [torch.from_numpy(ac).cuda(), torch.from_numpy(asc).cuda()]
    B = [torch.from_numpy(bc).cuda(), torch.from_numpy(bsc).cuda()]
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(1, ufp4.ufp4_gemm_workspace_size(M, N, K, desc)), dtype=torch.uint8, device="cuda")
    ufp4.ufp4_gemm(ufp4.qtensor(*A, M, K), ufp4.qtensor(*B, N, K), desc, D, ws)
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    return D.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape", [(256, 448, 256), (200, 300, 96), (1024, 768, 2048)])
def test_mxfp8_gemm_matches_oracle(shape):
    """Quantized operands (Q/K-projection-like X W^T), full and ragged tiles."""
    M, N, K = shape
    x = _outliers(M, K, 61)
    w = inputs.normal_bf16(N, K, 62, std=0.02)
    ac, asc = orc.quantize_mxfp8(x, n=16, sign_seed=inputs.SIGN_SEED)
    bc, bsc = orc.quantize_mxfp8(w, n=16, sign_seed=inputs.SIGN_SEED)
    D = _gemm(ac, asc, bc, bsc, M, N, K)
    ref = orc.gemm_reference_mxfp8(ac, asc, bc, bsc)
    assert np.linalg.norm(D - ref) / np.linalg.norm(ref) <= TOL


def test_mxfp8_gemm_exact_with_unit_scales():
    """Scale byte 127 and codes of small integers: every product and partial
    sum is an integer below 2^24, so D equals the fp64 product exactly."""
    M, N, K = 256, 448, 512
    rng = np.random.default_rng(63)
    ints = np.array([orc.e4m3_encode(float(v)) for v in range(0, 8)], dtype=np.uint8)
    def op(rows):
        c = ints[rng.integers(0, 8, size=(rows, K))] | (rng.integers(0, 2, size=(rows, K)) * 0x80).astype(np.uint8)
        c[(c & 0x7F) == 0] = 0
        return c, np.full((rows, K // 32), 127, dtype=np.uint8)
    ac, asc = op(M)
    bc, bsc = op(N)
    D = _gemm(ac, asc, bc, bsc, M, N, K)
    np.testing.assert_array_equal(D, orc.gemm_reference_mxfp8(ac, asc, bc, bsc))
