"""Parity of the quantized GEMM D = Q(A) Q(B)^T with the oracle's fp64 product
of the dequantized operands (UFP4 summary, section 方法, Eq. of the quantized
GEMM), called through the C ABI.  Bar: exact where every partial sum is an
integer below 2^24, else relative Frobenius error <= 1e-5."""
import numpy as np
import pytest
import torch

import oracle as orc
from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import gpu_quantize, to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-5
BLOCKS = [(1, 16), (1, 32), (32, 32)]


def _pack(nib):
    return (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)


def _rand_operand(rng, rows, K, grid, block, lo=127, hi=127):
    nib = rng.integers(0, 16, size=(rows, K)).astype(np.uint8)
    if grid == "int4":
        nib[nib == 8] = 0  # -8 is not a level
    sc = rng.integers(lo, hi + 1, size=(rows // block[0] if block[0] > 1 else rows, K // block[1])).astype(np.uint8)
    if block[0] > 1:
        sc = sc[: (rows + block[0] - 1) // block[0]]
    return _pack(nib), sc


def _gemm(ac, asc, bc, bsc, M, N, K, grid, block):
    desc = ufp4.make_desc(grid=grid, block=block, scale_fmt=ufp4.SCALE_UE8M0)
    dev = "cuda"
    A = [torch.from_numpy(ac).to(dev), torch.from_numpy(asc).to(dev)]
    B = [torch.from_numpy(bc).to(dev), torch.from_numpy(bsc).to(dev)]
    D = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(max(1, ufp4.ufp4_gemm_workspace_size(M, N, K, desc)), dtype=torch.uint8, device=dev)
    ufp4.ufp4_gemm(ufp4.qtensor(*A, M, K), ufp4.qtensor(*B, N, K), desc, D, ws)
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    return D.cpu().numpy().astype(np.float64)


def _rel(D, ref):
    return np.linalg.norm(D - ref) / max(np.linalg.norm(ref), 1e-300)


FP8_GRIDS = ("e1m2", "int4")


@pytest.mark.parametrize("block", [(1, 16), (1, 32), (32, 32)])
@pytest.mark.parametrize("shape", [(2560, 2304, 4096), (2500, 2200, 4160)])
def test_gemm_exact_integer_wide_fp4_tiles(shape, block):
    """Long K (16 or more K tiles): E2M1 1 x 16 takes the 256 x 256 tiles with
    one accumulator, 1 x 32 and 32 x 32 the 2X kind's double-buffered 256 x 224
    tiles.  More output tiles than CTA pairs (ragged in the second shape), so
    each pair hands its accumulators from one tile's epilogue to the next
    tile's MMAs.  Unit scales: exact."""
    rng = np.random.default_rng(23)
    M, N, K = shape
    if block[0] > 1:
        M, N = (M + 31) // 32 * 32, (N + 31) // 32 * 32
    ac, asc = _rand_operand(rng, M, K, "e2m1", block)
    bc, bsc = _rand_operand(rng, N, K, "e2m1", block)
    D = _gemm(ac, asc, bc, bsc, M, N, K, "e2m1", block)
    ref = orc.gemm_reference(ac, asc, bc, bsc, grid="e2m1", block=block)
    np.testing.assert_array_equal(D, ref)


@pytest.mark.parametrize("grid", FP8_GRIDS + ("e2m1", "e2m1r2"))
@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("shape", [(128, 256, 128), (256, 512, 512), (200, 300, 384), (200, 300, 160)])
def test_gemm_exact_integer_case(grid, block, shape):
    """Unit scales: every product and partial sum is an exact small dyadic,
    so the tensor-core result equals the fp64 reference bit for bit.  K = 160
    gives 5 or 10 scale bytes per row (odd rows start unaligned) and a partly
    filled last 128-element scale chunk."""
    M, N, K = shape
    if grid.startswith("e2m1") and K % 64:
        pytest.skip("FP4 operands need K % 64 == 0")
    if block[0] > 1 and (M % 32 or N % 32):
        M, N = (M + 31) // 32 * 32, (N + 31) // 32 * 32
    rng = np.random.default_rng(M + N + K)
    ac, asc = _rand_operand(rng, M, K, grid, block)
    bc, bsc = _rand_operand(rng, N, K, grid, block)
    D = _gemm(ac, asc, bc, bsc, M, N, K, grid, block)
    ref = orc.gemm_reference(ac, asc, bc, bsc, grid=grid, block=block)
    np.testing.assert_array_equal(D, ref)


@pytest.mark.parametrize("grid", FP8_GRIDS + ("e2m1",))
@pytest.mark.parametrize("block", BLOCKS)
@pytest.mark.parametrize("shape", [(384, 512, 1024), (200, 300, 160)])
def test_gemm_random_scales(grid, block, shape):
    """Block scales spread over 2^-9 .. 2^7 (pairs of 1 x 16 blocks differ by up
    to 16 binades, the exact range of the E5M2 fold).  K = 160: rows of 5 or 10
    scale bytes, so the scale bytes of odd rows start unaligned."""
    M, N, K = shape
    if grid.startswith("e2m1") and K % 64:
        pytest.skip("FP4 operands need K % 64 == 0")
    if block[0] > 1 and (M % 32 or N % 32):
        M, N = (M + 31) // 32 * 32, (N + 31) // 32 * 32
    rng = np.random.default_rng(31)
    ac, asc = _rand_operand(rng, M, K, grid, block, lo=118, hi=134)
    bc, bsc = _rand_operand(rng, N, K, grid, block, lo=118, hi=134)
    D = _gemm(ac, asc, bc, bsc, M, N, K, grid, block)
    ref = orc.gemm_reference(ac, asc, bc, bsc, grid=grid, block=block)
    assert _rel(D, ref) <= TOL


@pytest.mark.parametrize("grid", FP8_GRIDS)
def test_gemm_wide_scale_gap(grid):
    """Neighbouring 1 x 16 blocks 27 binades apart: the smaller block's
    elements fall below E5M2's range and round.  Besides the relative bar, each
    output stays within the stated bound: per product term at most 2^-17 of
    the pair's hardware scale (2^(e_max - 2) for E1M2, 2^e_max for INT4) times
    |B|, plus the fp32 accumulation."""
    M, N, K = 256, 256, 512
    rng = np.random.default_rng(5)
    ac, asc = _rand_operand(rng, M, K, grid, (1, 16), lo=127, hi=127)
    bc, bsc = _rand_operand(rng, N, K, grid, (1, 16), lo=127, hi=127)
    asc[:, 1::2] = 100
    D = _gemm(ac, asc, bc, bsc, M, N, K, grid, (1, 16))
    ref = orc.gemm_reference(ac, asc, bc, bsc, grid=grid, block=(1, 16))
    assert _rel(D, ref) <= TOL
    da = orc.dequantize_f64(ac, asc, grid=grid, block=(1, 16))
    db = orc.dequantize_f64(bc, bsc, grid=grid, block=(1, 16))
    e = asc.astype(np.int64) - 127
    e_pair = np.maximum(e[:, 0::2], e[:, 1::2])                       # per 32 elements
    gap = np.repeat(e_pair, 2, axis=1) - e                            # binades below the pair's max
    hw = 2.0 ** (np.repeat(e_pair, 2, axis=1) - (2 if grid == "e1m2" else 0))
    term = np.where(gap > 16, 2.0 ** -17 * hw, 0.0)  # per 16-element block: exact up to 16 binades
    bound = np.repeat(term, 16, axis=1) @ np.abs(db).T
    slack = 2.0 ** -20 * (np.abs(da) @ np.abs(db).T)
    assert (np.abs(D - ref) <= bound + slack).all()


def _quantized(x, grid, block, colwise=False, rounding=orc.RTNE):
    kw = dict(grid=grid, block=block, n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=orc.SCALE_UE8M0,
              rounding=rounding, sr_seed=inputs.SR_SEED)
    got = gpu_quantize(to_dev(x), out_mask=ufp4.OUT_COLWISE if colwise else ufp4.OUT_ROWWISE, **kw)
    return got["col" if colwise else "row"]


@pytest.mark.parametrize("grid", FP8_GRIDS + ("e2m1", "e2m1r2"))
def test_fprop_dense_small(grid):
    x, w = inputs.dense_fprop(m=1024, n=768, k=2048)
    ac, asc = _quantized(x, grid, (1, 16))
    bc, bsc = _quantized(w, grid, (1, 16))
    D = _gemm(ac, asc, bc, bsc, 1024, 768, 2048, grid, (1, 16))
    ref = orc.gemm_reference(ac, asc, bc, bsc, grid=grid, block=(1, 16))
    assert _rel(D, ref) <= TOL


def test_fprop_dense_full_size():
    """Dense-1.5B-like FPROP Y = X W^T (8192 x 5632 x 2048), E1M2 1 x 16 RTNE."""
    x, w = inputs.dense_fprop()
    ac, asc = _quantized(x, "e1m2", (1, 16))
    bc, bsc = _quantized(w, "e1m2", (1, 16))
    D = _gemm(ac, asc, bc, bsc, 8192, 5632, 2048, "e1m2", (1, 16))
    ref = orc.gemm_reference(ac, asc, bc, bsc, grid="e1m2", block=(1, 16))
    assert _rel(D, ref) <= TOL


def test_dgrad_and_wgrad_from_one_pass():
    """dY (1e-3 Student-t, SR) row-wise feeds DGRAD dX = dY W (B = W column-wise);
    its column-wise copy feeds WGRAD dW = dY^T X (B = X column-wise)."""
    m, n, k = 2048, 1024, 768
    dy = inputs.student_t_bf16(m, n, 301)
    w = inputs.normal_bf16(n, k, 302, std=0.02)
    x = inputs.normal_bf16(m, k, 303)
    desc_sr = dict(grid="e1m2", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=orc.SCALE_UE8M0,
                   rounding=orc.SR, sr_seed=inputs.SR_SEED)
    both = gpu_quantize(to_dev(dy), out_mask=3, **desc_sr)
    wc, wsc = _quantized(w, "e1m2", (1, 16), colwise=True)     # [k x n]
    xc, xsc = _quantized(x, "e1m2", (1, 16), colwise=True)     # [k x m]
    # DGRAD: [m x n] . [k x n]^T
    D = _gemm(*both["row"], wc, wsc, m, k, n, "e1m2", (1, 16))
    ref = orc.gemm_reference(*both["row"], wc, wsc, grid="e1m2", block=(1, 16))
    assert _rel(D, ref) <= TOL
    # WGRAD: [n x m] . [k x m]^T
    D = _gemm(*both["col"], xc, xsc, n, k, m, "e1m2", (1, 16))
    ref = orc.gemm_reference(*both["col"], xc, xsc, grid="e1m2", block=(1, 16))
    assert _rel(D, ref) <= TOL


@pytest.mark.parametrize("grid,block", [("e1m2", (1, 16)), ("int4", (32, 32)), ("e2m1", (1, 16)),
                                        ("e2m1", (32, 32))])
def test_large_fprop_sampled_rows(grid, block):
    """MoE-124B-like FPROP 16384 x 7168 x 7168 checked on 256 seeded rows of D."""
    x, w = inputs.large_sweep()
    ac, asc = _quantized(x, grid, block)
    bc, bsc = _quantized(w, grid, block)
    D = torch.empty((16384, 7168), dtype=torch.float32, device="cuda")
    desc = ufp4.make_desc(grid=grid, block=block, scale_fmt=ufp4.SCALE_UE8M0)
    A = [torch.from_numpy(ac).cuda(), torch.from_numpy(asc).cuda()]
    B = [torch.from_numpy(bc).cuda(), torch.from_numpy(bsc).cuda()]
    ws = torch.empty(max(1, ufp4.ufp4_gemm_workspace_size(16384, 7168, 7168, desc)), dtype=torch.uint8, device="cuda")
    ufp4.ufp4_gemm(ufp4.qtensor(*A, 16384, 7168), ufp4.qtensor(*B, 7168, 7168), desc, D, ws)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(7).choice(16384, 256, replace=False))
    got = D[torch.from_numpy(rows).cuda()].cpu().numpy().astype(np.float64)
    ref = orc.gemm_reference(ac, asc, bc, bsc, grid=grid, block=block, a_rows=rows)
    assert _rel(got, ref) <= TOL


@pytest.mark.parametrize("grid", ["e1m2", "e2m1"])
def test_prepare_then_prepared_equals_gemm(grid):
    """ufp4_gemm = ufp4_gemm_prepare + ufp4_gemm_prepared, bit for bit, and a
    prepared workspace can serve a second call."""
    M, N, K = 256, 384, 512
    rng = np.random.default_rng(77)
    ac, asc = _rand_operand(rng, M, K, grid, (1, 16), lo=120, hi=132)
    bc, bsc = _rand_operand(rng, N, K, grid, (1, 16), lo=120, hi=132)
    desc = ufp4.make_desc(grid=grid, block=(1, 16), scale_fmt=ufp4.SCALE_UE8M0)
    A = [torch.from_numpy(ac).cuda(), torch.from_numpy(asc).cuda()]
    B = [torch.from_numpy(bc).cuda(), torch.from_numpy(bsc).cuda()]
    qa, qb = ufp4.qtensor(*A, M, K), ufp4.qtensor(*B, N, K)
    ws = torch.empty(max(1, ufp4.ufp4_gemm_workspace_size(M, N, K, desc)), dtype=torch.uint8, device="cuda")
    D1 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    D2 = torch.empty_like(D1)
    D3 = torch.empty_like(D1)
    ufp4.ufp4_gemm(qa, qb, desc, D1, ws)
    ufp4.ufp4_gemm_prepare(qa, qb, desc, ws)
    ufp4.ufp4_gemm_prepared(qa, qb, desc, D2, ws)
    ufp4.ufp4_gemm_prepared(qa, qb, desc, D3, ws)
    torch.cuda.synchronize()
    assert torch.equal(D1, D2) and torch.equal(D1, D3)
