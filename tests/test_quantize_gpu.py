"""Parity of the CUDA quantizer with the oracle: codes, scales and packed
bytes must be bit-exact (integer/byte work), called through the C ABI.

Sizes span several 128 x 128 tiles plus ragged tails; the full workload
shapes are checked on sampled row bands (row-wise outputs depend on their
own row only) or in full where the oracle takes seconds."""
import numpy as np
import pytest
import torch

import oracle as orc
from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import assert_bitwise, gpu_quantize, to_dev

pytestmark = pytest.mark.gpu

GRIDS = ("e1m2", "int4", "e2m1", "e2m1r2")
SR = orc.SR
RTNE = orc.RTNE
PO2 = orc.SCALE_UE8M0
FP32 = orc.SCALE_FP32


def _check(x, *, colwise_too=False, ld=None, **kw):
    """Quantize x on the GPU (row-wise, and column-wise if asked) and compare with the oracle."""
    mask = ufp4.OUT_ROWWISE | (ufp4.OUT_COLWISE if colwise_too else 0)
    got = gpu_quantize(to_dev(x, ld=ld), out_mask=mask, **kw)
    okw = dict(grid=kw.get("grid", "e1m2"), block=kw.get("block", (1, 16)), n=kw.get("n", 16),
               sign_seed=kw.get("sign_seed", 0), rounding=kw.get("rounding", RTNE),
               sr_seed=kw.get("sr_seed", 0), scale_fmt=kw.get("scale_fmt", FP32), group=kw.get("group", 0))
    c, s = orc.quantize(x, **okw)
    assert_bitwise(got["row"][0], c, "row-wise codes")
    assert_bitwise(got["row"][1], s, "row-wise scales")
    if colwise_too:
        c, s = orc.quantize(x, colwise=True, **okw)
        assert_bitwise(got["col"][0], c, "column-wise codes")
        assert_bitwise(got["col"][1], s, "column-wise scales")


# ------------------------------------------------- tiny check, every mode
@pytest.mark.parametrize("grid", GRIDS)
@pytest.mark.parametrize("scale_fmt", [FP32, PO2])
@pytest.mark.parametrize("rounding", [RTNE, SR])
def test_tiny_check_all_modes(grid, scale_fmt, rounding):
    x = inputs.tiny_check()
    _check(x, grid=grid, n=16, sign_seed=inputs.SIGN_SEED, rounding=rounding, sr_seed=inputs.SR_SEED,
           scale_fmt=scale_fmt, colwise_too=True)


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128])
@pytest.mark.parametrize("grid", GRIDS)
def test_hadamard_sizes_row_and_col(n, grid):
    x = inputs.tiny_check(256, 512)
    _check(x, grid=grid, n=n, sign_seed=77, colwise_too=True, rounding=SR, sr_seed=5)


@pytest.mark.parametrize("grid", GRIDS)
@pytest.mark.parametrize("rounding", [RTNE, SR])
def test_hadamard_256_rowwise(grid, rounding):
    x = inputs.tiny_check(128, 1024)
    _check(x, grid=grid, n=256, sign_seed=9, rounding=rounding, sr_seed=11, scale_fmt=PO2)


@pytest.mark.parametrize("block", [(1, 32), (8, 8), (16, 16), (32, 32), (64, 64)])
@pytest.mark.parametrize("n", [16, 64])
def test_block_shapes(block, n):
    x = inputs.tiny_check(256, 512)
    fmt = PO2 if block[0] > 1 else FP32
    _check(x, grid="e1m2", block=block, n=n, sign_seed=3, scale_fmt=fmt, colwise_too=True)
    _check(x, grid="e2m1", block=block, n=n, sign_seed=3, scale_fmt=PO2, colwise_too=True, rounding=SR,
           sr_seed=2)


@pytest.mark.parametrize("b", [16, 32, 64])
@pytest.mark.parametrize("n", [1, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("rounding", [RTNE, SR])
def test_2d_blocks_rowwise_kernel(b, n, rounding):
    """Row-wise b x b blocks run in the row kernels (n = 64 and 256: the segment
    kernel; otherwise the row kernel, one row pair per thread; the block amax
    reduced across lanes and warps): ragged tiles (rows and columns multiples
    of b but not of the tile), every grid."""
    rows = 3 * b + 2 * 64 if b < 64 else 320
    cols = 768 if n == 256 else 384 + 2 * b
    cols = -(-cols // max(n, b)) * max(n, b)
    x = inputs.tiny_check(rows, cols)
    for grid in GRIDS:
        _check(x, grid=grid, block=(b, b), n=n, sign_seed=5, rounding=rounding, sr_seed=13, scale_fmt=PO2)


@pytest.mark.parametrize("block", [(8, 8), (32, 32)])
def test_2d_blocks_with_n256(block):
    x = inputs.tiny_check(128, 512)
    _check(x, grid="int4", block=block, n=256, sign_seed=3, scale_fmt=PO2)


def test_2d_transposition_invariance_on_gpu():
    """Without the RHT, b x b blocks give the transposed column-wise copy
    (2D-block tutorial, Eq. S(B) = S(B^T))."""
    x = inputs.tiny_check(256, 384)
    got = gpu_quantize(to_dev(x), grid="e1m2", block=(32, 32), n=1, scale_fmt=PO2,
                       out_mask=ufp4.OUT_ROWWISE | ufp4.OUT_COLWISE)
    unpack = lambda c: np.stack([c & 0xF, c >> 4], -1).reshape(c.shape[0], -1)
    np.testing.assert_array_equal(unpack(got["col"][0]), unpack(got["row"][0]).T)
    np.testing.assert_array_equal(got["col"][1], got["row"][1].T)


# ------------------------------------------------------- ragged / layout
@pytest.mark.parametrize("shape", [(272, 400), (16, 16), (144, 1408), (1, 64), (3, 2064)])
def test_ragged_shapes(shape):
    rows, cols = shape
    x = inputs.normal_bf16(rows, cols, 1234)
    _check(x, grid="int4", n=16, sign_seed=1, rounding=SR, sr_seed=3, colwise_too=(rows % 16 == 0))


def test_strided_input():
    x = inputs.tiny_check(192, 256)
    _check(x, ld=264, grid="e1m2", n=32, sign_seed=4, colwise_too=True)
    _check(x, ld=384, grid="e2m1", n=64, sign_seed=4, colwise_too=True, scale_fmt=PO2)


def test_group_id_enters_sr():
    x = inputs.tiny_check(64, 256)
    _check(x, grid="e1m2", rounding=SR, sr_seed=8, group=5)


def test_empty_input_is_a_no_op():
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    desc = ufp4.make_desc(out_mask=ufp4.OUT_ROWWISE)
    codes = torch.zeros((0, 32), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((0, 4), dtype=torch.float32, device="cuda")
    ufp4.ufp4_rht_quantize(x, desc, ufp4.qtensor(codes, scales, 0, 64), None)
    torch.cuda.synchronize()


def test_zero_and_extreme_blocks():
    x = np.zeros((32, 128), dtype=np.uint16)
    x[1::2] = 0x8000  # -0
    x[4, :16] = inputs.f32_to_bf16_bits(np.full(16, 1e30, np.float32))
    x[5, 16:32] = inputs.f32_to_bf16_bits(np.full(16, -3e-30, np.float32))
    x[6, :] = inputs.f32_to_bf16_bits(np.linspace(-4, 4, 128).astype(np.float32))
    for grid in GRIDS:
        for fmt in (FP32, PO2):
            _check(x, grid=grid, n=16, sign_seed=2, scale_fmt=fmt, colwise_too=True)


def test_exact_ties_round_to_even():
    """Scale 1 blocks (amax = qmax, n = 1) quantize the bf16 values themselves,
    including every exact midpoint between levels."""
    for grid, qmax, step in (("e1m2", 1.75, 0.125), ("int4", 7.0, 0.5), ("e2m1", 6.0, 0.25)):
        vals = np.arange(-qmax, qmax + step / 2, step / 2, dtype=np.float32)
        cols = 16 * int(np.ceil(vals.size / 15))
        row = np.zeros(cols, dtype=np.float32)
        for b in range(cols // 16):
            chunk = vals[b * 15:(b + 1) * 15]
            row[b * 16] = qmax
            row[b * 16 + 1:b * 16 + 1 + chunk.size] = chunk
        x = inputs.f32_to_bf16_bits(np.tile(row, (16, 1)))
        _check(x, grid=grid, n=1, scale_fmt=FP32)
        _check(x, grid=grid, n=1, scale_fmt=FP32, rounding=SR, sr_seed=99)


# ----------------------------------------------------------- RHT / dequant
@pytest.mark.parametrize("n", [2, 16, 64, 256])
def test_rht_transform_bit_exact(n):
    x = inputs.tiny_check(64, 512)
    z = torch.empty((64, 512), dtype=torch.float32, device="cuda")
    ufp4.ufp4_rht_transform(to_dev(x), n, 0x5EED0001, z)
    torch.cuda.synchronize()
    assert_bitwise(z.cpu().numpy(), orc.rht_rows(x, n, 0x5EED0001), "RHT output")


@pytest.mark.parametrize("grid", GRIDS)
@pytest.mark.parametrize("inverse", [False, True])
def test_dequantize_bit_exact(grid, inverse):
    x = inputs.tiny_check(64, 256)
    for block, fmt in (((1, 16), FP32), ((1, 32), PO2), ((16, 16), PO2)):
        c, s = orc.quantize(x, grid=grid, block=block, n=64, sign_seed=6, scale_fmt=fmt)
        desc = ufp4.make_desc(grid=grid, block=block, n=64, sign_seed=6, scale_fmt=fmt)
        cd, sd = torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda()
        out = torch.empty((64, 256), dtype=torch.float32, device="cuda")
        ufp4.ufp4_dequantize(ufp4.qtensor(cd, sd, 64, 256), desc, inverse, out)
        torch.cuda.synchronize()
        ref = orc.dequantize(c, s, grid=grid, block=block, scale_fmt=fmt, n=64, sign_seed=6,
                             inverse_rht=inverse)
        assert_bitwise(out.cpu().numpy(), ref, f"dequantize {block}")


# ------------------------------------------------------------ MoE grouped
def test_grouped_quantize_matches_per_group_oracle():
    lists = inputs.moe_routing(tokens=1024, experts=8)
    x_all = inputs.normal_bf16(1024, 256, 402)
    xs = np.concatenate([x_all[l] for l in lists])
    offsets = np.concatenate([[0], np.cumsum([len(l) for l in lists])])
    desc = ufp4.make_desc(grid="e1m2", n=16, sign_seed=inputs.SIGN_SEED, rounding=ufp4.ROUND_SR,
                          sr_seed=inputs.SR_SEED, scale_fmt=FP32, out_mask=3)
    pads = [ufp4.ufp4_grouped_padded_rows(int(offsets[g + 1] - offsets[g]), desc) for g in range(8)]
    ptot = int(sum(pads))
    xd = to_dev(xs)
    rc = torch.empty((xs.shape[0], 128), dtype=torch.uint8, device="cuda")
    rs = torch.empty((xs.shape[0], 16), dtype=torch.float32, device="cuda")
    cc = torch.full((256 * ptot // 2,), 0xAB, dtype=torch.uint8, device="cuda")
    cs = torch.empty((256 * ptot // 16,), dtype=torch.float32, device="cuda")
    rq = ufp4.QTensor(rc.data_ptr(), rs.data_ptr(), xs.shape[0], 256, 128, 16)
    cq = ufp4.QTensor(cc.data_ptr(), cs.data_ptr(), 256, ptot, 0, 0)
    ufp4.ufp4_rht_quantize_grouped(xd, offsets.tolist(), desc, rq, cq)
    torch.cuda.synchronize()
    rc, rs, cc, cs = rc.cpu().numpy(), rs.cpu().numpy(), cc.cpu().numpy(), cs.cpu().numpy()
    poff = 0
    for g in range(8):
        xe = xs[offsets[g]:offsets[g + 1]]
        kw = dict(grid="e1m2", n=16, sign_seed=inputs.SIGN_SEED, rounding=SR, sr_seed=inputs.SR_SEED,
                  scale_fmt=FP32, group=g)
        c, s = orc.quantize(xe, **kw)
        assert_bitwise(rc[offsets[g]:offsets[g + 1]], c, f"group {g} row-wise codes")
        assert_bitwise(rs[offsets[g]:offsets[g + 1]], s, f"group {g} row-wise scales")
        xp = np.zeros((pads[g], 256), dtype=np.uint16)
        xp[: xe.shape[0]] = xe
        c, s = orc.quantize(xp, colwise=True, **kw)
        got_c = cc[256 * poff // 2: 256 * (poff + pads[g]) // 2].reshape(256, pads[g] // 2)
        got_s = cs[256 * poff // 16: 256 * (poff + pads[g]) // 16].reshape(256, pads[g] // 16)
        assert_bitwise(got_c, c, f"group {g} column-wise codes")
        assert_bitwise(got_s, s, f"group {g} column-wise scales")
        poff += pads[g]


# ------------------------------------------------------------- workloads
def test_dense_fprop_operands_full_size():
    """Dense-1.5B-like FPROP operands (X 8192 x 2048, W 5632 x 2048), E1M2
    1 x 16 RTNE with fp32 scales and with UE8M0 scales, checked in full."""
    x, w = inputs.dense_fprop()
    for t in (x, w):
        for fmt in (FP32, PO2):
            _check(t, grid="e1m2", n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=fmt)


def test_dy_sr_row_and_col_full_size():
    """dY 8192 x 2048 (1e-3 Student-t), SR with seed 1234, row-wise and
    column-wise from one pass, in full; W column-wise RTNE."""
    dy, w = inputs.dy_sr()
    _check(dy, grid="e1m2", n=16, sign_seed=inputs.SIGN_SEED, rounding=SR, sr_seed=inputs.SR_SEED,
           colwise_too=True)
    got = gpu_quantize(to_dev(w), grid="e1m2", n=16, sign_seed=inputs.SIGN_SEED, out_mask=ufp4.OUT_COLWISE)
    c, s = orc.quantize(w, grid="e1m2", n=16, sign_seed=inputs.SIGN_SEED, colwise=True)
    assert_bitwise(got["col"][0], c, "W column-wise codes")
    assert_bitwise(got["col"][1], s, "W column-wise scales")


SWEEP_CELLS = [(grid, block, fmt, rnd) for grid in ("e1m2", "int4", "e2m1")
               for block, fmt in (((1, 16), FP32), ((1, 32), FP32), ((32, 32), PO2))
               for rnd in (RTNE, SR)]


@pytest.mark.parametrize("n", [16, 64, 256])
def test_large_sweep_sampled_rows(n):
    """MoE-124B-like X 16384 x 7168, every cell of the quantizer sweep (grid x
    block x rounding, here for one n): each checked on two seeded bands of 64
    rows (1-D blocks depend on their own row only; 2-D 32 x 32 blocks on
    their 32-row band)."""
    x, _ = inputs.large_sweep(k=7168, m=16384, n=7168)
    xd = to_dev(x)
    rng = np.random.default_rng(n)
    for grid, block, fmt, rnd in SWEEP_CELLS:
        kw = dict(grid=grid, block=block, n=n, sign_seed=inputs.SIGN_SEED, rounding=rnd,
                  sr_seed=inputs.SR_SEED, scale_fmt=fmt)
        got = gpu_quantize(xd, out_mask=ufp4.OUT_ROWWISE, **kw)
        for b in sorted(rng.choice(16384 // 64, size=2, replace=False)):
            r0 = int(b) * 64
            c, s = orc.quantize(x[r0:r0 + 64], row0=r0, **kw)
            what = f"{grid} {block} {'SR' if rnd else 'RTNE'} n={n} band {b}"
            assert_bitwise(got["row"][0][r0:r0 + 64], c, what + " codes")
            br = block[0]
            assert_bitwise(got["row"][1][r0 // br:(r0 + 64) // br], s, what + " scales")


# ----------------------------------------- row-wise kernel and batched calls
# Row-wise calls with 1-D blocks run the row kernels (n = 64 and n = 256: the
# segment kernel, 128 x 128 and 64 x 256 tiles); these cover their ragged row
# and column tiles, padded leading dimensions and every rounding and scale
# mode.
@pytest.mark.parametrize("grid", GRIDS)
@pytest.mark.parametrize("rounding", [RTNE, SR])
@pytest.mark.parametrize("block,n,cols", [((1, 16), 16, 576), ((1, 32), 64, 576), ((1, 16), 128, 640),
                                          ((1, 32), 1, 544), ((1, 16), 64, 704), ((1, 16), 256, 768),
                                          ((1, 32), 256, 512)])
def test_rowwise_ragged_tiles(grid, rounding, block, n, cols):
    x = inputs.tiny_check(300, cols)
    fmt = PO2 if grid.startswith("e2m1") else FP32
    _check(x, grid=grid, block=block, n=n, sign_seed=21, rounding=rounding, sr_seed=8, scale_fmt=fmt,
           ld=cols + 64, group=2)


@pytest.mark.parametrize("rounding", [RTNE, SR])
@pytest.mark.parametrize("grid", ["e1m2", "e2m1"])
@pytest.mark.parametrize("n", [16, 64, 256])
def test_batch_matches_oracle_and_single_calls(rounding, grid, n):
    """ufp4_rht_quantize_batch over tensors of different shapes (one empty)
    equals the oracle per tensor and the separate single calls, bit for bit
    (n = 16: the row kernel; n = 64, 256: the segment kernel)."""
    shapes = [(300, 576), (128, 1024), (0, 64), (1000, 192)] if n < 256 else [(300, 768), (64, 512), (0, 256),
                                                                             (200, 256)]
    xs = [inputs.tiny_check(r, c) if r else np.zeros((0, c), np.uint16) for r, c in shapes]
    kw = dict(grid=grid, block=(1, 16), n=n, sign_seed=inputs.SIGN_SEED, rounding=rounding,
              sr_seed=inputs.SR_SEED, scale_fmt=PO2, group=3)
    desc = ufp4.make_desc(out_mask=ufp4.OUT_ROWWISE, **kw)
    devs = [to_dev(x) for x in xs]
    bufs = [ufp4.alloc_quantized(r, c, desc, "cuda") for r, c in shapes]
    qts = [ufp4.qtensor(cb, sb, r, c) for (cb, sb), (r, c) in zip(bufs, shapes)]
    ufp4.ufp4_rht_quantize_batch(devs, desc, qts)
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    for x, dv, (cb, sb), (r, c) in zip(xs, devs, bufs, shapes):
        if r == 0:
            continue
        oc, osc = orc.quantize(x, **kw)
        assert_bitwise(cb.cpu().numpy(), oc, f"batch codes {r}x{c}")
        assert_bitwise(sb.cpu().numpy(), osc, f"batch scales {r}x{c}")
        single = gpu_quantize(dv, out_mask=ufp4.OUT_ROWWISE, **kw)["row"]
        assert_bitwise(cb.cpu().numpy(), single[0], "batch vs single codes")
        assert_bitwise(sb.cpu().numpy(), single[1], "batch vs single scales")


@pytest.mark.parametrize("block,fmt", [((1, 16), FP32), ((1, 32), PO2), ((32, 32), PO2)])
@pytest.mark.parametrize("rounding", [RTNE, SR])
def test_hadamard_256_code_rows_8_byte_aligned(block, fmt, rounding):
    """n = 256 stores each segment's two chunks of codes as one 16-byte word
    when the code rows are 16-byte aligned, else as two 8-byte words: a code
    leading dimension of 8 mod 16 bytes takes the second form.  The padding
    bytes of each code row stay untouched."""
    rows, cols = 128, 768
    x = inputs.tiny_check(rows, cols)
    kw = dict(grid="e1m2", block=block, n=256, sign_seed=4, rounding=rounding, sr_seed=6, scale_fmt=fmt)
    desc = ufp4.make_desc(out_mask=ufp4.OUT_ROWWISE, **ufp4_kw(kw))
    dev = torch.device("cuda", 0)
    codes_full = torch.full((rows, cols // 2 + 8), 0x5A, dtype=torch.uint8, device=dev)
    codes = codes_full[:, : cols // 2]
    _, scales = ufp4.alloc_quantized(rows, cols, desc, dev)
    q = ufp4.qtensor(codes, scales, rows, cols)
    assert q.codes_ld % 16 == 8
    ufp4.ufp4_rht_quantize(to_dev(x), desc, q, None)
    torch.cuda.synchronize()
    c, s = orc.quantize(x, **kw)
    assert_bitwise(codes.cpu().numpy(), c, "row-wise codes")
    assert_bitwise(scales.cpu().numpy(), s, "row-wise scales")
    assert torch.all(codes_full[:, cols // 2:] == 0x5A), "a code row's padding was written"


def ufp4_kw(kw):
    """The oracle's keyword names mapped to ufp4.make_desc's."""
    return dict(grid=kw["grid"], block=kw["block"], n=kw["n"], sign_seed=kw["sign_seed"], rounding=kw["rounding"],
                sr_seed=kw["sr_seed"], scale_fmt=kw["scale_fmt"])
