"""Out-of-bounds writes: every output buffer sits between guard bands of
canary bytes, and the canaries must be intact after the call (ragged shapes,
padded leading dimensions, every quantizer path and the GEMM).  A stray store
past a row's end, a tile's edge or a tensor's last row would land in a guard
band or in the padding between rows, which is canaried too."""
import ctypes

import numpy as np
import pytest
import torch

from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu

GUARD = 4096
CANARY = 0xA5


class Guarded:
    """A device byte buffer of rows x ld bytes (row-major, ld >= width) with
    guard bands before and after; the bytes between width and ld are canaried."""

    def __init__(self, rows, width, ld):
        self.rows, self.width, self.ld = rows, width, ld
        self.buf = torch.full((2 * GUARD + rows * ld,), CANARY, dtype=torch.uint8, device="cuda")
        self.body = self.buf[GUARD:GUARD + rows * ld]

    def ptr(self):
        return self.body.data_ptr()

    def check(self, what):
        h = self.buf.cpu().numpy()
        assert (h[:GUARD] == CANARY).all(), f"{what}: write before the buffer"
        assert (h[GUARD + self.rows * self.ld:] == CANARY).all(), f"{what}: write after the buffer"
        pad = h[GUARD:GUARD + self.rows * self.ld].reshape(self.rows, self.ld)[:, self.width:]
        assert (pad == CANARY).all(), f"{what}: write into the row padding"


def _quant_out(rows, cols, desc, pad_codes=16, pad_scales=8):
    bw = desc.block_cols
    br = desc.block_rows
    cw = cols if desc.grid == ufp4.GRID_MXFP8 else cols // 2
    sbytes = 4 if desc.scale_fmt == ufp4.SCALE_FP32 else 1
    srows = rows // br if br > 1 else rows
    codes = Guarded(rows, cw, cw + pad_codes)
    scales = Guarded(srows, (cols // bw) * sbytes, (cols // bw + pad_scales) * sbytes)
    q = ufp4.QTensor(codes.ptr(), scales.ptr(), rows, cols, cw + pad_codes, cols // bw + pad_scales)
    return codes, scales, q


@pytest.mark.parametrize("kw", [
    dict(grid="e1m2", block=(1, 16), n=16, scale_fmt=ufp4.SCALE_UE8M0),
    dict(grid="int4", block=(1, 32), n=64, scale_fmt=ufp4.SCALE_FP32, rounding=ufp4.ROUND_SR, sr_seed=3),
    dict(grid="e2m1", block=(1, 16), n=256, scale_fmt=ufp4.SCALE_UE8M0),
    dict(grid="e1m2", block=(32, 32), n=16, scale_fmt=ufp4.SCALE_UE8M0),
    dict(grid="int4", block=(16, 16), n=64, scale_fmt=ufp4.SCALE_UE8M0, rounding=ufp4.ROUND_SR, sr_seed=4),
    dict(grid="mxfp8", block=(1, 32), n=16, scale_fmt=ufp4.SCALE_UE8M0),
])
@pytest.mark.parametrize("colwise", [False, True])
def test_quantizer_writes_stay_inside(kw, colwise):
    if colwise and (kw["n"] == 256 or kw["grid"] == "mxfp8"):
        pytest.skip("the column-wise output keeps n <= 128 and 4-bit grids")
    # rows ragged against 128-row tiles; columns against 128-column tiles (n = 256
    # needs whole 256-column segments, so only its rows are ragged)
    rows, cols = 576, (768 if kw["n"] == 256 else 832)
    x = inputs.tiny_check(rows, cols)
    xd = to_dev(x, ld=cols + 64)
    desc = ufp4.make_desc(sign_seed=9, out_mask=ufp4.OUT_ROWWISE | (ufp4.OUT_COLWISE if colwise else 0), **kw)
    rc, rs, rq = _quant_out(rows, cols, desc)
    cc = cs = cq = None
    if colwise:
        cc, cs, cq = _quant_out(cols, rows, desc)
    ufp4.ufp4_rht_quantize(xd, desc, rq, cq)
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    for g, what in ((rc, "row-wise codes"), (rs, "row-wise scales"), (cc, "column-wise codes"),
                    (cs, "column-wise scales")):
        if g is not None:
            g.check(what)


@pytest.mark.parametrize("grid,block", [("e1m2", (1, 16)), ("e2m1", (1, 16)), ("int4", (32, 32))])
def test_gemm_writes_stay_inside(grid, block):
    M, N, K = 200, 300, 512  # ragged against 256 x 224 / 256 x 192 output tiles
    rng = np.random.default_rng(1)
    def operand(rows):
        c = torch.from_numpy(rng.integers(0, 256, (rows, K // 2), dtype=np.uint8) & 0x77).cuda()
        srows = -(-rows // block[0]) if block[0] > 1 else rows
        s = torch.from_numpy(rng.integers(120, 134, (srows, K // block[1]), dtype=np.uint8)).cuda()
        return c, s
    if block[0] > 1:
        M, N = 224, 320
    A, B = operand(M), operand(N)
    desc = ufp4.make_desc(grid=grid, block=block, scale_fmt=ufp4.SCALE_UE8M0)
    ldd = N + 12
    D = Guarded(M, N * 4, ldd * 4)
    ws = torch.empty(max(1, ufp4.ufp4_gemm_workspace_size(M, N, K, desc)), dtype=torch.uint8, device="cuda")
    st = ufp4.load().ufp4_gemm(ctypes.byref(ufp4.qtensor(*A, M, K)), ctypes.byref(ufp4.qtensor(*B, N, K)),
                               ctypes.byref(desc), D.ptr(), ldd, ws.data_ptr(), ws.numel(), None)
    assert st == 0
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    D.check("GEMM output")
