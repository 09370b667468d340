"""ufp4_rht_quantize_prepare: the two GEMM operands quantized and prepared in
one launch must equal ufp4_rht_quantize_batch followed by ufp4_gemm_prepare,
byte for byte (codes, scales and the whole workspace), and the GEMM that
reads the workspace must then give the same D bit for bit.  The quantized
codes and scales are checked against the oracle through the batch call
(tests/test_quantize_gpu.py); the GEMM on such a workspace against the
oracle's fp64 product (tests/test_gemm_gpu.py)."""
import pytest
import torch

from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu


def _two_routes(x, w, desc, x_ld=None):
    dev = torch.device("cuda", 0)
    M, K = x.shape
    N = w.shape[0]
    xd, wd = to_dev(x, ld=x_ld), to_dev(w)
    size = ufp4.ufp4_gemm_workspace_size(M, N, K, desc)
    outs = []
    for fused in (False, True):
        qa, qb = ufp4.alloc_quantized(M, K, desc, dev), ufp4.alloc_quantized(N, K, desc, dev)
        ta, tb = ufp4.qtensor(*qa, M, K), ufp4.qtensor(*qb, N, K)
        ws = torch.full((size,), 0xA5, dtype=torch.uint8, device=dev)  # bytes neither route writes stay equal
        D = torch.empty((M, N), dtype=torch.float32, device=dev)
        if fused:
            ufp4.ufp4_rht_quantize_prepare(xd, wd, desc, ta, tb, ws)
        else:
            ufp4.ufp4_rht_quantize_batch([xd, wd], desc, [ta, tb])
            ufp4.ufp4_gemm_prepare(ta, tb, desc, ws)
        ufp4.ufp4_gemm_prepared(ta, tb, desc, D, ws)
        torch.cuda.synchronize()
        outs.append((qa, qb, ws, D))
    assert ufp4.ufp4_device_error() == 0
    return outs


def _assert_same(outs):
    (qa0, qb0, ws0, D0), (qa1, qb1, ws1, D1) = outs
    for a, b, what in ((qa0[0], qa1[0], "A codes"), (qa0[1], qa1[1], "A scales"), (qb0[0], qb1[0], "B codes"),
                       (qb0[1], qb1[1], "B scales")):
        assert torch.equal(a, b), what
    if not torch.equal(ws0, ws1):
        bad = torch.nonzero(ws0 != ws1).flatten()
        raise AssertionError(f"workspace: {bad.numel()} bytes differ, first at {int(bad[0])}")
    assert torch.equal(D0, D1), "D"


# ragged M (not whole 128-row tiles), N not a multiple of the 224-row GEMM
# tile (scale cells past the quantizer's own rows), K not whole 128-element
# chunks; and a larger shape with several K chunks and GEMM tiles
@pytest.mark.parametrize("grid", ["e1m2", "int4"])
@pytest.mark.parametrize("block", [(1, 16), (1, 32)])
@pytest.mark.parametrize("mnk", [(300, 500, 416), (1024, 896, 2048)])
def test_fused_prepare_equals_quantize_then_prepare(grid, block, mnk):
    M, N, K = mnk
    x = inputs.with_element_outliers(inputs.normal_bf16(M, K, 601), 1e-3, 50.0, 602)
    w = inputs.normal_bf16(N, K, 603, std=0.02)
    desc = ufp4.make_desc(grid=grid, block=block, n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=ufp4.SCALE_UE8M0,
                          out_mask=ufp4.OUT_ROWWISE)
    _assert_same(_two_routes(x, w, desc))


def test_fused_prepare_wide_scale_gaps_and_strided_input():
    """Neighbouring 16-element blocks 20 binades apart: the pair shift d exceeds
    14 and both routes take the rounded fp32 path for the smaller block."""
    M, N, K = 256, 448, 512
    x = inputs.normal_bf16(M, K, 611)
    xf = inputs.bf16_bits_to_f32(x).reshape(M, K // 16, 16)
    xf[:, 1::2, :] *= 2.0 ** -20
    x = inputs.f32_to_bf16_bits(xf.reshape(M, K))
    w = inputs.normal_bf16(N, K, 612)
    for grid in ("e1m2", "int4"):
        desc = ufp4.make_desc(grid=grid, block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED,
                              scale_fmt=ufp4.SCALE_UE8M0, out_mask=ufp4.OUT_ROWWISE)
        _assert_same(_two_routes(x, w, desc, x_ld=K + 64))


@pytest.mark.parametrize("grid", ["e1m2", "int4"])
def test_fused_prepare_stochastic_rounding(grid):
    M, N, K = 384, 224, 1024
    x = inputs.student_t_bf16(M, K, 621)
    w = inputs.normal_bf16(N, K, 622, std=0.02)
    desc = ufp4.make_desc(grid=grid, block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=ufp4.SCALE_UE8M0,
                          rounding=ufp4.ROUND_SR, sr_seed=inputs.SR_SEED, out_mask=ufp4.OUT_ROWWISE)
    _assert_same(_two_routes(x, w, desc))


def test_fused_prepare_full_size_moe124b_operands():
    """The MoE-124B-like FPROP operands (X 16384 x 7168, W 7168 x 7168): the
    shape the benchmark step runs."""
    x, w = inputs.large_sweep(16384, 7168, 7168)
    desc = ufp4.make_desc(grid="e1m2", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=ufp4.SCALE_UE8M0,
                          out_mask=ufp4.OUT_ROWWISE)
    _assert_same(_two_routes(x, w, desc))
