"""Two-level scale (per-tensor fp32 x per-block E4M3) through the C ABI
against the oracle: codes, E4M3 scale bytes and the tensor amax bit for bit;
dequantize exact; the native FP4 GEMM with E4M3 block scales within 1e-5 of
the fp64 product of the dequantized operands."""
import numpy as np
import pytest
import torch

import oracle as orc
from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import assert_bitwise, to_dev

pytestmark = pytest.mark.gpu
E4M3 = ufp4.SCALE_E4M3


def _quantize(xd, **kw):
    desc = ufp4.make_desc(scale_fmt=E4M3, out_mask=ufp4.OUT_ROWWISE, **kw)
    out = ufp4.quantize(xd, desc)
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    return desc, out["row"][0], out["row"][1], out["row_amax"]


@pytest.mark.parametrize("grid", ["e2m1", "e1m2", "int4", "e2m1r2"])
@pytest.mark.parametrize("block,n", [((1, 16), 16), ((1, 32), 64), ((1, 16), 1)])
@pytest.mark.parametrize("rounding", [orc.RTNE, orc.SR])
def test_two_level_quantize_matches_oracle(grid, block, n, rounding):
    x = inputs.tiny_check(300, 1024)
    kw = dict(grid=grid, block=block, n=n, sign_seed=inputs.SIGN_SEED, rounding=rounding, sr_seed=inputs.SR_SEED)
    _, c, s, t = _quantize(to_dev(x), **kw)
    oc, os_, ot = orc.quantize_2level(x, **kw)
    assert float(t.item()) == ot
    assert_bitwise(c.cpu().numpy(), oc, "two-level codes")
    assert_bitwise(s.cpu().numpy(), os_, "two-level E4M3 scales")


def test_two_level_dequantize_and_stats():
    x = inputs.tiny_check(256, 512)
    kw = dict(grid="e2m1", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED)
    xd = to_dev(x)
    desc, c, s, t = _quantize(xd, **kw)
    q = ufp4.qtensor(c, s, 256, 512, t)
    out = torch.empty((256, 512), dtype=torch.float32, device="cuda")
    ufp4.ufp4_dequantize(q, desc, False, out)
    inv = torch.empty_like(out)
    ufp4.ufp4_dequantize(q, desc, True, inv)
    stats = torch.zeros(4, dtype=torch.float64, device="cuda")
    ufp4.ufp4_quant_error_stats(xd, desc, q, stats)
    torch.cuda.synchronize()
    cn, sn, T = c.cpu().numpy(), s.cpu().numpy(), float(t.item())
    assert_bitwise(out.cpu().numpy(), orc.dequantize_2level(cn, sn, T, **kw), "two-level dequantize")
    assert_bitwise(inv.cpu().numpy(), orc.dequantize_2level(cn, sn, T, inverse_rht=True, **kw),
                   "two-level inverse RHT")
    z = orc.rht_rows(x, 16, inputs.SIGN_SEED).astype(np.float64)
    qv = orc.dequantize_2level(cn, sn, T, **kw).astype(np.float64)
    ref = np.array([(z * z).sum(), ((qv - z) ** 2).sum(), (qv * z).sum(), (qv * qv).sum()])
    np.testing.assert_allclose(stats.cpu().numpy(), ref, rtol=1e-5)


@pytest.mark.parametrize("grid", ["e2m1", "e2m1r2"])
def test_two_level_gemm(grid):
    x, w = inputs.dense_fprop(m=1024, n=768, k=2048)
    kw = dict(grid=grid, block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED)
    _, ac, asc, at = _quantize(to_dev(x), **kw)
    _, bc, bsc, bt = _quantize(to_dev(w), **kw)
    desc = ufp4.make_desc(grid=grid, block=(1, 16), scale_fmt=E4M3)
    qa, qb = ufp4.qtensor(ac, asc, 1024, 2048, at), ufp4.qtensor(bc, bsc, 768, 2048, bt)
    D = torch.empty((1024, 768), dtype=torch.float32, device="cuda")
    ws = torch.empty(ufp4.ufp4_gemm_workspace_size(1024, 768, 2048, desc), dtype=torch.uint8, device="cuda")
    ufp4.ufp4_gemm(qa, qb, desc, D, ws)
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    ref = orc.gemm_reference_2level(ac.cpu().numpy(), asc.cpu().numpy(), float(at.item()), bc.cpu().numpy(),
                                    bsc.cpu().numpy(), float(bt.item()), grid=grid)
    d = D.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(d - ref) / np.linalg.norm(ref) <= 1e-5


def test_two_level_batch_equals_single_calls():
    xs = [inputs.tiny_check(200, 512), inputs.tiny_check(128, 1024)]
    kw = dict(grid="e2m1", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED)
    desc = ufp4.make_desc(scale_fmt=E4M3, out_mask=ufp4.OUT_ROWWISE, **kw)
    devs = [to_dev(x) for x in xs]
    bufs = [ufp4.alloc_quantized(x.shape[0], x.shape[1], desc, "cuda") for x in xs]
    amax = [torch.zeros(1, dtype=torch.float32, device="cuda") for _ in xs]
    qts = [ufp4.qtensor(cb, sb, x.shape[0], x.shape[1], a) for (cb, sb), x, a in zip(bufs, xs, amax)]
    ufp4.ufp4_rht_quantize_batch(devs, desc, qts)
    torch.cuda.synchronize()
    for x, (cb, sb), a in zip(xs, bufs, amax):
        oc, os_, ot = orc.quantize_2level(x, **kw)
        assert float(a.item()) == ot
        assert_bitwise(cb.cpu().numpy(), oc, "batch two-level codes")
        assert_bitwise(sb.cpu().numpy(), os_, "batch two-level scales")
