"""The MoE-7.9B-like expert FFN step at its full size (UFP4 summary, section
方法: RHT and the quantized GEMM on FPROP, DGRAD and WGRAD; section 实验: the
MoE 7.9B model): 16384 tokens routed top-2 over 8 experts (32768 routed rows,
an uneven split), hidden 2048, ffn 1408, with the seeded inputs of the
workload recipe (X seed 402, W_e seed 403, dY seed 404).

Quantizer: the grouped row-wise and column-wise outputs of X (RTNE), dY (SR)
and the stacked W_e (RTNE), all E1M2 1 x 16 UE8M0, n = 16, are compared bit
for bit with the oracle expert by expert (column-wise on the zero-padded
slabs).  GEMMs: the three grouped GEMMs are compared with the oracle's fp64
product of the dequantized operands, relative Frobenius <= 1e-5, on 384
sampled rows of A per expert (the first, the last and seeded ones; the fp64
product of every row takes minutes on the host) against all columns."""
import numpy as np
import pytest
import torch

import oracle as orc
from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import assert_bitwise, to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-5
DEV = "cuda"
SAMPLE_ROWS = 384


def _grouped(t_np, offsets, cols, desc, pads):
    """Grouped quantization on the GPU; returns per-group (codes, scales) host
    arrays of the row-wise and of the column-wise output."""
    total = int(offsets[-1])
    poff = np.concatenate([[0], np.cumsum(pads)]).astype(np.int64)
    ptot = int(poff[-1])
    rc = torch.empty((total, cols // 2), dtype=torch.uint8, device=DEV)
    rs = torch.empty((total, cols // 16), dtype=torch.uint8, device=DEV)
    cc = torch.empty((cols * ptot // 2,), dtype=torch.uint8, device=DEV)
    cs = torch.empty((cols * ptot // 16,), dtype=torch.uint8, device=DEV)
    ufp4.ufp4_rht_quantize_grouped(to_dev(t_np), [int(o) for o in offsets], desc, ufp4.qtensor(rc, rs, total, cols),
                                   ufp4.QTensor(cc.data_ptr(), cs.data_ptr(), cols, ptot, 0, 0))
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    rows = [(rc[offsets[g]:offsets[g + 1]], rs[offsets[g]:offsets[g + 1]]) for g in range(len(pads))]
    colq = [(cc[cols * poff[g] // 2: cols * poff[g + 1] // 2].view(cols, pads[g] // 2),
             cs[cols * poff[g] // 16: cols * poff[g + 1] // 16].view(cols, pads[g] // 16)) for g in range(len(pads))]
    return rows, colq


def _check_grouped(t_np, offsets, cols, pads, rows, colq, rounding, what):
    for g in range(len(pads)):
        xe = t_np[offsets[g]:offsets[g + 1]]
        kw = dict(grid="e1m2", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED, rounding=rounding,
                  sr_seed=inputs.SR_SEED, scale_fmt=orc.SCALE_UE8M0, group=g)
        c, s = orc.quantize(xe, **kw)
        assert_bitwise(rows[g][0].cpu().numpy(), c, f"{what} expert {g} row-wise codes")
        assert_bitwise(rows[g][1].cpu().numpy(), s, f"{what} expert {g} row-wise scales")
        xp = np.zeros((pads[g], cols), dtype=np.uint16)
        xp[: xe.shape[0]] = xe
        c, s = orc.quantize(xp, colwise=True, **kw)
        assert_bitwise(colq[g][0].cpu().numpy(), c, f"{what} expert {g} column-wise codes")
        assert_bitwise(colq[g][1].cpu().numpy(), s, f"{what} expert {g} column-wise scales")


def test_moe_step_full_size():
    lists, x_all, w_all, dy = inputs.moe_step()
    experts, ffn, hidden = w_all.shape
    counts = [len(l) for l in lists]
    assert sum(counts) == 32768 and len(set(counts)) > 1
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    xs = np.ascontiguousarray(np.concatenate([x_all[l] for l in lists]))
    kw = dict(grid="e1m2", block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=ufp4.SCALE_UE8M0, out_mask=3)
    x_desc = ufp4.make_desc(**kw)
    dy_desc = ufp4.make_desc(rounding=ufp4.ROUND_SR, sr_seed=inputs.SR_SEED, **kw)
    pads = [ufp4.ufp4_grouped_padded_rows(c, x_desc) for c in counts]

    xrow, xcol = _grouped(xs, off, hidden, x_desc, pads)
    _check_grouped(xs, off, hidden, pads, xrow, xcol, orc.RTNE, "X")
    yrow, ycol = _grouped(dy, off, ffn, dy_desc, pads)
    _check_grouped(dy, off, ffn, pads, yrow, ycol, orc.SR, "dY")
    w_stack = np.ascontiguousarray(w_all.reshape(experts * ffn, hidden))
    w_off = np.arange(experts + 1, dtype=np.int64) * ffn
    w_pads = [ufp4.ufp4_grouped_padded_rows(ffn, x_desc)] * experts
    assert w_pads[0] == ffn  # each expert's column-wise slab is its own W_e^T
    wrow, wcol = _grouped(w_stack, w_off, hidden, x_desc, w_pads)
    _check_grouped(w_stack, w_off, hidden, w_pads, wrow, wcol, orc.RTNE, "W_e")

    gdesc = ufp4.make_desc(grid="e1m2", block=(1, 16), scale_fmt=ufp4.SCALE_UE8M0)
    cases = {
        "FPROP Y = X W^T": ([(xrow[g], counts[g], hidden) for g in range(experts)],
                            [(wrow[g], ffn, hidden) for g in range(experts)]),
        "DGRAD dX = dY W": ([(yrow[g], counts[g], ffn) for g in range(experts)],
                            [(wcol[g], hidden, ffn) for g in range(experts)]),
        "WGRAD dW = dY^T X": ([(ycol[g], ffn, pads[g]) for g in range(experts)],
                              [(xcol[g], hidden, pads[g]) for g in range(experts)]),
    }
    rng = np.random.default_rng(4040)
    for name, (A, B) in cases.items():
        qa = [ufp4.qtensor(a[0][0], a[0][1], a[1], a[2]) for a in A]
        qb = [ufp4.qtensor(b[0][0], b[0][1], b[1], b[2]) for b in B]
        outs = [torch.full((a[1], b[1]), float("nan"), dtype=torch.float32, device=DEV) for a, b in zip(A, B)]
        ws = torch.empty(max(1, ufp4.ufp4_gemm_grouped_workspace_size(qa, qb, gdesc)), dtype=torch.uint8, device=DEV)
        ufp4.ufp4_gemm_grouped(qa, qb, gdesc, outs, ws)
        torch.cuda.synchronize()
        assert ufp4.ufp4_device_error() == 0
        for g in range(experts):
            m = A[g][1]
            rows = np.unique(np.concatenate([[0, m - 1], rng.choice(m, size=min(m, SAMPLE_ROWS - 2), replace=False)]))
            ac, asc = A[g][0][0].cpu().numpy()[rows], A[g][0][1].cpu().numpy()[rows]
            bc, bsc = B[g][0][0].cpu().numpy(), B[g][0][1].cpu().numpy()
            ref = orc.gemm_reference(ac, asc, bc, bsc, grid="e1m2", block=(1, 16))
            got = outs[g].cpu().numpy().astype(np.float64)[rows]
            rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
            assert rel <= TOL, (name, g, rel)
