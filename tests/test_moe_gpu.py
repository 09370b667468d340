"""MoE expert FFN step through the grouped entry points (MoE-7.9B-like shape,
scaled down): seeded top-2 routing, grouped RHT + 4-bit quantization of X and
dY (row-wise and column-wise from one pass, SR on dY), per-expert W_e, then
the grouped FPROP, DGRAD and WGRAD GEMMs.  Each expert's product is checked
against the oracle's fp64 product of the dequantized operands (UFP4 summary,
section 方法: RHT and the quantized GEMM on all three training GEMMs)."""
import numpy as np
import pytest
import torch

import oracle as orc
from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import to_dev

pytestmark = pytest.mark.gpu

TOL = 1e-5
DEV = "cuda"


class Op:
    """A quantized operand: torch views of its codes/scales plus its QTensor."""

    def __init__(self, codes, scales, rows, cols):
        self.codes, self.scales = codes, scales
        self.q = ufp4.qtensor(codes, scales, rows, cols)

    def host(self):
        return self.codes.cpu().numpy(), self.scales.cpu().numpy()


def _rel(d, ref):
    return np.linalg.norm(d - ref) / max(np.linalg.norm(ref), 1e-300)


@pytest.mark.parametrize("grid", ["e1m2", "e2m1"])
def test_moe_step_grouped(grid):
    tokens, experts, hidden, ffn = 1024, 8, 256, 192
    lists = inputs.moe_routing(tokens=tokens, experts=experts)
    x_all = inputs.normal_bf16(tokens, hidden, 402)
    w = inputs.normal_bf16(experts * ffn, hidden, 403, std=0.02).reshape(experts, ffn, hidden)
    counts = [len(l) for l in lists]
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    total = int(off[-1])
    xs = np.concatenate([x_all[l] for l in lists])
    dy = inputs.student_t_bf16(total, ffn, 404)
    kw = dict(grid=grid, block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED, scale_fmt=ufp4.SCALE_UE8M0, out_mask=3)
    x_desc = ufp4.make_desc(**kw)
    dy_desc = ufp4.make_desc(rounding=ufp4.ROUND_SR, sr_seed=inputs.SR_SEED, **kw)
    gdesc = ufp4.make_desc(grid=grid, block=(1, 16), scale_fmt=ufp4.SCALE_UE8M0)
    pads = [ufp4.ufp4_grouped_padded_rows(c, x_desc) for c in counts]
    assert all(p % 64 == 0 for p in pads)
    poff = np.concatenate([[0], np.cumsum(pads)]).astype(np.int64)
    ptot = int(poff[-1])

    def grouped_quant(t_np, cols, desc):
        d = to_dev(t_np)
        rc = torch.empty((total, cols // 2), dtype=torch.uint8, device=DEV)
        rs = torch.empty((total, cols // 16), dtype=torch.uint8, device=DEV)
        cc = torch.empty((cols * ptot // 2,), dtype=torch.uint8, device=DEV)
        cs = torch.empty((cols * ptot // 16,), dtype=torch.uint8, device=DEV)
        ufp4.ufp4_rht_quantize_grouped(d, off.tolist(), desc, ufp4.qtensor(rc, rs, total, cols),
                                       ufp4.QTensor(cc.data_ptr(), cs.data_ptr(), cols, ptot, 0, 0))
        row = [Op(rc[off[g]:off[g + 1]], rs[off[g]:off[g + 1]], counts[g], cols) for g in range(experts)]
        col = [Op(cc[cols * poff[g] // 2: cols * poff[g + 1] // 2].view(cols, pads[g] // 2),
                  cs[cols * poff[g] // 16: cols * poff[g + 1] // 16].view(cols, pads[g] // 16), cols, pads[g])
               for g in range(experts)]
        return row, col

    xrow, xcol = grouped_quant(xs, hidden, x_desc)
    yrow, ycol = grouped_quant(dy, ffn, dy_desc)
    wrow, wcol = [], []
    for e in range(experts):
        q = ufp4.quantize(to_dev(np.ascontiguousarray(w[e])), x_desc)
        wrow.append(Op(*q["row"], ffn, hidden))
        wcol.append(Op(*q["col"], hidden, ffn))

    def run(A, B, shapes):
        outs = [torch.full((m, n), float("nan"), dtype=torch.float32, device=DEV) for m, n in shapes]
        qa, qb = [a.q for a in A], [b.q for b in B]
        ws = torch.empty(max(1, ufp4.ufp4_gemm_grouped_workspace_size(qa, qb, gdesc)), dtype=torch.uint8, device=DEV)
        ufp4.ufp4_gemm_grouped(qa, qb, gdesc, outs, ws)
        torch.cuda.synchronize()
        assert ufp4.ufp4_device_error() == 0
        return [o.cpu().numpy().astype(np.float64) for o in outs]

    cases = {
        "FPROP Y = X W^T": (xrow, wrow, [(c, ffn) for c in counts]),
        "DGRAD dX = dY W": (yrow, wcol, [(c, hidden) for c in counts]),
        "WGRAD dW = dY^T X": (ycol, xcol, [(ffn, hidden)] * experts),
    }
    for name, (A, B, shapes) in cases.items():
        outs = run(A, B, shapes)
        for g in range(experts):
            ac, asc = A[g].host()
            bc, bsc = B[g].host()
            ref = orc.gemm_reference(ac, asc, bc, bsc, grid=grid, block=(1, 16))
            assert _rel(outs[g], ref) <= TOL, (name, g)


def test_gemm_empty_sum_and_empty_group():
    """K = 0 gives D = 0 (an expert that received no token, in WGRAD); a group
    with no rows is skipped."""
    desc = ufp4.make_desc(grid="e1m2", block=(1, 16), scale_fmt=ufp4.SCALE_UE8M0)
    D = torch.full((64, 32), float("nan"), dtype=torch.float32, device=DEV)
    ufp4.ufp4_gemm(ufp4.QTensor(0, 0, 64, 0, 0, 0), ufp4.QTensor(0, 0, 32, 0, 0, 0), desc, D)
    empty = torch.empty((0, 32), dtype=torch.float32, device=DEV)
    ufp4.ufp4_gemm_grouped([ufp4.QTensor(0, 0, 0, 64, 32, 4)], [ufp4.QTensor(0, 0, 32, 64, 32, 4)], desc, [empty])
    torch.cuda.synchronize()
    assert torch.count_nonzero(D).item() == 0
