"""ufp4_gemm_noalloc, the GEMM entry point for callers that cannot allocate
device memory (for example a plugin or custom op whose host framework owns
every device allocation, or a loop that must not risk the device-wide
synchronization an allocation can cause): through the C ABI it must give
exactly what ufp4_gemm gives with a caller-allocated workspace, call after
call.  The first call has the largest footprint, so the later, smaller calls
(other K and N) run over scratch bytes left behind by the earlier ones.  This
file is collected last on purpose."""
import numpy as np
import pytest
import torch

from rht_bit_block_gb300 import inputs, ufp4

pytestmark = pytest.mark.gpu


def _operands(seed, m, n, k, grid):
    desc = ufp4.make_desc(grid=grid, block=(1, 16), n=16, sign_seed=inputs.SIGN_SEED,
                          scale_fmt=ufp4.SCALE_UE8M0, out_mask=ufp4.OUT_ROWWISE)
    to_t = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    x = to_t(inputs.normal_bf16(m, k, seed))
    w = to_t(inputs.normal_bf16(n, k, seed + 1, std=0.02))
    qa = ufp4.quantize(x, desc)["row"]
    qb = ufp4.quantize(w, desc)["row"]
    return desc, ufp4.qtensor(*qa, m, k), ufp4.qtensor(*qb, n, k), (qa, qb)


@pytest.mark.parametrize("grid", ["e1m2", "e2m1"])
def test_noalloc_matches_workspace_gemm_call_after_call(grid):
    torch.cuda.init()
    shapes = [(11, 1024, 1280, 4096), (12, 384, 512, 2048), (13, 256, 448, 1024)]
    for call, (seed, m, n, k) in enumerate(shapes):
        desc, A, B, keep = _operands(seed, m, n, k, grid)
        ref = torch.empty((m, n), dtype=torch.float32, device="cuda")
        ws = torch.empty(max(1, ufp4.ufp4_gemm_workspace_size(m, n, k, desc)), dtype=torch.uint8, device="cuda")
        ufp4.ufp4_gemm(A, B, desc, ref, ws)
        got = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        ufp4.ufp4_gemm_noalloc(A, B, desc, got)
        torch.cuda.synchronize()
        assert ufp4.ufp4_device_error() == 0
        # the same kernels on the same operands: the results must agree bit for bit
        assert torch.equal(got, ref), f"call {call}: noalloc result differs from ufp4_gemm"


def test_noalloc_rejects_shapes_beyond_its_scratch():
    m, n, k = 8192, 8192, 2048  # E1M2 needs (m + n) * k bytes > 32 MiB
    desc = ufp4.make_desc(grid="e1m2", block=(1, 16), scale_fmt=ufp4.SCALE_UE8M0)
    assert ufp4.ufp4_gemm_workspace_size(m, n, k, desc) > 32 * 1024 * 1024
    codes = torch.zeros((m, k // 2), dtype=torch.uint8, device="cuda")
    scales = torch.zeros((m, k // 16), dtype=torch.uint8, device="cuda")
    D = torch.empty((m, n), dtype=torch.float32, device="cuda")
    A = ufp4.qtensor(codes, scales, m, k)
    with pytest.raises(ufp4.Ufp4Error) as e:
        ufp4.ufp4_gemm_noalloc(A, A, desc, D)
    assert e.value.status == 2  # UFP4_ERR_UNSUPPORTED
