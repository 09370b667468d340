"""ufp4_gemm_grouped deals its groups over the caller's stream and two internal
streams.  Checked here: every group equals the same GEMM run alone through
ufp4_gemm, bit for bit; work enqueued on the caller's stream right after the
call sees every group's output; and calls from two host threads on two
streams at the same time give the same bits."""
import threading

import pytest
import torch

from rht_bit_block_gb300 import ufp4

pytestmark = pytest.mark.gpu

DEV = "cuda"
K = 512


def _operands(gen, n_groups):
    """E1M2 1 x 16 UE8M0 operands of n_groups GEMMs with different shapes."""
    desc = ufp4.make_desc(grid="e1m2", block=(1, 16), scale_fmt=ufp4.SCALE_UE8M0)
    shapes = [(128 * (1 + i % 3) + 64, 256 + 32 * i) for i in range(n_groups)]
    A, B, keep = [], [], []
    for M, N in shapes:
        t = []
        for rows in (M, N):
            c = (torch.randint(0, 256, (rows, K // 2), generator=gen, dtype=torch.uint8) & 0x77).to(DEV)
            s = torch.randint(120, 134, (rows, K // 16), generator=gen, dtype=torch.uint8).to(DEV)
            t.append((c, s))
        keep += t
        A.append(ufp4.qtensor(*t[0], M, K))
        B.append(ufp4.qtensor(*t[1], N, K))
    return desc, shapes, A, B, keep


def _one_at_a_time(desc, shapes, A, B):
    outs = []
    for (M, N), a, b in zip(shapes, A, B):
        D = torch.empty((M, N), dtype=torch.float32, device=DEV)
        ws = torch.empty(max(1, ufp4.ufp4_gemm_workspace_size(M, N, K, desc)), dtype=torch.uint8, device=DEV)
        ufp4.ufp4_gemm(a, b, desc, D, ws)
        outs.append(D)
    torch.cuda.synchronize()
    return [d.cpu() for d in outs]


def _grouped(desc, shapes, A, B, stream, reps=1):
    outs = [torch.full((M, N), float("nan"), dtype=torch.float32, device=DEV) for M, N in shapes]
    ws = torch.empty(max(1, ufp4.ufp4_gemm_grouped_workspace_size(A, B, desc)), dtype=torch.uint8, device=DEV)
    for _ in range(reps):
        ufp4.ufp4_gemm_grouped(A, B, desc, outs, ws, stream=stream.cuda_stream)
    return outs, ws


def test_grouped_equals_one_at_a_time_and_orders_the_stream():
    gen = torch.Generator().manual_seed(11)
    desc, shapes, A, B, keep = _operands(gen, 7)
    ref = _one_at_a_time(desc, shapes, A, B)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        outs, ws = _grouped(desc, shapes, A, B, s)
        # enqueued on the caller's stream right after the call: must see every group's output
        early = torch.stack([o.sum() for o in outs])
    s.synchronize()
    for o, r in zip(outs, ref):
        assert torch.equal(o.cpu(), r)
    late = torch.stack([o.sum() for o in outs])
    torch.cuda.synchronize()
    assert torch.equal(early.cpu(), late.cpu())


def test_grouped_from_two_host_threads():
    gen = torch.Generator().manual_seed(12)
    sets = [_operands(gen, 5), _operands(gen, 6)]
    refs = [_one_at_a_time(*st[:4]) for st in sets]
    results, errors = [None, None], []
    barrier = threading.Barrier(2)

    def run(i):
        try:
            desc, shapes, A, B, _ = sets[i]
            s = torch.cuda.Stream()
            barrier.wait(timeout=60)
            outs, ws = _grouped(desc, shapes, A, B, s, reps=4)
            s.synchronize()
            results[i] = [o.cpu() for o in outs]
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=run, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for res, ref in zip(results, refs):
        assert res is not None
        for o, r in zip(res, ref):
            assert torch.equal(o, r)
