"""Helpers shared by the GPU tests: numpy bf16 bits <-> torch, and calls
through the library's C ABI (rht_bit_block_gb300.ufp4)."""
import numpy as np
import torch

from rht_bit_block_gb300 import ufp4


def to_dev(x_bits: np.ndarray, device="cuda:0", ld=None) -> torch.Tensor:
    """uint16 bf16 bit patterns -> bf16 CUDA tensor (optionally with a wider leading dimension)."""
    t = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16)
    if ld is not None and ld != x_bits.shape[1]:
        big = torch.zeros((x_bits.shape[0], ld), dtype=torch.bfloat16)
        big[:, : x_bits.shape[1]] = t
        return big.to(device)[:, : x_bits.shape[1]]
    return t.to(device)


def gpu_quantize(x_dev: torch.Tensor, **kw):
    desc = ufp4.make_desc(**kw)
    out = ufp4.quantize(x_dev, desc)
    torch.cuda.synchronize()
    res = {k: (v[0].cpu().numpy(), v[1].cpu().numpy()) for k, v in out.items() if k != "row_amax"}
    if "row_amax" in out:
        res["row_amax"] = float(out["row_amax"].cpu().item())
    return res


def assert_bitwise(a: np.ndarray, b: np.ndarray, what: str):
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    av = a.view(np.uint8).reshape(-1)
    bv = b.view(np.uint8).reshape(-1)
    bad = np.nonzero(av != bv)[0]
    if bad.size:
        i = bad[0] // a.itemsize
        raise AssertionError(f"{what}: {bad.size} bytes differ; first element {np.unravel_index(i, a.shape)}: "
                             f"gpu={a.reshape(-1)[i]!r} oracle={b.reshape(-1)[i]!r}")
