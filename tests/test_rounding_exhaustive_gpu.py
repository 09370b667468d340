"""The quantizer's rounding and packing step against the oracle's on every fp32
value a block can hold: all finite t with |t| <= qmax, both signs, for RTNE
and SR (draws a fixed function of each value) on every 4-bit grid, through
both arithmetic paths of the device code (fp32 scales and UE8M0 scales;
E2M1 takes the same path under both).  UFP4 summary, section 数据集: RTNE
(nearest level, ties to the even index) and SR to the codebook levels, the
4-bit encodings, a zero level written as +0.

The device side runs ufp4_round_levels, the quantizer's own code on blocks
whose reciprocal is 1.  The oracle side runs in spawned worker processes
(tests/oracle_sweep.py); each chunk is compared by the CRC-32 of its codes,
and a differing chunk is compared element by element to report the first
difference."""
import multiprocessing
import os
import zlib

import numpy as np
import pytest
import torch

import oracle as orc
from rht_bit_block_gb300 import ufp4
from tests import oracle_sweep

pytestmark = pytest.mark.gpu

CHUNK = 1 << 26
CASES = [(g, r, f) for r in (orc.RTNE, orc.SR)
         for g, f in (("e1m2", ufp4.SCALE_FP32), ("int4", ufp4.SCALE_FP32), ("e2m1", ufp4.SCALE_FP32),
                      ("e2m1r2", ufp4.SCALE_FP32), ("e1m2", ufp4.SCALE_UE8M0), ("int4", ufp4.SCALE_UE8M0))]


def _chunks(n: int):
    """[first, first + count) ranges covering 0 .. n - 1 (n >= CHUNK), each count a
    multiple of 32; the last one starts early enough to stay inside the range."""
    assert n >= CHUNK
    out, first = [], 0
    while first < n:
        count = min(CHUNK, n - first)
        if count % 32:
            count = min(n, (count + 31) // 32 * 32)
            first = n - count
        out.append((first, count))
        first += count
    return out


def _device_codes(grid, rounding, fmt, first, count, negative):
    dev = torch.device("cuda", 0)
    bits = torch.arange(first, first + count, dtype=torch.int32, device=dev)
    if negative:
        bits = bits | torch.tensor(-(1 << 31), dtype=torch.int32, device=dev)
    t = bits.view(torch.float32)
    u = None
    if rounding == orc.SR:
        b64 = bits.to(torch.int64) & 0xFFFFFFFF
        u = (((b64 * oracle_sweep.DRAW_MULT) >> 13) & 0xFFFF).to(torch.int32).to(torch.int16)
    codes = torch.empty(count // 2, dtype=torch.uint8, device=dev)
    ufp4.ufp4_round_levels(grid, rounding, fmt, t, codes, u)
    return codes.cpu().numpy()


def _first_difference(grid, rounding, fmt, first, count, negative):
    got = _device_codes(grid, rounding, fmt, first, count, negative)
    want = oracle_sweep.oracle_codes(grid, rounding, first, count, negative)
    i = int(np.nonzero(got != want)[0][0])
    bits = oracle_sweep.chunk_bits(first, count, negative)[2 * i: 2 * i + 2]
    return (f"{grid} {'SR' if rounding else 'RTNE'} scale_fmt {fmt}: t = {bits.view(np.float32).tolist()} "
            f"(bits {[hex(b) for b in bits.tolist()]}): device byte {got[i]:#04x}, oracle {want[i]:#04x}")


def test_rounding_matches_oracle_on_every_fp32_value():
    torch.cuda.init()
    work = []
    for grid, rounding, fmt in CASES:
        n = int(np.float32(orc.qmax(grid)).view(np.uint32)) + 1  # bit patterns 0 .. qmax
        for negative in (False, True):
            for first, count in _chunks(n):
                work.append((grid, rounding, fmt, first, count, negative))
    # the oracle does not depend on the scale format: one task per distinct chunk
    tasks = sorted({(g, r, f0, c, neg) for g, r, _, f0, c, neg in work})
    ctx = multiprocessing.get_context("spawn")
    with ctx.Pool(max(1, os.cpu_count() or 1)) as pool:
        pending = pool.map_async(oracle_sweep.oracle_crc, tasks, chunksize=1)
        got = {w: zlib.crc32(_device_codes(*w)) for w in work}
        assert ufp4.ufp4_device_error() == 0
        want = dict(zip(tasks, pending.get()))
    bad = [w for w in work if got[w] != want[(w[0], w[1], w[3], w[4], w[5])]]
    assert not bad, _first_difference(*bad[0])
    # the sweep reached the top level: +qmax and -qmax (the last values of the
    # two ranges) take the largest code of each grid
    top = {"e1m2": 7, "int4": 7, "e2m1": 7, "e2m1r2": 4}
    for grid, rounding, fmt in CASES:
        n = int(np.float32(orc.qmax(grid)).view(np.uint32)) + 1
        for negative in (False, True):
            last = int(_device_codes(grid, rounding, fmt, n - 32, 32, negative)[-1]) >> 4
            want_top = top[grid] if not negative else ((16 - top[grid]) if grid == "int4" else 8 | top[grid])
            assert last == want_top, (grid, rounding, fmt, negative, last)
