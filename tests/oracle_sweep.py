"""Oracle side of the exhaustive rounding check (tests/test_rounding_exhaustive_gpu.py).

A module of its own, so that the spawned worker processes import only numpy
and the oracle.  A chunk is `count` consecutive fp32 bit patterns from
`first`, with the sign bit set when `negative`; SR draws are a fixed
function of each value's bit pattern, computed the same way on the device."""
import zlib

import numpy as np

import oracle as orc

DRAW_MULT = 2654435761  # draw = bits 13..28 of (bit pattern * DRAW_MULT) mod 2^64


def chunk_bits(first: int, count: int, negative: bool) -> np.ndarray:
    bits = np.arange(first, first + count, dtype=np.uint32)
    if negative:
        bits |= np.uint32(0x80000000)
    return bits


def draws(bits: np.ndarray) -> np.ndarray:
    prod = bits.astype(np.uint64) * np.uint64(DRAW_MULT)
    return ((prod >> np.uint64(13)) & np.uint64(0xFFFF)).astype(np.uint16)


def oracle_codes(grid: str, rounding: int, first: int, count: int, negative: bool) -> np.ndarray:
    bits = chunk_bits(first, count, negative)
    u = draws(bits) if rounding == orc.SR else None
    return orc.round_encode_array(grid, rounding, bits.view(np.float32), u)


def oracle_crc(task) -> int:
    grid, rounding, first, count, negative = task
    return zlib.crc32(oracle_codes(grid, rounding, first, count, negative))
