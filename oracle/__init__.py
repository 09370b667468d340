"""UFP4 oracle (test infrastructure only).

A plain CPU restatement of the fused RHT + block-scaled 4-bit quantizer, used
to check the CUDA library.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import it; the product path never does.

The arithmetic lives in ``ufp4_oracle.c`` (single-threaded C, built with
``-O2 -ffp-contract=off -fno-fast-math``); this module builds it with gcc,
loads it with ctypes and adds the fp64 GEMM reference, which uses one library
matmul as its only step.

Parity pins: every function here is checked against closed forms, brute force
and a library routine by ``tests/test_oracle_pins.py``.  The conventions the
pages leave open (sign generator, packing order, -0 handling, the reciprocal
used to scale, SR bit allocation) are fixed here and in the C ABI header and
are "parity unpinned" by the pages.
"""
from .oracle import *  # noqa: F401,F403
