"""Failure detection without a GPU fault: the quantizer's bounded waits.

ufp4_set_quantize_wait_limit(0) makes the first tile wait of every quantizer
CTA give up at once.  The kernel must record the timeout, let the copies it
started land (with the normal limit), and return; ufp4_device_error must then
report UFP4_ERR_TIMEOUT, and the next calls must run normally and stay
bit-exact.  No wait is left unbounded and nothing faults, so the GPU stays
usable for the rest of the suite."""
import numpy as np
import pytest
import torch

import oracle as orc
from rht_bit_block_gb300 import inputs, ufp4
from tests.gpu_util import assert_bitwise, gpu_quantize, to_dev

pytestmark = pytest.mark.gpu


# row-only n = 16: the row kernel; row + column: the general kernel; row-only
# n = 64 and n = 256: the segment kernel (per-warp waits, empty barriers; with
# b x b blocks the failed waits meet the band's other warps at its barrier, and
# n = 64 with 16 x 16 blocks, a band of one warp, leaves like 1-D blocks)
@pytest.mark.parametrize("mask,n,block", [(ufp4.OUT_ROWWISE, 16, (1, 16)),
                                          (ufp4.OUT_ROWWISE | ufp4.OUT_COLWISE, 16, (1, 16)),
                                          (ufp4.OUT_ROWWISE, 64, (1, 16)), (ufp4.OUT_ROWWISE, 256, (1, 16)),
                                          (ufp4.OUT_ROWWISE, 64, (32, 32)), (ufp4.OUT_ROWWISE, 256, (32, 32)),
                                          (ufp4.OUT_ROWWISE, 64, (16, 16)), (ufp4.OUT_ROWWISE, 256, (64, 64))])
def test_quantizer_wait_timeout_is_reported_and_recovers(mask, n, block):
    x = inputs.tiny_check(256, 1024)
    kw = dict(grid="e1m2", block=block, n=n, sign_seed=inputs.SIGN_SEED, scale_fmt=ufp4.SCALE_UE8M0)
    xd = to_dev(x)
    torch.cuda.synchronize()
    assert ufp4.ufp4_device_error() == 0
    ufp4.ufp4_set_quantize_wait_limit(0)
    try:
        ufp4.quantize(xd, ufp4.make_desc(out_mask=mask, **kw))
        torch.cuda.synchronize()
        assert ufp4.ufp4_device_error_status() == ufp4.UFP4_ERR_TIMEOUT
        assert ufp4.ufp4_device_error() == 0  # the read cleared it
    finally:
        ufp4.ufp4_set_quantize_wait_limit(-1)
    got = gpu_quantize(xd, out_mask=mask, **kw)
    assert ufp4.ufp4_device_error_status() == ufp4.UFP4_OK
    c, s = orc.quantize(x, grid="e1m2", block=block, n=n, sign_seed=inputs.SIGN_SEED,
                        scale_fmt=orc.SCALE_UE8M0)
    assert_bitwise(got["row"][0], c, "row-wise codes after the timeout")
    assert_bitwise(got["row"][1], s, "row-wise scales after the timeout")
