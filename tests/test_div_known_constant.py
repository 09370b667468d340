"""The quantizer's fp32 block scale s = fp32(M / qmax) is computed by division
by a constant known in advance (csrc/ufp4_device.cuh, div_known_rn: q0 =
RN(M z) with z = RN(1/qmax), rem = fma(-q0, qmax, M), s = fma(rem, z, q0)).
This checks that restatement of the method against IEEE division on the CPU:
every 97th fp32 bit pattern from 2^-123 up, and three binades exhaustively
(the low end of that range, [1, 2) and [2^120, 2^121)), for qmax = 1.75
(E1M2), 7 (INT4) and 6 (E2M1).  The GPU side is bit-exact against the oracle
in every fp32-scale parity test."""
import shutil
import subprocess

import pytest

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>
static float f_of(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static float div_known(float x, float q, float z) {
    float q0 = x * z;
    float rem = fmaf(-q0, q, x);
    return fmaf(rem, z, q0);
}
static uint64_t check(float q, uint32_t lo, uint32_t hi, uint32_t stride) {
    volatile float qv = q;
    const float z = 1.0f / qv;
    uint64_t bad = 0;
    for (uint64_t u = lo; u < hi; u += stride) {
        const float x = f_of((uint32_t)u);
        if (div_known(x, qv, z) != x / qv) ++bad;
    }
    return bad;
}
int main(void) {
    const float qs[3] = {1.75f, 7.0f, 6.0f};
    const uint32_t lo = 0x02000000u;  /* 2^-123 */
    for (int i = 0; i < 3; ++i) {
        uint64_t bad = check(qs[i], lo, 0x7F800000u, 97);
        bad += check(qs[i], lo, lo + 0x800000u, 1);                  /* [2^-123, 2^-122) */
        bad += check(qs[i], 0x3F800000u, 0x40000000u, 1);            /* [1, 2) */
        bad += check(qs[i], 0x7B800000u, 0x7C000000u, 1);            /* [2^120, 2^121) */
        printf("%g %llu\n", (double)qs[i], (unsigned long long)bad);
    }
    return 0;
}
"""


def test_division_by_known_qmax_is_correctly_rounded(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "div_known.c"
    exe = tmp_path / "div_known"
    src.write_text(SRC)
    subprocess.run([cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-o", str(exe), str(src), "-lm"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    results = {float(out[i]): int(out[i + 1]) for i in range(0, len(out), 2)}
    assert results == {1.75: 0, 7.0: 0, 6.0: 0}
