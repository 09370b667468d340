"""The C ABI library builds, loads and exports every symbol include/ufp4.h
declares, and rejects bad arguments on the host (no GPU needed: nothing
here launches a kernel)."""
import ctypes
import os
import re

import pytest

from rht_bit_block_gb300 import build, ufp4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ufp4.load()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "ufp4.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z0-9_]+\*?\s+\**(ufp4_[a-z0-9_]+)\s*\(", text, re.M)))


def test_header_declares_the_binding_names():
    assert sorted(ufp4.EXPORTED) == declared_symbols()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code, name in ufp4.STATUS_NAMES.items():
        assert ufp4.ufp4_status_string(code) == name


def test_sign_vector_matches_oracle(lib):
    import oracle as orc
    for n in (1, 2, 16, 256):
        got = ufp4.ufp4_sign_vector(0x5EED0001, n)
        exp = [1] if n == 1 else orc.signs(0x5EED0001, n).tolist()
        assert got == exp


def _call_quantize(lib, desc, rows=64, cols=64, ld=64, x=0x1000, codes=0x2000, scales=0x3000):
    q = ufp4.QTensor(codes, scales, rows, cols, cols // 2, cols // 16)
    return lib.ufp4_rht_quantize(ctypes.c_void_p(x), rows, cols, ld, ctypes.byref(desc), ctypes.byref(q), None,
                                 None)


def test_host_validation_rejects_bad_arguments(lib):
    """Every rejection happens before a launch (fake device addresses are never touched)."""
    ok = ufp4.make_desc(out_mask=ufp4.OUT_ROWWISE)
    bad_n = ufp4.make_desc(n=12)
    bad_block = ufp4.make_desc(block=(2, 16))
    fp32_2d = ufp4.make_desc(block=(32, 32), scale_fmt=ufp4.SCALE_FP32)
    bad_grid = ufp4.make_desc(grid=7)
    assert _call_quantize(lib, bad_n) == 1
    assert _call_quantize(lib, bad_block) == 1
    assert _call_quantize(lib, fp32_2d) == 1
    assert _call_quantize(lib, bad_grid) == 1
    assert _call_quantize(lib, ok, x=0x1001) == 3           # misaligned input
    assert _call_quantize(lib, ok, cols=72, ld=72) == 1      # cols not a multiple of n/16
    assert _call_quantize(lib, ok, ld=32) == 1               # ld < cols
    assert lib.ufp4_rht_quantize(None, 16, 16, 16, ctypes.byref(ok), None, None, None) == 1
    col256 = ufp4.make_desc(n=256, out_mask=ufp4.OUT_COLWISE)
    q = ufp4.QTensor(0x2000, 0x3000, 256, 256, 128, 16)
    assert lib.ufp4_rht_quantize(ctypes.c_void_p(0x1000), 256, 256, 256, ctypes.byref(col256), None,
                                 ctypes.byref(q), None) == 2


def test_gemm_fp32_scales_need_128_element_k_tiles(lib):
    """fp32 block scales run the two-scale path, which walks 128-element K tiles."""
    desc = ufp4.make_desc(scale_fmt=ufp4.SCALE_FP32)
    A = ufp4.QTensor(0x2000, 0x3000, 128, 96, 48, 6)
    D = ctypes.c_void_p(0x4000)
    assert lib.ufp4_gemm(ctypes.byref(A), ctypes.byref(A), ctypes.byref(desc), D, 128, None, 0, None) == 2


def test_batch_validation_rejects_bad_arguments(lib):
    """ufp4_rht_quantize_batch checks every tensor before anything is launched."""
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    def call(desc, count=2, xs=(0x1000, 0x9000), rows=(64, 64), cols=(64, 64), lds=(64, 64)):
        q = (ufp4.QTensor * 2)(*[ufp4.QTensor(0x2000, 0x3000, r, c, c // 2, c // 16) for r, c in zip(rows, cols)])
        return lib.ufp4_rht_quantize_batch(count, (P * 2)(*xs), (I64 * 2)(*rows), (I64 * 2)(*cols),
                                           (I64 * 2)(*lds), ctypes.byref(desc), q, None)
    ok = ufp4.make_desc(out_mask=ufp4.OUT_ROWWISE)
    assert call(ok, count=0) == 0                                          # nothing to do
    assert call(ok, count=ufp4.MAX_BATCH + 1) == 1                          # too many tensors
    assert call(ufp4.make_desc(out_mask=ufp4.OUT_ROWWISE | ufp4.OUT_COLWISE)) == 1  # row-wise only
    assert call(ufp4.make_desc(n=256, out_mask=ufp4.OUT_ROWWISE)) == 1     # cols not a multiple of n
    mx256 = ufp4.make_desc(grid="mxfp8", block=(1, 32), n=256, scale_fmt=ufp4.SCALE_UE8M0, out_mask=ufp4.OUT_ROWWISE)
    assert call(mx256, cols=(256, 256), lds=(256, 256)) == 2                 # MXFP8 keeps n <= 128
    assert call(ufp4.make_desc(block=(32, 32), scale_fmt=ufp4.SCALE_UE8M0, out_mask=ufp4.OUT_ROWWISE)) == 2
    assert call(ok, xs=(0x1000, 0x9001)) == 3                              # second input misaligned
    assert call(ok, cols=(64, 72), lds=(64, 72)) == 1                      # cols not a multiple of 16
    assert call(ok, lds=(64, 32)) == 1                                     # ld < cols
    # an empty tensor's pointer and leading dimension are not looked at
    assert call(ok, count=1, xs=(0, 0), rows=(0, 0), lds=(1, 1)) == 0


def test_quantize_prepare_validation(lib):
    """ufp4_rht_quantize_prepare takes only what it fuses (E1M2 / INT4, UE8M0,
    1-D blocks, n = 16) and checks the GEMM's rules, before anything is launched."""
    P = ctypes.c_void_p
    def call(desc, M=256, N=256, K=256, ws_bytes=1 << 20, a=0x1000, lda=256):
        A = ufp4.QTensor(0x20000, 0x30000, M, K, K // 2, K // 16)
        B = ufp4.QTensor(0x40000, 0x50000, N, K, K // 2, K // 16)
        return lib.ufp4_rht_quantize_prepare(P(a), lda, P(0x9000), K, ctypes.byref(desc), ctypes.byref(A),
                                             ctypes.byref(B), P(0x100000), ws_bytes, None)
    ue8 = dict(scale_fmt=ufp4.SCALE_UE8M0, out_mask=ufp4.OUT_ROWWISE)
    assert call(ufp4.make_desc(grid="e2m1", **ue8)) == 2                  # native FP4: nothing to widen
    assert call(ufp4.make_desc(n=64, **ue8)) == 2                         # n = 16 only
    assert call(ufp4.make_desc(block=(32, 32), **ue8)) == 2               # 1-D blocks only
    assert call(ufp4.make_desc(out_mask=ufp4.OUT_ROWWISE)) == 2           # fp32 scales
    assert call(ufp4.make_desc(scale_fmt=ufp4.SCALE_UE8M0, out_mask=ufp4.OUT_ROWWISE | ufp4.OUT_COLWISE)) == 1
    assert call(ufp4.make_desc(**ue8), ws_bytes=256) == 1                 # workspace too small
    assert call(ufp4.make_desc(**ue8), a=0x1001) == 3                     # a misaligned
    assert call(ufp4.make_desc(**ue8), lda=128) == 1                      # lda < K


def test_round_levels_validation(lib):
    """ufp4_round_levels checks its arguments before anything is launched."""
    P = ctypes.c_void_p
    def call(grid=0, rnd=0, fmt=0, t=0x1000, u=0x2000, count=64, codes=0x3000):
        return lib.ufp4_round_levels(grid, rnd, fmt, P(t), P(u), count, P(codes), None)
    assert call(count=0) == 0                   # nothing to do
    assert call(grid=4) == 1                    # MXFP8 codes are bytes, not levels
    assert call(grid=-1) == 1
    assert call(rnd=2) == 1
    assert call(fmt=2) == 1                     # two-level scales: not a rounding path of their own
    assert call(count=48) == 1                  # a multiple of 32
    assert call(count=-32) == 1
    assert call(t=0) == 1
    assert call(codes=0) == 1
    assert call(rnd=1, u=0) == 1                # SR needs draws
    assert call(t=0x1004) == 3                  # t 16-byte aligned
    assert call(codes=0x3004) == 3              # codes 8-byte aligned
    assert call(rnd=1, u=0x2002) == 3           # draws 4-byte aligned


def test_diagnostics_validation(lib):
    desc = ufp4.make_desc(out_mask=ufp4.OUT_ROWWISE)
    q = ufp4.QTensor(0x2000, 0x3000, 64, 64, 32, 4)
    x = ctypes.c_void_p(0x1000)
    assert lib.ufp4_quant_error_stats(x, 64, 64, 64, ctypes.byref(desc), ctypes.byref(q), None, None) == 1
    assert lib.ufp4_quant_error_stats(x, 64, 64, 64, ctypes.byref(desc), ctypes.byref(q),
                                      ctypes.c_void_p(0x4004), None) == 3       # stats not 8-byte aligned
    assert lib.ufp4_quant_error_stats(x, 64, 72, 72, ctypes.byref(desc), ctypes.byref(q),
                                      ctypes.c_void_p(0x4000), None) == 1       # cols not a multiple of 16
    assert lib.ufp4_error_stats(None, 8, None, 8, 4, 8, None, None) == 1
    assert lib.ufp4_error_stats(ctypes.c_void_p(0x1000), 4, ctypes.c_void_p(0x2000), 8, 4, 8,
                                ctypes.c_void_p(0x4000), None) == 1            # ld < cols


def test_two_level_validation(lib):
    """The two-level scale is row-wise only, needs the tensor-amax slot, and the
    GEMM takes it only for E2M1 codes with 1 x 16 blocks."""
    two = ufp4.make_desc(grid="e2m1", scale_fmt=ufp4.SCALE_E4M3, out_mask=ufp4.OUT_ROWWISE)
    q = ufp4.QTensor(0x2000, 0x3000, 64, 64, 32, 4)  # no tensor_amax
    assert lib.ufp4_rht_quantize(ctypes.c_void_p(0x1000), 64, 64, 64, ctypes.byref(two), ctypes.byref(q), None,
                                 None) == 1
    both = ufp4.make_desc(grid="e2m1", scale_fmt=ufp4.SCALE_E4M3, out_mask=ufp4.OUT_ROWWISE | ufp4.OUT_COLWISE)
    qa = ufp4.QTensor(0x2000, 0x3000, 64, 64, 32, 4, 0x5000)
    assert lib.ufp4_rht_quantize(ctypes.c_void_p(0x1000), 64, 64, 64, ctypes.byref(both), ctypes.byref(qa),
                                 ctypes.byref(qa), None) == 2
    e1m2 = ufp4.make_desc(grid="e1m2", scale_fmt=ufp4.SCALE_E4M3)
    A = ufp4.QTensor(0x2000, 0x3000, 128, 128, 64, 8, 0x5000)
    assert lib.ufp4_gemm(ctypes.byref(A), ctypes.byref(A), ctypes.byref(e1m2), ctypes.c_void_p(0x4000), 128, None, 0,
                         None) == 2


def test_mxfp8_validation(lib):
    """MXFP8 takes 1 x 32 blocks, E8M0 (UE8M0) scales, RTNE and the row-wise
    output only, with byte codes (codes_ld >= cols, a multiple of 16)."""
    UNS, INV, ALN = 2, 1, 3
    mk = lambda **kw: ufp4.make_desc(grid="mxfp8", block=kw.pop("block", (1, 32)),
                                     scale_fmt=kw.pop("scale_fmt", ufp4.SCALE_UE8M0), **kw)
    x, codes, scales = 0x1000, 0x2000, 0x3000

    def call(desc, codes_ld=64, colwise=False, rows=64, cols=64):
        q = ufp4.QTensor(codes, scales, rows, cols, codes_ld, cols // 32)
        c = ufp4.QTensor(codes, scales, cols, rows, rows, rows // 32)
        return lib.ufp4_rht_quantize(ctypes.c_void_p(x), rows, cols, cols, ctypes.byref(desc), ctypes.byref(q),
                                     ctypes.byref(c) if colwise else None, None)
    assert call(mk(block=(1, 16))) == UNS
    assert call(mk(scale_fmt=ufp4.SCALE_FP32)) == UNS
    assert call(mk(rounding=ufp4.ROUND_SR)) == UNS
    assert call(mk(out_mask=3), colwise=True) == UNS
    assert call(mk(), codes_ld=32) == INV      # half-byte leading dimension is too small for byte codes
    assert call(mk(), codes_ld=72) == ALN      # not a multiple of 16
    stats = (ctypes.c_double * 4)()
    q = ufp4.QTensor(codes, scales, 64, 64, 64, 2)
    assert lib.ufp4_quant_error_stats(ctypes.c_void_p(x), 64, 64, 64, ctypes.byref(mk()), ctypes.byref(q),
                                      stats, None) == UNS


def test_grouped_workspace_is_the_sum_of_aligned_group_sizes(lib):
    """Each group takes its own 256-byte aligned region (groups may run side by
    side); a group with an empty product needs none.  A workspace smaller than
    the first group's share is rejected before anything is launched (fake
    device addresses: the first group alone needs its 200 x 160 FP8 copy)."""
    desc = ufp4.make_desc(grid="e1m2", block=(1, 16), scale_fmt=ufp4.SCALE_UE8M0)
    shapes = [(200, 300, 160), (0, 64, 128), (512, 256, 2048), (128, 0, 64), (64, 96, 0)]
    A = [ufp4.QTensor(0x10000, 0x20000, m, k, max(16, k // 2), max(1, k // 16)) for m, n, k in shapes]
    B = [ufp4.QTensor(0x30000, 0x40000, n, k, max(16, k // 2), max(1, k // 16)) for m, n, k in shapes]
    each = []
    for m, n, k in shapes:
        b = ufp4.ufp4_gemm_workspace_size(m, n, k, desc) if m and n and k else 0
        each.append((b + 255) // 256 * 256)
    need = ufp4.ufp4_gemm_grouped_workspace_size(A, B, desc)
    assert need == sum(each) and need > 0
    n = len(shapes)
    arrA, arrB = (ufp4.QTensor * n)(*A), (ufp4.QTensor * n)(*B)
    dptr = (ctypes.c_void_p * n)(*[0x50000] * n)
    ldd = (ctypes.c_int64 * n)(*[max(1, s[1]) for s in shapes])
    assert each[0] > 200 * 160
    rc = lib.ufp4_gemm_grouped(n, arrA, arrB, ctypes.byref(desc), dptr, ldd, ctypes.c_void_p(0x100000),
                               ctypes.c_size_t(256), None)
    assert rc == 1  # UFP4_ERR_INVALID_ARG
