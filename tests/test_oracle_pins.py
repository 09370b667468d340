"""Pins of the oracle to things other than itself (no GPU needed).

Each test ties one oracle function to what the pages or mathematics fix:
closed forms, identities, brute force, library routines and hand-derived
fixtures under tests/golden/.  Citations name the page and section:
  UFP4 summary  = hyper.ai summary of arXiv 2606.20381 (sections 数据集, 方法)
  2D-block page = "Stable FP4 Training via Transposition-Invariant Block Quantization"
"""
import ctypes
import os

import numpy as np
import pytest
import scipy.linalg

import oracle as orc
from rht_bit_block_gb300 import inputs
from tests.conftest import read_golden

GRIDS = ("e1m2", "int4", "e2m1", "e2m1r2")


# ------------------------------------------------------------------ Philox
def _curand():
    for path in ("/usr/local/cuda/lib64/libcurand.so", "libcurand.so", "libcurand.so.10"):
        try:
            return ctypes.CDLL(path)
        except OSError:
            continue
    pytest.skip("libcurand not found")


def _curand_host_philox(seed, nwords, offset_words=0):
    cr = _curand()
    g = ctypes.c_void_p()
    assert cr.curandCreateGeneratorHost(ctypes.byref(g), 161) == 0  # PHILOX4_32_10
    try:
        assert cr.curandSetPseudoRandomGeneratorSeed(g, ctypes.c_ulonglong(seed)) == 0
        assert cr.curandSetGeneratorOffset(g, ctypes.c_ulonglong(offset_words)) == 0
        out = np.zeros(nwords, dtype=np.uint32)
        assert cr.curandGenerate(g, out.ctypes.data_as(ctypes.c_void_p), ctypes.c_size_t(nwords)) == 0
    finally:
        cr.curandDestroyGenerator(g)
    return out.reshape(-1, 4)


@pytest.mark.parametrize("seed", [0, 1234, 0x5EED0001, 0x123456789ABCDEF0, (1 << 64) - 1])
def test_philox_matches_curand_host_generator(seed):
    """Philox4x32-10 (Salmon et al., SC'11) against the cuRAND host library.
    cuRAND's host stream block b is the generator at counter
    (b // 65536, 0, b % 65536, 0) with key = the 64-bit seed; an offset of
    4 * 65536 * 2^32 words carries into the second counter word."""
    key = [seed & 0xFFFFFFFF, seed >> 32]
    blocks = _curand_host_philox(seed, 4 * 8)
    for b in range(8):
        np.testing.assert_array_equal(orc.philox4x32_10([0, 0, b, 0], key), blocks[b])
    blocks = _curand_host_philox(seed, 4 * 4, offset_words=4 * 65536 * 3)
    np.testing.assert_array_equal(orc.philox4x32_10([3, 0, 0, 0], key), blocks[0])
    np.testing.assert_array_equal(orc.philox4x32_10([3, 0, 2, 0], key), blocks[2])
    blocks = _curand_host_philox(seed, 4 * 2, offset_words=4 * 65536 * ((1 << 32) + 5))
    np.testing.assert_array_equal(orc.philox4x32_10([5, 1, 0, 0], key), blocks[0])


def test_philox_fourth_counter_word_matters():
    """The fourth counter word (used for the expert id) enters every output
    word after ten rounds: flipping any one of its bits changes all four words."""
    base = orc.philox4x32_10([7, 0, 1, 0], [11, 13])
    for bit in range(32):
        other = orc.philox4x32_10([7, 0, 1, 1 << bit], [11, 13])
        assert (base != other).all()


def test_philox_bit_balance():
    words = np.concatenate([orc.philox4x32_10([i, 0, 0, 3], [0xDEAD, 0xBEEF]) for i in range(4096)])
    bits = np.unpackbits(words.view(np.uint8))
    n = bits.size
    assert abs(bits.mean() - 0.5) < 4 * 0.5 / np.sqrt(n)
    # each of the 32 bit positions is balanced as well
    per_pos = ((words[:, None] >> np.arange(32, dtype=np.uint32)) & 1).mean(axis=0)
    assert np.all(np.abs(per_pos - 0.5) < 5 * 0.5 / np.sqrt(words.size))


def test_signs_are_balanced_and_seeded():
    e = orc.signs(0x5EED0001, 256)
    assert set(np.unique(e)) <= {-1, 1}
    assert abs(int(e.sum())) < 4 * 16  # 4 sigma for 256 fair signs
    assert not np.array_equal(e, orc.signs(0x5EED0002, 256))
    # the first n signs do not depend on n
    np.testing.assert_array_equal(orc.signs(0x5EED0001, 16), e[:16])


# ----------------------------------------------------------------- Hadamard
def _unit_bf16(n):
    return inputs.f32_to_bf16_bits(np.eye(n, dtype=np.float32))


@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_fwht_reproduces_sylvester_matrix(n):
    """UFP4 summary, 方法: H'_n = S_n H_n with H_n the Sylvester matrix.  The
    oracle's butterfly applied to unit vectors must give S_n H_n entry by
    entry; scipy.linalg.hadamard is the Sylvester +-1 matrix."""
    eps = orc.signs(99, n).astype(np.float64) if n > 1 else np.ones(1)  # n = 1: transform off
    z = orc.rht_rows(_unit_bf16(n), n, 99).astype(np.float64)
    H = scipy.linalg.hadamard(n).astype(np.float64)
    inv = np.float64(np.float32(1.0 / np.sqrt(n)))  # fp32(1/sqrt n), exact for n = 4^j
    np.testing.assert_array_equal(z, eps[:, None] * H * inv)


def test_h4_matches_hand_expanded_recursion():
    H4 = np.array([[float(v) for v in row] for row in read_golden("sylvester_h4.txt")]) / 2.0
    z = orc.rht_rows(_unit_bf16(4), 4, 7).astype(np.float64)
    eps = orc.signs(7, 4).astype(np.float64)
    np.testing.assert_array_equal(z, eps[:, None] * H4)


@pytest.mark.parametrize("n", [2, 4, 16, 64, 256])
def test_hadamard_is_orthogonal(n):
    """UFP4 summary, 方法: H_n^T H_n = I for n = 2^k (fp64, exact for n = 4^j)."""
    eps = orc.signs(5, n).astype(np.float64)
    H = scipy.linalg.hadamard(n) / np.sqrt(n)
    Hp = eps[:, None] * H
    err = np.abs(Hp.T @ Hp - np.eye(n)).max()
    assert err <= (0.0 if n in (4, 16, 64, 256) else 1e-15)


def test_rht_small_integers_is_exact():
    """Small-integer inputs keep every butterfly sum exact, so the fp32 oracle
    equals the fp64 product x S_n H_n bit for bit (n = 16: 1/sqrt n = 1/4)."""
    rng = np.random.default_rng(3)
    x = rng.integers(-8, 9, size=(64, 256)).astype(np.float32)
    z = orc.rht_rows(inputs.f32_to_bf16_bits(x), 16, 1234).astype(np.float64)
    eps = orc.signs(1234, 16).astype(np.float64)
    Hp = eps[:, None] * scipy.linalg.hadamard(16) / 4.0
    ref = (x.astype(np.float64).reshape(64, 16, 16) @ Hp).reshape(64, 256)
    np.testing.assert_array_equal(z, ref)


@pytest.mark.parametrize("n", [16, 32, 64, 256])
def test_rht_random_within_fp32_rounding(n):
    x = inputs.tiny_check(32, 512)
    z = orc.rht_rows(x, n, 42).astype(np.float64)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    eps = orc.signs(42, n).astype(np.float64)
    Hp = eps[:, None] * scipy.linalg.hadamard(n) / np.sqrt(n)
    ref = (xf.reshape(32, -1, n) @ Hp).reshape(32, 512)
    rel = np.abs(z - ref).max(axis=1) / np.abs(ref).max(axis=1)
    assert rel.max() <= 1e-6


def test_rht_preserves_gemm():
    """UFP4 summary, 方法: Y = X W^T = (X H')(W H')^T when the same H' acts on the
    shared dimension.  Small integers make the oracle's transform exact, so
    the identity holds to fp64 rounding."""
    rng = np.random.default_rng(4)
    X = rng.integers(-4, 5, size=(48, 128)).astype(np.float32)
    W = rng.integers(-4, 5, size=(40, 128)).astype(np.float32)
    zx = orc.rht_rows(inputs.f32_to_bf16_bits(X), 64, 77).astype(np.float64)
    zw = orc.rht_rows(inputs.f32_to_bf16_bits(W), 64, 77).astype(np.float64)
    Y = X.astype(np.float64) @ W.astype(np.float64).T
    assert np.abs(zx @ zw.T - Y).max() <= 1e-12 * np.abs(Y).max()
    # different signs on the two operands break it
    zw2 = orc.rht_rows(inputs.f32_to_bf16_bits(W), 64, 78).astype(np.float64)
    assert np.abs(zx @ zw2.T - Y).max() > 1e-3 * np.abs(Y).max()


# ----------------------------------------------------------------- rounding
@pytest.mark.parametrize("grid", GRIDS)
def test_rtne_is_nearest_level_dense_sweep(grid):
    """RTNE picks a nearest level (brute force over the level list)."""
    levels = np.array([orc.level(grid, i) for i in range(orc.num_levels(grid))])
    qm = orc.qmax(grid)
    for a in np.linspace(0.0, qm, 4001, dtype=np.float32):
        idx = orc.round_rtne(grid, float(a))
        d = np.abs(levels - np.float64(a))
        assert d[idx] == d.min()


def test_rtne_ties_go_to_even_code():
    for grid, mid, expect in read_golden("rtne_ties.txt"):
        idx = orc.round_rtne(grid, float(mid))
        assert orc.level(grid, idx) == float(expect), (grid, mid)


def test_uniform_rtne_matches_numpy_rint():
    """On the uniform grids RTNE is numpy's round-half-even of a / step."""
    for grid, step in (("e1m2", 0.25), ("int4", 1.0), ("e2m1r2", 0.5)):
        qm = orc.qmax(grid)
        a = np.random.default_rng(8).uniform(0, qm, 20000).astype(np.float32)
        halves = int(round(2 * qm / step)) + 1  # every level and midpoint in [0, qmax]
        a = np.concatenate([a, (np.arange(0, halves) * 0.5 * step).astype(np.float32)])
        for v in a:
            assert orc.round_rtne(grid, float(v)) == int(np.rint(np.float64(v) / step))


@pytest.mark.parametrize("grid,q,expect", [(r[0], float(r[1]), float(r[2])) for r in read_golden("bin_bias.txt")])
def test_bin_bias_law(grid, q, expect):
    """UFP4 summary, 方法, bin-bias law: for t uniform on the RTNE bin of an
    interior level q_i, E[rho(t) - t] = (2 q_i - q_{i-1} - q_{i+1}) / 4."""
    levels = [orc.level(grid, i) for i in range(orc.num_levels(grid))]
    i = levels.index(q)
    lo, hi = (levels[i - 1] + q) / 2, (q + levels[i + 1]) / 2
    t = np.random.default_rng(int(q * 1000) + len(grid)).uniform(lo, hi, 200_000).astype(np.float32)
    err = np.array([orc.level(grid, orc.round_rtne(grid, float(v))) for v in t]) - t.astype(np.float64)
    sigma = (hi - lo) / np.sqrt(12) / np.sqrt(t.size)
    assert abs(err.mean() - expect) < 5 * sigma + 1e-9


def _sr_bins(grid):
    """The lowest and the highest bin of the grid, and one in the middle."""
    levels = [orc.level(grid, i) for i in range(orc.num_levels(grid))]
    m = len(levels) // 2
    return levels, [(0, 1), (m - 1, m), (len(levels) - 2, len(levels) - 1)]


def _sr_mean_check(grid, idx, levels, i_lo, x):
    lo, hi = levels[i_lo], levels[i_lo + 1]
    assert set(np.unique(idx).tolist()) <= {i_lo, i_lo + 1}, "SR left the two neighbouring levels"
    p = (np.float64(x) - lo) / (hi - lo)
    mean = np.asarray(levels, dtype=np.float64)[idx].mean()
    sigma = (hi - lo) * np.sqrt(p * (1 - p) / idx.size)
    # 16-bit draws: P(up) = ceil(65536 p) / 65536, a bias of at most 2^-16 of the gap
    assert abs(mean - np.float64(x)) < 4 * sigma + (hi - lo) * 2.0 ** -16, (grid, p, mean, np.float64(x))


@pytest.mark.parametrize("grid", GRIDS)
@pytest.mark.parametrize("p", [0.5 + 1e-6, 1e-3, 1 - 1e-3])
def test_sr_is_unbiased(grid, p):
    """2D-block page (stochastic rounding, E[roundS(x)] = x) and UFP4 summary
    (数据集, SR): the oracle's own SR function, applied to 10^6 uniform 16-bit
    draws at adversarial points of three bins per grid, averages to x within
    4 sigma (plus the 2^-16 resolution of the draws).  An 8-bit draw, a wrong
    threshold or a wrong neighbour would miss by far more at p = 1e-3."""
    levels, bins = _sr_bins(grid)
    u = np.random.default_rng(17).integers(0, 65536, 1_000_000).astype(np.uint16)
    for i_lo, i_hi in bins:
        x = np.float32(levels[i_lo] + p * (levels[i_hi] - levels[i_lo]))
        idx = orc.round_sr_array(grid, np.full(u.size, x, dtype=np.float32), u)
        _sr_mean_check(grid, idx, levels, i_lo, x)


@pytest.mark.parametrize("grid", GRIDS)
@pytest.mark.parametrize("p", [0.5 + 1e-6, 1e-3, 1 - 1e-3])
def test_sr_is_unbiased_with_the_quantizer_draws(grid, p):
    """The same law with the draws the quantizer itself uses (Philox4x32-10,
    the 16-bit halves of consecutive output elements), 10^6 elements in both
    the row-wise and the column-wise stream."""
    levels, bins = _sr_bins(grid)
    i_lo = bins[1][0]
    x = np.float32(levels[i_lo] + p * (levels[i_lo + 1] - levels[i_lo]))
    for stream in (0, 1):
        idx = orc.round_sr_philox(grid, float(x), inputs.SR_SEED, 12345 * 8, 1_000_000, stream=stream, group=3)
        _sr_mean_check(grid, idx, levels, i_lo, x)


def test_sr_draw_cross_check():
    """Cross-check of the rule on its own: counting u < p * 65536 over the same
    draws gives the same number of round-ups as the oracle."""
    u = np.random.default_rng(3).integers(0, 65536, 200_000).astype(np.uint16)
    for grid in GRIDS:
        levels = [orc.level(grid, i) for i in range(orc.num_levels(grid))]
        x = np.float32(levels[1] + 0.3141 * (levels[2] - levels[1]))
        thr = (np.float64(x) - levels[1]) / (levels[2] - levels[1]) * 65536.0
        idx = orc.round_sr_array(grid, np.full(u.size, x, dtype=np.float32), u)
        assert int((idx == 2).sum()) == int((u < thr).sum())


@pytest.mark.parametrize("grid", GRIDS)
def test_sr_only_picks_neighbours(grid):
    levels = np.array([orc.level(grid, i) for i in range(orc.num_levels(grid))])
    top = len(levels) - 1
    rng = np.random.default_rng(5)
    for a in rng.uniform(0, orc.qmax(grid), 3000).astype(np.float32):
        idx = orc.round_sr(grid, float(a), int(rng.integers(0, 65536)))
        assert levels[idx] >= a or idx == top or levels[idx + 1] > a
        lo = np.max(np.nonzero(levels <= a)[0])
        assert idx in (lo, min(lo + 1, top))


@pytest.mark.parametrize("v", [1.296875, 1.0078125, 1.9921875])
def test_sr_through_quantizer_is_unbiased(v):
    """Whole quantizer with SR (n = 1, E1M2, fp32 scales): blocks [7, v, ..., v]
    have s = 4, so v / 4 falls between the levels 0.25 and 0.5 at p = 0.297,
    2^-7 and 1 - 2^-7; the mean dequantized v over about 10^6 elements equals
    v within 4 sigma."""
    rows, cols = 1024, 1024
    base = np.tile(np.array([7.0] + [v] * 15, dtype=np.float32), (rows, cols // 16))
    x = inputs.f32_to_bf16_bits(base)
    codes, sc = orc.quantize(x, grid="e1m2", n=1, rounding=orc.SR, sr_seed=9)
    assert (sc == 4.0).all()
    deq = orc.dequantize(codes, sc, grid="e1m2", n=1).astype(np.float64)
    vals = deq.reshape(rows, cols // 16, 16)[:, :, 1:].ravel()
    assert set(np.unique(vals).tolist()) <= {1.0, 2.0}
    p = (v / 4 - 0.25) / 0.25
    sigma = 1.0 * np.sqrt(p * (1 - p) / vals.size)
    assert abs(vals.mean() - v) < 4 * sigma + 2.0 ** -16


# -------------------------------------------------------------------- scale
@pytest.mark.parametrize("grid", GRIDS)
def test_fp32_scale_maps_amax_to_qmax(grid):
    """UFP4 summary, 数据集: s_B = amax / qmax, so the block maximum lands on +-qmax."""
    x = inputs.tiny_check(64, 256)
    codes, sc = orc.quantize(x, grid=grid, n=16, sign_seed=1)
    mags = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(64, 256)
    if grid == "int4":
        k = np.where(mags >= 8, mags.astype(int) - 16, mags.astype(int))
        m = np.abs(k)
    else:
        m = mags & 7
    blockmax = m.reshape(64, 16, 16).max(axis=2)
    assert (blockmax[sc > 0] == orc.num_levels(grid) - 1).all()


@pytest.mark.parametrize("grid", GRIDS)
def test_po2_scale_is_truncation_free_and_tight(grid):
    """2D-block page, truncation-free scaling S = 2^ceil(log2(2M/(Qp-Qn))):
    every block satisfies qmax/2 < M/S <= qmax."""
    qm = orc.qmax(grid)
    rng = np.random.default_rng(6)
    Ms = np.concatenate([rng.lognormal(0, 6, 2000), 2.0 ** np.arange(-30, 30), qm * 2.0 ** np.arange(-30, 30)])
    for M in Ms.astype(np.float32):
        e = orc.po2_exponent(float(M), grid)
        r = np.float64(M) / 2.0 ** e
        assert qm / 2 < r <= qm, (M, e)
    assert orc.po2_exponent(0.0, grid) == -127


def test_e1m2_and_int4_codes_are_identical():
    """fp32(M/1.75) = 4 fp32(M/7) exactly, so E1M2 and INT4 pick the same signed
    integer level k in every mode; only the nibble encoding differs."""
    x = inputs.tiny_check(128, 512)
    for kw in (dict(), dict(scale_fmt=orc.SCALE_UE8M0), dict(rounding=orc.SR, sr_seed=3),
               dict(block=(32, 32), scale_fmt=orc.SCALE_UE8M0, n=64)):
        ce, se = orc.quantize(x, grid="e1m2", **kw)
        ci, si = orc.quantize(x, grid="int4", **kw)
        def k_e(c):
            nib = np.stack([c & 0xF, c >> 4], -1).astype(int)
            return np.where(nib & 8, -(nib & 7), nib & 7)
        def k_i(c):
            nib = np.stack([c & 0xF, c >> 4], -1).astype(int)
            return np.where(nib >= 8, nib - 16, nib)
        np.testing.assert_array_equal(k_e(ce), k_i(ci))
        if kw.get("scale_fmt") == orc.SCALE_UE8M0:
            np.testing.assert_array_equal(se.astype(int), si.astype(int) + 2)
        else:
            np.testing.assert_array_equal(se, si * np.float32(4))


def _quantizer_draws(sr_seed, count, stream=0, group=0):
    """16-bit SR draws of output elements 0 .. count - 1 (row-major), in the
    quantizer's counter layout: Philox4x32-10 with key = sr_seed and counter
    (g lo, g hi, stream, group), g = element / 8; element j of the eight takes
    the low half of word j/2 when j is even, the high half when odd."""
    key = np.array([sr_seed & 0xFFFFFFFF, sr_seed >> 32], dtype=np.uint32)
    out = np.empty(count, dtype=np.uint16)
    for g in range(count // 8):
        w = orc.philox4x32_10(np.array([g, 0, stream, group], dtype=np.uint32), key)
        for j in range(8):
            out[8 * g + j] = (int(w[j // 2]) >> (16 * (j % 2))) & 0xFFFF
    return out


@pytest.mark.parametrize("grid", GRIDS)
def test_round_encode_array_is_the_quantizer_element_step(grid):
    """round_encode_array applies the quantizer's own element step.  With n = 1
    (z = x) and every 1 x 16 block holding +-qmax, the block reciprocal is 1 in
    both scale formats (fp32: s = qmax / qmax; UE8M0: e = 0), so the
    quantizer's codes are the element step of x itself; for SR with the draws
    the quantizer takes for each element."""
    q = np.float32(orc.qmax(grid))
    x = np.random.default_rng(11).uniform(-q, q, size=(32, 64)).astype(np.float32)
    x[:, 0::16] = q
    x[:, 1::16] = -q
    x[:, 2::16] = np.float32(-1e-30)  # rounds to the zero level, written as +0
    xb = inputs.f32_to_bf16_bits(x)
    t = inputs.bf16_bits_to_f32(xb).ravel()
    for fmt in (orc.SCALE_FP32, orc.SCALE_UE8M0):
        c, _ = orc.quantize(xb, grid=grid, n=1, scale_fmt=fmt)
        np.testing.assert_array_equal(c.ravel(), orc.round_encode_array(grid, orc.RTNE, t))
        c, _ = orc.quantize(xb, grid=grid, n=1, scale_fmt=fmt, rounding=orc.SR, sr_seed=inputs.SR_SEED)
        u = _quantizer_draws(inputs.SR_SEED, t.size)
        np.testing.assert_array_equal(c.ravel(), orc.round_encode_array(grid, orc.SR, t, u))


@pytest.mark.parametrize("grid", GRIDS)
def test_zero_block_has_zero_scale_and_codes(grid):
    x = np.zeros((16, 64), dtype=np.uint16)
    x[::2] = 0x8000  # -0.0 in half the rows
    for fmt in (orc.SCALE_FP32, orc.SCALE_UE8M0):
        for rnd in (orc.RTNE, orc.SR):
            codes, sc = orc.quantize(x, grid=grid, scale_fmt=fmt, rounding=rnd, sign_seed=3)
            assert (codes == 0).all()
            assert (sc == 0).all()


# ------------------------------------------------------------- 2D blocks
@pytest.mark.parametrize("b", [8, 16, 32])
@pytest.mark.parametrize("grid", GRIDS)
def test_square_blocks_are_transposition_invariant(grid, b):
    """2D-block page, Eq. S(B) = S(B^T): without the RHT (n = 1) the
    column-wise quantization of X equals the transpose of the row-wise one,
    codes and scales, bit for bit."""
    x = inputs.tiny_check(96, 128)
    kw = dict(grid=grid, block=(b, b), n=1, scale_fmt=orc.SCALE_UE8M0)
    cr, sr = orc.quantize(x, **kw)
    cc, sc = orc.quantize(x, colwise=True, **kw)
    unpack = lambda c: np.stack([c & 0xF, c >> 4], -1).reshape(c.shape[0], -1)
    np.testing.assert_array_equal(unpack(cc), unpack(cr).T)
    np.testing.assert_array_equal(sc, sr.T)


def test_1d_blocks_are_not_transposition_invariant():
    """2D-block page, the transposition problem: 1 x 16 blocks give different
    scales to the same element in X and X^T."""
    x = inputs.tiny_check(64, 64)
    cr, sr = orc.quantize(x, grid="e1m2", n=1, scale_fmt=orc.SCALE_UE8M0)
    cc, sc = orc.quantize(x, grid="e1m2", n=1, scale_fmt=orc.SCALE_UE8M0, colwise=True)
    unpack = lambda c: np.stack([c & 0xF, c >> 4], -1).reshape(c.shape[0], -1)
    assert not np.array_equal(unpack(cc), unpack(cr).T)


# ----------------------------------------------------------- dequantize
@pytest.mark.parametrize("grid", GRIDS)
def test_dequantize_inverse_rht_undoes_rotation(grid):
    """Q_G(T) is the dequantized tensor (UFP4 summary, 数据集); the inverse RHT
    applies H'^T = H S.  Compared with an fp64 product built from scipy's
    Sylvester matrix and the oracle's signs."""
    x = inputs.tiny_check(32, 256)
    codes, sc = orc.quantize(x, grid=grid, n=64, sign_seed=21)
    deq = orc.dequantize(codes, sc, grid=grid, n=64).astype(np.float64)
    inv = orc.dequantize(codes, sc, grid=grid, n=64, sign_seed=21, inverse_rht=True).astype(np.float64)
    eps = orc.signs(21, 64).astype(np.float64)
    Hp = eps[:, None] * scipy.linalg.hadamard(64) / 8.0
    ref = (deq.reshape(32, -1, 64) @ Hp.T).reshape(32, 256)
    assert np.abs(inv - ref).max() <= 1e-6 * np.abs(ref).max()
    # and the reconstruction error is within the grid's resolution
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    seg_err = np.linalg.norm((inv - xf).reshape(32, -1, 16), axis=2)
    step = {"e1m2": 0.25, "int4": 1.0, "e2m1": 2.0, "e2m1r2": 0.5}[grid]
    s = np.repeat(sc.astype(np.float64), 1, axis=1)
    assert (seg_err <= np.sqrt(16) * step / 2 * s.max() * 1.01 + 1e-6).all()


def test_dequantize_values_are_level_times_scale():
    x = inputs.tiny_check(16, 64)
    codes, sc = orc.quantize(x, grid="e2m1", n=16, scale_fmt=orc.SCALE_UE8M0)
    d32 = orc.dequantize(codes, sc, grid="e2m1", scale_fmt=orc.SCALE_UE8M0)
    d64 = orc.dequantize_f64(codes, sc, grid="e2m1", scale_fmt=orc.SCALE_UE8M0)
    np.testing.assert_array_equal(d32.astype(np.float64), d64)
    allowed = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}
    s = np.repeat(2.0 ** (sc.astype(np.float64) - 127), 16, axis=1)
    assert set(np.unique(np.abs(d64 / s))) <= allowed


# ------------------------------------------------------------------ GEMM
def test_gemm_reference_exact_integer_case():
    """PO2 operands with scale 2^0 and integer levels: Q(A)Q(B)^T is an integer
    matrix, equal to numpy's int64 matmul of the signed levels."""
    rng = np.random.default_rng(12)
    M, N, K = 40, 24, 128
    ka = rng.integers(-7, 8, size=(M, K))
    kb = rng.integers(-7, 8, size=(N, K))
    pack = lambda k: ((k[:, 0::2] & 0xF) | ((k[:, 1::2] & 0xF) << 4)).astype(np.uint8)
    sa = np.full((M, K // 16), 127, dtype=np.uint8)
    sb = np.full((N, K // 16), 127, dtype=np.uint8)
    D = orc.gemm_reference(pack(ka), sa, pack(kb), sb, grid="int4", block=(1, 16))
    np.testing.assert_array_equal(D, (ka @ kb.T).astype(np.float64))


# ------------------------------------------------ range-limited E2M1 (E2M1_R2)
def test_range_limited_e2m1_uses_the_uniform_part_of_e2m1():
    """The range-limited grid rounds to E2M1's levels up to 2 and writes plain
    E2M1 codes: its level table is the first five entries of the E2M1
    codebook printed on the UFP4 summary (数据集: E2M1 = {0, 0.5, 1, 1.5, 2,
    3, 4, 6}), and no code above 4 (the level 2) ever appears."""
    e2m1_pages = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert orc.num_levels("e2m1r2") == 5 and orc.qmax("e2m1r2") == 2.0
    assert [orc.level("e2m1r2", i) for i in range(5)] == e2m1_pages[:5]
    x = inputs.tiny_check(128, 512)
    for kw in (dict(), dict(scale_fmt=orc.SCALE_UE8M0), dict(rounding=orc.SR, sr_seed=4)):
        codes, _ = orc.quantize(x, grid="e2m1r2", n=16, sign_seed=2, **kw)
        nib = np.stack([codes & 0xF, codes >> 4], -1)
        assert int((nib & 7).max()) == 4


def test_range_limited_e2m1_has_no_bin_bias_where_e2m1_does():
    """UFP4 summary, 方法 (bin-bias law): E2M1 is biased at q = 2 (its spacing
    changes there); on the range-limited grid the same level sits on a uniform
    run and the bias is zero.  Measured on locally uniform samples."""
    def bias(grid, q):
        levels = [orc.level(grid, i) for i in range(orc.num_levels(grid))]
        i = levels.index(q)
        lo, hi = (levels[i - 1] + q) / 2, (q + levels[i + 1]) / 2
        t = np.random.default_rng(44).uniform(lo, hi, 100_000).astype(np.float32)
        err = np.array([orc.level(grid, orc.round_rtne(grid, float(v))) for v in t]) - t.astype(np.float64)
        return err.mean(), (hi - lo) / np.sqrt(12) / np.sqrt(t.size)
    m, sig = bias("e2m1", 2.0)
    assert abs(m + 0.125) < 5 * sig
    for q in (0.5, 1.0, 1.5):
        m, sig = bias("e2m1r2", q)
        assert abs(m) < 5 * sig


# ----------------------------------------------------------- diagnostics
def test_shrinkage_follows_the_bin_bias_law():
    """UFP4 summary, 方法: with RTNE, E[Q(t) (Q(t) - t)] = sum_i q_i * bias_i
    over the bins.  On a uniform grid the interior biases vanish (E[Q^2] =
    E[Q t] up to sampling noise); E2M1's negative biases at 2 and 4 make
    E[Q^2] < E[Q t]: the values shrink toward zero.  Measured with n = 1 on
    magnitudes uniform up to a bin edge (so every bin is sampled evenly on
    both sides of its level) and one element per 1 x 16 block at amax."""
    edge = {"e1m2": 1.375, "int4": 6.5, "e2m1": 5.0, "e2m1r2": 1.75}  # bin edges below qmax
    res = {}
    for grid, e in edge.items():
        rng = np.random.default_rng(12)
        a = rng.uniform(0.0, e / orc.qmax(grid), (512, 1024)).astype(np.float32)
        a[:, ::16] = 1.0  # amax = 1 in every block: t = a * qmax
        x = inputs.f32_to_bf16_bits(a)
        codes, sc = orc.quantize(x, grid=grid, n=1)
        zz, dd, qz, qq = orc.quant_error_stats(x, codes, sc, grid=grid, n=1)
        res[grid] = ((qq - qz) / dd, qz / zz)
    for grid in ("e1m2", "int4", "e2m1r2"):
        assert abs(res[grid][0]) < 0.2, (grid, res[grid])
    assert res["e2m1"][0] < -1.0
    assert res["e2m1"][1] < min(res[g][1] for g in ("e1m2", "int4", "e2m1r2"))  # stronger shrinkage


# ------------------------------------------------ two-level scale (E4M3 x fp32)
def test_e4m3_rounding_matches_torch_float8():
    """The oracle's E4M3 rounding (written from the format's definition) equals
    torch's float8_e4m3fn conversion (a library routine) on [0, 448]: dense
    random values, every midpoint between neighbouring codes, subnormals."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    vals = [orc.e4m3_decode(b) for b in range(0, 0x7F)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    rng = np.random.default_rng(9)
    xs = np.concatenate([rng.uniform(0, 448, 5000), 2.0 ** rng.uniform(-12, 8.8, 5000), mids, vals])
    xs = xs.astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.e4m3_encode(float(v)) for v in xs], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)
    dec = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.array(vals), dec)


def test_e4m3_is_the_nearest_code_brute_force():
    vals = np.array([orc.e4m3_decode(b) for b in range(0, 0x7F)])  # all finite non-negative codes
    rng = np.random.default_rng(10)
    for a in rng.uniform(0, 448, 3000).astype(np.float32):
        b = orc.e4m3_encode(float(a))
        d = np.abs(vals - np.float64(a))
        assert d[b] == d.min()


def test_two_level_scale_properties():
    """The block holding the tensor amax gets the largest E4M3 scale (448); a
    band quantized with the whole tensor's T equals the same rows of the full
    run; every element is scaled by s = e4m3(b) * g."""
    x = inputs.tiny_check(128, 512)
    for grid in ("e2m1", "e1m2"):
        c, s, T = orc.quantize_2level(x, grid=grid, n=16, sign_seed=4)
        z = orc.rht_rows(x, 16, 4)
        assert T == np.abs(z).max()
        assert s.max() == 0x7E
        cb, sb, Tb = orc.quantize_2level(x[32:64], grid=grid, n=16, sign_seed=4, row0=32, tensor_amax=T)
        np.testing.assert_array_equal(cb, c[32:64])
        np.testing.assert_array_equal(sb, s[32:64])
        deq = orc.dequantize_2level(c, s, T, grid=grid, n=16)
        g = np.float32(orc.tensor_scale(T, grid))
        s_el = np.repeat(np.array([[np.float32(orc.e4m3_decode(b)) * g for b in row] for row in s],
                                  dtype=np.float32), 16, axis=1)
        nib = np.stack([c & 0xF, c >> 4], -1).reshape(c.shape[0], -1).astype(int)
        lev = np.array([orc.level(grid, k) for k in range(8)], dtype=np.float32)[nib & 7]
        lev = np.where(nib & 8, -lev, lev).astype(np.float32)
        np.testing.assert_array_equal(deq, lev * s_el)


# ------------------------------------------------------------------ MXFP8
# The 2D-block page keeps MXFP8 for the Query and Key projections (section on
# mixed precision); the oracle reads it as the OCP MX format: 32-element
# blocks, E8M0 scale 2^(floor(log2 amax) - 8), E4M3 elements, nearest-even,
# saturated at 448.

def _bf16_bits(values):
    return inputs.f32_to_bf16_bits(np.asarray(values, dtype=np.float32))


def test_mxfp8_scale_puts_the_block_amax_in_the_top_binade():
    """floor(log2 amax) - 8: the amax divided by the scale lies in [256, 512),
    the binade of E4M3's largest normal (checked with frexp in fp64)."""
    x = inputs.normal_bf16(64, 256, 11)
    codes, scales = orc.quantize_mxfp8(x)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    amax = np.abs(xf.reshape(64, 8, 32)).max(axis=2)
    ratio = amax / np.ldexp(1.0, scales.astype(np.int64) - 127)
    assert np.all((ratio >= 256.0) & (ratio < 512.0))


def test_mxfp8_elements_match_torch_float8_rounding():
    """Each element is z / X rounded by torch's float8_e4m3fn cast (a library
    routine), saturated at 448; zero stays +0."""
    import torch
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    x = inputs.with_element_outliers(inputs.normal_bf16(32, 512, 12), 0.001, 50.0, 14)
    codes, scales = orc.quantize_mxfp8(x)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    t = xf / np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    tc = np.clip(t, -448.0, 448.0)
    ref = torch.from_numpy(tc).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref = np.where((ref & 0x7F) == 0, 0, ref).astype(np.uint8)
    assert np.array_equal(codes, ref)


def test_mxfp8_is_exact_on_representable_blocks():
    """Blocks built from E4M3 values times 2^k, with the block amax in
    [256, 448] * 2^k, come back unchanged through quantize + dequantize."""
    rng = np.random.default_rng(13)
    e4m3 = np.array([orc.e4m3_decode(b) for b in range(0, 0x7F)])
    rows = []
    for k in (-20, -3, 0, 5, 30):
        vals = rng.choice(e4m3, size=32) * rng.choice([-1.0, 1.0], size=32)
        vals[rng.integers(32)] = rng.choice(e4m3[e4m3 >= 256.0])
        rows.append(np.ldexp(vals, k))
    x = _bf16_bits(np.array(rows))
    codes, scales = orc.quantize_mxfp8(x)
    back = orc.dequantize_mxfp8(codes, scales)
    assert np.array_equal(back, np.array(rows))


def test_mxfp8_saturates_and_keeps_zero_positive():
    """amax / X in (448, 512): the largest element becomes 448 * X; a zero
    block has scale byte 0 and zero codes; -tiny rounds to +0."""
    row = np.zeros(64, dtype=np.float32)
    row[0] = 480.0
    row[1] = -1e-6
    x = _bf16_bits(row[None, :])
    codes, scales = orc.quantize_mxfp8(x)
    assert scales[0, 0] == 127 + 0 and codes[0, 0] == 0x7E
    assert codes[0, 1] == 0x00
    assert scales[0, 1] == 0 and not codes[0, 32:].any()
