"""ctypes binding of the C oracle plus the fp64 GEMM reference (test infrastructure)."""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ufp4_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

E1M2, INT4, E2M1, E2M1_R2 = 0, 1, 2, 3
RTNE, SR = 0, 1
SCALE_FP32, SCALE_UE8M0, SCALE_E4M3 = 0, 1, 2
GRID_NAMES = {"e1m2": E1M2, "int4": INT4, "e2m1": E2M1, "e2m1r2": E2M1_R2}

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-shared", "-fPIC"]


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast math)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i64, u64, u32, i32 = ctypes.c_int64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int
        L.orc_philox4x32_10.argtypes = [P, P, P]
        L.orc_signs.argtypes = [u64, i32, P]
        L.orc_rht_rows.argtypes = [P, i64, i64, i64, i32, u64, P]
        L.orc_rht_rows.restype = i32
        L.orc_quantize_rows.argtypes = [P, i64, i64, i64, i32, i32, i32, i32, u64, i32, u64, i32,
                                        u32, u32, u64, P, P]
        L.orc_quantize_rows.restype = i32
        L.orc_quantize_cols.argtypes = [P, i64, i64, i64, i32, i32, i32, i32, u64, i32, u64, i32,
                                        u32, P, P]
        L.orc_quantize_cols.restype = i32
        L.orc_dequantize.argtypes = [P, P, i64, i64, i32, i32, i32, i32, i32, u64, i32, P]
        L.orc_dequantize.restype = i32
        L.orc_dequantize_f64.argtypes = [P, P, i64, i64, i32, i32, i32, i32, P]
        L.orc_dequantize_f64.restype = i32
        L.orc_level.argtypes = [i32, i32]
        L.orc_level.restype = ctypes.c_double
        L.orc_qmax.argtypes = [i32]
        L.orc_qmax.restype = ctypes.c_double
        L.orc_num_levels.argtypes = [i32]
        L.orc_num_levels.restype = i32
        L.orc_e4m3_encode.argtypes = [ctypes.c_double]
        L.orc_e4m3_encode.restype = ctypes.c_uint8
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_decode.restype = ctypes.c_double
        L.orc_tensor_scale.argtypes = [ctypes.c_float, i32]
        L.orc_tensor_scale.restype = ctypes.c_float
        L.orc_quantize_rows_2level.argtypes = [P, i64, i64, i64, i32, i32, i32, i32, u64, i32, u64, ctypes.c_uint32,
                                               u64, ctypes.c_float, P, P, P]
        L.orc_quantize_rows_2level.restype = i32
        L.orc_dequantize_2level.argtypes = [P, P, i64, i64, i32, i32, i32, ctypes.c_float, i32, u64, i32, P]
        L.orc_dequantize_2level.restype = i32
        L.orc_dequantize_f64_2level.argtypes = [P, P, i64, i64, i32, i32, i32, ctypes.c_float, P]
        L.orc_dequantize_f64_2level.restype = i32
        L.orc_po2_exponent.argtypes = [ctypes.c_float, i32]
        L.orc_po2_exponent.restype = i32
        L.orc_round_rtne.argtypes = [i32, ctypes.c_float]
        L.orc_round_rtne.restype = i32
        L.orc_round_sr.argtypes = [i32, ctypes.c_float, u32]
        L.orc_round_sr.restype = i32
        L.orc_round_sr_array.argtypes = [i32, P, P, i64, P]
        L.orc_round_sr_array.restype = None
        L.orc_round_sr_philox.argtypes = [i32, ctypes.c_float, u64, u64, i64, u32, u32, P]
        L.orc_round_encode_array.argtypes = [i32, i32, P, P, i64, P]
        L.orc_round_sr_philox.restype = None
        L.orc_quantize_rows_mxfp8.argtypes = [P, i64, i64, i64, i32, u64, P, P]
        L.orc_quantize_rows_mxfp8.restype = i32
        L.orc_dequantize_f64_mxfp8.argtypes = [P, P, i64, i64, P]
        L.orc_dequantize_f64_mxfp8.restype = i32
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _grid(g) -> int:
    return GRID_NAMES[g] if isinstance(g, str) else int(g)


# ---------------------------------------------------------------- primitives
def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.asarray(ctr, dtype=np.uint32).copy()
    k = np.asarray(key, dtype=np.uint32).copy()
    out = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def signs(sign_seed: int, n: int) -> np.ndarray:
    out = np.zeros(n, dtype=np.int8)
    lib().orc_signs(sign_seed, n, _ptr(out))
    return out


def level(grid, idx: int) -> float:
    return lib().orc_level(_grid(grid), idx)


def qmax(grid) -> float:
    return lib().orc_qmax(_grid(grid))


def num_levels(grid) -> int:
    """Number of non-negative levels the grid rounds to (qmax is the last)."""
    return lib().orc_num_levels(_grid(grid))


def po2_exponent(M: float, grid) -> int:
    return lib().orc_po2_exponent(M, _grid(grid))


def round_rtne(grid, a: float) -> int:
    return lib().orc_round_rtne(_grid(grid), a)


def round_sr(grid, a: float, u16: int) -> int:
    return lib().orc_round_sr(_grid(grid), a, u16)


def round_sr_array(grid, a: np.ndarray, u16: np.ndarray) -> np.ndarray:
    """orc_round_sr over arrays of magnitudes and 16-bit draws (level indices)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = np.ascontiguousarray(u16, dtype=np.uint16)
    assert a.shape == u.shape
    idx = np.empty(a.shape, dtype=np.uint8)
    lib().orc_round_sr_array(_grid(grid), _ptr(a), _ptr(u), a.size, _ptr(idx))
    return idx


def round_encode_array(grid, rounding, t: np.ndarray, u16: np.ndarray | None = None) -> np.ndarray:
    """The quantizer's element step (clamp to qmax, round, encode with the sign)
    over given scaled values t, packed two per byte like the codes."""
    t = np.ascontiguousarray(t, dtype=np.float32).ravel()
    assert t.size % 2 == 0
    if rounding == SR:
        u = np.ascontiguousarray(u16, dtype=np.uint16).ravel()
        assert u.size == t.size
        up = _ptr(u)
    else:
        up = None
    codes = np.empty(t.size // 2, dtype=np.uint8)
    lib().orc_round_encode_array(_grid(grid), int(rounding), _ptr(t), up, t.size, _ptr(codes))
    return codes


def round_sr_philox(grid, a: float, sr_seed: int, lin0: int, count: int, stream: int = 0,
                    group: int = 0) -> np.ndarray:
    """orc_round_sr of one magnitude with the quantizer's Philox draws of output
    elements lin0 .. lin0 + count - 1 (level indices)."""
    idx = np.empty(count, dtype=np.uint8)
    lib().orc_round_sr_philox(_grid(grid), a, sr_seed, lin0, count, stream, group, _ptr(idx))
    return idx


# ---------------------------------------------------------------- tensors
def _as_bf16(x: np.ndarray) -> np.ndarray:
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns held in uint16 arrays")
    return np.ascontiguousarray(x)


def rht_rows(x_bf16: np.ndarray, n: int, sign_seed: int) -> np.ndarray:
    x = _as_bf16(x_bf16)
    rows, cols = x.shape
    z = np.zeros((rows, cols), dtype=np.float32)
    if lib().orc_rht_rows(_ptr(x), rows, cols, cols, n, sign_seed, _ptr(z)):
        raise ValueError("unsupported RHT arguments")
    return z


def quantize(x_bf16: np.ndarray, *, grid="e1m2", block=(1, 16), n=16, sign_seed=0, rounding=RTNE,
             sr_seed=0, scale_fmt=SCALE_FP32, colwise=False, group=0, row0=0):
    """Quantize a bf16 matrix; returns (codes uint8, scales float32|uint8).

    Row-wise: codes [rows x cols/2], scales [rows/br x cols/bc].
    Column-wise: the quantization of x^T, in x^T's layout.
    row0 (row-wise only): index of x's first row in the whole tensor, used by
    the SR counters when a band of rows is checked on its own."""
    x = _as_bf16(x_bf16)
    rows, cols = x.shape
    g = _grid(grid)
    br, bc = block
    orows, ocols = (cols, rows) if colwise else (rows, cols)
    codes = np.zeros((orows, ocols // 2), dtype=np.uint8)
    sdt = np.float32 if scale_fmt == SCALE_FP32 else np.uint8
    scales = np.zeros((orows // br, ocols // bc), dtype=sdt)
    if colwise:
        rc = lib().orc_quantize_cols(_ptr(x), rows, cols, cols, g, br, bc, n, sign_seed, rounding,
                                     sr_seed, scale_fmt, group, _ptr(codes), _ptr(scales))
    else:
        rc = lib().orc_quantize_rows(_ptr(x), rows, cols, cols, g, br, bc, n, sign_seed, rounding,
                                     sr_seed, scale_fmt, 0, group, row0, _ptr(codes), _ptr(scales))
    if rc:
        raise ValueError("unsupported quantize arguments")
    return codes, scales


def dequantize(codes, scales, *, grid="e1m2", block=(1, 16), scale_fmt=SCALE_FP32, n=16,
               sign_seed=0, inverse_rht=False) -> np.ndarray:
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    rows, half = codes.shape
    cols = 2 * half
    out = np.zeros((rows, cols), dtype=np.float32)
    if lib().orc_dequantize(_ptr(codes), _ptr(scales), rows, cols, _grid(grid), block[0], block[1],
                            scale_fmt, n, sign_seed, int(inverse_rht), _ptr(out)):
        raise ValueError("unsupported dequantize arguments")
    return out


def dequantize_f64(codes, scales, *, grid="e1m2", block=(1, 16), scale_fmt=SCALE_UE8M0) -> np.ndarray:
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    rows, half = codes.shape
    cols = 2 * half
    out = np.zeros((rows, cols), dtype=np.float64)
    if lib().orc_dequantize_f64(_ptr(codes), _ptr(scales), rows, cols, _grid(grid), block[0],
                                block[1], scale_fmt, _ptr(out)):
        raise ValueError("unsupported dequantize arguments")
    return out


def gemm_reference(a_codes, a_scales, b_codes, b_scales, *, grid="e1m2", block=(1, 16),
                   scale_fmt=SCALE_UE8M0, a_rows=None) -> np.ndarray:
    """D = Q(A) Q(B)^T in fp64 [UFP4 summary, section 方法: the quantized GEMM
    Y^ = Q_G(X H') Q_G(W H')^T with Q_G the dequantized operand].  a_rows
    optionally selects a subset of A's rows (sampled check of large shapes)."""
    A = dequantize_f64(a_codes, a_scales, grid=grid, block=block, scale_fmt=scale_fmt)
    if a_rows is not None:
        A = A[np.asarray(a_rows)]
    B = dequantize_f64(b_codes, b_scales, grid=grid, block=block, scale_fmt=scale_fmt)
    return A @ B.T


def quant_error_stats(x_bf16: np.ndarray, codes, scales, *, grid="e1m2", block=(1, 16), scale_fmt=SCALE_FP32, n=16,
                      sign_seed=0) -> np.ndarray:
    """Diagnostics of one row-wise quantization (UFP4 summary, 数据集: Q_G(T) is
    the dequantized tensor; 方法: RTNE shrinkage bin by bin).  z = the RHT of x
    with the quantizer's fp32 arithmetic, q = level * scale (fp32); returns the
    fp64 sums [sum z^2, sum (q - z)^2, sum q z, sum q^2]."""
    z = rht_rows(x_bf16, n, sign_seed).astype(np.float64)
    q = dequantize(codes, scales, grid=grid, block=block, scale_fmt=scale_fmt, n=n).astype(np.float64)
    d = q - z
    return np.array([(z * z).sum(), (d * d).sum(), (q * z).sum(), (q * q).sum()])


# ------------------------------------------------------ two-level scale
def e4m3_encode(a: float) -> int:
    """E4M3 byte of a >= 0, rounded to nearest even, saturated at 448."""
    return int(lib().orc_e4m3_encode(float(a)))


def e4m3_decode(b: int) -> float:
    return float(lib().orc_e4m3_decode(int(b)))


def tensor_scale(tensor_amax: float, grid) -> float:
    """g = fp32(T / fp32(qmax * 448))."""
    return float(lib().orc_tensor_scale(tensor_amax, _grid(grid)))


def quantize_2level(x_bf16: np.ndarray, *, grid="e2m1", block=(1, 16), n=16, sign_seed=0, rounding=RTNE,
                    sr_seed=0, group=0, row0=0, tensor_amax=-1.0):
    """Row-wise quantization with the two-level scale (E4M3 block scales x the
    fp32 tensor scale g): returns (codes, E4M3 scale bytes, tensor amax T).
    tensor_amax < 0 takes T from this call's rows."""
    x = _as_bf16(x_bf16)
    rows, cols = x.shape
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.zeros((rows // block[0], cols // block[1]), dtype=np.uint8)
    t_out = np.zeros(1, dtype=np.float32)
    if lib().orc_quantize_rows_2level(_ptr(x), rows, cols, cols, _grid(grid), block[0], block[1], n, sign_seed,
                                      rounding, sr_seed, group, row0, tensor_amax, _ptr(codes), _ptr(scales),
                                      _ptr(t_out)):
        raise ValueError("unsupported quantizer arguments")
    return codes, scales, float(t_out[0])


def dequantize_2level(codes, scales, tensor_amax: float, *, grid="e2m1", block=(1, 16), n=16, sign_seed=0,
                      inverse_rht=False) -> np.ndarray:
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    rows, half = codes.shape
    out = np.zeros((rows, 2 * half), dtype=np.float32)
    if lib().orc_dequantize_2level(_ptr(codes), _ptr(scales), rows, 2 * half, _grid(grid), block[0], block[1],
                                   tensor_amax, n, sign_seed, int(inverse_rht), _ptr(out)):
        raise ValueError("unsupported dequantize arguments")
    return out


def gemm_reference_2level(a_codes, a_scales, a_amax, b_codes, b_scales, b_amax, *, grid="e2m1",
                          block=(1, 16)) -> np.ndarray:
    """fp64 product of the two-level dequantized operands (level * e4m3 * g)."""
    def deq(c, sc, t):
        c = np.ascontiguousarray(c)
        sc = np.ascontiguousarray(sc)
        rows, half = c.shape
        out = np.zeros((rows, 2 * half), dtype=np.float64)
        if lib().orc_dequantize_f64_2level(_ptr(c), _ptr(sc), rows, 2 * half, _grid(grid), block[0], block[1],
                                           t, _ptr(out)):
            raise ValueError("unsupported arguments")
        return out
    return deq(a_codes, a_scales, a_amax) @ deq(b_codes, b_scales, b_amax).T


def quantize_mxfp8(x_bf16: np.ndarray, *, n=1, sign_seed=0):
    """MXFP8 (E4M3 elements, one E8M0 scale per 32 along the row) of the
    row-wise RHT of x, the format the 2D-block page keeps for the Query and
    Key projections (mixed-precision section), read as the OCP MX
    definition.  Returns (codes [rows x cols] E4M3 bytes, scales [rows x
    cols/32] E8M0 bytes)."""
    x = _as_bf16(x_bf16)
    rows, cols = x.shape
    codes = np.zeros((rows, cols), dtype=np.uint8)
    scales = np.zeros((rows, cols // 32), dtype=np.uint8)
    if lib().orc_quantize_rows_mxfp8(_ptr(x), rows, cols, x.strides[0] // 2, n, sign_seed, _ptr(codes),
                                     _ptr(scales)):
        raise ValueError("unsupported arguments")
    return codes, scales


def dequantize_mxfp8(codes, scales) -> np.ndarray:
    """Exact fp64 values e4m3(code) * 2^(scale byte - 127)."""
    c = np.ascontiguousarray(codes)
    sc = np.ascontiguousarray(scales)
    rows, cols = c.shape
    out = np.zeros((rows, cols), dtype=np.float64)
    if lib().orc_dequantize_f64_mxfp8(_ptr(c), _ptr(sc), rows, cols, _ptr(out)):
        raise ValueError("unsupported arguments")
    return out


def gemm_reference_mxfp8(a_codes, a_scales, b_codes, b_scales, a_rows=None) -> np.ndarray:
    """fp64 product of two dequantized MXFP8 operands (both K-major)."""
    a = dequantize_mxfp8(a_codes, a_scales)
    if a_rows is not None:
        a = a[np.asarray(a_rows)]
    return a @ dequantize_mxfp8(b_codes, b_scales).T
