"""Thin ctypes binding of libufp4.so (the C ABI in include/ufp4.h).

Argument marshalling only: every step of the quantizer and the GEMM runs in
the library's CUDA kernels.  Functions keep the C names; torch tensors supply
device memory (``data_ptr``) and the current CUDA stream.  The library is
required: importing this module on a machine without it raises.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libufp4.so")

UFP4_OK = 0
UFP4_ERR_TIMEOUT = 5
STATUS_NAMES = {0: "UFP4_OK", 1: "UFP4_ERR_INVALID_ARG", 2: "UFP4_ERR_UNSUPPORTED",
                3: "UFP4_ERR_ALIGNMENT", 4: "UFP4_ERR_CUDA", 5: "UFP4_ERR_TIMEOUT"}
GRID_E1M2, GRID_INT4, GRID_E2M1 = 0, 1, 2
GRID_E2M1_R2 = 3
GRID_MXFP8 = 4  # E4M3 byte codes, 1 x 32 blocks with E8M0 scales
GRIDS = {"e1m2": GRID_E1M2, "int4": GRID_INT4, "e2m1": GRID_E2M1, "e2m1r2": GRID_E2M1_R2, "mxfp8": GRID_MXFP8}
ROUND_RTNE, ROUND_SR = 0, 1
SCALE_FP32, SCALE_UE8M0, SCALE_E4M3 = 0, 1, 2
OUT_ROWWISE, OUT_COLWISE = 1, 2

# Every symbol include/ufp4.h declares (checked by the tests).
EXPORTED = (
    "ufp4_rht_quantize", "ufp4_rht_quantize_grouped", "ufp4_grouped_padded_rows",
    "ufp4_rht_transform", "ufp4_dequantize", "ufp4_gemm_workspace_size", "ufp4_gemm",
    "ufp4_sign_vector", "ufp4_device_error", "ufp4_status_string", "ufp4_gemm_noalloc",
    "ufp4_gemm_grouped_workspace_size", "ufp4_gemm_grouped", "ufp4_gemm_prepare", "ufp4_gemm_prepared",
    "ufp4_rht_quantize_batch", "ufp4_quant_error_stats", "ufp4_error_stats", "ufp4_set_quantize_wait_limit",
    "ufp4_rht_quantize_prepare", "ufp4_round_levels",
)
MAX_BATCH = 4


class QuantDesc(ctypes.Structure):
    _fields_ = [("grid", ctypes.c_int32), ("block_rows", ctypes.c_int32), ("block_cols", ctypes.c_int32),
                ("hadamard_n", ctypes.c_int32), ("sign_seed", ctypes.c_uint64), ("round", ctypes.c_int32),
                ("scale_fmt", ctypes.c_int32), ("sr_seed", ctypes.c_uint64), ("out_mask", ctypes.c_int32),
                ("group", ctypes.c_int32)]


class QTensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("rows", ctypes.c_int64),
                ("cols", ctypes.c_int64), ("codes_ld", ctypes.c_int64), ("scales_ld", ctypes.c_int64),
                ("tensor_amax", ctypes.c_void_p)]


class Ufp4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libufp4.so (build it with rht_bit_block_gb300.build.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: run `python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(path)
    P, i64, i32, u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64
    QD, QT = ctypes.POINTER(QuantDesc), ctypes.POINTER(QTensor)
    L.ufp4_rht_quantize.argtypes = [P, i64, i64, i64, QD, QT, QT, P]
    L.ufp4_rht_quantize_grouped.argtypes = [P, i64, i64, ctypes.POINTER(i64), i32, QD, QT, QT, P]
    L.ufp4_quant_error_stats.argtypes = [P, i64, i64, i64, QD, QT, P, P]
    L.ufp4_error_stats.argtypes = [P, i64, P, i64, i64, i64, P, P]
    L.ufp4_rht_quantize_batch.argtypes = [i32, ctypes.POINTER(P), ctypes.POINTER(i64), ctypes.POINTER(i64),
                                          ctypes.POINTER(i64), QD, QT, P]
    L.ufp4_grouped_padded_rows.argtypes = [i64, QD]
    L.ufp4_grouped_padded_rows.restype = i64
    L.ufp4_rht_transform.argtypes = [P, i64, i64, i64, i32, u64, P, i64, P]
    L.ufp4_dequantize.argtypes = [QT, QD, i32, P, i64, P]
    L.ufp4_gemm_workspace_size.argtypes = [i64, i64, i64, QD, ctypes.POINTER(ctypes.c_size_t)]
    L.ufp4_gemm.argtypes = [QT, QT, QD, P, i64, P, ctypes.c_size_t, P]
    L.ufp4_gemm_noalloc.argtypes = [QT, QT, QD, P, i64, P]
    L.ufp4_gemm_prepare.argtypes = [QT, QT, QD, P, ctypes.c_size_t, P]
    L.ufp4_gemm_prepared.argtypes = [QT, QT, QD, P, i64, P, ctypes.c_size_t, P]
    L.ufp4_rht_quantize_prepare.argtypes = [P, i64, P, i64, QD, QT, QT, P, ctypes.c_size_t, P]
    L.ufp4_gemm_grouped_workspace_size.argtypes = [i32, QT, QT, QD, ctypes.POINTER(ctypes.c_size_t)]
    L.ufp4_gemm_grouped.argtypes = [i32, QT, QT, QD, ctypes.POINTER(P), ctypes.POINTER(i64), P, ctypes.c_size_t, P]
    L.ufp4_sign_vector.argtypes = [u64, i32, P]
    L.ufp4_round_levels.argtypes = [i32, i32, i32, P, P, i64, P, P]
    L.ufp4_device_error.argtypes = [ctypes.POINTER(i32)]
    L.ufp4_set_quantize_wait_limit.argtypes = [i64]
    L.ufp4_set_quantize_wait_limit.restype = ctypes.c_int
    L.ufp4_status_string.argtypes = [ctypes.c_int]
    L.ufp4_status_string.restype = ctypes.c_char_p
    for name in ("ufp4_rht_quantize", "ufp4_rht_quantize_grouped", "ufp4_rht_transform", "ufp4_dequantize",
                 "ufp4_gemm_workspace_size", "ufp4_gemm", "ufp4_sign_vector", "ufp4_device_error",
                 "ufp4_gemm_noalloc", "ufp4_gemm_grouped_workspace_size", "ufp4_gemm_grouped",
                 "ufp4_gemm_prepare", "ufp4_gemm_prepared", "ufp4_rht_quantize_prepare", "ufp4_round_levels"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


def _check(status: int, what: str):
    if status != UFP4_OK:
        raise Ufp4Error(status, what)


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return ctypes.c_void_p(int(stream))


def make_desc(grid="e1m2", block=(1, 16), n=16, sign_seed=0, rounding=ROUND_RTNE, sr_seed=0,
              scale_fmt=SCALE_FP32, out_mask=OUT_ROWWISE, group=0) -> QuantDesc:
    g = GRIDS[grid] if isinstance(grid, str) else int(grid)
    return QuantDesc(g, block[0], block[1], n, sign_seed, rounding, scale_fmt, sr_seed, out_mask, group)


def qtensor(codes, scales, rows: int, cols: int, tensor_amax=None) -> QTensor:
    """Describe a quantized matrix held in torch tensors codes [rows, cols/2]
    (uint8; [rows, cols] for MXFP8) and scales [rows/br, cols/bc] (float32 or uint8); tensor_amax: a
    1-element float32 tensor for the two-level scale format."""
    return QTensor(codes.data_ptr(), scales.data_ptr(), rows, cols, codes.stride(0) * codes.element_size(),
                   scales.stride(0), tensor_amax.data_ptr() if tensor_amax is not None else None)


# ------------------------------------------------------------- C entry points
def ufp4_rht_quantize(x, desc: QuantDesc, rowwise: QTensor | None, colwise: QTensor | None, stream=None):
    rows, cols = x.shape
    _check(load().ufp4_rht_quantize(x.data_ptr(), rows, cols, x.stride(0), ctypes.byref(desc),
                                    ctypes.byref(rowwise) if rowwise is not None else None,
                                    ctypes.byref(colwise) if colwise is not None else None,
                                    _stream(stream)), "ufp4_rht_quantize")


def ufp4_rht_quantize_batch(xs, desc: QuantDesc, rowwise, stream=None):
    """Row-wise quantization of several 2-D bf16 tensors sharing `desc`, one launch."""
    k = len(xs)
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    ptrs = (P * max(k, 1))(*[x.data_ptr() for x in xs])
    rows = (I64 * max(k, 1))(*[x.shape[0] for x in xs])
    cols = (I64 * max(k, 1))(*[x.shape[1] for x in xs])
    lds = (I64 * max(k, 1))(*[x.stride(0) for x in xs])
    outs = (QTensor * max(k, 1))(*rowwise)
    _check(load().ufp4_rht_quantize_batch(k, ptrs, rows, cols, lds, ctypes.byref(desc), outs, _stream(stream)),
           "ufp4_rht_quantize_batch")


def ufp4_quant_error_stats(x, desc: QuantDesc, rowwise: QTensor, stats, stream=None):
    """fp64 sums [sum z^2, sum (q-z)^2, sum q z, sum q^2] of a row-wise quantization, into `stats` (4 doubles)."""
    rows, cols = x.shape
    _check(load().ufp4_quant_error_stats(x.data_ptr(), rows, cols, x.stride(0), ctypes.byref(desc),
                                         ctypes.byref(rowwise), stats.data_ptr(), _stream(stream)),
           "ufp4_quant_error_stats")


def ufp4_error_stats(ref, approx, stats, stream=None):
    """fp64 sums [sum ref^2, sum (approx-ref)^2, sum ref*approx, sum approx^2] of two fp32 matrices."""
    rows, cols = ref.shape
    _check(load().ufp4_error_stats(ref.data_ptr(), ref.stride(0), approx.data_ptr(), approx.stride(0), rows, cols,
                                   stats.data_ptr(), _stream(stream)), "ufp4_error_stats")


def ufp4_rht_quantize_grouped(x, offsets, desc: QuantDesc, rowwise: QTensor | None, colwise: QTensor | None,
                              stream=None):
    cols = x.shape[1]
    arr = (ctypes.c_int64 * len(offsets))(*[int(o) for o in offsets])
    _check(load().ufp4_rht_quantize_grouped(x.data_ptr(), cols, x.stride(0), arr, len(offsets) - 1,
                                            ctypes.byref(desc),
                                            ctypes.byref(rowwise) if rowwise is not None else None,
                                            ctypes.byref(colwise) if colwise is not None else None,
                                            _stream(stream)), "ufp4_rht_quantize_grouped")


def ufp4_grouped_padded_rows(rows: int, desc: QuantDesc) -> int:
    return int(load().ufp4_grouped_padded_rows(rows, ctypes.byref(desc)))


def ufp4_rht_transform(x, n: int, sign_seed: int, z, stream=None):
    rows, cols = x.shape
    _check(load().ufp4_rht_transform(x.data_ptr(), rows, cols, x.stride(0), n, sign_seed, z.data_ptr(),
                                     z.stride(0), _stream(stream)), "ufp4_rht_transform")


def ufp4_dequantize(q: QTensor, desc: QuantDesc, inverse_rht: bool, out, stream=None):
    _check(load().ufp4_dequantize(ctypes.byref(q), ctypes.byref(desc), int(inverse_rht), out.data_ptr(),
                                  out.stride(0), _stream(stream)), "ufp4_dequantize")


def ufp4_gemm_workspace_size(M: int, N: int, K: int, desc: QuantDesc) -> int:
    out = ctypes.c_size_t(0)
    _check(load().ufp4_gemm_workspace_size(M, N, K, ctypes.byref(desc), ctypes.byref(out)),
           "ufp4_gemm_workspace_size")
    return int(out.value)


def ufp4_gemm(A: QTensor, B: QTensor, desc: QuantDesc, D, workspace=None, stream=None):
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().ufp4_gemm(ctypes.byref(A), ctypes.byref(B), ctypes.byref(desc), D.data_ptr(), D.stride(0),
                            ws_ptr, ws_bytes, _stream(stream)), "ufp4_gemm")


def ufp4_gemm_prepare(A: QTensor, B: QTensor, desc: QuantDesc, workspace, stream=None):
    _check(load().ufp4_gemm_prepare(ctypes.byref(A), ctypes.byref(B), ctypes.byref(desc), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "ufp4_gemm_prepare")


def ufp4_rht_quantize_prepare(a, b, desc: QuantDesc, A: QTensor, B: QTensor, workspace, stream=None):
    """Row-wise quantization of the GEMM operands a and b into A and B, and their prepared form in
    `workspace` (what ufp4_gemm_prepare writes), in one launch."""
    _check(load().ufp4_rht_quantize_prepare(a.data_ptr(), a.stride(0), b.data_ptr(), b.stride(0), ctypes.byref(desc),
                                            ctypes.byref(A), ctypes.byref(B), workspace.data_ptr(),
                                            workspace.numel() * workspace.element_size(), _stream(stream)),
           "ufp4_rht_quantize_prepare")


def ufp4_gemm_prepared(A: QTensor, B: QTensor, desc: QuantDesc, D, workspace, stream=None):
    _check(load().ufp4_gemm_prepared(ctypes.byref(A), ctypes.byref(B), ctypes.byref(desc), D.data_ptr(),
                                     D.stride(0), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                     _stream(stream)), "ufp4_gemm_prepared")


def ufp4_gemm_grouped_workspace_size(A, B, desc: QuantDesc) -> int:
    n = len(A)
    arrA, arrB = (QTensor * max(n, 1))(*A), (QTensor * max(n, 1))(*B)
    out = ctypes.c_size_t(0)
    _check(load().ufp4_gemm_grouped_workspace_size(n, arrA, arrB, ctypes.byref(desc), ctypes.byref(out)),
           "ufp4_gemm_grouped_workspace_size")
    return int(out.value)


def ufp4_gemm_grouped(A, B, desc: QuantDesc, D, workspace=None, stream=None):
    """A, B: lists of QTensor; D: list of float32 CUDA tensors (one per group)."""
    n = len(A)
    arrA, arrB = (QTensor * max(n, 1))(*A), (QTensor * max(n, 1))(*B)
    dptr = (ctypes.c_void_p * max(n, 1))(*[d.data_ptr() for d in D])
    ldd = (ctypes.c_int64 * max(n, 1))(*[d.stride(0) if d.dim() == 2 else 1 for d in D])
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().ufp4_gemm_grouped(n, arrA, arrB, ctypes.byref(desc), dptr, ldd, ws_ptr, ws_bytes,
                                    _stream(stream)), "ufp4_gemm_grouped")


def ufp4_gemm_noalloc(A: QTensor, B: QTensor, desc: QuantDesc, D, stream=None):
    """ufp4_gemm without a workspace: the library's fixed device scratch is used
    (for callers that cannot allocate device memory; calls must not overlap)."""
    _check(load().ufp4_gemm_noalloc(ctypes.byref(A), ctypes.byref(B), ctypes.byref(desc), D.data_ptr(),
                                    D.stride(0), _stream(stream)), "ufp4_gemm_noalloc")


def ufp4_sign_vector(sign_seed: int, n: int):
    buf = (ctypes.c_int8 * n)()
    _check(load().ufp4_sign_vector(sign_seed, n, buf), "ufp4_sign_vector")
    return list(buf)


def ufp4_round_levels(grid, rounding: int, scale_fmt: int, t, codes, u16=None, stream=None):
    """The quantizer's rounding and packing step on the scaled values t (device
    float32, |t| <= qmax, numel a multiple of 32) into codes (device uint8,
    numel / 2); u16: device draws for SR."""
    g = GRIDS[grid] if isinstance(grid, str) else int(grid)
    _check(load().ufp4_round_levels(g, rounding, scale_fmt, t.data_ptr(), None if u16 is None else u16.data_ptr(),
                                    t.numel(), codes.data_ptr(), _stream(stream)), "ufp4_round_levels")


def ufp4_device_error() -> int:
    """The device error code (0: no bounded wait gave up since the last read);
    the C call returns UFP4_ERR_TIMEOUT exactly when the code is nonzero."""
    code = ctypes.c_int32(0)
    st = load().ufp4_device_error(ctypes.byref(code))
    if st not in (UFP4_OK, UFP4_ERR_TIMEOUT) or (st == UFP4_ERR_TIMEOUT) != (code.value != 0):
        raise Ufp4Error(st, "ufp4_device_error")
    return int(code.value)


def ufp4_device_error_status() -> int:
    """The status ufp4_device_error returns (UFP4_OK or UFP4_ERR_TIMEOUT)."""
    code = ctypes.c_int32(0)
    return int(load().ufp4_device_error(ctypes.byref(code)))


def ufp4_set_quantize_wait_limit(polls: int):
    """Failure-detection hook: polls of a tile barrier before the quantizer
    kernels give up (negative: the default)."""
    _check(load().ufp4_set_quantize_wait_limit(polls), "ufp4_set_quantize_wait_limit")


def ufp4_status_string(status: int) -> str:
    return load().ufp4_status_string(status).decode()


# ------------------------------------------------------------- conveniences
def alloc_quantized(rows: int, cols: int, desc: QuantDesc, device):
    """torch buffers for one quantized matrix (rows x cols in its own layout)."""
    import torch
    br, bc = desc.block_rows, desc.block_cols
    code_cols = cols if desc.grid == GRID_MXFP8 else cols // 2
    codes = torch.empty((rows, code_cols), dtype=torch.uint8, device=device)
    sdt = torch.float32 if desc.scale_fmt == SCALE_FP32 else torch.uint8
    scales = torch.empty((rows // br, cols // bc), dtype=sdt, device=device)
    return codes, scales


def quantize(x, desc: QuantDesc, stream=None):
    """Quantize a bf16 CUDA tensor; returns {"row": (codes, scales)?, "col": (codes, scales)?}
    (and "row_amax", the tensor amax, for the two-level scale format)."""
    rows, cols = x.shape
    out = {}
    rq = cq = None
    if desc.out_mask & OUT_ROWWISE:
        out["row"] = alloc_quantized(rows, cols, desc, x.device)
        amax = None
        if desc.scale_fmt == SCALE_E4M3:
            import torch
            amax = torch.zeros(1, dtype=torch.float32, device=x.device)
            out["row_amax"] = amax
        rq = qtensor(*out["row"], rows, cols, amax)
    if desc.out_mask & OUT_COLWISE:
        out["col"] = alloc_quantized(cols, rows, desc, x.device)
        cq = qtensor(*out["col"], cols, rows)
    ufp4_rht_quantize(x, desc, rq, cq, stream)
    return out
