// E1M2 / INT4 levels as FP8 E5M2 operands of the block-scaled FP8 MMA, and
// the replicated scale-chunk layout of the CTA-pair GEMM kernel.  Shared by
// the GEMM's operand prep (gemm.cu) and the quantizer that writes the
// prepared operands itself (quantize_rows.cu), so both produce the same bytes.
//
// The levels are integers k (|k| <= 7) times the block's step: E1M2 k/4 of
// its scale, INT4 k.  Two 1 x 16 blocks with UE8M0 exponents e0, e1 share one
// hardware scale per 32 elements, hw = max(max(e0, e1) + step_log2, 0), and
// the elements of block b are k * 2^-d_b with d_b = hw - step_log2 - e_b >= 0
// (UFP4 summary, section 方法: the quantized GEMM Y^ = Q_G(X H') Q_G(W H')^T,
// each product exact in the block-scaled MMA while d_b <= 14).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace ufp4 {

__device__ __forceinline__ uint32_t cvt_e5m2x2(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float pow2f(int e) {  // 2^e for e in [-149, 127]
    if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
    if (e < -149) return 0.0f;
    return __uint_as_float(1u << (e + 149));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// Eight sign-magnitude codes (one 32-bit word) -> eight E5M2 bytes of
// k * 2^-d, d <= 14 (two words).  lo and hi hold the E5M2 bytes of 0, 1, ..., 7
// with d already subtracted from the exponent field of the nonzero ones
// (e5m2_tables); the magnitudes select from them and the sign bits select
// 0x80 or 0 (byte permutes).  Exact: every k * 2^-d with |k| <= 7, d <= 14 is
// an E5M2 normal number.
__device__ __forceinline__ void e5m2x8(uint32_t w, uint32_t lo, uint32_t hi, uint32_t& o0, uint32_t& o1) {
    const uint32_t mw = w & 0x77777777u;
    const uint32_t sw = (w >> 3) & 0x11111111u;  // each nibble: its sign bit
    o0 = prmt(lo, hi, mw) | prmt(0x00008000u, 0u, sw);
    o1 = prmt(lo, hi, mw >> 16) | prmt(0x00008000u, 0u, sw >> 16);
}

// E5M2 bytes of 0, 1.0, 2.0, 3.0 (lo) and 4.0 .. 7.0 (hi), each nonzero one
// scaled by 2^-d (d <= 14: every byte stays >= 4 d, so no borrow crosses bytes).
__device__ __forceinline__ void e5m2_tables(int d, uint32_t& lo, uint32_t& hi) {
    const uint32_t sub = (uint32_t)d * 0x04040404u;
    lo = 0x42403C00u - (sub & 0xFFFFFF00u);
    hi = 0x47464544u - sub;
}

// Eight two's complement INT4 nibbles -> sign-magnitude (no -8 code occurs).
__device__ __forceinline__ uint32_t twos_to_signmag8(uint32_t v) {
    const uint32_t neg = (v >> 3) & 0x11111111u;
    const uint32_t mag = ((v ^ (neg * 15u)) + neg) & 0x77777777u;
    return mag | (neg << 3);
}

// The 16 elements of one block (two words of sign-magnitude nibbles, element
// i in bits 4i..4i+3 of the pair) as 16 E5M2 bytes of k * 2^-d.  Beyond
// d = 14 the values leave E5M2's normal range: they are formed in fp32
// (exact) and rounded to E5M2 (nearest even), which is exact down to its
// smallest subnormal 2^-16.
__device__ __forceinline__ uint4 widen16_e5m2(uint32_t w0, uint32_t w1, int d) {
    uint32_t o[4];
    if (d <= 14) {
        uint32_t lo, hi;
        e5m2_tables(d, lo, hi);
        e5m2x8(w0, lo, hi, o[0], o[1]);
        e5m2x8(w1, lo, hi, o[2], o[3]);
    } else {
        const float mult = pow2f(-d);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t v = ((k < 2 ? w0 : w1) >> (16 * (k & 1))) & 0xFFFFu;
            float f[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t nib = (v >> (4 * u)) & 0xFu;
                const float m = (float)(int)(nib & 7u);
                f[u] = ((nib & 8u) ? -m : m) * mult;
            }
            o[k] = cvt_e5m2x2(f[1], f[0]) | (cvt_e5m2x2(f[3], f[2]) << 16);
        }
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

// Byte offset of the scale cell of (row w of the 128-row part h of GEMM tile
// t, 32-element group g) in the replicated chunk array of the CTA-pair
// kernel: chunk g / 4 along K of that part (parts = ceil(tile_rows / 128)
// per tile), stored four times (copy 0..3, 512 bytes apart), cell j = g % 4
// at (w % 32) * 16 + (w / 32) * 4 + j in each copy (the tcgen05.cp 32x128b
// chunk layout).  Operand row r is t = r / tile_rows, h = (r % tile_rows) /
// 128, w = r % tile_rows % 128.
// A tile's last part may hold fewer than 128 rows (part_rows); the cells of
// its rows w >= part_rows belong to no operand row and are written as zero.
__device__ __forceinline__ int64_t chunk_cell_offset_twh(int t, int h, int w, int g, int parts, int chunks_k) {
    return ((((int64_t)t * chunks_k + (g >> 2)) * parts + h) * 4) * 512 + (w & 31) * 16 + (w >> 5) * 4 + (g & 3);
}

}  // namespace ufp4
