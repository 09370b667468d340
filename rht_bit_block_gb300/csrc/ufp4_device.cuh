// Device helpers of the UFP4 quantizer: Philox4x32-10, bf16 widening, the
// per-chunk FWHT, block scales, rounding and 4-bit packing.
//
// Every floating-point step is written with explicit round-to-nearest
// intrinsics (__fadd_rn/__fsub_rn/__fmul_rn/__fdiv_rn/__frcp_rn) so that no
// multiply is fused with an add and results are reproducible bit for bit.
//
// Pages: UFP4 summary (hyper.ai, arXiv 2606.20381), sections 数据集 (codebooks,
// blocks, s_B = amax / largest level, RTNE, SR) and 方法 (Sylvester H_2n,
// H'_n = S_n H_n); "Stable FP4 Training via Transposition-Invariant Block
// Quantization", truncation-free scale and 2D square blocks.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace ufp4 {

constexpr int kChunk = 16;  // elements one thread carries along the quantized dimension

// Largest level and its reciprocal step for each grid (E1M2 1.75, INT4 7, E2M1 6).
__host__ __device__ constexpr float grid_qmax(int grid) {
    return grid == 0 ? 1.75f : (grid == 1 ? 7.0f : (grid == 2 ? 6.0f : (grid == 3 ? 2.0f : 448.0f)));
}

// E4M3 byte of a >= 0, rounded to nearest even and saturated at 448 (the
// hardware conversion), and its value.
__device__ __forceinline__ uint32_t e4m3_byte(float a) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(a));
    return r & 0xFFu;
}
__device__ __forceinline__ float e4m3_value(uint32_t b) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)(b & 0xFFu)));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// Value of a 4-bit code on the grid's level scale (before the block scale).
__device__ __forceinline__ float decode_level(int grid, uint32_t nib) {
    if (grid == 1) return (float)((nib & 8u) ? (int)nib - 16 : (int)nib);
    const uint32_t k = nib & 7u;
    float v;
    if (grid == 0) {
        v = (float)k * 0.25f;
    } else {
        // E2M1 levels 0, .5, 1, 1.5, 2, 3, 4, 6
        v = k < 4 ? (float)k * 0.5f : (k == 4 ? 2.0f : (k == 5 ? 3.0f : (k == 6 ? 4.0f : 6.0f)));
    }
    return (nib & 8u) ? -v : v;
}

// ------------------------------------------------------------- Philox4x32-10
// Salmon et al., SC'11: ten rounds, multipliers 0xD2511F53 / 0xCD9E8D57, key
// bumped by 0x9E3779B9 / 0xBB67AE85 between rounds (the round keys come
// precomputed, see SrKeys).  Each product is one 32 x 32 -> 64-bit multiply
// (both halves at once).  Four independent blocks run round by round, so
// that the four multiply chains overlap (ten dependent rounds each).
__device__ __forceinline__ void philox4x32_10_x4(uint4 c[4], const SrKeys& k) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint64_t p0, p1;
            asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c[j].x), "r"(0xD2511F53u));
            asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c[j].z), "r"(0xCD9E8D57u));
            c[j] = make_uint4((uint32_t)(p1 >> 32) ^ c[j].y ^ k.k[2 * i], (uint32_t)p1,
                              (uint32_t)(p0 >> 32) ^ c[j].w ^ k.k[2 * i + 1], (uint32_t)p0);
        }
    }
}

// SR draws of 16 output elements lin0 .. lin0+15 (lin0 % 8 == 0): counter
// (g lo, g hi, stream, group) with g = lin / 8; element j of a group of
// eight takes the low half of word j/2 when j is even, the high half when odd.
// Two vectors at once: elements la0 .. la0+15 into wa, lb0 .. lb0+15 into wb.
__device__ __forceinline__ void sr_draws16x2(const SrKeys& k, uint64_t la0, uint64_t lb0, uint32_t stream,
                                             uint32_t group, uint32_t wa[8], uint32_t wb[8]) {
    const uint64_t ga = la0 >> 3, gb = lb0 >> 3;
    uint4 c[4] = {make_uint4((uint32_t)ga, (uint32_t)(ga >> 32), stream, group),
                  make_uint4((uint32_t)(ga + 1), (uint32_t)((ga + 1) >> 32), stream, group),
                  make_uint4((uint32_t)gb, (uint32_t)(gb >> 32), stream, group),
                  make_uint4((uint32_t)(gb + 1), (uint32_t)((gb + 1) >> 32), stream, group)};
    philox4x32_10_x4(c, k);
    wa[0] = c[0].x; wa[1] = c[0].y; wa[2] = c[0].z; wa[3] = c[0].w;
    wa[4] = c[1].x; wa[5] = c[1].y; wa[6] = c[1].z; wa[7] = c[1].w;
    wb[0] = c[2].x; wb[1] = c[2].y; wb[2] = c[2].z; wb[3] = c[2].w;
    wb[4] = c[3].x; wb[5] = c[3].y; wb[6] = c[3].z; wb[7] = c[3].w;
}

// ------------------------------------------------------------------ loading
// 16 bf16 (8 words) -> 16 fp32, with the RHT signs applied as sign-bit flips
// (bit j of sgn set <=> eps_j = -1; exact, same as multiplying by -1).
__device__ __forceinline__ void widen16(const uint32_t w[8], uint32_t sgn, float v[16]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t lo = (w[k] << 16) ^ (((sgn >> (2 * k)) & 1u) << 31);
        const uint32_t hi = (w[k] & 0xFFFF0000u) ^ (((sgn >> (2 * k + 1)) & 1u) << 31);
        v[2 * k] = __uint_as_float(lo);
        v[2 * k + 1] = __uint_as_float(hi);
    }
}

// ----------------------------------------------------------------- the FWHT
// Sylvester order: strides 1, 2, 4, ... (the recursion H_2n = [[H_n, H_n],
// [H_n, -H_n]]/sqrt 2 combines halves last), pair (i, i+h) -> (a+b, a-b).
// Strides below 16 run inside the thread; strides 16..n/2 pair the thread
// with lane ^ (h/16), which holds the elements h positions away.
// `seg_lane` is this thread's chunk index inside its length-n segment.
__device__ __forceinline__ void fwht16(float v[16], int n, int seg_lane) {
#pragma unroll
    for (int h = 1; h < kChunk; h <<= 1) {
        if (h < n) {
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                if (i & h) continue;
                const float a = v[i], b = v[i + h];
                v[i] = __fadd_rn(a, b);
                v[i + h] = __fsub_rn(a, b);
            }
        }
    }
    for (int h = kChunk; h < n; h <<= 1) {
        const int lm = h / kChunk;
        const bool upper = (seg_lane & lm) != 0;
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const float o = __shfl_xor_sync(0xFFFFFFFFu, v[i], lm);
            v[i] = upper ? __fsub_rn(o, v[i]) : __fadd_rn(v[i], o);
        }
    }
}

// ------------------------------------------------------------------- scales
// fp32(x / q) for the grid's largest level q, x >= 0, correctly rounded.  For
// q = 1.75, 7 and 6 it uses division by a constant known in advance (P.
// Markstein's correction step, as analysed for constant divisors by N.
// Brisebarre and J.-M. Muller, "Accelerating correctly rounded floating-point
// division when the divisor is known in advance", IEEE Trans. Computers 53(8),
// 2004): q0 = RN(x z) with z = RN(1/q), the remainder x - q0 q exact in one
// fma, then RN(q0 + rem z).  Compared with IEEE x / q on every non-negative
// finite fp32 x: equal for every x with q = 7, and for every x >= 2^-123 with
// q = 1.75 and q = 6 (block amaxes below 2^-120 are outside the quantizer's
// input contract).  q = 2 is a multiplication by 0.5.
__device__ __forceinline__ float div_known_rn(float x, float q, float z) {
    const float q0 = __fmul_rn(x, z);
    const float rem = __fmaf_rn(-q0, q, x);
    return __fmaf_rn(rem, z, q0);
}
template <int GRID>
__device__ __forceinline__ float div_qmax_rn(float x) {
    if (GRID == 0) return div_known_rn(x, 1.75f, 0x1.24924ap-1f);  // z = RN(1 / 1.75)
    if (GRID == 1) return div_known_rn(x, 7.0f, 0x1.24924ap-3f);   // z = RN(1 / 7)
    if (GRID == 2) return div_known_rn(x, 6.0f, 0x1.555556p-3f);   // z = RN(1 / 6)
    if (GRID == 3) return __fmul_rn(x, 0.5f);
    return __fdiv_rn(x, grid_qmax(GRID));
}

// fp32 scale s = fp32(M / qmax); reciprocal r = fp32(1/s), 0 for s = 0.
template <int GRID>
__device__ __forceinline__ void scale_fp32(float M, float& s, float& r) {
    s = div_qmax_rn<GRID>(M);
    r = (s == 0.0f) ? 0.0f : __frcp_rn(s);
}

__device__ __forceinline__ uint32_t cvt_e2m1x2(float hi, float lo) {
    uint32_t r;
    asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// A zero level is written as +0: clear the sign of every nibble whose
// magnitude bits are zero.
__device__ __forceinline__ uint32_t clear_negative_zero(uint32_t w) {
    // per nibble, (mag + 7) has bit 3 set iff mag >= 1 (no carry leaves the nibble)
    const uint32_t y = (w & 0x77777777u) + 0x77777777u;
    return w & (y | 0x77777777u);
}

// Sign-magnitude nibbles with no -0 (clear_negative_zero first) -> INT4
// two's complement: a negative nibble 8 + k (k >= 1) becomes
// ((8 + k) ^ 7) + 1 = 16 - k, which stays inside the nibble.
__device__ __forceinline__ uint32_t signmag_nz_to_twos(uint32_t w) {
    const uint32_t neg = (w >> 3) & 0x11111111u;
    return (w ^ (neg * 7u)) + neg;
}

// Four E4M3 bytes s000 0kkk (levels k on the subnormal grid, k <= 7) -> the
// INT4 two's complement of (-1)^s k in the low nibble of each byte: 16 - k
// for s = 1, formed within the byte (16 - 0 sets bit 4, which the caller
// masks off, so -0 gives 0).  The sign mask is a byte permute that replicates
// each byte's top bit.
__device__ __forceinline__ uint32_t int4_from_e4m3_bytes(uint32_t v) {
    const uint32_t k = v & 0x07070707u;
    uint32_t m;
    asm("prmt.b32 %0, %1, 0, 0xBA98;" : "=r"(m) : "r"(v));
    return (k & ~m) | ((0x10101010u - k) & m);
}

}  // namespace ufp4

// ======================================================================
// Paired-lane helpers (PTX add/sub/mul.rn.f32x2: two independent IEEE
// binary32 operations, round to nearest even).  On sm_103a each issues as one
// instruction: the fp32 instruction counts of the quantizers match one per
// pair.  The pairing keeps two vectors in step through the same code.
namespace ufp4 {

__device__ __forceinline__ uint64_t pk2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void up2(uint64_t v, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Sign masks of a 16-element chunk: bit j of sgn set <=> eps_j = -1.
struct SignMasks {
    uint32_t lo[8], hi[8];  // 0 or 0x80000000 for elements 2k and 2k+1
};
__device__ __forceinline__ void make_masks(uint32_t sgn, SignMasks& m) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m.lo[k] = ((sgn >> (2 * k)) & 1u) << 31;
        m.hi[k] = ((sgn >> (2 * k + 1)) & 1u) << 31;
    }
}

__device__ __forceinline__ float pow2_exact(int e) {  // 2^e, e in [-149, 127]
    if (e >= -126) return __uint_as_float((uint32_t)(e + 127) << 23);
    return __uint_as_float(1u << (e + 149));
}

// Four e4m3 conversions packed into one word of bytes.
__device__ __forceinline__ uint32_t cvt_e4m3x4(float b0, float b1, float b2, float b3) {
    uint32_t r;
    asm("{ .reg .b16 lo, hi;\n"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n"
        "mov.b32 %0, {lo, hi}; }"
        : "=r"(r)
        : "f"(b0), "f"(b1), "f"(b2), "f"(b3));
    return r;
}

__device__ __forceinline__ uint32_t cvt_e2m1x8(float t0, float t1, float t2, float t3, float t4, float t5,
                                               float t6, float t7) {
    uint32_t r;
    asm("{ .reg .b8 b0, b1, b2, b3;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
        "mov.b32 %0, {b0, b1, b2, b3}; }"
        : "=r"(r)
        : "f"(t0), "f"(t1), "f"(t2), "f"(t3), "f"(t4), "f"(t5), "f"(t6), "f"(t7));
    return r;
}

// RTNE of 8 scaled values (already multiplied by the folded reciprocal) to one
// word of packed sign-magnitude codes.  Uniform grids: the values are k * 2^-9
// with |k| <= 7 exactly on e4m3's subnormals, so an e4m3 conversion rounds to
// nearest with ties to even k; the even-indexed elements land in word E and
// the odd ones in word O, and each byte of E | O becomes one packed byte
// (INT4: two's complement codes, formed per byte before packing).
template <int GRID>
__device__ __forceinline__ uint32_t rtne8(float t0, float t1, float t2, float t3, float t4, float t5, float t6,
                                          float t7) {
    uint32_t w;
    if (GRID >= 2) {
        w = cvt_e2m1x8(t0, t1, t2, t3, t4, t5, t6, t7);
    } else {
        const uint32_t E = cvt_e4m3x4(t0, t2, t4, t6);  // bytes: s000 0kkk
        const uint32_t O = cvt_e4m3x4(t1, t3, t5, t7);
        if (GRID == 1)
            return (int4_from_e4m3_bytes(E) & 0x0F0F0F0Fu) | ((int4_from_e4m3_bytes(O) << 4) & 0xF0F0F0F0u);
        w = ((E | (E >> 4)) & 0x0F0F0F0Fu) | ((O | (O << 4)) & 0xF0F0F0F0u);
    }
    return clear_negative_zero(w);
}

}  // namespace ufp4

// ======================================================================
// Two independent 16-element vectors a and b carried together: e[i] holds
// (a_i, b_i) in one 64-bit register pair, so every butterfly stage, the
// 1/sqrt(n) multiply and the scaling are paired fp32 operations.
namespace ufp4 {

struct Dest {
    uint8_t* codes;    // 8 bytes of packed codes
    uint8_t* s0;       // scale of elements 0..7 (byte address)
    uint8_t* s1;       // scale of elements 8..15
    bool valid, w0, w1;
    uint64_t lin0;     // SR: linear index of element 0 in the output tensor
};

// Rows: two chunks (8 words each) sharing the same sign masks.
__device__ __forceinline__ void widen_rows(const uint32_t wa[8], const uint32_t wb[8], const SignMasks& m,
                                           uint64_t e[16]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        e[2 * k] = pk2(__uint_as_float(wa[k] * 65536u + m.lo[k]), __uint_as_float(wb[k] * 65536u + m.lo[k]));
        e[2 * k + 1] = pk2(__uint_as_float((wa[k] & 0xFFFF0000u) ^ m.hi[k]),
                           __uint_as_float((wb[k] & 0xFFFF0000u) ^ m.hi[k]));
    }
}

// The same with the masks of the 16 elements read from kernel parameters
// (constant bank) instead of registers: mask[j] is 0x80000000 when eps_j = -1.
__device__ __forceinline__ void widen_rows_c(const uint32_t wa[8], const uint32_t wb[8], const uint32_t* mask,
                                             uint64_t e[16]) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        e[2 * k] = pk2(__uint_as_float(wa[k] * 65536u + mask[2 * k]), __uint_as_float(wb[k] * 65536u + mask[2 * k]));
        e[2 * k + 1] = pk2(__uint_as_float((wa[k] & 0xFFFF0000u) ^ mask[2 * k + 1]),
                           __uint_as_float((wb[k] & 0xFFFF0000u) ^ mask[2 * k + 1]));
    }
}
__device__ __forceinline__ void widen_cols_c(const uint32_t g[16], const uint32_t* mask, uint64_t e[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i)
        e[i] = pk2(__uint_as_float(g[i] * 65536u + mask[i]), __uint_as_float((g[i] & 0xFFFF0000u) ^ mask[i]));
}

// Columns: word g[i] holds row i of column a (low half) and column b (high half).
__device__ __forceinline__ void widen_cols(const uint32_t g[16], const SignMasks& m, uint64_t e[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t mi = (i & 1) ? m.hi[i >> 1] : m.lo[i >> 1];
        e[i] = pk2(__uint_as_float(g[i] * 65536u + mi), __uint_as_float((g[i] & 0xFFFF0000u) ^ mi));
    }
}

// Sylvester butterfly, strides 1, 2, ..., n/2 in that order (strides >= 16
// with the lane holding the chunk h/16 away).
__device__ __forceinline__ void fwht_pair(uint64_t e[16], int n, int seg_lane) {
#pragma unroll
    for (int h = 1; h < kChunk; h <<= 1) {
        if (h < n) {
#pragma unroll
            for (int i = 0; i < kChunk; ++i) {
                if (i & h) continue;
                const uint64_t a = e[i], b = e[i + h];
                e[i] = add2(a, b);
                e[i + h] = sub2(a, b);
            }
        }
    }
    // across lanes: the lower lane of a pair forms a + b, the upper one a - b,
    // i.e. o + s e with s = +1 or -1, one fma each (the product is exact, so
    // the single rounding equals that of the add or subtract)
    for (int h = kChunk; h < n; h <<= 1) {
        const int lm = h / kChunk;
        const float sgn = (seg_lane & lm) != 0 ? -1.0f : 1.0f;
        const uint64_t s2 = pk2(sgn, sgn);
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            const uint64_t o = (uint64_t)__shfl_xor_sync(0xFFFFFFFFu, (unsigned long long)e[i], lm);
            e[i] = fma2(s2, e[i], o);
        }
    }
}

// The same for n = 16: strides 1, 2, 4, 8, all inside the thread.
__device__ __forceinline__ void fwht_pair16(uint64_t e[16]) {
#pragma unroll
    for (int h = 1; h < kChunk; h <<= 1) {
#pragma unroll
        for (int i = 0; i < kChunk; ++i) {
            if (i & h) continue;
            const uint64_t a = e[i], b = e[i + h];
            e[i] = add2(a, b);
            e[i + h] = sub2(a, b);
        }
    }
}


// Tree amax of |a_i| and |b_i| over i in [lo, hi) (lo, hi multiples of 8).
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ void amax_pair(const uint64_t e[16], int lo, int hi, float& ma, float& mb) {
    float ta[16], tb[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) up2(e[i], ta[i], tb[i]);
    float ra = 0.0f, rb = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        if (i < lo || i >= hi) continue;
        ra = max3(ra, fabsf(ta[i]), fabsf(ta[i + 1]));
        rb = max3(rb, fabsf(tb[i]), fabsf(tb[i + 1]));
    }
    ma = ra;
    mb = rb;
}

}  // namespace ufp4
