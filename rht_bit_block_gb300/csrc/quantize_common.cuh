// Device code shared by the two quantizer units (quantize.cu: the general
// kernel; quantize_rows.cu: the row-wise kernel): ring waits, block scales,
// rounding and packing of 16-element vectors held as pairs.  See those units
// for the pages each step follows.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ufp4_device.cuh"

namespace ufp4 {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = 6;               // TMA ring depth
constexpr uint32_t kWaitLimit = 1u << 24;   // bounded mbarrier polling

__device__ __forceinline__ int find_group(const QuantParams& p, int row_tile) {
    int g = 0;
    for (int i = 1; i < p.num_groups; ++i)
        if (p.grp_tile0[i] <= row_tile) g = i;
    return g;
}

// Non-negative floats order like their bit patterns, so a 2-D block amax is
// an atomicMax on the bits in shared memory.
__device__ __forceinline__ void post_amax(uint32_t* slot, float m) {
    atomicMax(slot, __float_as_uint(m));
}

__device__ __forceinline__ uint32_t chunk_signs(const QuantParams& p, int pos) {
    pos &= 255;
    return (p.sign_bits[pos >> 5] >> (pos & 31)) & 0xFFFFu;
}

__device__ __forceinline__ uint32_t smem_addr(const void* ptr) {
    return (uint32_t)__cvta_generic_to_shared(ptr);
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred q; mbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2; selp.u32 %0, 1, 0, q; }"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// Constants of a launch that the per-chunk code needs.
struct Fold {
    float g;       // two-level scale: the tensor scale fp32(T / fp32(qmax * 448))
    float inv_s;   // fp32(1/sqrt n)
    bool pow4;     // n = 4^j: 1/sqrt n = 2^-j folds exactly into the block reciprocal
    int j;         // log4 n when pow4
};

// The UE8M0 byte e + 127 of a block amax M: e is the smallest integer with
// M <= qmax * 2^e (exact form of the truncation-free scale).  With M = m 2^E
// (m in [1,2)) and qmax = mq 2^Eq: e = E - Eq + (m > mq), and the comparison
// is the carry of M's mantissa + (2^23 - 1 - mq) into the exponent field, so
// the byte is one add and one shift of M's bits; a zero block gives 0.
// MXFP8 (GRID 4) takes e = floor(log2 M) - 8 instead: the same formula with
// Eq = 8 and mq = 2^23 - 1 (no carry).  Blocks whose amax is nonzero but
// below 2^-120 or above 2^120 are outside the input contract and are not
// special-cased.
template <int GRID>
__device__ __forceinline__ int po2_byte(float M) {
    constexpr int Eq = (GRID == 0) ? 0 : (GRID == 3 ? 1 : (GRID == 4 ? 8 : 2));
    constexpr uint32_t mq = (GRID == 2) ? 0x400000u : (GRID == 3 ? 0u : (GRID == 4 ? 0x7FFFFFu : 0x600000u));
    constexpr uint32_t add = (0x7FFFFFu - mq) - ((uint32_t)Eq << 23);
    return max((int)(__float_as_uint(M) + add) >> 23, 0);
}

// Eight level offsets o_i = k_i + 8 (the low nibbles of v_i = bits of
// fp32(1.5 * 2^23 + 8 + k_i)) packed into one word, element i in bits 4i..4i+3.
// Every v_i is E + o_i with E = 0x4B400000 and o_i < 16, so a tree of
// multiply-adds (x16, x256, x65536) lines the nibbles up and leaves the
// constant E (17 * 257 * ...) in bits 22 and up, removed at the end.
template <uint32_t E = 0x4B400000u>
__device__ __forceinline__ uint32_t pack_offsets8(const uint32_t* v) {
    constexpr uint32_t bias = E * 17u * 257u;  // mod 2^32; the low 22 bits are zero
    const uint32_t p0 = v[1] * 16u + v[0], p1 = v[3] * 16u + v[2];
    const uint32_t p2 = v[5] * 16u + v[4], p3 = v[7] * 16u + v[6];
    const uint32_t q0 = p1 * 256u + p0, q1 = p3 * 256u + p2;
    return q1 * 65536u + q0 - bias;
}

// Paired subtractions with directed rounding (round up / round down).
__device__ __forceinline__ uint64_t sub2_rp(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rp.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2_rm(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rm.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Scale, round, pack and store two 16-element vectors a and b held as pairs
// e[i] = (a_i, b_i) of transformed values before the 1/sqrt(n) multiply
// (y = H S x).  MA0/MA1 (MB0/MB1): amax of |y| over the blocks holding
// elements 0..7 / 8..15 of a (of b).  The block amax of z = y/sqrt n is
// fp32(My * fp32(1/sqrt n)) (rounding is monotone), exact for n = 4^j.
//
// RTNE multiplies y by one folded reciprocal per block, rr = r * 2^-j * f,
// where f = 2^-7 (E1M2: k/4 -> k * 2^-9) or 2^-9 (INT4: k -> k * 2^-9) puts
// the uniform levels on e4m3's subnormals, and f = 1 for E2M1; with UE8M0
// scales the uniform grids are rounded by an fma instead, with f = 1/step
// (E1M2 4, INT4 1); every factor is a power of
// two, so fp32(y * rr) = fp32(z * r) * f exactly.  SR uses
// f = 1/step (E1M2 4, INT4 1, E2M1 1).  For other n, z = fp32(y * 1/sqrt n)
// is formed first, as in the definition.
// SF: 0 fp32 scale, 1 UE8M0, 2 two-level (E4M3 block byte x tensor scale g).
template <int GRID, int SF>
__device__ __forceinline__ float block_recip(float My, const Fold& fd, int lf, bool write, uint8_t* sptr,
                                             int* byte_out = nullptr) {
    constexpr float qmax = grid_qmax(GRID);
    const float Mz = __fmul_rn(My, fd.inv_s);
    const int lj = fd.pow4 ? -fd.j : 0;
    if (SF == 2) {
        // b = E4M3(fp32(fp32(M / qmax) / g)), s = fp32(e4m3(b) * g), r = fp32(1 / s)
        const float sb = div_qmax_rn<GRID>(Mz);
        const uint32_t b8 = fd.g == 0.0f ? 0u : e4m3_byte(__fdiv_rn(sb, fd.g));
        const float s = __fmul_rn(e4m3_value(b8), fd.g);
        if (write) *sptr = (uint8_t)b8;
        const float r = s == 0.0f ? 0.0f : __frcp_rn(s);
        return __fmul_rn(r, pow2_exact(lf + lj));
    } else if (SF == 1) {
        const int eb = po2_byte<GRID>(Mz);  // e + 127
        if (write) *sptr = (uint8_t)eb;
        if (byte_out) *byte_out = eb;
        // 2^(-e + lf + lj) from its biased exponent: a normal number for every
        // block inside the input contract (|lf + lj| <= 6, eb <= 248)
        return __uint_as_float((uint32_t)(254 + lf + lj - eb) << 23);
    } else {
        float sc, r;
        scale_fp32<GRID>(Mz, sc, r);
        if (write) *reinterpret_cast<float*>(sptr) = sc;
        return __fmul_rn(r, pow2_exact(lf + lj));
    }
}

// Stochastic rounding of 16 scaled values to packed E2M1 codes (the uniform
// grids take the fma path in emit_pair).  With a = min(|t|, qmax) in units of
// the local level gap g (v = a / g, between the levels floor(v) and
// floor(v) + 1), round up iff u < (v - floor(v)) * 2^16, u the element's 16
// random bits.  For integer u that is u < ceil(v * 2^16) - floor(v) * 2^16, so
// the level index is k = (ceil(v * 2^16) + 2^16 - 1 - u) >> 16 (floor(v) or
// floor(v) + 1), and ceil(v * 2^16) is the low mantissa bits of one fma
// rounded upward, v * 2^16 + 2^23 (exact: v * 2^16 < 2^23).  Each nibble is
// sign * 8 + k (sign-magnitude), the nibbles line up through a tree of
// multiply-adds, and a zero level loses its sign word-wise.
template <int GRID>
__device__ __forceinline__ uint2 sr_vec(const float t[16], const uint32_t w[8]) {
    static_assert(GRID == 2 || GRID == 3, "E2M1 grids only");
    constexpr float qmax = grid_qmax(GRID);
    uint32_t nib[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t u = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu);
        const float ti = t[i];
        // E2M1 gaps: 0.5 below 2, 1 on [2,4), 2 on [4,6]
        const float a = fminf(fabsf(ti), qmax);
        const float gap = a < 2.0f ? 0.5f : (a < 4.0f ? 1.0f : 2.0f);
        const float inv = a < 2.0f ? 2.0f : (a < 4.0f ? 1.0f : 0.5f);
        const uint32_t vb = __float_as_uint(__fmaf_ru(__fmul_rn(a, inv), 65536.0f, 8388608.0f));
        const uint32_t k = (vb - 0x4B000000u + 0xFFFFu - u) >> 16;
        const uint32_t idx = cvt_e2m1x2(0.0f, __fmul_rn((float)k, gap)) & 7u;
        nib[i] = (__float_as_uint(ti) >> 31) * 8u + idx;
    }
    auto pack8 = [](const uint32_t* v) {
        const uint32_t q0 = (v[3] * 16u + v[2]) * 256u + (v[1] * 16u + v[0]);
        const uint32_t q1 = (v[7] * 16u + v[6]) * 256u + (v[5] * 16u + v[4]);
        return q1 * 65536u + q0;
    };
    return make_uint2(clear_negative_zero(pack8(nib)), clear_negative_zero(pack8(nib + 8)));
}

// SR draws of the two vectors of one emit_pair call (16 elements each).  The
// caller draws them before it widens and transforms the input: they depend
// only on the output positions, and the generator's registers are then free
// again when the transformed values are live.
struct SrDraws {
    uint32_t a[8], b[8];
};
__device__ __forceinline__ void draw_pair(SrDraws& d, const SrKeys& keys, const Dest& A, const Dest& B,
                                          uint32_t stream, uint32_t group) {
    sr_draws16x2(keys, A.lin0, B.lin0, stream, group, d.a, d.b);
}

// What one emit_pair call stored, for callers that derive more from it:
// the packed code words of A and B and (UE8M0 scales) their scale bytes.
struct EmitOut {
    uint2 ca, cb;
    int sa, sb;
};

// nega / negb: the sign bit (0 or 0x80000000) of a vector held negated; its
// reciprocal then carries that sign, so that t = y r is the value of the
// unnegated vector (exact: IEEE products are sign-symmetric).  join: B's codes
// follow A's (A.codes + 8, 16-byte aligned, A.valid == B.valid), stored as one
// 16-byte word.  out: if given, receives the codes and scale bytes (1-D
// blocks of 16 or 32, split false).  b_in_a: B is the second half of A's
// block (a 32-wide block over both vectors: MB0 == MA0, split false, B writes
// no scale), so B takes A's reciprocal instead of computing it again.
template <int GRID, bool SR, int SF>
__device__ __forceinline__ void emit_pair(uint64_t e[16], float MA0, float MA1, float MB0, float MB1, bool split,
                                          const Fold& fd, const Dest& A, const Dest& B, const SrDraws& dr,
                                          uint32_t nega = 0u, uint32_t negb = 0u, bool join = false,
                                          EmitOut* out = nullptr, bool b_in_a = false) {
    // the uniform grids with power-of-two scales round by adding 1.5 * 2^23 + 8
    // to the value in units of the grid step (below): INT4 k, E1M2 4 t
    constexpr bool kMagic = GRID <= 1 && !SR && SF == 1;
    constexpr int lf = GRID == 4 ? 0
                     : kMagic    ? (GRID == 0 ? 2 : 0)
                                 : (SR ? (GRID == 0 ? 2 : 0) : (GRID == 0 ? -7 : (GRID == 1 ? -9 : 0)));  // log2 f
    const float ra0 = block_recip<GRID, SF>(MA0, fd, lf, A.valid && A.w0, A.s0, out ? &out->sa : nullptr);
    const float rb0 = b_in_a ? ra0 : block_recip<GRID, SF>(MB0, fd, lf, B.valid && B.w0, B.s0, out ? &out->sb : nullptr);
    if (b_in_a && out) out->sb = out->sa;
    float ra1 = ra0, rb1 = rb0;
    if (split) {
        ra1 = block_recip<GRID, SF>(MA1, fd, lf, A.valid && A.w1, A.s1);
        rb1 = block_recip<GRID, SF>(MB1, fd, lf, B.valid && B.w1, B.s1);
    }
    const float sa0 = __uint_as_float(__float_as_uint(ra0) ^ nega), sa1 = __uint_as_float(__float_as_uint(ra1) ^ nega);
    const float sb0 = __uint_as_float(__float_as_uint(rb0) ^ negb), sb1 = __uint_as_float(__float_as_uint(rb1) ^ negb);
    auto store_pair = [&](uint2 ca, uint2 cb) {
        if (out) {
            out->ca = ca;
            out->cb = cb;
        }
        if (join) {
            if (A.valid) *reinterpret_cast<uint4*>(A.codes) = make_uint4(ca.x, ca.y, cb.x, cb.y);
        } else {
            if (A.valid) *reinterpret_cast<uint2*>(A.codes) = ca;
            if (B.valid) *reinterpret_cast<uint2*>(B.codes) = cb;
        }
    };
    if (!fd.pow4) {
        const uint64_t is2 = pk2(fd.inv_s, fd.inv_s);
#pragma unroll
        for (int i = 0; i < 16; ++i) e[i] = mul2(e[i], is2);
    }
    if (GRID == 4) {
        // MXFP8: t = z * 2^-e (exact), one E4M3 byte per element, nearest
        // even, saturated at 448; a zero byte keeps no sign
        const uint64_t q = pk2(sa0, sb0);
        float ta[16], tb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) up2(mul2(e[i], q), ta[i], tb[i]);
        uint32_t wa[4], wb[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t va = cvt_e4m3x4(ta[4 * k], ta[4 * k + 1], ta[4 * k + 2], ta[4 * k + 3]);
            const uint32_t vb = cvt_e4m3x4(tb[4 * k], tb[4 * k + 1], tb[4 * k + 2], tb[4 * k + 3]);
            // per byte: keep bit 7 only where the magnitude bits are nonzero
            wa[k] = va & (((va & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | 0x7F7F7F7Fu);
            wb[k] = vb & (((vb & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | 0x7F7F7F7Fu);
        }
        if (A.valid) *reinterpret_cast<uint4*>(A.codes) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
        if (B.valid) *reinterpret_cast<uint4*>(B.codes) = make_uint4(wb[0], wb[1], wb[2], wb[3]);
        return;
    }
    if (kMagic) {
        // t = z r is exact (r a power of two; for E1M2 r also carries the
        // factor 4 = 1 / step), so one fma t + (1.5 * 2^23 + 8) rounds t to the
        // nearest integer k, ties to even (the addend is even and the result's
        // unit is 1), and its low nibble is o = k + 8 (|k| <= 7: the
        // truncation-free scale keeps |t| <= 7).  The offsets line up through
        // a tree of multiply-adds (pack_offsets8).  INT4: flipping
        // bit 3 of o gives the two's complement nibble of k.  E1M2: o >= 8
        // (k >= 0) becomes o - 8 = k; o < 8 (k < 0) becomes (o ^ 15) + 1 =
        // 8 + |k|, the sign-magnitude nibble, and k = 0 is +0.
        const uint64_t q0 = pk2(sa0, sb0), q1 = pk2(sa1, sb1), cc = pk2(12582920.0f, 12582920.0f);
        uint32_t va[16], vb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float a, b;
            up2(fma2(e[i], i < 8 ? q0 : q1, cc), a, b);
            va[i] = __float_as_uint(a);
            vb[i] = __float_as_uint(b);
        }
        auto finish = [](uint32_t w) {
            if (GRID == 1) return w ^ 0x88888888u;
            const uint32_t neg = ((w >> 3) & 0x11111111u) ^ 0x11111111u;  // per nibble: 1 iff o < 8
            return (w ^ (neg * 7u + 0x88888888u)) + neg;
        };
        store_pair(make_uint2(finish(pack_offsets8<>(va)), finish(pack_offsets8<>(va + 8))),
                   make_uint2(finish(pack_offsets8<>(vb)), finish(pack_offsets8<>(vb + 8))));
        return;
    }
    if (SR && GRID <= 1) {
        // SR on the uniform grids (t in units of the step, largest level 7),
        // on the fma pipe.  With C = ceil(|t| 2^16) and u the element's 16-bit
        // draw, the level index is k = ceil((C - u) / 2^16) (u < the fraction
        // of |t| above floor(|t|), times 2^16, rounds up; see sr_vec).
        //  X = rm(192 + u 2^-16 - |t|) = 192 + (u - C) 2^-16: the addend's
        //      bits are 0x4340 above u, and its unit 2^-16 sets the grid;
        //  K = rp(2^23 + 196 - X) = 2^23 + 4 + k;
        //  V = K - copysign(4, t) = 2^23 + 8 s + k, s the sign bit.
        // The low nibbles of V are sign-magnitude codes (a zero level with
        // s = 1 is cleared below).  With UE8M0 scales t = y r is exact, so
        // the first step is one fma on y; otherwise t = fp32(y r) is formed
        // and clamped to 7 first, as in the definition.
        const uint32_t* wa = dr.a;
        const uint32_t* wb = dr.b;
        const uint64_t c196 = pk2(8388804.0f, 8388804.0f);
        const uint64_t q0 = pk2(sa0, sb0), q1 = pk2(sa1, sb1);
        // the sign of t: y's sign bit flipped for a negated vector (the
        // SF == 1 form takes |y| times the unsigned reciprocal)
        const uint32_t csa = (SF == 1 ? nega : 0u) | 0x40800000u, csb = (SF == 1 ? negb : 0u) | 0x40800000u;
        uint32_t va[16], vb[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t sel = (i & 1) ? 0x7632u : 0x7610u;
            const float ua = __uint_as_float(__byte_perm(wa[i >> 1], 0x43400000u, sel));
            const float ub = __uint_as_float(__byte_perm(wb[i >> 1], 0x43400000u, sel));
            float ya, yb;
            uint64_t x;
            if (SF == 1) {
                up2(e[i], ya, yb);
                x = pk2(__fmaf_rd(-fabsf(ya), i < 8 ? ra0 : ra1, ua), __fmaf_rd(-fabsf(yb), i < 8 ? rb0 : rb1, ub));
            } else {
                up2(mul2(e[i], i < 8 ? q0 : q1), ya, yb);
                x = sub2_rm(pk2(ua, ub), pk2(fminf(fabsf(ya), 7.0f), fminf(fabsf(yb), 7.0f)));
            }
            const uint64_t cs = pk2(__uint_as_float((__float_as_uint(ya) & 0x80000000u) ^ csa),
                                    __uint_as_float((__float_as_uint(yb) & 0x80000000u) ^ csb));
            float a, b;
            up2(sub2(sub2_rp(c196, x), cs), a, b);
            va[i] = __float_as_uint(a);
            vb[i] = __float_as_uint(b);
        }
        uint32_t oa[2] = {clear_negative_zero(pack_offsets8<0x4B000000u>(va)),
                          clear_negative_zero(pack_offsets8<0x4B000000u>(va + 8))};
        uint32_t ob[2] = {clear_negative_zero(pack_offsets8<0x4B000000u>(vb)),
                          clear_negative_zero(pack_offsets8<0x4B000000u>(vb + 8))};
        if (GRID == 1) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                oa[h] = signmag_nz_to_twos(oa[h]);
                ob[h] = signmag_nz_to_twos(ob[h]);
            }
        }
        store_pair(make_uint2(oa[0], oa[1]), make_uint2(ob[0], ob[1]));
        return;
    }
    const uint64_t q0 = pk2(sa0, sb0), q1 = pk2(sa1, sb1);
    float ta[16], tb[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) up2(mul2(e[i], i < 8 ? q0 : q1), ta[i], tb[i]);
    uint2 ca, cb;
    if constexpr (SR && (GRID == 2 || GRID == 3)) {
        ca = sr_vec<GRID>(ta, dr.a);
        cb = sr_vec<GRID>(tb, dr.b);
    } else {
        ca = make_uint2(rtne8<GRID>(ta[0], ta[1], ta[2], ta[3], ta[4], ta[5], ta[6], ta[7]),
                        rtne8<GRID>(ta[8], ta[9], ta[10], ta[11], ta[12], ta[13], ta[14], ta[15]));
        cb = make_uint2(rtne8<GRID>(tb[0], tb[1], tb[2], tb[3], tb[4], tb[5], tb[6], tb[7]),
                        rtne8<GRID>(tb[8], tb[9], tb[10], tb[11], tb[12], tb[13], tb[14], tb[15]));
    }
    store_pair(ca, cb);
}

// 1-D block amax over bw/16 neighbouring lanes (bw >= 16), for both vectors.
__device__ __forceinline__ void amax_1d_pair(const uint64_t e[16], int bw, float& ma, float& mb) {
    amax_pair(e, 0, 16, ma, mb);
    for (int k = 1; k < bw / kChunk; k <<= 1) {
        ma = fmaxf(ma, __shfl_xor_sync(0xFFFFFFFFu, ma, k));
        mb = fmaxf(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, k));
    }
}

// Row pass: 16 consecutive elements of tile row trow from shared memory.
template <int TC>
__device__ __forceinline__ void load_row_chunk(const uint16_t* tile, int trow, int cchunk, uint32_t w[8]) {
    const uint4* src = reinterpret_cast<const uint4*>(tile + trow * TC + cchunk * kChunk);
    const uint4 a = src[0], b = src[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
    w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}

// Column pass: rows rchunk*16 .. +15 of the column pair (tcol, tcol+1), one
// 32-bit shared load per row (column tcol in the low half).
template <int TC>
__device__ __forceinline__ void gather_pair(const uint16_t* tile, int tcol, int rchunk, uint32_t g[16]) {
    const uint32_t* src = reinterpret_cast<const uint32_t*>(tile + (rchunk * kChunk) * TC + tcol);
#pragma unroll
    for (int i = 0; i < 16; ++i) g[i] = src[i * (TC / 2)];
}

}  // namespace ufp4
