// Fused RHT + block-scaled 4-bit quantizer for sm_103a.
//
// Persistent CTAs walk TR x TC tiles of the bf16 input.  Each tile arrives by
// one TMA copy into a 3-stage shared-memory ring, and from that single HBM
// read the CTA produces the row-wise quantization (RHT and blocks along the
// columns) and the column-wise quantization of the transpose (RHT and blocks
// along the rows), as required for FPROP, DGRAD and WGRAD (UFP4 summary,
// section 方法: RHT on all three training GEMMs; 2D-block tutorial: dX = dY W
// and dW = dY^T X need transposed operands).
//
//  * row pass: a thread carries 16 consecutive elements of a row, widened to
//    fp32 with the random signs folded into the widening, transformed with
//    paired fp32 butterflies (shuffles for strides >= 16), scaled by one
//    folded reciprocal per block, rounded and packed;
//  * column pass: a thread gathers two adjacent columns, 16 rows each, with
//    one 32-bit shared load per row, and runs them through the same steps;
//  * 2-D b x b blocks reduce their amax through shared-memory atomics.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "ufp4_device.cuh"

namespace ufp4 {

__device__ int g_quant_error;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxStages = 6;               // TMA ring depth
constexpr int kCtasPerSm = 2;               // 16 warps per SM, up to 128 registers a thread; about 96 KB of ring per CTA
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

// Polls of a tile's barrier before a quantizer kernel gives up (a failure-
// detection hook can lower it; the drain of copies in flight always uses
// kWaitLimit).
__device__ uint32_t g_quant_wait_limit = kWaitLimit;

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
__device__ __forceinline__ uint32_t pack_offsets8(const uint32_t* v) {
    constexpr uint32_t E = 0x4B400000u;
    constexpr uint32_t bias = E * 17u * 257u;  // mod 2^32; the low 22 bits are zero
    const uint32_t p0 = v[1] * 16u + v[0], p1 = v[3] * 16u + v[2];
    const uint32_t p2 = v[5] * 16u + v[4], p3 = v[7] * 16u + v[6];
    const uint32_t q0 = p1 * 256u + p0, q1 = p3 * 256u + p2;
    return q1 * 65536u + q0 - bias;
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
__device__ __forceinline__ float block_recip(float My, const Fold& fd, int lf, bool write, uint8_t* sptr) {
    constexpr float qmax = grid_qmax(GRID);
    const float Mz = __fmul_rn(My, fd.inv_s);
    const int lj = fd.pow4 ? -fd.j : 0;
    if (SF == 2) {
        // b = E4M3(fp32(fp32(M / qmax) / g)), s = fp32(e4m3(b) * g), r = fp32(1 / s)
        const float sb = __fdiv_rn(Mz, qmax);
        const uint32_t b8 = fd.g == 0.0f ? 0u : e4m3_byte(__fdiv_rn(sb, fd.g));
        const float s = __fmul_rn(e4m3_value(b8), fd.g);
        if (write) *sptr = (uint8_t)b8;
        const float r = s == 0.0f ? 0.0f : __frcp_rn(s);
        return __fmul_rn(r, pow2_exact(lf + lj));
    } else if (SF == 1) {
        const int eb = po2_byte<GRID>(Mz);  // e + 127
        if (write) *sptr = (uint8_t)eb;
        // 2^(-e + lf + lj) from its biased exponent: a normal number for every
        // block inside the input contract (|lf + lj| <= 6, eb <= 248)
        return __uint_as_float((uint32_t)(254 + lf + lj - eb) << 23);
    } else {
        float sc, r;
        scale_fp32(Mz, qmax, sc, r);
        if (write) *reinterpret_cast<float*>(sptr) = sc;
        return __fmul_rn(r, pow2_exact(lf + lj));
    }
}

// Stochastic rounding of 16 scaled values to packed codes.  With a =
// min(|t|, qmax) in units of the local level gap g (v = a / g, between the
// levels floor(v) and floor(v) + 1), round up iff u < (v - floor(v)) * 2^16,
// u the element's 16 random bits.  For integer u that is u < ceil(v * 2^16) -
// floor(v) * 2^16, so the level index is k = (ceil(v * 2^16) + 2^16 - 1 - u)
// >> 16 (floor(v) or floor(v) + 1), and ceil(v * 2^16) is the low mantissa
// bits of one fma rounded upward, v * 2^16 + 2^23 (exact: v * 2^16 < 2^23).
// Each nibble is sign * 8 + k (sign-magnitude), the nibbles line up through a
// tree of multiply-adds, and a zero level loses its sign word-wise.  CLAMP:
// |t| may exceed the largest level by an ulp (fp32 and two-level scales);
// with UE8M0 scales |t| <= qmax holds exactly.
template <int GRID, bool CLAMP>
__device__ __forceinline__ uint2 sr_vec(const float t[16], const SrKeys& keys, uint64_t lin0, uint32_t stream,
                                        uint32_t group) {
    constexpr float qmax = grid_qmax(GRID);
    uint32_t w[8];
    sr_draws16(keys, lin0, stream, group, w);
    uint32_t nib[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const uint32_t u = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu);
        const float ti = t[i];
        uint32_t idx;
        if (GRID >= 2) {
            // E2M1 gaps: 0.5 below 2, 1 on [2,4), 2 on [4,6]
            const float a = fminf(fabsf(ti), qmax);
            const float gap = a < 2.0f ? 0.5f : (a < 4.0f ? 1.0f : 2.0f);
            const float inv = a < 2.0f ? 2.0f : (a < 4.0f ? 1.0f : 0.5f);
            const uint32_t vb = __float_as_uint(__fmaf_ru(__fmul_rn(a, inv), 65536.0f, 8388608.0f));
            const uint32_t k = (vb - 0x4B000000u + 0xFFFFu - u) >> 16;
            idx = cvt_e2m1x2(0.0f, __fmul_rn((float)k, gap)) & 7u;
        } else {
            // uniform grids: t is already in units of the step (largest level 7)
            const float a = CLAMP ? fminf(fabsf(ti), 7.0f) : fabsf(ti);
            const uint32_t vb = __float_as_uint(__fmaf_ru(a, 65536.0f, 8388608.0f));
            idx = (vb - 0x4B000000u + 0xFFFFu - u) >> 16;
        }
        nib[i] = (__float_as_uint(ti) >> 31) * 8u + idx;
    }
    auto pack8 = [](const uint32_t* v) {
        const uint32_t q0 = (v[3] * 16u + v[2]) * 256u + (v[1] * 16u + v[0]);
        const uint32_t q1 = (v[7] * 16u + v[6]) * 256u + (v[5] * 16u + v[4]);
        return q1 * 65536u + q0;
    };
    uint32_t out[2] = {clear_negative_zero(pack8(nib)), clear_negative_zero(pack8(nib + 8))};
    if (GRID == 1) {
        out[0] = signmag_to_twos(out[0]);
        out[1] = signmag_to_twos(out[1]);
    }
    return make_uint2(out[0], out[1]);
}

template <int GRID, bool SR, int SF>
__device__ __forceinline__ void emit_pair(uint64_t e[16], float MA0, float MA1, float MB0, float MB1, bool split,
                                          const Fold& fd, const Dest& A, const Dest& B,
                                          const SrKeys& sr_keys, uint32_t stream, uint32_t group) {
    // the uniform grids with power-of-two scales round by adding 1.5 * 2^23 + 8
    // to the value in units of the grid step (below): INT4 k, E1M2 4 t
    constexpr bool kMagic = GRID <= 1 && !SR && SF == 1;
    constexpr int lf = GRID == 4 ? 0
                     : kMagic    ? (GRID == 0 ? 2 : 0)
                                 : (SR ? (GRID == 0 ? 2 : 0) : (GRID == 0 ? -7 : (GRID == 1 ? -9 : 0)));  // log2 f
    const float ra0 = block_recip<GRID, SF>(MA0, fd, lf, A.valid && A.w0, A.s0);
    const float rb0 = block_recip<GRID, SF>(MB0, fd, lf, B.valid && B.w0, B.s0);
    float ra1 = ra0, rb1 = rb0;
    if (split) {
        ra1 = block_recip<GRID, SF>(MA1, fd, lf, A.valid && A.w1, A.s1);
        rb1 = block_recip<GRID, SF>(MB1, fd, lf, B.valid && B.w1, B.s1);
    }
    if (!fd.pow4) {
        const uint64_t is2 = pk2(fd.inv_s, fd.inv_s);
#pragma unroll
        for (int i = 0; i < 16; ++i) e[i] = mul2(e[i], is2);
    }
    if (GRID == 4) {
        // MXFP8: t = z * 2^-e (exact), one E4M3 byte per element, nearest
        // even, saturated at 448; a zero byte keeps no sign
        const uint64_t q = pk2(ra0, rb0);
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
        const uint64_t q0 = pk2(ra0, rb0), q1 = pk2(ra1, rb1), cc = pk2(12582920.0f, 12582920.0f);
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
        if (A.valid)
            *reinterpret_cast<uint2*>(A.codes) = make_uint2(finish(pack_offsets8(va)), finish(pack_offsets8(va + 8)));
        if (B.valid)
            *reinterpret_cast<uint2*>(B.codes) = make_uint2(finish(pack_offsets8(vb)), finish(pack_offsets8(vb + 8)));
        return;
    }
    const uint64_t q0 = pk2(ra0, rb0), q1 = pk2(ra1, rb1);
    float ta[16], tb[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) up2(mul2(e[i], i < 8 ? q0 : q1), ta[i], tb[i]);
    uint2 ca, cb;
    if (SR) {
        ca = sr_vec<GRID, SF != 1>(ta, sr_keys, A.lin0, stream, group);
        cb = sr_vec<GRID, SF != 1>(tb, sr_keys, B.lin0, stream, group);
    } else {
        ca = make_uint2(rtne8<GRID>(ta[0], ta[1], ta[2], ta[3], ta[4], ta[5], ta[6], ta[7]),
                        rtne8<GRID>(ta[8], ta[9], ta[10], ta[11], ta[12], ta[13], ta[14], ta[15]));
        cb = make_uint2(rtne8<GRID>(tb[0], tb[1], tb[2], tb[3], tb[4], tb[5], tb[6], tb[7]),
                        rtne8<GRID>(tb[8], tb[9], tb[10], tb[11], tb[12], tb[13], tb[14], tb[15]));
    }
    if (A.valid) *reinterpret_cast<uint2*>(A.codes) = ca;
    if (B.valid) *reinterpret_cast<uint2*>(B.codes) = cb;
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

template <int GRID, bool SR, bool PO2, int TC>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
quantize_kernel(const __grid_constant__ CUtensorMap tmap, const QuantParams p, const int num_tiles) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int SZ = PO2 ? 1 : 4;         // bytes per scale
    const int TR = p.tile_rows;             // 64 or 128 (runtime)
    const int tile_bytes = TR * TC * 2;
    const int kStages = p.stages;           // ring depth (runtime, <= kMaxStages)
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 127u) & ~127u) - raw;
    uint8_t* base = smem_raw + pad;
    uint32_t* amax2d = reinterpret_cast<uint32_t*>(base + kStages * tile_bytes);
    const uint32_t bars = smem_addr(base + kStages * tile_bytes + 4 * p.amax_slots);  // 8-byte aligned

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int n = p.n;
    Fold fd;
    fd.g = 0.0f;
    fd.inv_s = p.inv_sqrt_n;
    fd.pow4 = p.pow4;
    fd.j = p.log4n;

    auto issue = [&](int tile, int s) {
        const int row_tile = tile / p.col_tiles;
        const int g = find_group(p, row_tile);
        const int64_t lr0 = (int64_t)(row_tile - p.grp_tile0[g]) * TR;
        const int64_t c0 = (int64_t)(tile - row_tile * p.col_tiles) * TC;
        const uint32_t bar = bars + 8u * s;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(tile_bytes)
                     : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
            ::"r"(smem_addr(base + s * tile_bytes)), "l"((uint64_t)&tmap), "r"((int)c0),
            "r"((int)(p.grp_row0[g] + lr0)), "r"(bar)
            : "memory");
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8u * s));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // the input may come from the previous kernel, and that kernel may still
    // read buffers this one writes: wait for it before the first copy
    griddep_wait();
    griddep_launch();
    const uint32_t wait_limit = g_quant_wait_limit;
    if (tid == 0)
        for (int s = 0; s < kStages; ++s) {
            const int tile = blockIdx.x + s * gridDim.x;
            if (tile < num_tiles) issue(tile, s);
        }

    // row pass: a thread owns chunk column cchunk of the row pairs
    // (r, r + kRPI), r = r0 + 2 * kRPI * it
    constexpr int kCPR = TC / kChunk;       // chunks per tile row
    constexpr int kRPI = kThreads / kCPR;   // tile rows per thread step
    const int pairs = TR / (2 * kRPI);
    const int cchunk = tid % kCPR;
    const int r0 = tid / kCPR;
    const int seg_row = (cchunk * kChunk % (n > kChunk ? n : kChunk)) / kChunk;
    SignMasks mrow;
    make_masks(chunk_signs(p, cchunk * kChunk), mrow);
    const int lbw = p.lbw_row, lbwc = p.lbw_col, lb = p.lb2d;
    // column pass: S = 2^lS lanes share one column segment; a warp task is
    // 32/S column pairs x S row chunks
    const int lS = p.lseg;
    const int S = 1 << lS;
    const int lncb = 1 + lS;                 // log2((TC/2) / (32/S)) for TC = 128
    const int ncb_mask = (1 << lncb) - 1;
    const int col_tasks = TR * TC / (kChunk * 64 * kWarps);  // per warp
    // a thread's row chunks are all lane % S modulo S, and the signs repeat
    // every n = 16 S elements (or every 16 when n <= 16): one mask set serves
    SignMasks mc;
    make_masks(chunk_signs(p, (lane & (S - 1)) * kChunk), mc);
    const int nslot = p.amax_slots;
    // tile coordinates advance by gridDim.x tiles per step, without division
    const int step_r = gridDim.x / p.col_tiles, step_c = gridDim.x - step_r * p.col_tiles;
    int row_tile = blockIdx.x / p.col_tiles, col_tile = blockIdx.x - row_tile * p.col_tiles;
    int g = p.num_groups > 1 ? find_group(p, row_tile) : 0;

    int i = 0;
    int s = 0;            // ring stage of tile i
    uint32_t phase = 0;   // parity of that stage's current use
    for (;; ++i) {
        const int tile = blockIdx.x + i * gridDim.x;
        if (tile >= num_tiles) break;
        if (i) {
            col_tile += step_c;
            row_tile += step_r;
            if (col_tile >= p.col_tiles) {
                col_tile -= p.col_tiles;
                ++row_tile;
            }
            if (p.num_groups > 1) g = find_group(p, row_tile);
        }
        const bool landed = wait_phase(bars + 8u * s, phase, wait_limit);
        if (!__syncthreads_and(landed)) {
            if (tid == 0) atomicExch(&g_quant_error, 1);
            break;
        }
        const int64_t lr0 = (int64_t)(row_tile - p.grp_tile0[g]) * TR;
        const int64_t c0 = (int64_t)col_tile * TC;
        const int64_t grow0 = p.grp_row0[g];
        const int64_t cnt = p.grp_row0[g + 1] - grow0;
        const int64_t padded = p.grp_pad0[g + 1] - p.grp_pad0[g];
        const uint32_t grp_id = (uint32_t)(p.group_base + g);
        uint16_t* tile_s = reinterpret_cast<uint16_t*>(base + s * tile_bytes);
        if (p.do_col && lr0 + TR > cnt) {
            // rows past the group's end belong to the next group (or the
            // padding): the column pass must see zeros there
            const int first = cnt - lr0 > 0 ? (int)(cnt - lr0) : 0;
            uint4* t4 = reinterpret_cast<uint4*>(tile_s + first * TC);
            for (int q = tid; q < (TR - first) * TC / 8; q += kThreads) t4[q] = make_uint4(0, 0, 0, 0);
            __syncthreads();
        }

        // -------------------------------------------------------- row pass
        if (p.do_row) {
            const int64_t col = c0 + cchunk * kChunk;
            const bool col_ok = col < p.cols;
            // rows of this tile that exist, counted from this thread's first row
            const int64_t left = cnt - lr0 - r0;
            const uint16_t* src = tile_s + r0 * TC + cchunk * kChunk;
            if (p.is2d) {
                const int lnbc = 7 + (TC == 256) - lb;  // log2(TC / b)
                const int bmask = (1 << lb) - 1;
                for (int q = tid; q < nslot; q += kThreads) amax2d[q] = 0u;
                __syncthreads();
                // with one row pair per thread (64-row tiles) the transformed values
                // stay in registers while the block amax settles in shared memory;
                // with two, the second pass transforms them again
                uint64_t keep[16];
                for (int it = 0; it < pairs; ++it) {
                    const int ra = r0 + 2 * kRPI * it, rb = ra + kRPI;
                    uint32_t wa[8], wb[8];
                    uint64_t e[16];
                    load_row_chunk<TC>(tile_s, ra, cchunk, wa);
                    load_row_chunk<TC>(tile_s, rb, cchunk, wb);
                    widen_rows(wa, wb, mrow, e);
                    fwht_pair(e, n, seg_row);
                    if (pairs == 1)
#pragma unroll
                        for (int i = 0; i < 16; ++i) keep[i] = e[i];
                    const int sa = (ra >> lb) << lnbc, sb = (rb >> lb) << lnbc;
                    if (lb == 3) {
                        float a0, b0, a1, b1;
                        amax_pair(e, 0, 8, a0, b0);
                        amax_pair(e, 8, 16, a1, b1);
                        post_amax(&amax2d[sa + 2 * cchunk], a0);
                        post_amax(&amax2d[sa + 2 * cchunk + 1], a1);
                        post_amax(&amax2d[sb + 2 * cchunk], b0);
                        post_amax(&amax2d[sb + 2 * cchunk + 1], b1);
                    } else {
                        float a0, b0;
                        amax_pair(e, 0, 16, a0, b0);
                        post_amax(&amax2d[sa + ((cchunk * kChunk) >> lb)], a0);
                        post_amax(&amax2d[sb + ((cchunk * kChunk) >> lb)], b0);
                    }
                }
                __syncthreads();
                for (int it = 0; it < pairs; ++it) {
                    const int ra = r0 + 2 * kRPI * it, rb = ra + kRPI;
                    uint64_t e[16];
                    if (pairs == 1) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) e[i] = keep[i];
                    } else {
                        uint32_t wa[8], wb[8];
                        load_row_chunk<TC>(tile_s, ra, cchunk, wa);
                        load_row_chunk<TC>(tile_s, rb, cchunk, wb);
                        widen_rows(wa, wb, mrow, e);
                        fwht_pair(e, n, seg_row);
                    }
                    const int off = lb == 3 ? 2 * cchunk : ((cchunk * kChunk) >> lb);
                    const int sa = ((ra >> lb) << lnbc) + off, sb = ((rb >> lb) << lnbc) + off;
                    const float MA0 = __uint_as_float(amax2d[sa]);
                    const float MA1 = __uint_as_float(amax2d[lb == 3 ? sa + 1 : sa]);
                    const float MB0 = __uint_as_float(amax2d[sb]);
                    const float MB1 = __uint_as_float(amax2d[lb == 3 ? sb + 1 : sb]);
                    Dest A, B;
                    const int64_t la = lr0 + ra, lbr = lr0 + rb;
                    const bool colfirst = lb == 3 || (col & bmask) == 0;
                    uint8_t* sbase = (uint8_t*)p.row.scales;
                    A.codes = (uint8_t*)p.row.codes + (grow0 + la) * p.row.codes_ld + (col >> 1);
                    B.codes = (uint8_t*)p.row.codes + (grow0 + lbr) * p.row.codes_ld + (col >> 1);
                    A.s0 = sbase + ((la >> lb) * p.row.scales_ld + (col >> lb)) * SZ;
                    B.s0 = sbase + ((lbr >> lb) * p.row.scales_ld + (col >> lb)) * SZ;
                    A.s1 = A.s0 + SZ;
                    B.s1 = B.s0 + SZ;
                    A.valid = la < cnt && col_ok;
                    B.valid = lbr < cnt && col_ok;
                    A.w0 = (la & bmask) == 0 && colfirst;
                    B.w0 = (lbr & bmask) == 0 && colfirst;
                    A.w1 = (la & bmask) == 0 && lb == 3;
                    B.w1 = (lbr & bmask) == 0 && lb == 3;
                    A.lin0 = (uint64_t)la * (uint64_t)p.cols + (uint64_t)col;
                    B.lin0 = (uint64_t)lbr * (uint64_t)p.cols + (uint64_t)col;
                    emit_pair<GRID, SR, PO2 ? 1 : 0>(e, MA0, MA1, MB0, MB1, lb == 3, fd, A, B, p.sr_keys, 0u, grp_id);
                }
            } else {
                const bool wsc = (col & ((1 << lbw) - 1)) == 0;
                // output pointers of this thread's first row, stepped per pair
                const int64_t orow0 = grow0 + lr0 + r0;  // row-wise output rows follow the input rows
                uint8_t* cp = (uint8_t*)p.row.codes + orow0 * p.row.codes_ld + (col >> 1);
                uint8_t* sp = (uint8_t*)p.row.scales + (orow0 * p.row.scales_ld + (col >> lbw)) * SZ;
                const int64_t cstep = (int64_t)kRPI * p.row.codes_ld;
                const int64_t sstep = (int64_t)kRPI * p.row.scales_ld * SZ;
                uint64_t lin = (uint64_t)(lr0 + r0) * (uint64_t)p.cols + (uint64_t)col;
                const uint64_t lstep = (uint64_t)kRPI * (uint64_t)p.cols;
                for (int it = 0; it < pairs; ++it) {
                    const int ra = 2 * kRPI * it;
                    uint32_t wa[8], wb[8];
                    uint64_t e[16];
                    const uint4* pa = reinterpret_cast<const uint4*>(src + ra * TC);
                    const uint4* pb = reinterpret_cast<const uint4*>(src + (ra + kRPI) * TC);
                    const uint4 a0 = pa[0], a1 = pa[1], b0 = pb[0], b1 = pb[1];
                    wa[0] = a0.x; wa[1] = a0.y; wa[2] = a0.z; wa[3] = a0.w;
                    wa[4] = a1.x; wa[5] = a1.y; wa[6] = a1.z; wa[7] = a1.w;
                    wb[0] = b0.x; wb[1] = b0.y; wb[2] = b0.z; wb[3] = b0.w;
                    wb[4] = b1.x; wb[5] = b1.y; wb[6] = b1.z; wb[7] = b1.w;
                    widen_rows(wa, wb, mrow, e);
                    fwht_pair(e, n, seg_row);
                    float Ma, Mb;
                    amax_1d_pair(e, 1 << lbw, Ma, Mb);
                    Dest A, B;
                    A.codes = cp + (2 * it) * cstep;
                    B.codes = A.codes + cstep;
                    A.s0 = A.s1 = sp + (2 * it) * sstep;
                    B.s0 = B.s1 = A.s0 + sstep;
                    A.valid = ra < left && col_ok;
                    B.valid = ra + kRPI < left && col_ok;
                    A.w0 = B.w0 = wsc;
                    A.w1 = B.w1 = false;
                    A.lin0 = lin + (uint64_t)(2 * it) * lstep;
                    B.lin0 = A.lin0 + lstep;
                    emit_pair<GRID, SR, PO2 ? 1 : 0>(e, Ma, Ma, Mb, Mb, false, fd, A, B, p.sr_keys, 0u, grp_id);
                }
            }
        }

        // ----------------------------------------------------- column pass
        if (p.do_col) {
            const int64_t out_ld = p.col_grouped ? padded / 2 : p.col.codes_ld;
            const int lsd = p.is2d ? lb : lbwc;
            const int64_t sc_ld = p.col_grouped ? (padded >> lsd) : p.col.scales_ld;
            uint8_t* gcodes = (uint8_t*)p.col.codes + (p.col_grouped ? p.cols * (p.grp_pad0[g] / 2) : 0);
            uint8_t* gscales = (uint8_t*)p.col.scales + (p.col_grouped ? p.cols * (p.grp_pad0[g] >> lsd) * SZ : 0);
            if (p.is2d) {
                const int lnbq = (TR == 128 ? 7 : 6) - lb;  // log2(TR / b)
                const int bmask = (1 << lb) - 1;
                for (int q = tid; q < nslot; q += kThreads) amax2d[q] = 0u;
                __syncthreads();
                uint64_t keep[16];
                for (int k = 0; k < col_tasks; ++k) {
                    const int t = warp + kWarps * k;
                    const int tcol = 2 * (((t & ncb_mask) << (5 - lS)) + (lane >> lS));
                    const int rchunk = ((t >> lncb) << lS) + (lane & (S - 1));
                    uint32_t gw[16];
                    uint64_t e[16];
                    gather_pair<TC>(tile_s, tcol, rchunk, gw);
                    widen_cols(gw, mc, e);
                    fwht_pair(e, n, rchunk & (S - 1));
                    if (col_tasks == 1)
#pragma unroll
                        for (int i = 0; i < 16; ++i) keep[i] = e[i];
                    const int sa = (tcol >> lb) << lnbq, sb = ((tcol + 1) >> lb) << lnbq;
                    if (lb == 3) {
                        float a0, b0, a1, b1;
                        amax_pair(e, 0, 8, a0, b0);
                        amax_pair(e, 8, 16, a1, b1);
                        post_amax(&amax2d[sa + 2 * rchunk], a0);
                        post_amax(&amax2d[sa + 2 * rchunk + 1], a1);
                        post_amax(&amax2d[sb + 2 * rchunk], b0);
                        post_amax(&amax2d[sb + 2 * rchunk + 1], b1);
                    } else {
                        float a0, b0;
                        amax_pair(e, 0, 16, a0, b0);
                        post_amax(&amax2d[sa + ((rchunk * kChunk) >> lb)], a0);
                        post_amax(&amax2d[sb + ((rchunk * kChunk) >> lb)], b0);
                    }
                }
                __syncthreads();
                for (int k = 0; k < col_tasks; ++k) {
                    const int t = warp + kWarps * k;
                    const int tcol = 2 * (((t & ncb_mask) << (5 - lS)) + (lane >> lS));
                    const int rchunk = ((t >> lncb) << lS) + (lane & (S - 1));
                    uint64_t e[16];
                    if (col_tasks == 1) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) e[i] = keep[i];
                    } else {
                        uint32_t gw[16];
                        gather_pair<TC>(tile_s, tcol, rchunk, gw);
                        widen_cols(gw, mc, e);
                        fwht_pair(e, n, rchunk & (S - 1));
                    }
                    const int off = lb == 3 ? 2 * rchunk : ((rchunk * kChunk) >> lb);
                    const int sa = ((tcol >> lb) << lnbq) + off, sb = (((tcol + 1) >> lb) << lnbq) + off;
                    const float MA0 = __uint_as_float(amax2d[sa]);
                    const float MA1 = __uint_as_float(amax2d[lb == 3 ? sa + 1 : sa]);
                    const float MB0 = __uint_as_float(amax2d[sb]);
                    const float MB1 = __uint_as_float(amax2d[lb == 3 ? sb + 1 : sb]);
                    const int64_t lrow = lr0 + rchunk * kChunk;
                    const int64_t ca = c0 + tcol, cb = ca + 1;
                    const bool rowfirst = lb == 3 || (lrow & bmask) == 0;
                    Dest A, B;
                    A.codes = gcodes + ca * out_ld + (lrow >> 1);
                    B.codes = gcodes + cb * out_ld + (lrow >> 1);
                    A.s0 = gscales + ((ca >> lb) * sc_ld + (lrow >> lb)) * SZ;
                    B.s0 = gscales + ((cb >> lb) * sc_ld + (lrow >> lb)) * SZ;
                    A.s1 = A.s0 + SZ;
                    B.s1 = B.s0 + SZ;
                    A.valid = lrow < padded && ca < p.cols;
                    B.valid = lrow < padded && cb < p.cols;
                    A.w0 = (ca & bmask) == 0 && rowfirst;
                    B.w0 = (cb & bmask) == 0 && rowfirst;
                    A.w1 = (ca & bmask) == 0 && lb == 3;
                    B.w1 = (cb & bmask) == 0 && lb == 3;
                    A.lin0 = (uint64_t)ca * (uint64_t)padded + (uint64_t)lrow;
                    B.lin0 = A.lin0 + (uint64_t)padded;
                    emit_pair<GRID, SR, PO2 ? 1 : 0>(e, MA0, MA1, MB0, MB1, lb == 3, fd, A, B, p.sr_keys, 1u, grp_id);
                }
            } else {
                const int bwc = 1 << lbwc;
                for (int k = 0; k < col_tasks; ++k) {
                    const int t = warp + kWarps * k;
                    const int tcol = 2 * (((t & ncb_mask) << (5 - lS)) + (lane >> lS));
                    const int rchunk = ((t >> lncb) << lS) + (lane & (S - 1));
                    uint32_t gw[16];
                    uint64_t e[16];
                    gather_pair<TC>(tile_s, tcol, rchunk, gw);
                    widen_cols(gw, mc, e);
                    fwht_pair(e, n, rchunk & (S - 1));
                    float Ma, Mb;
                    amax_1d_pair(e, bwc, Ma, Mb);
                    const int64_t lrow = lr0 + rchunk * kChunk;
                    const bool wsc = (lrow & (bwc - 1)) == 0;
                    const int64_t ca = c0 + tcol, cb = ca + 1;
                    Dest A, B;
                    A.codes = gcodes + ca * out_ld + (lrow >> 1);
                    B.codes = A.codes + out_ld;
                    A.s0 = A.s1 = gscales + (ca * sc_ld + (lrow >> lbwc)) * SZ;
                    B.s0 = B.s1 = A.s0 + sc_ld * SZ;
                    A.valid = lrow < padded && ca < p.cols;
                    B.valid = lrow < padded && cb < p.cols;
                    A.w0 = B.w0 = wsc;
                    A.w1 = B.w1 = false;
                    A.lin0 = (uint64_t)ca * (uint64_t)padded + (uint64_t)lrow;
                    B.lin0 = A.lin0 + (uint64_t)padded;
                    emit_pair<GRID, SR, PO2 ? 1 : 0>(e, Ma, Ma, Mb, Mb, false, fd, A, B, p.sr_keys, 1u, grp_id);
                }
            }
        }
        // everyone is done with stage s: refill it (the fence orders this
        // CTA's generic shared-memory accesses before the async-proxy write)
        __syncthreads();
        if (tid == 0) {
            const int next = tile + kStages * gridDim.x;
            if (next < num_tiles) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(next, s);
            }
        }
        if (++s == kStages) {
            s = 0;
            phase ^= 1u;
        }
    }
    // a broken-off loop leaves copies in flight: let them land (bounded)
    if (tid == 0)
        for (int k = i; k < i + kStages; ++k) {
            const int tile = blockIdx.x + k * gridDim.x;
            if (tile >= num_tiles) break;
            wait_phase(bars + 8u * (k % kStages), (uint32_t)((k / kStages) & 1), kWaitLimit);
        }
}

// ------------------------------------------------------ row-wise (lean)
// Row-wise quantization with 1-D blocks and n <= 128, the FPROP operands'
// case, over up to kMaxBatch independent tensors in one launch (their tiles
// are numbered one after the other).  Same steps as the row pass above, with
// 128 x 128 tiles fixed at compile time, tile coordinates and output pointers
// advanced without division, and per-row bounds checks only on ragged tiles.
struct RowsMaps {
    CUtensorMap m[kMaxBatch];
};

// N16: n = 16 (the FPROP operands' case), with the four butterfly strides
// fixed at compile time.
// TC: tile columns, 128, or 256 for n = 256 (whose segments span 16 chunks);
// the tiles hold 16 K elements either way.
template <int GRID, bool SR, int SF, bool N16, int CTAS, int TC>
__global__ void __launch_bounds__(kThreads, CTAS)
quantize_rows_kernel(const __grid_constant__ RowsMaps maps, const RowsParams p) {
    constexpr int TR = 16384 / TC;
    constexpr int kTileBytes = TR * TC * 2;
    constexpr int SZ = SF == 0 ? 4 : 1;
    constexpr int kCPR = TC / kChunk;      // 16-element chunks per tile row
    constexpr int kRPI = kThreads / kCPR;  // tile rows per thread step
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 127u) & ~127u) - raw;
    uint8_t* base = smem_raw + pad;
    const int kStages = p.stages;
    const uint32_t bars = smem_addr(base + kStages * kTileBytes);
    const int tid = threadIdx.x;
    const int cchunk = tid % kCPR;
    const int r0 = tid / kCPR;
    const int n = p.n;
    Fold fd;
    fd.inv_s = p.inv_sqrt_n;
    fd.pow4 = p.pow4;
    fd.j = p.log4n;
    fd.g = 0.0f;
    const int seg_row = (cchunk * kChunk % (n > kChunk ? n : kChunk)) / kChunk;
    SignMasks mrow;
    {
        const int pos = (cchunk * kChunk) & 255;
        make_masks((p.sign_bits[pos >> 5] >> (pos & 31)) & 0xFFFFu, mrow);
    }
    const int lbw = p.lbw;

    // tensor and tile coordinates of a tile index
    auto locate = [&](int tile, int& t, int& rt, int& ct) {
        t = 0;
        while (t + 1 < p.count && tile >= p.t[t + 1].tile0) ++t;
        const int local = tile - p.t[t].tile0;
        rt = local / p.t[t].col_tiles;
        ct = local - rt * p.t[t].col_tiles;
    };
    auto issue = [&](int tile, int s) {
        int t, rt, ct;
        locate(tile, t, rt, ct);
        const uint32_t bar = bars + 8u * s;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kTileBytes) : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
            ::"r"(smem_addr(base + s * kTileBytes)), "l"((uint64_t)&maps.m[t]), "r"(ct * TC), "r"(rt * TR), "r"(bar)
            : "memory");
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s)
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8u * s));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    griddep_wait();
    griddep_launch();
    const uint32_t wait_limit = g_quant_wait_limit;
    if (tid == 0)
        for (int s = 0; s < kStages; ++s) {
            const int tile = blockIdx.x + s * gridDim.x;
            if (tile < p.num_tiles) issue(tile, s);
        }

    int t = 0, rt = 0, ct = 0, step_r = 0, step_c = 0;
    auto relocate = [&](int tile) {
        locate(tile, t, rt, ct);
        step_r = (int)gridDim.x / p.t[t].col_tiles;
        step_c = (int)gridDim.x - step_r * p.t[t].col_tiles;
        // two-level scale: the tensor amax was written by the pre-pass (before this launch)
        if (SF == 2) fd.g = __fdiv_rn(*p.t[t].amax, grid_qmax(GRID) * 448.0f);
    };
    if ((int)blockIdx.x < p.num_tiles) relocate(blockIdx.x);
    int s = 0;
    uint32_t phase = 0;
    int i = 0;
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++i) {
        if (i) {
            ct += step_c;
            rt += step_r;
            if (ct >= p.t[t].col_tiles) {
                ct -= p.t[t].col_tiles;
                ++rt;
            }
            if (rt >= p.t[t].row_tiles) relocate(tile);  // into the next tensor
        }
        const bool landed = wait_phase(bars + 8u * s, phase, wait_limit);
        if (!__syncthreads_and(landed)) {
            if (tid == 0) atomicExch(&g_quant_error, 1);
            break;
        }
        const RowsTensor& T = p.t[t];
        const uint16_t* tile_s = reinterpret_cast<const uint16_t*>(base + s * kTileBytes);
        const int row0 = rt * TR;
        const int col = ct * TC + cchunk * kChunk;
        const bool col_ok = col < T.cols;
        const int left = T.rows - row0 - r0;  // rows of this thread's first row onward
        const bool full = T.rows - row0 >= TR;
        uint8_t* cp = T.codes + (int64_t)(row0 + r0) * T.codes_ld + (GRID == 4 ? col : col >> 1);
        uint8_t* sp = T.scales + ((int64_t)(row0 + r0) * T.scales_ld + (col >> lbw)) * SZ;
        const int64_t cstep = (int64_t)kRPI * T.codes_ld;
        const int64_t sstep = (int64_t)kRPI * T.scales_ld * SZ;
        const bool wsc = (col & ((1 << lbw) - 1)) == 0;
        const uint16_t* src = tile_s + r0 * TC + cchunk * kChunk;
#pragma unroll
        for (int it = 0; it < TR / (2 * kRPI); ++it) {
            const int ra = 2 * kRPI * it;
            uint32_t wa[8], wb[8];
            uint64_t e[16];
            const uint4* pa = reinterpret_cast<const uint4*>(src + ra * TC);
            const uint4* pb = reinterpret_cast<const uint4*>(src + (ra + kRPI) * TC);
            const uint4 a0 = pa[0], a1 = pa[1], b0 = pb[0], b1 = pb[1];
            wa[0] = a0.x; wa[1] = a0.y; wa[2] = a0.z; wa[3] = a0.w;
            wa[4] = a1.x; wa[5] = a1.y; wa[6] = a1.z; wa[7] = a1.w;
            wb[0] = b0.x; wb[1] = b0.y; wb[2] = b0.z; wb[3] = b0.w;
            wb[4] = b1.x; wb[5] = b1.y; wb[6] = b1.z; wb[7] = b1.w;
            widen_rows(wa, wb, mrow, e);
            float Ma, Mb;
            if (N16) {
                fwht_pair16(e);
                amax_pair(e, 0, 16, Ma, Mb);
                if (lbw == 5) {  // 1 x 32 blocks: the neighbouring lane holds the other half
                    Ma = fmaxf(Ma, __shfl_xor_sync(0xFFFFFFFFu, Ma, 1));
                    Mb = fmaxf(Mb, __shfl_xor_sync(0xFFFFFFFFu, Mb, 1));
                }
            } else {
                fwht_pair(e, n, seg_row);
                amax_1d_pair(e, 1 << lbw, Ma, Mb);
            }
            Dest A, B;
            A.codes = cp + (2 * it) * cstep;
            B.codes = A.codes + cstep;
            A.s0 = A.s1 = sp + (2 * it) * sstep;
            B.s0 = B.s1 = A.s0 + sstep;
            A.valid = col_ok && (full || ra < left);
            B.valid = col_ok && (full || ra + kRPI < left);
            A.w0 = B.w0 = wsc;
            A.w1 = B.w1 = false;
            A.lin0 = (uint64_t)(row0 + r0 + ra) * (uint64_t)T.cols + (uint64_t)col;
            B.lin0 = A.lin0 + (uint64_t)kRPI * (uint64_t)T.cols;
            emit_pair<GRID, SR, SF>(e, Ma, Ma, Mb, Mb, false, fd, A, B, p.sr_keys, 0u, (uint32_t)p.group);
        }
        // everyone is done with stage s: refill it
        __syncthreads();
        if (tid == 0) {
            const int next = tile + kStages * gridDim.x;
            if (next < p.num_tiles) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(next, s);
            }
        }
        if (++s == kStages) {
            s = 0;
            phase ^= 1u;
        }
    }
    // a broken-off loop leaves copies in flight: let them land (bounded)
    if (tid == 0)
        for (int k = i; k < i + kStages; ++k) {
            const int tile = blockIdx.x + k * gridDim.x;
            if (tile >= p.num_tiles) break;
            wait_phase(bars + 8u * (k % kStages), (uint32_t)((k / kStages) & 1), kWaitLimit);
        }
}

// ------------------------------------------------------------- RHT only
__global__ void __launch_bounds__(kThreads)
rht_kernel(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int n, float inv_sqrt_n,
           SignBits sb, float* z, int64_t ldz) {
    const int64_t chunks_per_row = cols / kChunk;
    const int64_t total = rows * chunks_per_row;
    // grid-stride over whole warps so that shuffles see full warps
    for (int64_t base = (int64_t)blockIdx.x * kThreads; base < total; base += (int64_t)gridDim.x * kThreads) {
        const int64_t q = base + threadIdx.x;
        const bool valid = q < total;
        const int64_t r = valid ? q / chunks_per_row : 0;
        const int64_t cc = valid ? q % chunks_per_row : 0;
        uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (valid) {
            const uint4* src = reinterpret_cast<const uint4*>(x + r * ld + cc * kChunk);
            const uint4 a = __ldg(src), b = __ldg(src + 1);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
            w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        }
        const int pos = (int)((cc * kChunk) % 256);
        const uint32_t sgn = (sb.bits[pos / 32] >> (pos % 32)) & 0xFFFFu;
        float v[16];
        const int seg_lane = (int)((cc * kChunk) % (n > kChunk ? n : kChunk)) / kChunk;
        widen16(w, sgn, v);
        fwht16(v, n, seg_lane);
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = __fmul_rn(v[k], inv_sqrt_n);
        if (valid) {
            float4* dst = reinterpret_cast<float4*>(z + r * ldz + cc * kChunk);
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        }
    }
}

// ------------------------------------------------------------- launchers
template <int GRID, bool SR, bool PO2, int TC>
static cudaError_t launch_q(const CUtensorMap& map, const QuantParams& p, int num_tiles, int num_sms,
                            cudaStream_t st) {
    const size_t smem = (size_t)p.stages * p.tile_rows * TC * 2 + 4 * (size_t)p.amax_slots + 8 * p.stages + 128;
    auto k = quantize_kernel<GRID, SR, PO2, TC>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = num_tiles < kCtasPerSm * num_sms ? num_tiles : kCtasPerSm * num_sms;
    return launch_pdl(k, dim3(grid), dim3(kThreads), smem, st, map, p, num_tiles);
}

template <int GRID, bool SR, bool PO2>
static cudaError_t launch_q_tiles(const CUtensorMap& map, const QuantParams& p, int tc, int num_tiles, int num_sms,
                                  cudaStream_t st) {
    if (tc == 256) return launch_q<GRID, SR, PO2, 256>(map, p, num_tiles, num_sms, st);
    return launch_q<GRID, SR, PO2, 128>(map, p, num_tiles, num_sms, st);
}

cudaError_t launch_quantize(const QuantParams& p, int grid, bool sr, bool po2, int tc, int tr, int num_tiles,
                            int64_t total_rows, int num_sms, cudaStream_t st) {
    CUtensorMap map;
    if (!encode_map_2d(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, p.x, (uint64_t)p.cols, (uint64_t)total_rows,
                       (uint64_t)p.ld * 2, (uint32_t)tc, (uint32_t)tr, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
#define UFP4_Q(G)                                                                                   \
    if (grid == G) {                                                                                \
        if (sr) return po2 ? launch_q_tiles<G, true, true>(map, p, tc, num_tiles, num_sms, st)      \
                           : launch_q_tiles<G, true, false>(map, p, tc, num_tiles, num_sms, st);    \
        return po2 ? launch_q_tiles<G, false, true>(map, p, tc, num_tiles, num_sms, st)             \
                   : launch_q_tiles<G, false, false>(map, p, tc, num_tiles, num_sms, st);           \
    }
    UFP4_Q(0)
    UFP4_Q(1)
    UFP4_Q(2)
    UFP4_Q(3)
#undef UFP4_Q
    return cudaErrorInvalidValue;
}

// CTAs per SM and ring depth of the row kernel (128 x 128 tiles): two CTAs
// of up to 128 registers a thread, each with three 32 KB stages (measured on
// the 16384 x 7168 + 7168 x 7168 batch: 6.13 TB/s, against 5.87 TB/s for
// three CTAs of two stages, whose 80-register cap costs 1.6 instructions per
// element in register moves).
constexpr int kRowsCtas = 2, kRowsStages = 3;

template <int GRID, bool SR, int SF, bool N16, int CTAS, int TC>
static cudaError_t launch_rows_cfg(const RowsMaps& maps, const RowsParams& p, int num_sms, cudaStream_t st) {
    const size_t smem = (size_t)p.stages * 16384 * 2 + 8 * p.stages + 128;
    auto k = quantize_rows_kernel<GRID, SR, SF, N16, CTAS, TC>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = p.num_tiles < CTAS * num_sms ? p.num_tiles : CTAS * num_sms;
    return launch_pdl(k, dim3(grid), dim3(kThreads), smem, st, maps, p);
}

template <int GRID, bool SR, int SF>
static cudaError_t launch_rows(const RowsMaps& maps, RowsParams& p, int num_sms, cudaStream_t st) {
    p.stages = kRowsStages;
    if (p.tc == 256) return launch_rows_cfg<GRID, SR, SF, false, kRowsCtas, 256>(maps, p, num_sms, st);
    if (p.n == 16) return launch_rows_cfg<GRID, SR, SF, true, kRowsCtas, 128>(maps, p, num_sms, st);
    return launch_rows_cfg<GRID, SR, SF, false, kRowsCtas, 128>(maps, p, num_sms, st);
}

cudaError_t launch_quantize_rows(RowsParams& p, int grid, bool sr, int sf, int num_sms, cudaStream_t st) {
    RowsMaps maps;
    memset(&maps, 0, sizeof(maps));
    for (int t = 0; t < p.count; ++t) {
        const RowsTensor& T = p.t[t];
        if (!encode_map_2d(&maps.m[t], CU_TENSOR_MAP_DATA_TYPE_UINT16, T.x, (uint64_t)T.cols, (uint64_t)T.rows,
                           (uint64_t)T.ld * 2, (uint32_t)p.tc, (uint32_t)(16384 / p.tc), CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
#define UFP4_R(G)                                                                              \
    if (grid == G) {                                                                           \
        if (sr) return sf == 2 ? launch_rows<G, true, 2>(maps, p, num_sms, st)                 \
                     : sf == 1 ? launch_rows<G, true, 1>(maps, p, num_sms, st)                 \
                               : launch_rows<G, true, 0>(maps, p, num_sms, st);                \
        return sf == 2 ? launch_rows<G, false, 2>(maps, p, num_sms, st)                        \
             : sf == 1 ? launch_rows<G, false, 1>(maps, p, num_sms, st)                        \
                       : launch_rows<G, false, 0>(maps, p, num_sms, st);                       \
    }
    UFP4_R(0)
    UFP4_R(1)
    UFP4_R(2)
    UFP4_R(3)
#undef UFP4_R
    if (grid == 4 && !sr && sf == 1) return launch_rows<4, false, 1>(maps, p, num_sms, st);  // MXFP8
    return cudaErrorInvalidValue;
}

uint32_t quant_wait_limit_default() { return kWaitLimit; }

cudaError_t set_quant_wait_limit(uint32_t polls) {
    return cudaMemcpyToSymbol(g_quant_wait_limit, &polls, sizeof(polls));
}

cudaError_t quant_error_read_clear(int* value) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_quant_error, sizeof(int));
    if (e != cudaSuccess) return e;
    if (v) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_quant_error, &zero, sizeof(int));
    }
    *value = v;
    return e;
}

cudaError_t launch_rht(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int n,
                       float inv_sqrt_n, const SignBits& sb, float* z, int64_t ldz, int num_sms,
                       cudaStream_t st) {
    const int64_t total = rows * (cols / kChunk);
    int64_t blocks = (total + kThreads - 1) / kThreads;
    const int64_t cap = (int64_t)num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    rht_kernel<<<(unsigned)blocks, kThreads, 0, st>>>(x, rows, cols, ld, n, inv_sqrt_n, sb, z, ldz);
    return cudaGetLastError();
}

// Loads every kernel of this unit (cudaFuncGetAttributes loads a function
// that has not been loaded yet).
template <int G, bool SR, bool PO2>
static void preload_q(cudaFuncAttributes* a) {
    cudaFuncGetAttributes(a, quantize_kernel<G, SR, PO2, 128>);
    cudaFuncGetAttributes(a, quantize_kernel<G, SR, PO2, 256>);
}
template <int G, bool SR>
static void preload_rows(cudaFuncAttributes* a) {
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 0, false, kRowsCtas, 128>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 1, false, kRowsCtas, 128>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 2, false, kRowsCtas, 128>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 0, true, kRowsCtas, 128>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 1, true, kRowsCtas, 128>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 2, true, kRowsCtas, 128>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 0, false, kRowsCtas, 256>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 1, false, kRowsCtas, 256>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 2, false, kRowsCtas, 256>);
}
template <int G>
static void preload_grid(cudaFuncAttributes* a) {
    preload_q<G, false, false>(a);
    preload_q<G, false, true>(a);
    preload_q<G, true, false>(a);
    preload_q<G, true, true>(a);
    preload_rows<G, false>(a);
    preload_rows<G, true>(a);
}
cudaError_t preload_quantize_kernels() {
    cudaFuncAttributes a;
    preload_grid<0>(&a);
    preload_grid<1>(&a);
    preload_grid<2>(&a);
    preload_grid<3>(&a);
    cudaFuncGetAttributes(&a, quantize_rows_kernel<4, false, 1, false, kRowsCtas, 128>);
    cudaFuncGetAttributes(&a, quantize_rows_kernel<4, false, 1, true, kRowsCtas, 128>);
    cudaFuncGetAttributes(&a, quantize_rows_kernel<4, false, 1, false, kRowsCtas, 256>);
    return cudaFuncGetAttributes(&a, rht_kernel);
}

}  // namespace ufp4
