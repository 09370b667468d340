// Fused RHT + block-scaled 4-bit quantizer for sm_103a.
//
// One CTA owns a TR x TC tile of the bf16 input and produces, from a single
// read of it, the row-wise quantization (RHT and blocks along the columns)
// and the column-wise quantization of the transpose (RHT and blocks along the
// rows), as required for FPROP, DGRAD and WGRAD (UFP4 summary, section 方法:
// RHT on all three training GEMMs; 2D-block tutorial: dX = dY W and
// dW = dY^T X need transposed operands).
//
//  * row pass: each thread carries 16 consecutive elements of a row, loaded
//    with one 256-bit (or two 128-bit) coalesced load, widened to fp32,
//    transformed (in-register butterflies for strides < 16, warp shuffles
//    above), scaled, rounded and packed straight from registers;
//  * column pass: the same bf16 values are parked in shared memory with an
//    XOR swizzle of 16-byte units by (row / 16), so that a warp reading 16
//    consecutive rows of 32/S columns hits distinct banks; each thread then
//    carries 16 consecutive rows of one column through the same steps;
//  * 2-D b x b blocks reduce their amax through shared-memory atomics.
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ufp4_device.cuh"

namespace ufp4 {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

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

// Scale, round, pack and store one 16-element chunk of transformed values z.
// M0 is the amax of the block holding elements 0..7, M1 of 8..15 (equal
// unless blocks are 8 wide).  w0 / w1: this thread writes the block's scale.
template <int GRID, bool SR, bool PO2>
__device__ __forceinline__ void emit_chunk(const float z[16], float M0, float M1, bool valid,
                                           bool w0, bool w1, uint8_t* codes_ptr, void* scales,
                                           int64_t si0, int64_t si1, uint64_t sr_seed,
                                           uint64_t lin0, uint32_t stream, uint32_t group) {
    constexpr float qmax = grid_qmax(GRID);
    float r0, r1;
    if (PO2) {
        const int e0 = scale_po2<GRID>(M0, r0);
        const int e1 = scale_po2<GRID>(M1, r1);
        if (valid) {
            uint8_t* sb = (uint8_t*)scales;
            if (w0) sb[si0] = (uint8_t)(e0 + 127);
            if (w1) sb[si1] = (uint8_t)(e1 + 127);
        }
    } else {
        float s0, s1;
        scale_fp32(M0, qmax, s0, r0);
        scale_fp32(M1, qmax, s1, r1);
        if (valid) {
            float* sb = (float*)scales;
            if (w0) sb[si0] = s0;
            if (w1) sb[si1] = s1;
        }
    }
    uint2 packed;
    if (SR) {
        uint32_t w[8];
        sr_draws16(sr_seed, lin0, stream, group, w);
        packed = round_sr16<GRID>(z, r0, r1, w);
    } else {
        packed = round_rtne16<GRID>(z, r0, r1);
    }
    if (valid) *reinterpret_cast<uint2*>(codes_ptr) = packed;
}

// widen + signs + FWHT + 1/sqrt(n)
__device__ __forceinline__ void build_z(const uint32_t w[8], uint32_t sgn, int n, int seg_lane,
                                        float inv_sqrt_n, float z[16]) {
    widen16(w, sgn, z);
    fwht16(z, n, seg_lane);
#pragma unroll
    for (int i = 0; i < 16; ++i) z[i] = __fmul_rn(z[i], inv_sqrt_n);
}

// Amax of a 1-D block of width bw >= 16 spread over bw/16 neighbouring lanes.
__device__ __forceinline__ float amax_1d(const float z[16], int bw) {
    float m = amax_range(z, 0, 16);
    for (int k = 1; k < bw / kChunk; k <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, k));
    return m;
}

// Read 16 consecutive rows (rchunk*16 ..) of tile column tcol from the
// swizzled tile (row r's 16-byte unit u lives at u ^ (((r/16) & 7) << 1)).
template <int TC>
__device__ __forceinline__ void gather_column(const uint16_t* tile, int tcol, int rchunk, uint32_t w[8]) {
    const int sw = (rchunk & 7) << 1;
    const int u = (tcol >> 3) ^ sw;
    const uint16_t* base = tile + (rchunk * kChunk) * TC + u * 8 + (tcol & 7);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t ea = base[(2 * j) * TC];
        const uint32_t eb = base[(2 * j + 1) * TC];
        w[j] = ea | (eb << 16);
    }
}

template <int GRID, bool SR, bool PO2, int TR, int TC>
__global__ void __launch_bounds__(kThreads)
quantize_kernel(const QuantParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    uint16_t* tile = reinterpret_cast<uint16_t*>(smem_raw);
    uint32_t* amax2d = reinterpret_cast<uint32_t*>(smem_raw + (p.do_col ? TR * TC * 2 : 0));

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int row_tile = blockIdx.x / p.col_tiles;
    const int col_tile = blockIdx.x % p.col_tiles;
    const int g = find_group(p, row_tile);
    const int64_t grow0 = p.grp_row0[g];                       // group's first input row
    const int64_t cnt = p.grp_row0[g + 1] - grow0;             // real rows of the group
    const int64_t padded = p.grp_pad0[g + 1] - p.grp_pad0[g];  // column-pass length
    const int64_t lr0 = (int64_t)(row_tile - p.grp_tile0[g]) * TR;  // tile's first row in the group
    const int64_t c0 = (int64_t)col_tile * TC;
    const int n = p.n;
    const int nslot = p.is2d ? (TR / p.b2d) * (TC / p.b2d) : 0;

    constexpr int kCPR = TC / kChunk;       // chunks per tile row
    constexpr int kRPI = kThreads / kCPR;   // tile rows per iteration
    constexpr int kIters = TR / kRPI;

    // ------------------------------------------------ load (one HBM read)
    const int cchunk = tid % kCPR;
    const int64_t col = c0 + cchunk * kChunk;
    uint32_t w[kIters][8];
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
        const int trow = it * kRPI + tid / kCPR;
        const int64_t lrow = lr0 + trow;
#pragma unroll
        for (int j = 0; j < 8; ++j) w[it][j] = 0u;
        if (lrow < cnt && col < p.cols) {
            const uint16_t* src = p.x + (grow0 + lrow) * p.ld + col;
            if (p.vec256) {
                asm volatile("ld.global.nc.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                             : "=r"(w[it][0]), "=r"(w[it][1]), "=r"(w[it][2]), "=r"(w[it][3]),
                               "=r"(w[it][4]), "=r"(w[it][5]), "=r"(w[it][6]), "=r"(w[it][7])
                             : "l"(src));
            } else {
                const uint4 a = __ldg(reinterpret_cast<const uint4*>(src));
                const uint4 b = __ldg(reinterpret_cast<const uint4*>(src) + 1);
                w[it][0] = a.x; w[it][1] = a.y; w[it][2] = a.z; w[it][3] = a.w;
                w[it][4] = b.x; w[it][5] = b.y; w[it][6] = b.z; w[it][7] = b.w;
            }
        }
    }
    if (p.do_col) {
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
            const int trow = it * kRPI + tid / kCPR;
            const int sw = ((trow >> 4) & 7) << 1;
            uint4* rowp = reinterpret_cast<uint4*>(tile + trow * TC);
            const uint4 lo = make_uint4(w[it][0], w[it][1], w[it][2], w[it][3]);
            const uint4 hi = make_uint4(w[it][4], w[it][5], w[it][6], w[it][7]);
            // alternate the store order over lane quads to spread the banks
            if ((cchunk >> 2) & 1) {
                rowp[(2 * cchunk + 1) ^ sw] = hi;
                rowp[(2 * cchunk) ^ sw] = lo;
            } else {
                rowp[(2 * cchunk) ^ sw] = lo;
                rowp[(2 * cchunk + 1) ^ sw] = hi;
            }
        }
    }

    // ------------------------------------------------------------ row pass
    if (p.do_row) {
        const int seg_lane = (cchunk * kChunk % (n > kChunk ? n : kChunk)) / kChunk;
        const uint32_t sgn = chunk_signs(p, cchunk * kChunk);
        const int bw = p.bw_row;
        if (p.is2d) {
            const int b = p.b2d;
            const int nbc = TC / b;
            for (int i = tid; i < nslot; i += kThreads) amax2d[i] = 0u;
            __syncthreads();
#pragma unroll
            for (int it = 0; it < kIters; ++it) {
                const int trow = it * kRPI + tid / kCPR;
                float z[16];
                build_z(w[it], sgn, n, seg_lane, p.inv_sqrt_n, z);
                if (b == 8) {
                    post_amax(&amax2d[(trow / b) * nbc + 2 * cchunk], amax_range(z, 0, 8));
                    post_amax(&amax2d[(trow / b) * nbc + 2 * cchunk + 1], amax_range(z, 8, 16));
                } else {
                    post_amax(&amax2d[(trow / b) * nbc + (cchunk * kChunk) / b], amax_range(z, 0, 16));
                }
            }
            __syncthreads();
#pragma unroll
            for (int it = 0; it < kIters; ++it) {
                const int trow = it * kRPI + tid / kCPR;
                const int64_t lrow = lr0 + trow;
                float z[16];
                build_z(w[it], sgn, n, seg_lane, p.inv_sqrt_n, z);
                const int s0 = (trow / b) * nbc + (b == 8 ? 2 * cchunk : (cchunk * kChunk) / b);
                const float M0 = __uint_as_float(amax2d[s0]);
                const float M1 = __uint_as_float(amax2d[b == 8 ? s0 + 1 : s0]);
                const int64_t sidx = (lrow / b) * p.row.scales_ld + col / b;
                const bool first_row = (lrow % b) == 0;
                const bool w0 = first_row && (b == 8 || (col % b) == 0);
                const bool w1 = first_row && b == 8;
                uint8_t* cp = (uint8_t*)p.row.codes + (grow0 + lrow) * p.row.codes_ld + col / 2;
                const uint64_t lin0 = (uint64_t)lrow * (uint64_t)p.cols + (uint64_t)col;
                emit_chunk<GRID, SR, PO2>(z, M0, M1, lrow < cnt && col < p.cols, w0, w1, cp,
                                          p.row.scales, sidx, sidx + 1, p.sr_seed, lin0, 0u, (uint32_t)(p.group_base + g));
            }
        } else {
#pragma unroll
            for (int it = 0; it < kIters; ++it) {
                const int trow = it * kRPI + tid / kCPR;
                const int64_t lrow = lr0 + trow;
                const int64_t orow = grow0 + lrow;  // row-wise output rows follow the input rows
                float z[16];
                build_z(w[it], sgn, n, seg_lane, p.inv_sqrt_n, z);
                const float M = amax_1d(z, bw);
                const int64_t sidx = orow * p.row.scales_ld + col / bw;
                uint8_t* cp = (uint8_t*)p.row.codes + orow * p.row.codes_ld + col / 2;
                const uint64_t lin0 = (uint64_t)lrow * (uint64_t)p.cols + (uint64_t)col;
                emit_chunk<GRID, SR, PO2>(z, M, M, lrow < cnt && col < p.cols, (col % bw) == 0, false,
                                          cp, p.row.scales, sidx, sidx, p.sr_seed, lin0, 0u, (uint32_t)(p.group_base + g));
            }
        }
    }
    if (!p.do_col) return;

    // --------------------------------------------------------- column pass
    __syncthreads();
    // S lanes share one column segment (S consecutive 16-row chunks of one
    // column); a warp task covers 32/S columns x S chunks.
    const int S = p.col_seg_lanes;
    const int cpw = 32 / S;
    const int ncb = TC / cpw;
    constexpr int kTasks = (TR / kChunk) * TC / 32 / kWarps;  // tasks per warp
    const int bwc = p.bw_col;
    const int64_t out_ld = p.col_grouped ? padded / 2 : p.col.codes_ld;
    const int sdiv = p.is2d ? p.b2d : bwc;
    const int64_t sc_ld = p.col_grouped ? padded / sdiv : p.col.scales_ld;
    uint8_t* gcodes = (uint8_t*)p.col.codes + (p.col_grouped ? p.cols * (p.grp_pad0[g] / 2) : 0);
    uint8_t* gscales = (uint8_t*)p.col.scales +
                       (p.col_grouped ? p.cols * (p.grp_pad0[g] / sdiv) * (PO2 ? 1 : 4) : 0);
    if (p.is2d) {
        const int b = p.b2d;
        const int nbq = TR / b;  // blocks along the quantized dimension (tile rows)
        for (int i = tid; i < nslot; i += kThreads) amax2d[i] = 0u;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kTasks; ++k) {
            const int t = warp + kWarps * k;
            const int tcol = (t % ncb) * cpw + lane / S;
            const int rchunk = (t / ncb) * S + lane % S;
            uint32_t wc[8];
            gather_column<TC>(tile, tcol, rchunk, wc);
            float z[16];
            build_z(wc, chunk_signs(p, rchunk * kChunk), n, rchunk % S, p.inv_sqrt_n, z);
            if (b == 8) {
                post_amax(&amax2d[(tcol / b) * nbq + 2 * rchunk], amax_range(z, 0, 8));
                post_amax(&amax2d[(tcol / b) * nbq + 2 * rchunk + 1], amax_range(z, 8, 16));
            } else {
                post_amax(&amax2d[(tcol / b) * nbq + (rchunk * kChunk) / b], amax_range(z, 0, 16));
            }
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kTasks; ++k) {
            const int t = warp + kWarps * k;
            const int tcol = (t % ncb) * cpw + lane / S;
            const int rchunk = (t / ncb) * S + lane % S;
            uint32_t wc[8];
            gather_column<TC>(tile, tcol, rchunk, wc);
            float z[16];
            build_z(wc, chunk_signs(p, rchunk * kChunk), n, rchunk % S, p.inv_sqrt_n, z);
            const int s0 = (tcol / b) * nbq + (b == 8 ? 2 * rchunk : (rchunk * kChunk) / b);
            const float M0 = __uint_as_float(amax2d[s0]);
            const float M1 = __uint_as_float(amax2d[b == 8 ? s0 + 1 : s0]);
            const int64_t colg = c0 + tcol;
            const int64_t lrow = lr0 + rchunk * kChunk;
            const int64_t sidx = (colg / b) * sc_ld + lrow / b;
            const bool first_col = (colg % b) == 0;
            const bool w0 = first_col && (b == 8 || (lrow % b) == 0);
            const bool w1 = first_col && b == 8;
            uint8_t* cp = gcodes + colg * out_ld + lrow / 2;
            const uint64_t lin0 = (uint64_t)colg * (uint64_t)padded + (uint64_t)lrow;
            emit_chunk<GRID, SR, PO2>(z, M0, M1, lrow < padded && colg < p.cols, w0, w1, cp, gscales,
                                      sidx, sidx + 1, p.sr_seed, lin0, 1u, (uint32_t)(p.group_base + g));
        }
    } else {
#pragma unroll
        for (int k = 0; k < kTasks; ++k) {
            const int t = warp + kWarps * k;
            const int tcol = (t % ncb) * cpw + lane / S;
            const int rchunk = (t / ncb) * S + lane % S;
            uint32_t wc[8];
            gather_column<TC>(tile, tcol, rchunk, wc);
            float z[16];
            build_z(wc, chunk_signs(p, rchunk * kChunk), n, rchunk % S, p.inv_sqrt_n, z);
            const float M = amax_1d(z, bwc);
            const int64_t colg = c0 + tcol;
            const int64_t lrow = lr0 + rchunk * kChunk;
            const int64_t sidx = colg * sc_ld + lrow / bwc;
            uint8_t* cp = gcodes + colg * out_ld + lrow / 2;
            const uint64_t lin0 = (uint64_t)colg * (uint64_t)padded + (uint64_t)lrow;
            emit_chunk<GRID, SR, PO2>(z, M, M, lrow < padded && colg < p.cols, (lrow % bwc) == 0, false,
                                      cp, gscales, sidx, sidx, p.sr_seed, lin0, 1u, (uint32_t)(p.group_base + g));
        }
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
        build_z(w, sgn, n, seg_lane, inv_sqrt_n, v);
        if (valid) {
            float4* dst = reinterpret_cast<float4*>(z + r * ldz + cc * kChunk);
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        }
    }
}

// ------------------------------------------------------------- launchers
template <int GRID, bool SR, bool PO2, int TR, int TC>
static cudaError_t launch_q(const QuantParams& p, int num_tiles, cudaStream_t st) {
    const int amax_bytes = p.is2d ? (TR / p.b2d) * (TC / p.b2d) * 4 : 0;
    const size_t smem = (p.do_col ? (size_t)TR * TC * 2 : 0) + amax_bytes;
    auto k = quantize_kernel<GRID, SR, PO2, TR, TC>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    k<<<num_tiles, kThreads, smem, st>>>(p);
    return cudaGetLastError();
}

template <int GRID, bool SR, bool PO2>
static cudaError_t launch_q_tiles(const QuantParams& p, int tc, int num_tiles, cudaStream_t st) {
    if (tc == 256) return launch_q<GRID, SR, PO2, 64, 256>(p, num_tiles, st);
    return launch_q<GRID, SR, PO2, 128, 128>(p, num_tiles, st);
}

cudaError_t launch_quantize(const QuantParams& p, int grid, bool sr, bool po2, int tc, int num_tiles,
                            cudaStream_t st) {
#define UFP4_Q(G)                                                                  \
    if (grid == G) {                                                               \
        if (sr) return po2 ? launch_q_tiles<G, true, true>(p, tc, num_tiles, st)   \
                           : launch_q_tiles<G, true, false>(p, tc, num_tiles, st); \
        return po2 ? launch_q_tiles<G, false, true>(p, tc, num_tiles, st)          \
                   : launch_q_tiles<G, false, false>(p, tc, num_tiles, st);        \
    }
    UFP4_Q(0)
    UFP4_Q(1)
    UFP4_Q(2)
#undef UFP4_Q
    return cudaErrorInvalidValue;
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

}  // namespace ufp4
