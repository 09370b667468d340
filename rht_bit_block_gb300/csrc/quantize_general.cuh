// Fused RHT + block-scaled 4-bit quantizer for sm_103a: the general kernel.
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
// Row-wise calls with 1-D blocks take the leaner kernel of quantize_rows.cu;
// the steps both share are in quantize_common.cuh.  This header holds the
// kernel template and its launcher; quantize.cu instantiates the RTNE
// kernels and quantize_sr.cu the SR ones, so the two compile in parallel.
#pragma once

#include <algorithm>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "quantize_common.cuh"
#include "ufp4_device.cuh"

namespace ufp4 {

// Error word and wait limit of the general kernel, one copy per unit that
// instantiates it (quantize.cu: RTNE, quantize_sr.cu: SR).
static __device__ int g_quant_error;

// CTAs per SM: 2-D blocks 2 (16 warps, up to 128 registers a thread, about
// 96 KB of ring each); 1-D blocks 3 (24 warps, up to 80 registers, about
// 64 KB of ring each)
__host__ __device__ constexpr int general_ctas(bool two_d) { return two_d ? 2 : 3; }

// Polls of a tile's barrier before a general-kernel CTA gives up (a failure-
// detection hook can lower it; the drain of copies in flight always uses
// kWaitLimit).
static __device__ uint32_t g_quant_wait_limit = kWaitLimit;

// TWO_D: b x b blocks (compile-time, so that each instantiation carries only
// its own block path); they need power-of-two scales (PO2).
template <int GRID, bool SR, bool PO2, int TC, bool N16, bool TWO_D>
__global__ void __launch_bounds__(kThreads, general_ctas(TWO_D))
quantize_kernel(const __grid_constant__ CUtensorMap tmap, const QuantParams p, const int num_tiles) {
    extern __shared__ uint8_t smem_raw[];
    constexpr int SZ = PO2 ? 1 : 4;         // bytes per scale
    const int TR = p.tile_rows;             // 64 or 128 (runtime)
    const int tile_bytes = TR * TC * 2;
    const int kStages = p.stages;           // ring depth (runtime, <= kMaxStages)
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 127u) & ~127u) - raw;
    uint8_t* base = smem_raw + pad;
    uint32_t* amax2d = reinterpret_cast<uint32_t*>(base + kStages * tile_bytes);  // 2-D: 4 sets of amax_slots
    const uint32_t bars = smem_addr(base + kStages * tile_bytes + 16 * p.amax_slots);  // 8-byte aligned
    const uint32_t empties = bars + 8u * kStages;  // 1-D blocks: every warp done with the stage

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
        for (int s = 0; s < kStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8u * s));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empties + 8u * s), "r"(kWarps));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (TWO_D)
        for (int q = tid; q < 4 * p.amax_slots; q += kThreads) amax2d[q] = 0u;
    __syncthreads();
    // the input may come from the previous kernel, and that kernel may still
    // read buffers this one writes: wait for it before the first copy
    griddep_wait();
    griddep_launch();
    const uint32_t wait_limit = g_quant_wait_limit;
    int issued = 0;  // tiles of this CTA issued so far (thread 0)
    if (tid == 0)
        for (int s = 0; s < kStages; ++s) {
            const int tile = blockIdx.x + s * gridDim.x;
            if (tile < num_tiles) {
                issue(tile, s);
                issued = s + 1;
            }
        }

    // row pass: a thread owns chunk column cchunk of the row pairs
    // (r, r + kRPI), r = r0 + 2 * kRPI * it
    constexpr int kCPR = TC / kChunk;       // chunks per tile row
    constexpr int kRPI = kThreads / kCPR;   // tile rows per thread step
    const int pairs = TR / (2 * kRPI);
    const int cchunk = tid % kCPR;
    const int r0 = tid / kCPR;
    const int seg_row = (cchunk * kChunk % (n > kChunk ? n : kChunk)) / kChunk;
    // n = 16: every chunk of either pass has the same 16 signs, read from the
    // kernel parameters (p.smask16); otherwise masks in registers
    SignMasks mrow;
    if (!N16) make_masks(chunk_signs(p, cchunk * kChunk), mrow);
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
    if (!N16) make_masks(chunk_signs(p, (lane & (S - 1)) * kChunk), mc);
    const int nslot = p.amax_slots;
    // tile coordinates advance by gridDim.x tiles per step, without division
    const int step_r = gridDim.x / p.col_tiles, step_c = gridDim.x - step_r * p.col_tiles;
    int row_tile = blockIdx.x / p.col_tiles, col_tile = blockIdx.x - row_tile * p.col_tiles;
    int g = p.num_groups > 1 ? find_group(p, row_tile) : 0;
    // values of the current group, reloaded only when the group changes
    int gt0;                 // first row tile of the group
    int64_t grow0, cnt;      // first input row and row count
    int64_t padded;          // padded row count (column-wise output)
    uint32_t grp_id;         // SR counter group id
    int64_t out_ld1, sc_ld1; // 1-D column-wise output: code and scale leading dimensions
    uint8_t* gcodes1;        // 1-D column-wise output: the group's codes and scales
    uint8_t* gscales1;
    auto load_group = [&](int gg) {
        gt0 = p.grp_tile0[gg];
        grow0 = p.grp_row0[gg];
        cnt = p.grp_row0[gg + 1] - grow0;
        padded = p.grp_pad0[gg + 1] - p.grp_pad0[gg];
        grp_id = (uint32_t)(p.group_base + gg);
        out_ld1 = p.col_grouped ? padded / 2 : p.col.codes_ld;
        sc_ld1 = p.col_grouped ? (padded >> p.lbw_col) : p.col.scales_ld;
        gcodes1 = (uint8_t*)p.col.codes + (p.col_grouped ? p.cols * (p.grp_pad0[gg] / 2) : 0);
        gscales1 = (uint8_t*)p.col.scales + (p.col_grouped ? p.cols * (p.grp_pad0[gg] >> p.lbw_col) * SZ : 0);
    };
    load_group(g);

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
            if (p.num_groups > 1) {
                const int ng = find_group(p, row_tile);
                if (ng != g) {
                    g = ng;
                    load_group(g);
                }
            }
        }
        // 1-D blocks: no CTA barrier per tile; each warp waits for the copy
        // itself, and a warp whose wait gave up leaves the loop (the others
        // then give up on the stages it no longer releases).  2-D blocks keep
        // the CTA barrier, which their block amax needs anyway.
        const bool landed = wait_phase(bars + 8u * s, phase, wait_limit);
        if (TWO_D) {
            if (!__syncthreads_and(landed)) {
                if (tid == 0) atomicExch(&g_quant_error, 1);
                break;
            }
        } else if (!__all_sync(0xFFFFFFFFu, landed)) {
            if (lane == 0) atomicExch(&g_quant_error, 1);
            break;
        }
        const int64_t lr0 = (int64_t)(row_tile - gt0) * TR;
        const int64_t c0 = (int64_t)col_tile * TC;
        uint16_t* tile_s = reinterpret_cast<uint16_t*>(base + s * tile_bytes);
        if (p.do_col && lr0 + TR > cnt) {
            // rows past the group's end belong to the next group (or the
            // padding): the column pass must see zeros there
            const int first = cnt - lr0 > 0 ? (int)(cnt - lr0) : 0;
            uint4* t4 = reinterpret_cast<uint4*>(tile_s + first * TC);
            for (int q = tid; q < (TR - first) * TC / 8; q += kThreads) t4[q] = make_uint4(0, 0, 0, 0);
            __syncthreads();
        }

        if (!TWO_D) {
            // ------------------------------------------ 1-D blocks, both passes
            // the row pairs and the column tasks of this tile go through one
            // emit site, so that the scale, rounding and packing code (long
            // with SR) has one inlined copy
            const int64_t col = c0 + cchunk * kChunk;
            const bool col_ok = col < p.cols;
            // rows of this tile that exist, counted from this thread's first row
            const int64_t left = cnt - lr0 - r0;
            const uint16_t* src = tile_s + r0 * TC + cchunk * kChunk;
            const int64_t out_ld = out_ld1, sc_ld = sc_ld1;
            uint8_t* gcodes = gcodes1;
            uint8_t* gscales = gscales1;
            const bool wsc = (col & ((1 << lbw) - 1)) == 0;
            // output pointers of this thread's first row, stepped per pair
            const int64_t orow0 = grow0 + lr0 + r0;  // row-wise output rows follow the input rows
            uint8_t* cp = (uint8_t*)p.row.codes + orow0 * p.row.codes_ld + (col >> 1);
            uint8_t* sp = (uint8_t*)p.row.scales + (orow0 * p.row.scales_ld + (col >> lbw)) * SZ;
            const int64_t cstep = (int64_t)kRPI * p.row.codes_ld;
            const int64_t sstep = (int64_t)kRPI * p.row.scales_ld * SZ;
            uint64_t lin = (uint64_t)(lr0 + r0) * (uint64_t)p.cols + (uint64_t)col;
            const uint64_t lstep = (uint64_t)kRPI * (uint64_t)p.cols;
            const int bwc = 1 << lbwc;
            const int nrow = p.do_row ? pairs : 0;
            const int items = nrow + (p.do_col ? col_tasks : 0);
#pragma unroll(SR ? 1 : 2)
            for (int w = 0; w < items; ++w) {
                const bool is_row = w < nrow;
                // output positions first: the SR draws depend on them only
                Dest A, B;
                uint32_t stream;
                int ra = 0, tcol = 0, rchunk = 0;
                if (is_row) {
                    const int it = w;
                    ra = 2 * kRPI * it;
                    A.codes = cp + (2 * it) * cstep;
                    B.codes = A.codes + cstep;
                    A.s0 = A.s1 = sp + (2 * it) * sstep;
                    B.s0 = B.s1 = A.s0 + sstep;
                    A.valid = ra < left && col_ok;
                    B.valid = ra + kRPI < left && col_ok;
                    A.w0 = B.w0 = wsc;
                    A.lin0 = lin + (uint64_t)(2 * it) * lstep;
                    B.lin0 = A.lin0 + lstep;
                    stream = 0u;
                } else {
                    const int t = warp + kWarps * (w - nrow);
                    tcol = 2 * (((t & ncb_mask) << (5 - lS)) + (lane >> lS));
                    rchunk = ((t >> lncb) << lS) + (lane & (S - 1));
                    const int64_t lrow = lr0 + rchunk * kChunk;
                    const int64_t ca = c0 + tcol, cb = ca + 1;
                    A.codes = gcodes + ca * out_ld + (lrow >> 1);
                    B.codes = A.codes + out_ld;
                    A.s0 = A.s1 = gscales + (ca * sc_ld + (lrow >> lbwc)) * SZ;
                    B.s0 = B.s1 = A.s0 + sc_ld * SZ;
                    A.valid = lrow < padded && ca < p.cols;
                    B.valid = lrow < padded && cb < p.cols;
                    A.w0 = B.w0 = (lrow & (bwc - 1)) == 0;
                    A.lin0 = (uint64_t)ca * (uint64_t)padded + (uint64_t)lrow;
                    B.lin0 = A.lin0 + (uint64_t)padded;
                    stream = 1u;
                }
                A.w1 = B.w1 = false;
                SrDraws dr;
                if (SR) draw_pair(dr, p.sr_keys, A, B, stream, grp_id);
                uint64_t e[16];
                float Ma, Mb;
                if (is_row) {
                    uint32_t wa[8], wb[8];
                    const uint4* pa = reinterpret_cast<const uint4*>(src + ra * TC);
                    const uint4* pb = reinterpret_cast<const uint4*>(src + (ra + kRPI) * TC);
                    const uint4 a0 = pa[0], a1 = pa[1], b0 = pb[0], b1 = pb[1];
                    wa[0] = a0.x; wa[1] = a0.y; wa[2] = a0.z; wa[3] = a0.w;
                    wa[4] = a1.x; wa[5] = a1.y; wa[6] = a1.z; wa[7] = a1.w;
                    wb[0] = b0.x; wb[1] = b0.y; wb[2] = b0.z; wb[3] = b0.w;
                    wb[4] = b1.x; wb[5] = b1.y; wb[6] = b1.z; wb[7] = b1.w;
                    if (N16) widen_rows_c(wa, wb, p.smask16, e);
                    else widen_rows(wa, wb, mrow, e);
                    if (N16) fwht_pair16(e);
                    else fwht_pair(e, n, seg_row);
                    amax_1d_pair(e, 1 << lbw, Ma, Mb);
                } else {
                    uint32_t gw[16];
                    gather_pair<TC>(tile_s, tcol, rchunk, gw);
                    if (N16) widen_cols_c(gw, p.smask16, e);
                    else widen_cols(gw, mc, e);
                    if (N16) fwht_pair16(e);
                    else fwht_pair(e, n, rchunk & (S - 1));
                    amax_1d_pair(e, bwc, Ma, Mb);
                }
                emit_pair<GRID, SR, PO2 ? 1 : 0>(e, Ma, Ma, Mb, Mb, false, fd, A, B, dr);
            }
        } else {
            // ------------------------------------------------ 2-D blocks
            if (p.do_row) {
                const int64_t col = c0 + cchunk * kChunk;
                const bool col_ok = col < p.cols;
                {
                    const int lnbc = 7 + (TC == 256) - lb;  // log2(TC / b)
                    const int bmask = (1 << lb) - 1;
                    // two slot sets per pass, used by alternate tiles: the set of
                    // this tile was cleared during the previous one
                    uint32_t* slots = amax2d + (i & 1) * nslot;
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
                        if (N16) widen_rows_c(wa, wb, p.smask16, e);
                        else widen_rows(wa, wb, mrow, e);
                        if (N16) fwht_pair16(e);
                        else fwht_pair(e, n, seg_row);
                        if (pairs == 1)
#pragma unroll
                            for (int i = 0; i < 16; ++i) keep[i] = e[i];
                        const int sa = (ra >> lb) << lnbc, sb = (rb >> lb) << lnbc;
                        if (lb == 3) {
                            float a0, b0, a1, b1;
                            amax_pair(e, 0, 8, a0, b0);
                            amax_pair(e, 8, 16, a1, b1);
                            post_amax(&slots[sa + 2 * cchunk], a0);
                            post_amax(&slots[sa + 2 * cchunk + 1], a1);
                            post_amax(&slots[sb + 2 * cchunk], b0);
                            post_amax(&slots[sb + 2 * cchunk + 1], b1);
                        } else {
                            float a0, b0;
                            amax_pair(e, 0, 16, a0, b0);
                            post_amax(&slots[sa + ((cchunk * kChunk) >> lb)], a0);
                            post_amax(&slots[sb + ((cchunk * kChunk) >> lb)], b0);
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
                            if (N16) widen_rows_c(wa, wb, p.smask16, e);
                            else widen_rows(wa, wb, mrow, e);
                            if (N16) fwht_pair16(e);
                            else fwht_pair(e, n, seg_row);
                        }
                        const int off = lb == 3 ? 2 * cchunk : ((cchunk * kChunk) >> lb);
                        const int sa = ((ra >> lb) << lnbc) + off, sb = ((rb >> lb) << lnbc) + off;
                        const float MA0 = __uint_as_float(slots[sa]);
                        const float MA1 = __uint_as_float(slots[lb == 3 ? sa + 1 : sa]);
                        const float MB0 = __uint_as_float(slots[sb]);
                        const float MB1 = __uint_as_float(slots[lb == 3 ? sb + 1 : sb]);
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
                        SrDraws dr;
                        if (SR) draw_pair(dr, p.sr_keys, A, B, 0u, grp_id);
                        emit_pair<GRID, SR, PO2 ? 1 : 0>(e, MA0, MA1, MB0, MB1, lb == 3, fd, A, B, dr);
                    }
                    // the other set serves the next tile: every read of it (the
                    // previous tile's) happened before this tile's first barrier
                    uint32_t* other = amax2d + ((i & 1) ^ 1) * nslot;
                    for (int q = tid; q < nslot; q += kThreads) other[q] = 0u;
                }
            }
            if (p.do_col) {
                const int64_t out_ld = p.col_grouped ? padded / 2 : p.col.codes_ld;
                const int lsd = TWO_D ? lb : lbwc;
                const int64_t sc_ld = p.col_grouped ? (padded >> lsd) : p.col.scales_ld;
                uint8_t* gcodes = (uint8_t*)p.col.codes + (p.col_grouped ? p.cols * (p.grp_pad0[g] / 2) : 0);
                uint8_t* gscales = (uint8_t*)p.col.scales + (p.col_grouped ? p.cols * (p.grp_pad0[g] >> lsd) * SZ : 0);
                {
                    const int lnbq = (TR == 128 ? 7 : 6) - lb;  // log2(TR / b)
                    const int bmask = (1 << lb) - 1;
                    uint32_t* slots = amax2d + (2 + (i & 1)) * nslot;  // the column pass's two sets
                    uint64_t keep[16];
                    for (int k = 0; k < col_tasks; ++k) {
                        const int t = warp + kWarps * k;
                        const int tcol = 2 * (((t & ncb_mask) << (5 - lS)) + (lane >> lS));
                        const int rchunk = ((t >> lncb) << lS) + (lane & (S - 1));
                        uint32_t gw[16];
                        uint64_t e[16];
                        gather_pair<TC>(tile_s, tcol, rchunk, gw);
                        if (N16) widen_cols_c(gw, p.smask16, e);
                        else widen_cols(gw, mc, e);
                        if (N16) fwht_pair16(e);
                        else fwht_pair(e, n, rchunk & (S - 1));
                        if (col_tasks == 1)
#pragma unroll
                            for (int i = 0; i < 16; ++i) keep[i] = e[i];
                        const int sa = (tcol >> lb) << lnbq, sb = ((tcol + 1) >> lb) << lnbq;
                        if (lb == 3) {
                            float a0, b0, a1, b1;
                            amax_pair(e, 0, 8, a0, b0);
                            amax_pair(e, 8, 16, a1, b1);
                            post_amax(&slots[sa + 2 * rchunk], a0);
                            post_amax(&slots[sa + 2 * rchunk + 1], a1);
                            post_amax(&slots[sb + 2 * rchunk], b0);
                            post_amax(&slots[sb + 2 * rchunk + 1], b1);
                        } else {
                            float a0, b0;
                            amax_pair(e, 0, 16, a0, b0);
                            post_amax(&slots[sa + ((rchunk * kChunk) >> lb)], a0);
                            post_amax(&slots[sb + ((rchunk * kChunk) >> lb)], b0);
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
                            if (N16) widen_cols_c(gw, p.smask16, e);
                            else widen_cols(gw, mc, e);
                            if (N16) fwht_pair16(e);
                            else fwht_pair(e, n, rchunk & (S - 1));
                        }
                        const int off = lb == 3 ? 2 * rchunk : ((rchunk * kChunk) >> lb);
                        const int sa = ((tcol >> lb) << lnbq) + off, sb = (((tcol + 1) >> lb) << lnbq) + off;
                        const float MA0 = __uint_as_float(slots[sa]);
                        const float MA1 = __uint_as_float(slots[lb == 3 ? sa + 1 : sa]);
                        const float MB0 = __uint_as_float(slots[sb]);
                        const float MB1 = __uint_as_float(slots[lb == 3 ? sb + 1 : sb]);
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
                        SrDraws dr;
                        if (SR) draw_pair(dr, p.sr_keys, A, B, 1u, grp_id);
                        emit_pair<GRID, SR, PO2 ? 1 : 0>(e, MA0, MA1, MB0, MB1, lb == 3, fd, A, B, dr);
                    }
                    uint32_t* other = amax2d + (2 + ((i & 1) ^ 1)) * nslot;
                    for (int q = tid; q < nslot; q += kThreads) other[q] = 0u;
                }
            }
        }
        // the fence orders this CTA's generic shared-memory accesses (reads,
        // and the zero rows of a group's end) before the async-proxy refill
        const int next = tile + kStages * gridDim.x;
        if (TWO_D) {
            // everyone is done with stage s: refill it
            __syncthreads();
            if (tid == 0 && next < num_tiles) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(next, s);
                issued = i + kStages + 1;
            }
        } else {
            // this warp is done with stage s; thread 0 refills it once all are
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empties + 8u * s) : "memory");
            bool refill_failed = false;
            if (tid == 0 && next < num_tiles) {
                if (wait_phase(empties + 8u * s, phase, kWaitLimit)) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(next, s);
                    issued = i + kStages + 1;
                } else {
                    atomicExch(&g_quant_error, 1);
                    refill_failed = true;
                }
            }
            if (__shfl_sync(0xFFFFFFFFu, (int)refill_failed, 0)) {  // warp 0 stops with its producer
                ++i;
                break;
            }
        }
        if (++s == kStages) {
            s = 0;
            phase ^= 1u;
        }
    }
    // copies this CTA issued and thread 0 has not seen land (a broken-off
    // loop): let them land before the CTA exits (bounded)
    if (tid == 0)
        for (int k = i; k < issued; ++k)
            wait_phase(bars + 8u * (k % kStages), (uint32_t)((k / kStages) & 1), kWaitLimit);
}

// ------------------------------------------------------------- launchers
template <int GRID, bool SR, bool PO2, int TC, bool N16>
static cudaError_t launch_q(const CUtensorMap& map, const QuantParams& p, int num_tiles, int num_sms,
                            cudaStream_t st) {
    // ring: about 96 KB of tiles per CTA with 2-D blocks (2 CTAs per SM), 64 KB with 1-D ones (3)
    const int ctas = general_ctas(p.is2d);
    QuantParams q = p;
    q.stages = std::max(2, std::min(kMaxStages, (p.is2d ? 96 : 64) * 1024 / (p.tile_rows * TC * 2)));
    const size_t smem = (size_t)q.stages * q.tile_rows * TC * 2 + 16 * (size_t)q.amax_slots + 16 * q.stages + 128;
    auto k = quantize_kernel<GRID, SR, PO2, TC, N16, false>;
    if constexpr (PO2) {
        if (p.is2d) k = quantize_kernel<GRID, SR, PO2, TC, N16, true>;
    }
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = num_tiles < ctas * num_sms ? num_tiles : ctas * num_sms;
    return launch_pdl(k, dim3(grid), dim3(kThreads), smem, st, map, q, num_tiles);
}

// Tile shapes: 128 columns with the n = 16 butterflies fixed at compile
// time, 128 columns for any other n <= 128, 256 columns for n = 256.
template <int GRID, bool SR, bool PO2>
static cudaError_t launch_q_shape(const CUtensorMap& map, const QuantParams& p, int tc, int num_tiles,
                                  int num_sms, cudaStream_t st) {
    if (tc == 256) return launch_q<GRID, SR, PO2, 256, false>(map, p, num_tiles, num_sms, st);
    if (p.n == 16) return launch_q<GRID, SR, PO2, 128, true>(map, p, num_tiles, num_sms, st);
    return launch_q<GRID, SR, PO2, 128, false>(map, p, num_tiles, num_sms, st);
}

template <bool SR>
static cudaError_t launch_general(const CUtensorMap& map, const QuantParams& p, int grid, bool po2, int tc,
                                  int num_tiles, int num_sms, cudaStream_t st) {
#define UFP4_Q(G)                                                                                              \
    if (grid == G)                                                                                             \
        return po2 ? launch_q_shape<G, SR, true>(map, p, tc, num_tiles, num_sms, st)                          \
                   : launch_q_shape<G, SR, false>(map, p, tc, num_tiles, num_sms, st);
    UFP4_Q(0)
    UFP4_Q(1)
    UFP4_Q(2)
    UFP4_Q(3)
#undef UFP4_Q
    return cudaErrorInvalidValue;
}

// Reads and clears this unit's error word.
static cudaError_t general_error_read_clear(int* value) {
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

static cudaError_t general_set_wait_limit(uint32_t polls) {
    return cudaMemcpyToSymbol(g_quant_wait_limit, &polls, sizeof(polls));
}

// Loads every kernel this unit instantiates (cudaFuncGetAttributes loads a
// function that has not been loaded yet).
template <int G, bool SR, bool PO2>
static void preload_q(cudaFuncAttributes* a) {
    cudaFuncGetAttributes(a, quantize_kernel<G, SR, PO2, 128, true, false>);
    cudaFuncGetAttributes(a, quantize_kernel<G, SR, PO2, 128, false, false>);
    cudaFuncGetAttributes(a, quantize_kernel<G, SR, PO2, 256, false, false>);
    if constexpr (PO2) {
        cudaFuncGetAttributes(a, quantize_kernel<G, SR, PO2, 128, true, true>);
        cudaFuncGetAttributes(a, quantize_kernel<G, SR, PO2, 128, false, true>);
        cudaFuncGetAttributes(a, quantize_kernel<G, SR, PO2, 256, false, true>);
    }
}
template <bool SR>
static cudaError_t preload_general() {
    cudaFuncAttributes a;
    preload_q<0, SR, false>(&a);
    preload_q<0, SR, true>(&a);
    preload_q<1, SR, false>(&a);
    preload_q<1, SR, true>(&a);
    preload_q<2, SR, false>(&a);
    preload_q<2, SR, true>(&a);
    preload_q<3, SR, false>(&a);
    preload_q<3, SR, true>(&a);
    return cudaGetLastError();
}

}  // namespace ufp4
