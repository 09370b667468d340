// Row-wise fused RHT + block-scaled 4-bit quantizer for sm_103a: the FPROP
// operands' case (RHT and 1-D blocks along the rows), over up to four
// tensors in one launch.
//
// Pages: UFP4 summary (hyper.ai, arXiv 2606.20381), sections 数据集 (codebooks,
// blocks, s_B = amax / largest level, RTNE, SR) and 方法 (Sylvester H_2n,
// H'_n = S_n H_n, the quantized GEMM's operands quantized along K);
// "Stable FP4 Training via Transposition-Invariant Block Quantization",
// truncation-free scale.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "quantize_common.cuh"
#include "ufp4_device.cuh"
#include "widen_e5m2.cuh"

namespace ufp4 {

__device__ int g_rows_error;

// Polls of a tile's barrier before a row-kernel CTA gives up (see
// set_quant_wait_limit; the drain of copies in flight always uses kWaitLimit).
__device__ uint32_t g_rows_wait_limit = kWaitLimit;

// ------------------------------------------------------ row-wise (lean)
// Row-wise quantization (1-D blocks, or row-wise b x b blocks), over up to
// kMaxBatch independent tensors in one launch (their tiles are numbered one
// after the other).  The same steps as the general kernel's row pass, with the
// tile shape fixed at compile time, tile coordinates and output pointers
// advanced without division, and per-row bounds checks only on ragged tiles.
struct RowsMaps {
    CUtensorMap m[kMaxBatch];
};

// N16: n = 16 (the FPROP operands' case), with the four butterfly strides
// fixed at compile time.
// TC: tile columns, 128 (n = 256 and n = 64 take the segment kernel below;
// the template also takes 256 for segments of 16 chunks).
//
// With 1-D blocks no CTA barrier separates the tiles: each warp waits on the
// stage's TMA barrier itself and arrives on the stage's "empty" barrier when
// it is done with it; thread 0 waits on that one before it refills the stage.
//
// TWO_D: b x b blocks (b = 16, 32 or 64, UE8M0 scales).  The tile then has 2 kRPI rows, so each thread holds one
// row pair; the block amax is reduced across the lanes of a warp that share
// the block, then across warps with a shared-memory atomicMax, while the
// transformed values wait in registers.  The amax slots come in two sets
// used by alternate tiles, so a set is cleared during the tile before its use.
//
// PREP (E1M2 / INT4, UE8M0, 1-D blocks, n = 16): each tensor is also written
// in the prepared form ufp4_gemm_prepared reads (widen_e5m2.cuh): every chunk
// of 16 codes as 16 E5M2 bytes, shifted by its block's distance d to the
// hardware scale of its 32-element group (the other block of the group is in
// lane ^ 1), and the hardware scales as cells of the replicated chunk array.
// A tile's 128 columns are one chunk along K, so lane 0 of each row gathers
// its four cells (lanes 0, 2, 4, 6) into one word per copy.  The launch runs
// over the tensor's rows rounded up to whole GEMM tiles (rows_cover): the
// rows past the tensor read zeros and get zero cells.
template <int GRID, bool SR, int SF, bool N16, int CTAS, int TC, bool TWO_D, bool PREP = false>
__global__ void __launch_bounds__(kThreads, CTAS)
quantize_rows_kernel(const __grid_constant__ RowsMaps maps, const RowsParams p) {
    static_assert(!PREP || (GRID <= 1 && SF == 1 && N16 && TC == 128 && !TWO_D), "prepared FP8 operands");
    constexpr int kCPR = TC / kChunk;      // 16-element chunks per tile row
    constexpr int kRPI = kThreads / kCPR;  // tile rows per thread step
    constexpr int TR = TWO_D ? 2 * kRPI : 16384 / TC;
    constexpr int kTileBytes = TR * TC * 2;
    constexpr int SZ = SF == 0 ? 4 : 1;
    constexpr int kSlots = TWO_D ? (TR / 16) * (TC / 16) : 0;  // amax slots per set (b = 16 at most)
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 127u) & ~127u) - raw;
    uint8_t* base = smem_raw + pad;
    const int kStages = p.stages;
    uint32_t* amax2d = reinterpret_cast<uint32_t*>(base + kStages * kTileBytes);  // 2 sets of kSlots
    const uint32_t bars = smem_addr(base + kStages * kTileBytes + 8 * kSlots);
    const uint32_t empties = bars + 8u * kStages;  // 1-D blocks: every warp done with the stage
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
    SignMasks mrow;  // n = 16 reads its masks from the kernel parameters (p.smask)
    if (!N16) {
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
        for (int s = 0; s < kStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8u * s));
            if (!TWO_D) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empties + 8u * s), "r"(kWarps));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (TWO_D)
        for (int q = tid; q < 2 * kSlots; q += kThreads) amax2d[q] = 0u;
    const int lb = p.lb2d;  // log2 b (2-D blocks)
    __syncthreads();
    griddep_wait();
    griddep_launch();
    const uint32_t wait_limit = g_rows_wait_limit;
    const int lane = tid & 31;
    int issued = 0;  // tiles of this CTA issued so far (thread 0)
    if (tid == 0)
        for (int s = 0; s < kStages; ++s) {
            const int tile = blockIdx.x + s * gridDim.x;
            if (tile < p.num_tiles) {
                issue(tile, s);
                issued = s + 1;
            }
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
        if (TWO_D) {
            if (!__syncthreads_and(landed)) {
                if (tid == 0) atomicExch(&g_rows_error, 1);
                break;
            }
        } else if (!__all_sync(0xFFFFFFFFu, landed)) {
            // 1-D blocks: no CTA barrier per tile; a warp whose wait gave up
            // leaves the loop (the others then give up on the stages it no
            // longer releases)
            if (lane == 0) atomicExch(&g_rows_error, 1);
            break;
        }
        const RowsTensor& T = p.t[t];
        const uint16_t* tile_s = reinterpret_cast<const uint16_t*>(base + s * kTileBytes);
        const int row0 = rt * TR;
        const int col = ct * TC + cchunk * kChunk;
        // PREP: the GEMM tile holding the quantizer tile's first row, and its first row
        const int ptile = PREP ? row0 / T.prep.tile_rows : 0, prow0 = PREP ? ptile * T.prep.tile_rows : 0;
        const bool col_ok = col < T.cols;
        const int left = T.rows - row0 - r0;  // rows of this thread's first row onward
        const bool full = T.rows - row0 >= TR;
        uint8_t* cp = T.codes + (int64_t)(row0 + r0) * T.codes_ld + (GRID == 4 ? col : col >> 1);
        uint8_t* sp = T.scales + ((int64_t)(row0 + r0) * T.scales_ld + (col >> lbw)) * SZ;
        const int64_t cstep = (int64_t)kRPI * T.codes_ld;
        const int64_t sstep = (int64_t)kRPI * T.scales_ld * SZ;
        const bool wsc = (col & ((1 << lbw) - 1)) == 0;
        const uint16_t* src = tile_s + r0 * TC + cchunk * kChunk;
        // one copy of the step for SR (its Philox rounds make the step long;
        // two copies crowd the instruction cache), two otherwise
#pragma unroll(SR ? 1 : 2)
        for (int it = 0; it < TR / (2 * kRPI); ++it) {
            const int ra = 2 * kRPI * it;
            Dest A, B;
            A.codes = cp + (2 * it) * cstep;
            B.codes = A.codes + cstep;
            if (TWO_D) {
                // one UE8M0 byte per b x b block, written by its top-left thread
                const int rA = row0 + r0, rB = rA + kRPI;
                A.s0 = A.s1 = T.scales + (int64_t)(rA >> lb) * T.scales_ld + (col >> lb);
                B.s0 = B.s1 = T.scales + (int64_t)(rB >> lb) * T.scales_ld + (col >> lb);
                const bool cfirst = (col & ((1 << lb) - 1)) == 0;
                A.w0 = cfirst && (rA & ((1 << lb) - 1)) == 0;
                B.w0 = cfirst && (rB & ((1 << lb) - 1)) == 0;
            } else {
                A.s0 = A.s1 = sp + (2 * it) * sstep;
                B.s0 = B.s1 = A.s0 + sstep;
                A.w0 = B.w0 = wsc;
            }
            A.valid = col_ok && (full || ra < left);
            B.valid = col_ok && (full || ra + kRPI < left);
            A.w1 = B.w1 = false;
            A.lin0 = (uint64_t)(row0 + r0 + ra) * (uint64_t)T.cols + (uint64_t)col;
            B.lin0 = A.lin0 + (uint64_t)kRPI * (uint64_t)T.cols;
            SrDraws dr;
            if (SR) draw_pair(dr, p.sr_keys, A, B, 0u, (uint32_t)p.group);
            uint32_t wa[8], wb[8];
            uint64_t e[16];
            const uint4* pa = reinterpret_cast<const uint4*>(src + ra * TC);
            const uint4* pb = reinterpret_cast<const uint4*>(src + (ra + kRPI) * TC);
            const uint4 a0 = pa[0], a1 = pa[1], b0 = pb[0], b1 = pb[1];
            wa[0] = a0.x; wa[1] = a0.y; wa[2] = a0.z; wa[3] = a0.w;
            wa[4] = a1.x; wa[5] = a1.y; wa[6] = a1.z; wa[7] = a1.w;
            wb[0] = b0.x; wb[1] = b0.y; wb[2] = b0.z; wb[3] = b0.w;
            wb[4] = b1.x; wb[5] = b1.y; wb[6] = b1.z; wb[7] = b1.w;
            if (N16) widen_rows_c(wa, wb, p.smask, e);
            else widen_rows(wa, wb, mrow, e);
            float Ma, Mb;
            if (TWO_D) {
                if (N16) fwht_pair16(e);
                else fwht_pair(e, n, seg_row);
                amax_pair(e, 0, 16, Ma, Mb);
                // the lanes of this warp in the same block: the b/16 neighbouring
                // chunks (lane bits below log2 kCPR) and the warp's 32/kCPR rows
                // (the lane bits above); when b > kRPI the thread's two rows
                // share the block as well
                for (int k = 1; k < (1 << lb) / kChunk; k <<= 1) {
                    Ma = fmaxf(Ma, __shfl_xor_sync(0xFFFFFFFFu, Ma, k));
                    Mb = fmaxf(Mb, __shfl_xor_sync(0xFFFFFFFFu, Mb, k));
                }
                const bool shared_rows = (1 << lb) > kRPI;
                if (shared_rows) Ma = Mb = fmaxf(Ma, Mb);
#pragma unroll
                for (int k = kCPR; k < 32; k <<= 1) {
                    Ma = fmaxf(Ma, __shfl_xor_sync(0xFFFFFFFFu, Ma, k));
                    Mb = fmaxf(Mb, __shfl_xor_sync(0xFFFFFFFFu, Mb, k));
                }
                uint32_t* set = amax2d + (i & 1) * kSlots;
                const int lnbc = (TC == 256 ? 8 : 7) - lb;  // log2(TC / b): block columns per tile
                const int bc = (cchunk * kChunk) >> lb;
                const int sa = ((r0 >> lb) << lnbc) + bc, sb = (((r0 + kRPI) >> lb) << lnbc) + bc;
                if ((r0 & (32 / kCPR - 1)) == 0 && ((cchunk * kChunk) & ((1 << lb) - 1)) == 0) {
                    atomicMax(&set[sa], __float_as_uint(Ma));
                    if (!shared_rows) atomicMax(&set[sb], __float_as_uint(Mb));
                }
                __syncthreads();
                Ma = __uint_as_float(set[sa]);
                Mb = __uint_as_float(set[sb]);
                // the other set serves the next tile: every read of it (the
                // previous tile's) happened before this tile's first barrier
                uint32_t* other = amax2d + ((i & 1) ^ 1) * kSlots;
                for (int q = tid; q < kSlots; q += kThreads) other[q] = 0u;
            } else if (N16) {
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
            EmitOut eo;
            emit_pair<GRID, SR, SF>(e, Ma, Ma, Mb, Mb, false, fd, A, B, dr, 0u, 0u, false, PREP ? &eo : nullptr);
            if constexpr (PREP) {
                const PrepTarget& P = T.prep;
                constexpr int kStep = GRID == 0 ? -2 : 0;  // log2 of the level step in scale units: E1M2 k/4, INT4 k
                const int pa = __shfl_xor_sync(0xFFFFFFFFu, eo.sa, 1), pb = __shfl_xor_sync(0xFFFFFFFFu, eo.sb, 1);
                const int hwa = max(max(eo.sa, pa) + kStep, 0), hwb = max(max(eo.sb, pb) + kStep, 0);
                const int rA = row0 + r0 + ra, rB = rA + kRPI;
                uint32_t wa0 = eo.ca.x, wa1 = eo.ca.y, wb0 = eo.cb.x, wb1 = eo.cb.y;
                if (GRID == 1) {
                    wa0 = twos_to_signmag8(wa0);
                    wa1 = twos_to_signmag8(wa1);
                    wb0 = twos_to_signmag8(wb0);
                    wb1 = twos_to_signmag8(wb1);
                }
                if (A.valid)
                    *reinterpret_cast<uint4*>(P.fp8 + (int64_t)rA * P.K + col) =
                        widen16_e5m2(wa0, wa1, hwa - kStep - eo.sa);
                if (B.valid)
                    *reinterpret_cast<uint4*>(P.fp8 + (int64_t)rB * P.K + col) =
                        widen16_e5m2(wb0, wb1, hwb - kStep - eo.sb);
                // cells of the groups (col / 32): lanes with an even chunk index
                // hold them; every lane of the row's eight gets both rows' words
                const uint32_t ca = A.valid ? (uint32_t)hwa : 0u, cb = B.valid ? (uint32_t)hwb : 0u;
                uint32_t wa = 0u, wb = 0u;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    wa |= __shfl_sync(0xFFFFFFFFu, ca, (lane & ~7) + 2 * k) << (8 * k);
                    wb |= __shfl_sync(0xFFFFFFFFu, cb, (lane & ~7) + 2 * k) << (8 * k);
                }
                // lane c of the eight stores copy c % 4 of row A (c < 4) or B; when
                // the row's part is a tile's short last part (part_rows < 128),
                // row w also stores the zero cells of the part's row w + part_rows
                // if that row lies past the part's end
                const int r = cchunk < 4 ? rA : rB;
                if (r < P.rows_cover) {
                    // the GEMM tile of r from that of the quantizer tile's first row
                    // (tiles are at least 128 rows, so r is in it or the next)
                    int tt = ptile, rr = r - prow0;
                    if (rr >= P.tile_rows) {
                        ++tt;
                        rr -= P.tile_rows;
                    }
                    const int h = rr >> 7, w = rr & 127;
                    const int part_rows = min(128, P.tile_rows - 128 * h);
                    const int g0 = (col >> 5) & ~3;  // the first group of the chunk (the tile's 128 columns)
                    uint8_t* c = P.chunks + (cchunk & 3) * 512;
                    *reinterpret_cast<uint32_t*>(c + chunk_cell_offset_twh(tt, h, w, g0, P.parts, P.chunks_k)) =
                        cchunk < 4 ? wa : wb;
                    if (w + part_rows < 128)
                        *reinterpret_cast<uint32_t*>(
                            c + chunk_cell_offset_twh(tt, h, w + part_rows, g0, P.parts, P.chunks_k)) = 0u;
                }
            }
        }
        const int next = tile + kStages * gridDim.x;
        if (TWO_D) {
            // everyone is done with stage s: refill it
            __syncthreads();
            if (tid == 0 && next < p.num_tiles) {
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue(next, s);
                issued = i + kStages + 1;
            }
        } else {
            // this warp is done with stage s; thread 0 refills it once all are
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empties + 8u * s) : "memory");
            bool refill_failed = false;
            if (tid == 0 && next < p.num_tiles) {
                if (wait_phase(empties + 8u * s, phase, kWaitLimit)) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(next, s);
                    issued = i + kStages + 1;
                } else {
                    atomicExch(&g_rows_error, 1);
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

// CTAs per SM and ring depth of the row kernel (128 x 128 tiles): two CTAs
// of up to 128 registers a thread, each with three 32 KB stages (measured on
// the 16384 x 7168 + 7168 x 7168 batch: 6.13 TB/s, against 5.87 TB/s for
// three CTAs of two stages, whose 80-register cap costs 1.6 instructions per
// element in register moves).
constexpr int kRowsCtas = 2, kRowsStages = 3;

// Barrier of the nthreads threads (a multiple of 32) of the warps that use
// named barrier id (1..15); returns the AND of v over them.  Barrier
// semantics order the shared-memory accesses of those threads.
__device__ __forceinline__ bool band_sync_and(uint32_t id, uint32_t nthreads, bool v) {
    uint32_t r;
    asm volatile("{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.and.pred q, %2, %3, p; selp.u32 %0, 1, 0, q; }"
                 : "=r"(r)
                 : "r"((uint32_t)v), "r"(id), "r"(nthreads)
                 : "memory");
    return r != 0;
}

// n = 64 and n = 256, 1-D or b x b blocks: a thread owns one 64-element segment of
// a row.  QN segments make one tile row (QN = 2: 128 columns, n = 64; QN = 4:
// 256 columns, n = 256), so the tile is 128 x 128 or 64 x 256.  It arrives as
// QN 64-column TMA boxes with the 128-byte swizzle (16-byte unit u of row r at
// u ^ (r % 8)).  The eight threads of a quarter-warp take the same segment of
// eight consecutive rows, so their 16-byte loads fall on eight different bank
// groups.  The 64 values are held as pairs (v_i, v_i+32): strides 1 .. 16 are
// paired adds, stride 32 adds the two halves of each pair, and for n = 256
// strides 64 and 128 pair the thread with the lanes holding the neighbouring
// segments (lane ^ 8, lane ^ 16), each lane keeping half of the values.  The
// random signs: n = 64 reads a per-element mask table from the kernel
// parameters (the same for every segment); n = 256 from a table in shared
// memory, one 64-entry set per segment.
// 1-D blocks: no CTA barrier per tile; each warp waits on the stage's TMA
// barrier itself and, when done with the stage, arrives on the stage's
// "empty" barrier; thread 0 waits on that one before it refills the stage.
// TWO_D (b = 16, 32, 64; UE8M0): the block amax is reduced over the rows a
// warp holds (lanes ^ 1, 2, 4, and ^ 16 for two segments a row), then across
// the warps of its b-row band (the b / 16 or b / 8 warps holding those rows)
// with a shared-memory atomicMax and one named barrier of the band per tile;
// a band of one warp (n = 64, b = 16) needs neither.  The ring runs as for
// 1-D blocks.  The amax slots come in three sets used in turn: after tile
// i's barrier the band clears its slots of the set of tile i + 2.  Their
// last reads (tile i - 1) precede tile i's barrier in every warp of the
// band, and their next atomicMax (tile i + 2) follows tile i + 1's barrier,
// which the clearing threads reach only after the clear.
template <int GRID, bool SR, int SF, int CTAS, int QN, bool TWO_D>
__global__ void __launch_bounds__(kThreads, CTAS)
quantize_rows_seg_kernel(const __grid_constant__ RowsMaps maps, const RowsParams p) {
    static_assert(QN == 2 || QN == 4, "two or four segments per tile row");
    constexpr int kSlots = 64;  // amax slots per set: (TR / b) x (TC / b) <= 64 for b >= 16
    constexpr int TC = 64 * QN, TR = 16384 / TC;
    constexpr int kLQ = QN == 2 ? 1 : 2;
    constexpr int kTileBytes = TR * TC * 2;
    constexpr int kBoxBytes = TR * 128;
    constexpr int SZ = SF == 0 ? 4 : 1;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t pad = ((raw + 1023u) & ~1023u) - raw;  // 128-byte swizzle: 1024-byte aligned stages
    uint8_t* base = smem_raw + pad;
    const int kStages = p.stages;
    // full barriers (TMA landed) at bars + 8 s, empty barriers (every warp
    // done with the stage) at bars + 32 + 8 s, s < kStages <= 4
    const uint32_t bars = smem_addr(base + kStages * kTileBytes);
    const uint32_t empties = bars + 32u;
    uint32_t* sgn_tab = reinterpret_cast<uint32_t*>(base + kStages * kTileBytes + 64);  // n = 256: [segment][j], 16-byte aligned
    uint32_t* amax2d = sgn_tab + 256;  // 2-D blocks: three sets of kSlots
    const int tid = threadIdx.x;
    const int seg = (tid >> 3) & (QN - 1);
    const int r = (tid & 7) + 8 * (tid >> (3 + kLQ));
    Fold fd;
    fd.inv_s = p.inv_sqrt_n;
    fd.pow4 = p.pow4;
    fd.j = p.log4n;
    fd.g = 0.0f;
    const int lbw = p.lbw;

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
        const uint32_t dst = smem_addr(base + s * kTileBytes);
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(kTileBytes) : "memory");
#pragma unroll
        for (int h = 0; h < QN; ++h)
            asm volatile(
                "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
                ::"r"(dst + h * kBoxBytes), "l"((uint64_t)&maps.m[t]), "r"(ct * TC + 64 * h), "r"(rt * TR),
                "r"(bar)
                : "memory");
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8u * s));
            asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(empties + 8u * s), "r"(kWarps));
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (QN == 4)  // mask of element j of segment q: 0x80000000 when eps_(64 q + j) = -1
        sgn_tab[tid] = ((p.sign_bits[tid >> 5] >> (tid & 31)) & 1u) << 31;
    if (TWO_D && tid < 3 * kSlots) amax2d[tid] = 0u;
    const int lb = p.lb2d;  // log2 b (2-D blocks)
    __syncthreads();
    griddep_wait();
    griddep_launch();
    const uint32_t wait_limit = g_rows_wait_limit;
    const int lane = tid & 31;
    int issued = 0;  // tiles of this CTA issued so far (thread 0)
    if (tid == 0)
        for (int s = 0; s < kStages; ++s) {
            const int tile = blockIdx.x + s * gridDim.x;
            if (tile < p.num_tiles) {
                issue(tile, s);
                issued = s + 1;
            }
        }

    int t = 0, rt = 0, ct = 0, step_r = 0, step_c = 0;
    auto relocate = [&](int tile) {
        locate(tile, t, rt, ct);
        step_r = (int)gridDim.x / p.t[t].col_tiles;
        step_c = (int)gridDim.x - step_r * p.t[t].col_tiles;
        if (SF == 2) fd.g = __fdiv_rn(*p.t[t].amax, grid_qmax(GRID) * 448.0f);
    };
    if ((int)blockIdx.x < p.num_tiles) relocate(blockIdx.x);
    int s = 0;
    uint32_t phase = 0;
    int i = 0;
    bool refill_failed = false;  // 2-D: thread 0 could not refill a stage (carried to the next barrier)
    for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++i) {
        if (i) {
            ct += step_c;
            rt += step_r;
            if (ct >= p.t[t].col_tiles) {
                ct -= p.t[t].col_tiles;
                ++rt;
            }
            if (rt >= p.t[t].row_tiles) relocate(tile);
        }
        // Each warp waits for the copy itself.  1-D blocks: a warp whose
        // wait gave up leaves the loop (the others then give up on the stages
        // it no longer releases).  2-D blocks: it goes on to the tile's CTA
        // barrier (reading a stage that may not have landed, writing nothing
        // global before it), where every warp learns of it and leaves.
        const bool ok = __all_sync(0xFFFFFFFFu, wait_phase(bars + 8u * s, phase, wait_limit)) &&
                        !(TWO_D && __shfl_sync(0xFFFFFFFFu, (int)refill_failed, 0));
        if (!TWO_D && !ok) {
            if (lane == 0) atomicExch(&g_rows_error, 1);
            break;
        }
        const RowsTensor& T = p.t[t];
        const int row = rt * TR + r;
        const int col = ct * TC + 64 * seg;
        const bool valid = col < T.cols && row < T.rows;
        // the segment: eight 16-byte units of row r in box seg
        const uint8_t* box = base + s * kTileBytes + seg * kBoxBytes + r * 128;
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 u = *reinterpret_cast<const uint4*>(box + ((k ^ (r & 7)) << 4));
            w[4 * k] = u.x; w[4 * k + 1] = u.y; w[4 * k + 2] = u.z; w[4 * k + 3] = u.w;
        }
        // pairs (v_i, v_i+32) with the signs folded into the widening
        uint64_t e[32];
        uint32_t msk[QN == 4 ? 64 : 1];
        if (QN == 4) {
            const uint4* sm4 = reinterpret_cast<const uint4*>(sgn_tab + 64 * seg);
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint4 v = sm4[k];
                msk[4 * k] = v.x; msk[4 * k + 1] = v.y; msk[4 * k + 2] = v.z; msk[4 * k + 3] = v.w;
            }
        }
#pragma unroll
        for (int q = 0; q < 32; ++q) {
            const uint32_t wl = w[q >> 1], wh = w[(q + 32) >> 1];
            // n = 64: the parameter array indexed directly (constant-bank operands)
            const uint32_t ml = QN == 4 ? msk[q] : p.smask[q];
            const uint32_t mh = QN == 4 ? msk[q + 32] : p.smask[q + 32];
            const float lo = (q & 1) ? __uint_as_float((wl & 0xFFFF0000u) ^ ml) : __uint_as_float(wl * 65536u + ml);
            const float hi = (q & 1) ? __uint_as_float((wh & 0xFFFF0000u) ^ mh) : __uint_as_float(wh * 65536u + mh);
            e[q] = pk2(lo, hi);
        }
#pragma unroll
        for (int h = 1; h < 32; h <<= 1) {
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                if (q & h) continue;
                const uint64_t a = e[q], b = e[q + h];
                e[q] = add2(a, b);
                e[q + h] = sub2(a, b);
            }
        }
        if constexpr (QN == 4) {
            // Strides 32, 64 and 128 with half exchanges.  Lane (b1, b0) of a
            // row's four (segment S = 2 b1 + b0) keeps half of what it holds at
            // each step and sends the other half, one shuffle per kept value:
            //  * stride 32 (in the pair): keep position q + 32 b0 of S, send
            //    q + 32 (1 - b0): a + s b and a - s b with s = +1 (b0 = 0) or -1;
            //  * stride 64 (lane ^ 8, segments 2 b1 and 2 b1 + 1, same positions):
            //    keep = mine + t recv, send = mine - t recv, t = +1 (b1 = 0) or -1,
            //    so b1 = 0 keeps the sums and b1 = 1 the differences (negated
            //    where b0 = 1, as is the sent difference of b0 = 1, b1 = 0);
            //  * stride 128 (lane ^ 16): out1 = keep + recv, out2 = keep - recv.
            // Lane (b1, b0) ends with segments b1 (out1) and 2 + b1 (out2) at
            // positions 32 b0 + j (.x) and 32 b0 + 16 + j (.y), j < 16: chunks
            // 2 b0 and 2 b0 + 1 of each.  Every value equals the butterfly's
            // up to its sign (RN(a - b) = -RN(b - a)): out1 is negated on lane
            // (1, 1) and out2 on lane (1, 0), which the reciprocal's sign undoes.
            const int b0 = seg & 1, b1 = seg >> 1;
            const float s0 = b0 ? -1.0f : 1.0f;
            uint64_t K[16], S[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                float a0, c0, a1, c1;
                up2(e[j], a0, c0);
                up2(e[j + 16], a1, c1);
                K[j] = pk2(__fmaf_rn(s0, c0, a0), __fmaf_rn(s0, c1, a1));
                S[j] = pk2(__fmaf_rn(-s0, c0, a0), __fmaf_rn(-s0, c1, a1));
            }
            const float tau = b1 ? -1.0f : 1.0f;
            const uint64_t t2 = pk2(tau, tau), nt2 = pk2(-tau, -tau);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint64_t o = (uint64_t)__shfl_xor_sync(0xFFFFFFFFu, (unsigned long long)S[j], 8);
                S[j] = fma2(nt2, o, K[j]);
                K[j] = fma2(t2, o, K[j]);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint64_t o = (uint64_t)__shfl_xor_sync(0xFFFFFFFFu, (unsigned long long)S[j], 16);
                S[j] = sub2(K[j], o);
                K[j] = add2(K[j], o);
            }
            const uint32_t neg1 = (b1 & b0) ? 0x80000000u : 0u;
            const uint32_t neg2 = (b1 & (b0 ^ 1)) ? 0x80000000u : 0u;
            // chunk amax: (2 b0, 2 b0 + 1) of segment b1 (MA1, MB1) and of 2 + b1 (MA2, MB2)
            float MA1, MB1, MA2, MB2;
            amax_pair(K, 0, 16, MA1, MB1);
            amax_pair(S, 0, 16, MA2, MB2);
            const bool b32 = TWO_D ? lb >= 5 : lbw == 5;
            if (b32) {
                MA1 = MB1 = fmaxf(MA1, MB1);
                MA2 = MB2 = fmaxf(MA2, MB2);
            }
            const int c1 = 64 * b1 + 32 * b0;  // tile column of chunk 2 b0 of segment b1 (+128: of 2 + b1)
            if (TWO_D) {
                if (lb == 6) {  // a 64-wide block: both halves of the segment (lane ^ 8)
                    MA1 = MB1 = fmaxf(MA1, __shfl_xor_sync(0xFFFFFFFFu, MA1, 8));
                    MA2 = MB2 = fmaxf(MA2, __shfl_xor_sync(0xFFFFFFFFu, MA2, 8));
                }
                // the eight rows of this warp (lanes ^ 1, 2, 4): one b-row band for b >= 16
#pragma unroll
                for (int k = 1; k <= 4; k <<= 1) {
                    MA1 = fmaxf(MA1, __shfl_xor_sync(0xFFFFFFFFu, MA1, k));
                    MB1 = fmaxf(MB1, __shfl_xor_sync(0xFFFFFFFFu, MB1, k));
                    MA2 = fmaxf(MA2, __shfl_xor_sync(0xFFFFFFFFu, MA2, k));
                    MB2 = fmaxf(MB2, __shfl_xor_sync(0xFFFFFFFFu, MB2, k));
                }
                // then across the warps of the band (b / 8 warps of eight rows):
                // slot (row block = band, column block)
                uint32_t* set = amax2d + (i % 3) * kSlots;
                const int band = (tid >> 5) >> (lb - 3);
                const int bthreads = 32 << (lb - 3);
                const int rs = band << (8 - lb);
                const int sA1 = rs + (c1 >> lb), sB1 = rs + ((c1 + 16) >> lb);
                const int sA2 = rs + ((c1 + 128) >> lb), sB2 = rs + ((c1 + 144) >> lb);
                if ((lane & 7) == 0 && (lb < 6 || b0 == 0)) {
                    atomicMax(&set[sA1], __float_as_uint(MA1));
                    atomicMax(&set[sA2], __float_as_uint(MA2));
                    if (lb == 4) {
                        atomicMax(&set[sB1], __float_as_uint(MB1));
                        atomicMax(&set[sB2], __float_as_uint(MB2));
                    }
                }
                if (!band_sync_and(1 + band, bthreads, ok)) {
                    if (lane == 0) atomicExch(&g_rows_error, 1);
                    break;
                }
                MA1 = __uint_as_float(set[sA1]);
                MB1 = __uint_as_float(set[sB1]);
                MA2 = __uint_as_float(set[sA2]);
                MB2 = __uint_as_float(set[sB2]);
                // the band's slots of the set of tile i + 2 (last read in tile i - 1)
                const int bl = tid - band * bthreads;
                if (bl < (256 >> lb)) amax2d[((i + 2) % 3) * kSlots + rs + bl] = 0u;
            }
            const bool join = GRID != 4 && (T.codes_ld & 15) == 0;
            const int64_t rowlin = (int64_t)row * T.cols;
            uint8_t* const crow = T.codes + (int64_t)row * T.codes_ld;
            uint8_t* const sp2 = T.scales + (int64_t)(row >> lb) * T.scales_ld;
            const bool rfirst = (row & ((1 << lb) - 1)) == 0;
            auto dest = [&](int cc, Dest& D) {  // cc: column of the chunk
                D.codes = crow + (GRID == 4 ? cc : cc >> 1);
                if (TWO_D) {
                    D.s0 = sp2 + (cc >> lb);
                    D.w0 = rfirst && (cc & ((1 << lb) - 1)) == 0;
                } else {
                    D.s0 = T.scales + ((int64_t)row * T.scales_ld + (cc >> lbw)) * SZ;
                    D.w0 = !b32 || (cc & 31) == 0;
                }
                D.s1 = D.s0;
                D.w1 = false;
                D.lin0 = (uint64_t)(rowlin + cc);
            };
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int cc = ct * TC + c1 + 128 * h;
                Dest A, B;
                dest(cc, A);
                dest(cc + 16, B);
                A.valid = B.valid = row < T.rows && cc < T.cols;
                SrDraws dr;
                if (SR) draw_pair(dr, p.sr_keys, A, B, 0u, (uint32_t)p.group);
                // a 32-wide block (b32) covers both chunks: B (chunk + 16) writes no scale
                if (h == 0)
                    emit_pair<GRID, SR, SF>(K, MA1, MA1, MB1, MB1, false, fd, A, B, dr, neg1, neg1, join, nullptr, b32);
                else
                    emit_pair<GRID, SR, SF>(S, MA2, MA2, MB2, MB2, false, fd, A, B, dr, neg2, neg2, join, nullptr, b32);
            }
        } else {
    #pragma unroll
            for (int q = 0; q < 32; ++q) {  // stride 32: the two halves of each pair
                float a, b;
                up2(e[q], a, b);
                e[q] = pk2(__fadd_rn(a, b), __fsub_rn(a, b));
            }
            // block amax: (chunk 0, chunk 2) from pairs 0..15, (chunk 1, chunk 3) from pairs 16..31
            float M0, M2, M1, M3;
            amax_pair(e, 0, 16, M0, M2);
            amax_pair(e + 16, 0, 16, M1, M3);
            const bool b32 = TWO_D ? lb >= 5 : lbw == 5;
            if (b32) {
                M0 = M1 = fmaxf(M0, M1);
                M2 = M3 = fmaxf(M2, M3);
            }
            if (TWO_D) {
                if (lb == 6) M0 = M1 = M2 = M3 = fmaxf(M0, M2);
                // the rows of this warp in the same b-row band: lanes ^ 1, 2, 4 (and
                // ^ 16: rows + 8 with two segments a row); b >= 16 covers them all
    #pragma unroll
                for (int k = 1; k <= (QN == 2 ? 16 : 4); k <<= 1) {
                    if (k == 8) continue;
                    M0 = fmaxf(M0, __shfl_xor_sync(0xFFFFFFFFu, M0, k));
                    M1 = fmaxf(M1, __shfl_xor_sync(0xFFFFFFFFu, M1, k));
                    M2 = fmaxf(M2, __shfl_xor_sync(0xFFFFFFFFu, M2, k));
                    M3 = fmaxf(M3, __shfl_xor_sync(0xFFFFFFFFu, M3, k));
                }
                // then across the warps of the band (b / 16 warps of sixteen rows):
                // slot (row block = band, column block); a band of one warp
                // (b = 16) has its block amax already
                static_assert(QN == 2, "n = 64 here");
                if (lb == 4) {
                    if (!ok) {
                        if (lane == 0) atomicExch(&g_rows_error, 1);
                        break;
                    }
                } else {
                    uint32_t* set = amax2d + (i % 3) * kSlots;
                    const int band = (tid >> 5) >> (lb - 4);
                    const int bthreads = 32 << (lb - 4);
                    const int lnbc = 7 - lb;  // log2(TC / b)
                    const int slot0 = (band << lnbc) + ((64 * seg) >> lb);
                    const int cpb = (1 << lb) >> 4;  // chunks per block column
                    if ((lane & 0x17) == 0) {
                        atomicMax(&set[slot0], __float_as_uint(M0));
                        if (cpb <= 2) atomicMax(&set[slot0 + 1], __float_as_uint(M2));
                    }
                    if (!band_sync_and(1 + band, bthreads, ok)) {
                        if (lane == 0) atomicExch(&g_rows_error, 1);
                        break;
                    }
                    M0 = M1 = __uint_as_float(set[slot0]);
                    M2 = M3 = __uint_as_float(set[slot0 + (cpb == 2 ? 1 : 0)]);
                    // the band's slots of the set of tile i + 2 (last read in tile i - 1)
                    const int bl = tid - band * bthreads;
                    if (bl < (128 >> lb)) amax2d[((i + 2) % 3) * kSlots + (band << lnbc) + bl] = 0u;
                }
            }
            uint8_t* cp = T.codes + (int64_t)row * T.codes_ld + (GRID == 4 ? col : col >> 1);
            uint8_t* sp = T.scales + ((int64_t)row * T.scales_ld + (col >> lbw)) * SZ;
            const int cstride = GRID == 4 ? 16 : 8;  // code bytes per 16 elements
            const uint64_t lin0 = (uint64_t)row * (uint64_t)T.cols + (uint64_t)col;
            Dest A, B;
            // 2-D: one UE8M0 byte per b x b block at (row / b, column / b), written
            // by the thread holding its top-left chunk
            uint8_t* sp2 = T.scales + (int64_t)(row >> lb) * T.scales_ld;
            const bool rfirst = (row & ((1 << lb) - 1)) == 0;
            auto chunk_scale = [&](int c, uint8_t*& sptr, bool& w) {
                const int cc = col + 16 * c;
                if (TWO_D) {
                    sptr = sp2 + (cc >> lb);
                    w = rfirst && (cc & ((1 << lb) - 1)) == 0;
                } else {
                    sptr = sp + (cc - col) / (b32 ? 32 : 16) * SZ;
                    w = !b32 || (c & 1) == 0;
                }
            };
            // chunks 0 and 2
            A.codes = cp;
            B.codes = cp + 2 * cstride;
            chunk_scale(0, A.s0, A.w0);
            chunk_scale(2, B.s0, B.w0);
            A.s1 = A.s0;
            B.s1 = B.s0;
            A.valid = B.valid = valid;
            A.w1 = B.w1 = false;
            A.lin0 = lin0;
            B.lin0 = lin0 + 32;
            {
                SrDraws dr;
                if (SR) draw_pair(dr, p.sr_keys, A, B, 0u, (uint32_t)p.group);
                emit_pair<GRID, SR, SF>(e, M0, M0, M2, M2, false, fd, A, B, dr);
            }
            // chunks 1 and 3 (their 1 x 32 scales were written with chunks 0 and 2)
            A.codes = cp + cstride;
            B.codes = cp + 3 * cstride;
            chunk_scale(1, A.s0, A.w0);
            chunk_scale(3, B.s0, B.w0);
            A.s1 = A.s0;
            B.s1 = B.s0;
            A.lin0 = lin0 + 16;
            B.lin0 = lin0 + 48;
            {
                SrDraws dr;
                if (SR) draw_pair(dr, p.sr_keys, A, B, 0u, (uint32_t)p.group);
                emit_pair<GRID, SR, SF>(e + 16, M1, M1, M3, M3, false, fd, A, B, dr);
            }
        }
        const int next = tile + kStages * gridDim.x;
        {
            // this warp is done with stage s; thread 0 refills it once all are
            __syncwarp();
            if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(empties + 8u * s) : "memory");
            if (tid == 0 && next < p.num_tiles && !refill_failed) {
                if (wait_phase(empties + 8u * s, phase, kWaitLimit)) {
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    issue(next, s);
                    issued = i + kStages + 1;
                } else {
                    atomicExch(&g_rows_error, 1);
                    refill_failed = true;
                }
            }
            // 1-D: warp 0 stops with its producer; 2-D: every warp stops at the next barrier
            if (!TWO_D && __shfl_sync(0xFFFFFFFFu, (int)refill_failed, 0)) {
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

template <int GRID, bool SR, int SF>
static cudaError_t launch_rows_seg(const RowsMaps& maps, RowsParams& p, int num_sms, cudaStream_t st) {
    constexpr int kCtas = kRowsCtas;
    p.stages = kRowsStages;
    // ring, barriers, sign table, 2-D amax slots, alignment
    const size_t smem = (size_t)p.stages * 16384 * 2 + 64 + 1024 + 768 + 1024;
    auto k = p.n == 256 ? quantize_rows_seg_kernel<GRID, SR, SF, kCtas, 4, false>
                        : quantize_rows_seg_kernel<GRID, SR, SF, kCtas, 2, false>;
    if constexpr (SF == 1 && GRID < 4) {
        if (p.lb2d)
            k = p.n == 256 ? quantize_rows_seg_kernel<GRID, SR, SF, kCtas, 4, true>
                           : quantize_rows_seg_kernel<GRID, SR, SF, kCtas, 2, true>;
    }
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = p.num_tiles < kCtas * num_sms ? p.num_tiles : kCtas * num_sms;
    return launch_pdl(k, dim3(grid), dim3(kThreads), smem, st, maps, p);
}


template <int GRID, bool SR, int SF, bool N16, int CTAS, int TC, bool TWO_D, bool PREP = false>
static cudaError_t launch_rows_cfg(const RowsMaps& maps, const RowsParams& p, int num_sms, cudaStream_t st) {
    constexpr int kTileElems = TWO_D ? 2 * (kThreads / (TC / kChunk)) * TC : 16384;
    constexpr int kSlots = TWO_D ? (kTileElems / TC / 16) * (TC / 16) : 0;
    const size_t smem = (size_t)p.stages * kTileElems * 2 + 8 * kSlots + 16 * p.stages + 128;
    auto k = quantize_rows_kernel<GRID, SR, SF, N16, CTAS, TC, TWO_D, PREP>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = p.num_tiles < CTAS * num_sms ? p.num_tiles : CTAS * num_sms;
    return launch_pdl(k, dim3(grid), dim3(kThreads), smem, st, maps, p);
}

template <int GRID, bool SR, int SF>
static cudaError_t launch_rows(const RowsMaps& maps, RowsParams& p, int num_sms, cudaStream_t st) {
    if constexpr (SF == 1 && GRID < 4) {
        if (p.lb2d) {
            // 2-D blocks: 8 K-element tiles (one row pair per thread), six stages
            p.stages = 2 * kRowsStages;
            if (p.n == 16) return launch_rows_cfg<GRID, SR, SF, true, kRowsCtas, 128, true>(maps, p, num_sms, st);
            return launch_rows_cfg<GRID, SR, SF, false, kRowsCtas, 128, true>(maps, p, num_sms, st);
        }
    }
    p.stages = kRowsStages;
    if constexpr (SF == 1 && GRID <= 1) {
        if (p.prep) {
            if (p.n != 16) return cudaErrorNotSupported;
            return launch_rows_cfg<GRID, SR, SF, true, kRowsCtas, 128, false, true>(maps, p, num_sms, st);
        }
    }
    if (p.prep) return cudaErrorNotSupported;
    if (p.n == 16) return launch_rows_cfg<GRID, SR, SF, true, kRowsCtas, 128, false>(maps, p, num_sms, st);
    return launch_rows_cfg<GRID, SR, SF, false, kRowsCtas, 128, false>(maps, p, num_sms, st);
}

cudaError_t launch_quantize_rows(RowsParams& p, int grid, bool sr, int sf, int num_sms, cudaStream_t st) {
    // n = 64 and n = 256: the segment kernel, fed by 64-column boxes with the 128-byte swizzle
    const bool seg_kernel = (p.n == 64 && p.tc == 128) || (p.n == 256 && p.tc == 256);
    if (p.prep && (seg_kernel || p.lb2d || sf != 1 || grid > 1)) return cudaErrorNotSupported;
    RowsMaps maps;
    memset(&maps, 0, sizeof(maps));
    for (int t = 0; t < p.count; ++t) {
        const RowsTensor& T = p.t[t];
        if (!encode_map_2d(&maps.m[t], CU_TENSOR_MAP_DATA_TYPE_UINT16, T.x, (uint64_t)T.cols, (uint64_t)T.rows,
                           (uint64_t)T.ld * 2, seg_kernel ? 64u : (uint32_t)p.tc, seg_kernel ? (p.n == 256 ? 64u : 128u) : (uint32_t)p.tr,
                           seg_kernel ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
#define UFP4_R(G, FN)                                                                          \
    if (grid == G) {                                                                           \
        if (sr) return sf == 2 ? FN<G, true, 2>(maps, p, num_sms, st)                          \
                     : sf == 1 ? FN<G, true, 1>(maps, p, num_sms, st)                          \
                               : FN<G, true, 0>(maps, p, num_sms, st);                         \
        return sf == 2 ? FN<G, false, 2>(maps, p, num_sms, st)                                 \
             : sf == 1 ? FN<G, false, 1>(maps, p, num_sms, st)                                 \
                       : FN<G, false, 0>(maps, p, num_sms, st);                                \
    }
    if (seg_kernel) {
        UFP4_R(0, launch_rows_seg)
        UFP4_R(1, launch_rows_seg)
        UFP4_R(2, launch_rows_seg)
        UFP4_R(3, launch_rows_seg)
        if (grid == 4 && !sr && sf == 1) return launch_rows_seg<4, false, 1>(maps, p, num_sms, st);  // MXFP8
        return cudaErrorInvalidValue;
    }
    UFP4_R(0, launch_rows)
    UFP4_R(1, launch_rows)
    UFP4_R(2, launch_rows)
    UFP4_R(3, launch_rows)
#undef UFP4_R
    if (grid == 4 && !sr && sf == 1) return launch_rows<4, false, 1>(maps, p, num_sms, st);  // MXFP8
    return cudaErrorInvalidValue;
}

cudaError_t rows_error_read_clear(int* value) {
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_rows_error, sizeof(int));
    if (e != cudaSuccess) return e;
    if (v) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_rows_error, &zero, sizeof(int));
    }
    *value = v;
    return e;
}

cudaError_t set_rows_wait_limit(uint32_t polls) {
    return cudaMemcpyToSymbol(g_rows_wait_limit, &polls, sizeof(polls));
}

// Loads every kernel of this unit (cudaFuncGetAttributes loads a function
// that has not been loaded yet).
template <int G, bool SR>
static void preload_rows(cudaFuncAttributes* a) {
    constexpr int kSegCtas = kRowsCtas;
    cudaFuncGetAttributes(a, quantize_rows_seg_kernel<G, SR, 0, kSegCtas, 2, false>);
    cudaFuncGetAttributes(a, quantize_rows_seg_kernel<G, SR, 1, kSegCtas, 2, false>);
    cudaFuncGetAttributes(a, quantize_rows_seg_kernel<G, SR, 2, kSegCtas, 2, false>);
    cudaFuncGetAttributes(a, quantize_rows_seg_kernel<G, SR, 0, kSegCtas, 4, false>);
    cudaFuncGetAttributes(a, quantize_rows_seg_kernel<G, SR, 1, kSegCtas, 4, false>);
    cudaFuncGetAttributes(a, quantize_rows_seg_kernel<G, SR, 2, kSegCtas, 4, false>);
    cudaFuncGetAttributes(a, quantize_rows_seg_kernel<G, SR, 1, kSegCtas, 2, true>);
    cudaFuncGetAttributes(a, quantize_rows_seg_kernel<G, SR, 1, kSegCtas, 4, true>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 0, false, kRowsCtas, 128, false>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 1, false, kRowsCtas, 128, false>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 2, false, kRowsCtas, 128, false>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 0, true, kRowsCtas, 128, false>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 1, true, kRowsCtas, 128, false>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 2, true, kRowsCtas, 128, false>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 1, false, kRowsCtas, 128, true>);
    cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 1, true, kRowsCtas, 128, true>);
    if constexpr (G <= 1) cudaFuncGetAttributes(a, quantize_rows_kernel<G, SR, 1, true, kRowsCtas, 128, false, true>);
}

cudaError_t preload_rows_kernels() {
    cudaFuncAttributes a;
    preload_rows<0, false>(&a);
    preload_rows<0, true>(&a);
    preload_rows<1, false>(&a);
    preload_rows<1, true>(&a);
    preload_rows<2, false>(&a);
    preload_rows<2, true>(&a);
    preload_rows<3, false>(&a);
    preload_rows<3, true>(&a);
    cudaFuncGetAttributes(&a, quantize_rows_kernel<4, false, 1, false, kRowsCtas, 128, false>);
    cudaFuncGetAttributes(&a, quantize_rows_kernel<4, false, 1, true, kRowsCtas, 128, false>);
    cudaFuncGetAttributes(&a, quantize_rows_seg_kernel<4, false, 1, kRowsCtas, 2, false>);
    cudaFuncGetAttributes(&a, quantize_rows_seg_kernel<4, false, 1, kRowsCtas, 4, false>);
    return cudaGetLastError();
}

}  // namespace ufp4
