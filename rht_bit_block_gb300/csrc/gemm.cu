// Quantized GEMM consumer D = Q(A) Q(B)^T (UFP4 summary, section 方法, the
// quantized GEMM Y^ = Q_G(X H') Q_G(W H')^T) on the sm_103a tensor cores.
//
// Both operands are K-major 4-bit codes with UE8M0 (power-of-two) block
// scales, so every product is exact in a block-scaled MMA:
//  * E2M1 codes are native FP4: kind::mxf4nvf4 reads the packed nibbles
//    straight from the quantizer's output (1 x 16 blocks: scale_vec::4X, one
//    scale per 16 elements; 1 x 32 and 32 x 32 blocks: scale_vec::2X).
//  * E1M2 / INT4 levels are integers k (|k| <= 7) times a power of two.  A
//    prep kernel widens them into FP8 E5M2 (exact) in the workspace and folds
//    the block scales into one UE8M0 scale per 32 elements (kind::mxf8f6f4,
//    scale_vec::1X): for a pair of 1 x 16 blocks with exponents e0, e1 the
//    hardware scale is max(e0, e1) and the elements of the smaller block are
//    shifted down by the difference d (exact for d <= 16 in E5M2).
//  * The two-level format's E4M3 block scales (E2M1, 1 x 16) ride in
//    kind::mxf4nvf4 as UE4M3 (never negative); the product of the two fp32
//    tensor scales multiplies the accumulator in the epilogue.
//
// Kernel: persistent CTA pairs (clusters of two CTAs on two SMs, 8 warps
// each) walking 256 x BN output tiles with tcgen05.mma .cta_group::2.  Warp 0
// lane 0 of each CTA drives TMA (128B-swizzled 2-D tiles of A and B, boxes of
// replicated scale chunks) through a ring of mbarriers; warp 1 lane 0 of the
// even CTA copies the scales into tensor memory (tcgen05.cp) and issues the
// MMAs for both CTAs into one of two tensor-memory accumulators; warps 4..7
// of both CTAs read the other accumulator back (tcgen05.ld) and store fp32,
// so a tile's epilogue overlaps the next tile's main loop.  Every wait is
// bounded: on expiry the kernel records an error code, lets its copies and
// MMAs finish and returns.
//
// Plain fp32 block scales cannot ride in a block-scaled MMA; they take the
// two-scale kernel at the end of this file.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/ufp4.h"
#include "internal.h"
#include "widen_e5m2.cuh"

namespace ufp4 {

__device__ int g_device_error;

namespace {

constexpr int kBM = 128;
constexpr int kBKBytes = 128;          // bytes of K per stage per row (one 128B swizzle row)
constexpr int kGemmThreads = 256;
constexpr int kChunkBytes = 512;       // 128 rows x 4 scale bytes, tcgen05.cp 32x128b layout
constexpr uint32_t kWaitLimit = 1u << 22;  // bounded polling; each poll may sleep up to kSuspendNs
constexpr uint32_t kSuspendNs = 1000;
constexpr int kErrTimeout = 1;

// Output tile widths.  Both paths run on CTA pairs.  FP8: 256 x 224 tiles, two
// 224-column accumulators plus two sets of scale columns fit the 512
// tensor-memory columns, and the wider tile gives each MMA instruction more
// work (issuing a tcgen05 instruction costs a fixed time).  FP4 needs two
// (2X kind) to four (4X kind) times the scale columns per K tile: the 2X
// kind's two scale sets still fit beside two 224-column accumulators
// (448 + 48 <= 512).  The 4X kind's do not: kind 2 runs 256 x 192 tiles
// with two accumulators (384 + 96), kind 4 256 x 256 tiles with one (256 +
// 96).  Each stage's six scale copies and its hand-off cost the same time
// whatever the tile width, so the wide tile does a third more MMA work per
// stage, but a tile's epilogue then holds up the next tile's first MMA:
// the plan takes kind 4 for long K (16 or more K tiles per output tile).
constexpr int kBnFp8 = 224, kBnFp4 = 192, kBnFp4Wide = 256;
constexpr int kBnFp4x2 = 224;
__host__ __device__ constexpr int pair_bn(int kind) {
    return kind == 0 ? kBnFp8 : (kind == 1 ? kBnFp4x2 : (kind == 4 ? kBnFp4Wide : kBnFp4));
}
// accumulator buffers in tensor memory: two (a tile's epilogue overlaps the
// next tile's main loop), or one for kind 4's 256-wide tiles
__host__ __device__ constexpr int pair_nacc(int kind) { return kind == 4 ? 1 : 2; }
constexpr int kWideFp4MinKTiles = 16;
// CTA-pair rings: stages of KPS K tiles each (FP4 stages hold one K tile of
// 256 elements, as much MMA work as two FP8 K tiles of 128)
constexpr int kPairKps = 2, kPairStages = 3;          // FP8
constexpr int kPairStagesFp4x2 = 5, kPairStagesFp4x4 = 4;
// Scale chunks of the FP4 kinds: stored once and copied to tensor memory
// with one .32x128b.warpx4 per 512-byte chunk (false), or stored four times
// and copied two chunks per .128x256b (true, the FP8 layout)
constexpr bool kFp4Replicated = true;
// Pair rows per tile group (see pair_tile_coords).  With 16 on the
// 16384 x 7168 x 7168 FPROP, the tiles in flight touch about 16 A panels
// (29 MB of FP8) and 5 B panels, A is read from DRAM once and B four times.
constexpr int kPairGroupM = 16;
__host__ __device__ constexpr bool pair_replicated(int kind) { return kind == 0 || kFp4Replicated; }

// ------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Bounded wait on an mbarrier phase.  Returns false (and records the error)
// when the limit is reached.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        uint32_t ok;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
            : "=r"(ok)
            : "r"(bar), "r"(parity), "r"(kSuspendNs)
            : "memory");
        if (ok) return true;
    }
    atomicExch(&g_device_error, kErrTimeout);
    return false;
}

// L2 policies: operand tiles are re-read by many CTAs (keep them), the fp32
// output is written once (let it leave first).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar,
                                            uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(dst), "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void st_out4(float* dst, const uint32_t* r, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;"
                 ::"l"(dst), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "l"(pol)
                 : "memory");
}

// 32-byte store: one whole L2 sector per instruction (needs a 32-byte aligned address).
__device__ __forceinline__ void st_out8(float* dst, const uint32_t* r, uint64_t pol) {
    asm volatile("st.global.L1::no_allocate.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;"
                 ::"l"(dst), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                   "r"(r[7]), "l"(pol)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major, 128-byte swizzle shared-memory matrix descriptor: 8-row groups
// 1024 bytes apart (stride byte offset), fixed version bits 0b001 at 46..48,
// swizzle mode 2 (128B) at 61..63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t r[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Instruction descriptor of the block-scaled kinds: B scale id at 4..5,
// A/B formats at 7..9 / 10..12, N>>3 at 17..22, UE8M0 scale type at 23,
// M>>4 at 24..28, A scale id at 29..30; both operands K-major.
__host__ __device__ constexpr uint32_t make_idesc(int afmt, int bfmt, int M, int N, int sf_id, bool ue8m0 = true) {
    return ((uint32_t)sf_id << 4) | ((uint32_t)afmt << 7) | ((uint32_t)bfmt << 10) |
           ((uint32_t)(N >> 3) << 17) | ((ue8m0 ? 1u : 0u) << 23) | ((uint32_t)(M >> 4) << 24) |
           ((uint32_t)sf_id << 29);
}

// kind::f16 instruction descriptor: fp32 accumulator (bits 4..5 = 1), bf16 A
// and B (bits 7..9, 10..12 = 1), both K-major, N>>3 at 17..22, M>>4 at 24..28.
__host__ __device__ constexpr uint32_t make_idesc_f16(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------ CTA-pair kernel
// A cluster of two CTAs on two SMs computes a 256 x BN output tile with
// tcgen05.mma .cta_group::2: the FP8 path (E1M2 / INT4 widened to E5M2) and
// the native FP4 kinds (E2M1 codes straight from the quantizer).  Each CTA
// holds its own 128 rows of A and half (BN/2 rows) of B, so per SM the
// shared-memory and L2 traffic per MMA FLOP drops by about 30 % against a
// single-CTA 128 x BN tile; the accumulator rows of a CTA sit in its own
// tensor memory.  Both CTAs hold the scale chunks of all BN rows of B.  The
// even CTA ("leader") issues the MMAs for both; both CTAs' copies complete on
// the leader's stage barrier, and the leader's commits arrive on the barriers
// of both CTAs.

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// shared::cluster address of the same shared-memory offset in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// arrive on an mbarrier given by its shared::cluster address (own or peer CTA)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}

// TMA tile load into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_pair(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t cbar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        ::"r"(dst), "l"((uint64_t)map), "r"(x), "r"(y), "r"(cbar), "l"(pol)
        : "memory");
}

template <int KIND>  // 0: mxf8f6f4 scale_vec::1X, 1: mxf4 scale_vec::2X, 2 and 4: mxf4nvf4 scale_vec::4X
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t accumulate) {
    if (KIND == 0) {
        asm volatile(
            "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p; }"
            ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    } else if (KIND == 1) {
        asm volatile(
            "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p; }"
            ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p; }"
            ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    }
}

// arrives on the mbarrier at this offset in both CTAs once every MMA / copy
// issued so far by this thread has completed
__device__ __forceinline__ void tc_commit_pair_both(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"((uint16_t)3)
        : "memory");
}

__device__ __forceinline__ void tc_commit_pair_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 128 lanes x 32 bytes (8 columns) from a 4 KB replicated-chunk block:
// lane L reads 16-byte line L of the first 2 KB and of the second 2 KB.
__device__ __forceinline__ void tc_cp_scales_pair_256(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 32 lanes x 16 bytes of one 512-byte chunk, to all four lane quadrants
__device__ __forceinline__ void tc_cp_scales_pair_x4(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// No-swizzle descriptor of one 512-byte chunk: 8-row core matrices 128 bytes apart
__device__ __forceinline__ uint64_t sf512_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// No-swizzle K-major descriptor of that block: 8-row core matrices (128 B)
// 128 bytes apart, the second 16-byte column 2048 bytes after the first.
__device__ __forceinline__ uint64_t sf256_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(2048u >> 4) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// A stage holds KPS consecutive 128-byte K tiles ("atoms") of each operand,
// and the scale chunks of those K tiles in the replicated layout the prep
// kernels write for this path: each 512-byte chunk (128 rows x 4 scale bytes)
// stored four times, so that one tcgen05.cp .128x256b fills 8 tensor-memory
// columns of all 128 lanes from two chunks.  A K tile has CPK chunks per 128
// rows (FP8 1X: 1; FP4 2X: 2, one per two MMAs; FP4 4X: 4, one per MMA);
// chunk u = j * CPK + c of the stage (K tile j, chunk c):
//  * A: chunks 2v and 2v+1 side by side in copy v (columns 4u of the A set);
//  * B: its two 128-row parts side by side in copy u (columns 8u, 8u + 4).
// The scale stages come first in shared memory, the 1024-aligned operand
// stages after; stages alternate between two sets of scale columns.
template <int KIND, int STAGES, int KPS>
struct PairCfg {
    static constexpr int CPK = KIND == 0 ? 1 : (KIND == 1 ? 2 : 4);
    static constexpr int BN = pair_bn(KIND);  // output columns of a pair tile
    static constexpr int kBRows = BN / 2;                // B rows held per CTA
    static constexpr int kAAtom = kBM * kBKBytes;        // 16 KB
    static constexpr int kBAtom = kBRows * kBKBytes;
    static constexpr int kABytes = KPS * kAAtom;
    static constexpr int kBBytes = KPS * kBAtom;
    static constexpr int kChunks = KPS * CPK;                // chunks per 128 rows per stage
    static constexpr bool kRepl = pair_replicated(KIND);
    static constexpr int kRep = (kRepl ? 4 : 1) * kChunkBytes;  // one stored chunk: 2 KB replicated, else 512 B
    static constexpr int kSfaBytes = kChunks * kRep;         // this CTA's 128 rows
    static constexpr int kSfbBytes = 2 * kChunks * kRep;     // both 128-row parts of B
    static constexpr int kTxPerAtom = kAAtom + kBAtom;       // operand bytes per CTA per K tile
    static constexpr int kTxScales = kSfaBytes + kSfbBytes;  // scale bytes per CTA per stage (full boxes)
    static constexpr int kOffSfa = 0;
    static constexpr int kOffSfb = STAGES * kSfaBytes;
    static constexpr int kOffA = kOffSfb + STAGES * kSfbBytes;
    static constexpr int kOffB = kOffA + STAGES * kABytes;
    static constexpr int kOffBars = kOffB + STAGES * kBBytes;
    static constexpr int kNumBars = 2 * STAGES + 4 + 1;  // full, empty, acc_full x2, acc_empty x2, drain
    static constexpr int kSmem = kOffBars + 8 * kNumBars + 16 + 1024;
    static constexpr int kTmemCols = 512;
    static constexpr int kASet = 4 * kChunks;            // scale columns of A per set
    static constexpr int kBSet = 8 * kChunks;            // scale columns of B per set
    static constexpr int NACC = pair_nacc(KIND);
    static constexpr int kSfaCol = NACC * BN;
    static constexpr int kSfbCol = kSfaCol + 2 * kASet;
    static_assert(kSfbCol + 2 * kBSet <= kTmemCols, "tensor memory overflow");
    static_assert(kSmem <= 232448, "shared memory overflow");
    static_assert(kOffA % 1024 == 0 && kAAtom % 1024 == 0 && kBAtom % 1024 == 0,
                  "128B-swizzled tiles need 1024-byte alignment");
    static_assert(BN % 32 == 0 && BN > 128 && BN <= 256, "two scale parts of B; 32-column epilogue reads");
    static_assert(kChunks % 2 == 0, "A's scale copies hold two chunks");
};

// One GEMM of a launch.  A launch walks the tiles of up to G GEMMs sharing
// the kind and the descriptor (the groups of ufp4_gemm_grouped), numbered
// one GEMM after the other.
struct PairGroup {
    int M, N, k_tiles, m_pairs, n_tiles;
    int group_m;          // tile order: groups of group_m pair rows, n fastest inside a group
    int tile0;            // index of this GEMM's first tile in the launch
    int64_t sf_chunks_k;  // chunks along K per 128-row block
    float* D;
    int64_t ldd;
    int vec8;
    // two-level scale: D = acc * g_A * g_B, g = fp32(T / den), den = fp32(qmax * 448)
    const float* amax_a;
    const float* amax_b;
};
template <int G>
struct PairMaps {
    CUtensorMap m[G][4];  // A, B and their scale chunks, per GEMM
};
template <int G>
struct PairKParams {
    PairGroup g[G];
    int ngroups, num_tiles;
    uint32_t idesc[4];
    float den;
    int two_level;
};

// Output tile (pair row mp, column block nb) of the GEMM's local tile index.
// Tiles run in groups of group_m pair rows, the column block advancing
// fastest inside a group: the 76 or so tiles in flight at a time then touch
// about group_m A panels and a few B panels, which stay in L2 while the group
// sweeps N, so A comes from DRAM once and B once per group (in plain
// column-major order every column block re-read all of A).
__device__ __forceinline__ void pair_tile_coords(const PairGroup& pg, int local, int& mp, int& nb) {
    const int span = pg.group_m * pg.n_tiles;
    const int g = local / span;
    const int first = g * pg.group_m;
    const int rows = min(pg.group_m, pg.m_pairs - first);
    const int l = local - g * span;
    nb = l / rows;
    mp = first + (l - nb * rows);
}

template <int KIND, int STAGES, int KPS, int G>
__global__ void __launch_bounds__(kGemmThreads, 1)
gemm_pair_kernel(const __grid_constant__ PairMaps<G> maps, const __grid_constant__ PairKParams<G> p) {
    using C = PairCfg<KIND, STAGES, KPS>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t bars = base + C::kOffBars;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (STAGES + s); };
    auto accf_bar = [&](int b) { return bars + 8u * (2 * STAGES + b); };
    auto acce_bar = [&](int b) { return bars + 8u * (2 * STAGES + 2 + b); };
    const uint32_t drain_bar = bars + 8u * (2 * STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBars + 8 * C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBars + 8 * C::kNumBars + 4);
    auto stage_a = [&](int s) { return base + C::kOffA + s * C::kABytes; };
    auto stage_b = [&](int s) { return base + C::kOffB + s * C::kBBytes; };
    auto stage_sfa = [&](int s) { return base + C::kOffSfa + s * C::kSfaBytes; };
    auto stage_sfb = [&](int s) { return base + C::kOffSfb + s * C::kSfbBytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const uint32_t peer = rank & 1u;       // 0: leader (even CTA), 1: the other CTA of the pair
    const uint32_t leader = rank & ~1u;
    const int num_tiles = p.num_tiles;
    const int cluster_id = blockIdx.x >> 1;
    const int num_clusters = gridDim.x >> 1;
    // the GEMM a tile belongs to, and the tile's index inside it
    auto locate = [&](int tile, int& local) {
        int gi = 0;
        while (gi + 1 < p.ngroups && tile >= p.g[gi + 1].tile0) ++gi;
        local = tile - p.g[gi].tile0;
        return gi;
    };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);   // the leader's expect_tx arrival (both CTAs' bytes)
            mbar_init(empty_bar(s), 1);  // the leader's commit
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);   // the leader's commit
            mbar_init(acce_bar(b), 8);   // four epilogue warps of each CTA
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        // one warp of each CTA of the pair allocates, collectively
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(C::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs' barriers exist before any copy or commit targets them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_wait();
    griddep_launch();

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer (both CTAs)
        int s = 0;
        uint32_t ph = 0;
        const uint64_t keep = policy_evict_last();
        for (int tile = cluster_id; tile < num_tiles && !*abort_flag; tile += num_clusters) {
            int local;
            const int gi = locate(tile, local);
            const PairGroup& q = p.g[gi];
            const CUtensorMap* tm = maps.m[gi];
            int mp, nb;
            pair_tile_coords(q, local, mp, nb);
            const int k_stages = (q.k_tiles + KPS - 1) / KPS;
            const int ablk = 2 * mp + (int)peer;            // this CTA's 128-row block of A
            const int arow = ablk * kBM;
            const int brow = nb * C::BN + (int)peer * C::kBRows;
            // 512-byte rows of the chunk arrays: R per chunk for A, 2R for B (R = 4 replicated, else 1)
            constexpr int R = C::kRep / kChunkBytes;
            const int sfa_row = ablk * (int)q.sf_chunks_k * R;
            const int sfb_row = nb * (int)q.sf_chunks_k * 2 * R;
            for (int ks = 0; ks < k_stages; ++ks) {
                if (!mbar_wait(empty_bar(s), ph ^ 1u)) {
                    *abort_flag = 1;
                    break;
                }
                const int kt0 = ks * KPS;
                const int nk = q.k_tiles - kt0 < KPS ? q.k_tiles - kt0 : KPS;
                const uint32_t fb = map_to_rank(full_bar(s), leader);
                if (peer == 0) mbar_expect_tx(full_bar(s), 2 * (nk * C::kTxPerAtom + C::kTxScales));
                for (int j = 0; j < nk; ++j) {
                    tma_load_pair(stage_a(s) + j * C::kAAtom, &tm[0], (kt0 + j) * kBKBytes, arow, fb, keep);
                    tma_load_pair(stage_b(s) + j * C::kBAtom, &tm[1], (kt0 + j) * kBKBytes, brow, fb, keep);
                }
                // the scales of the stage's K tiles are contiguous: one box each
                tma_load_pair(stage_sfa(s), &tm[2], 0, sfa_row + kt0 * C::CPK * R, fb, keep);
                tma_load_pair(stage_sfb(s), &tm[3], 0, sfb_row + kt0 * C::CPK * 2 * R, fb, keep);
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 1 && lane == 0 && peer == 0) {
        // ------------------------------------------------ MMA issuer (leader only)
        int s = 0, tc = 0;
        uint32_t ph = 0;
        int sc = 0;  // stages issued so far (alternates the scale sets)
        bool ok = true;
        for (int tile = cluster_id; tile < num_tiles && ok; tile += num_clusters, ++tc) {
            // buffer buf of NACC, in its (tc / NACC)-th use
            const int buf = C::NACC == 2 ? (tc & 1) : 0;
            const uint32_t use_par = C::NACC == 2 ? ((tc >> 1) & 1) : (tc & 1);
            if (!mbar_wait(acce_bar(buf), use_par ^ 1)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t acc = tmem + buf * C::BN;
            int local;
            const int k_tiles = p.g[locate(tile, local)].k_tiles;
            const int k_stages = (k_tiles + KPS - 1) / KPS;
            for (int ks = 0; ks < k_stages; ++ks) {
                if (!mbar_wait(full_bar(s), ph) || *abort_flag) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int kt0 = ks * KPS;
                const int nk = k_tiles - kt0 < KPS ? k_tiles - kt0 : KPS;
                const uint32_t sfa_t = tmem + C::kSfaCol + (sc & 1) * C::kASet;
                const uint32_t sfb_t = tmem + C::kSfbCol + (sc & 1) * C::kBSet;
                ++sc;
                for (int j = 0; j < nk; ++j) {
                    const uint64_t da = sw128_desc(stage_a(s) + j * C::kAAtom);
                    const uint64_t db = sw128_desc(stage_b(s) + j * C::kBAtom);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        // chunk of MMA q: FP8 1X -> 0 (byte q), FP4 2X -> q/2 (bytes 0-1 / 2-3), FP4 4X -> q
                        const int cq = C::CPK == 1 ? 0 : (C::CPK == 2 ? q >> 1 : q);
                        const int u = j * C::CPK + cq;
                        if (C::CPK == 4 || q == 0 || (C::CPK == 2 && q == 2)) {
                            if (C::kRepl) {
                                // first MMA of chunk u: A's copy of chunks u, u+1 (u even), B's copy of chunk u
                                if ((u & 1) == 0)
                                    tc_cp_scales_pair_256(sfa_t + 4 * u,
                                                          sf256_desc(stage_sfa(s) + (u >> 1) * 2 * C::kRep));
                                tc_cp_scales_pair_256(sfb_t + 8 * u, sf256_desc(stage_sfb(s) + u * 2 * C::kRep));
                            } else {
                                // one copy per 512-byte chunk: A's chunk u, B's chunk u of parts 0 and 1
                                tc_cp_scales_pair_x4(sfa_t + 4 * u, sf512_desc(stage_sfa(s) + u * C::kRep));
                                tc_cp_scales_pair_x4(sfb_t + 8 * u, sf512_desc(stage_sfb(s) + 2 * u * C::kRep));
                                tc_cp_scales_pair_x4(sfb_t + 8 * u + 4, sf512_desc(stage_sfb(s) + (2 * u + 1) * C::kRep));
                            }
                        }
                        // each MMA consumes 32 bytes of K: advance the start address by two 16-byte units
                        mma_pair<KIND>(acc, da + 2 * q, db + 2 * q, p.idesc[q], sfa_t + 4 * u, sfb_t + 8 * u,
                                       (kt0 + j > 0 || q > 0) ? 1u : 0u);
                    }
                }
                tc_commit_pair_both(empty_bar(s));  // frees stage s in both CTAs
                if (++s == STAGES) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (ok) tc_commit_pair_both(accf_bar(buf));
        }
        if (!ok) *abort_flag = 1;
        tc_commit_pair_local(drain_bar);
        mbar_wait(drain_bar, 0);
    } else if (warp >= 4) {
        // ------------------------------------------------- epilogue (both CTAs)
        const int q = warp - 4;
        const uint64_t stream_out = policy_evict_first();
        int tc = 0;
        for (int tile = cluster_id; tile < num_tiles; tile += num_clusters, ++tc) {
            const int buf = C::NACC == 2 ? (tc & 1) : 0;
            const uint32_t use_par = C::NACC == 2 ? ((tc >> 1) & 1) : (tc & 1);
            const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(accf_bar(buf), use_par));
            if (!ok || *abort_flag) break;
            tc_fence_after();
            int local;
            const PairGroup& pg = p.g[locate(tile, local)];
            int mp, nb;
            pair_tile_coords(pg, local, mp, nb);
            const int row = (2 * mp + (int)peer) * kBM + q * 32 + lane;
            // two-level scale: the product of the tensor scales (written by the quantizer before this launch)
            const float gab =
                p.two_level ? __fmul_rn(__fdiv_rn(*pg.amax_a, p.den), __fdiv_rn(*pg.amax_b, p.den)) : 1.0f;
            const int n0 = nb * C::BN;
            for (int c = 0; c < C::BN; c += 32) {
                uint32_t r[32];
                tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + buf * C::BN + c, r);
                if (p.two_level)
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__fmul_rn(__uint_as_float(r[i]), gab));
                if (row < pg.M) {
                    float* dst = pg.D + (int64_t)row * pg.ldd + n0 + c;
                    if (n0 + c + 32 <= pg.N) {
                        if (pg.vec8) {
#pragma unroll
                            for (int i = 0; i < 32; i += 8) st_out8(dst + i, r + i, stream_out);
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i += 4) st_out4(dst + i, r + i, stream_out);
                        }
                    } else {
                        for (int i = 0; i < 32; ++i)
                            if (n0 + c + i < pg.N) dst[i] = __uint_as_float(r[i]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(acce_bar(buf), leader));
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // neither CTA leaves while the other may still use its memory or barriers
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols));
    }
}

// ------------------------------------------- fp32-scale GEMM (two-scale)
// D = sum over K blocks b of s_A[m,b] s_B[n,b] P_b[m,n], P_b = the block's
// product of the plain grid levels (UFP4 summary, 数据集: s_B = amax / qmax in
// fp32; 方法: the quantized GEMM Y^ = Q_G(XH') Q_G(WH')^T).  Plain fp32 block
// scales cannot be folded into a block-scaled MMA exactly, so each 16- or
// 32-element block runs as its own bf16 MMA (tcgen05.mma kind::f16, the
// levels are exact in bf16) into one of four tensor-memory partial buffers,
// and sixteen rescaler warps (4 lane quadrants x 4 groups of 32 columns) fold
// s_A s_B P_b into fp32 register accumulators.
// The CUDA-core multiply-adds bound it (two per output element and block).
constexpr int kF32sBN = 128;        // output tile 128 x 128
constexpr int kF32sStages = 3;
constexpr int kF32sThreads = 640;   // warps 0-3: TMA, MMA, idle; warps 4-19: rescalers
constexpr int kF32sPBufs = 4;       // 128-column partial buffers in tensor memory

struct F32sCfg {
    static constexpr int kAtom = kBM * kBKBytes;                 // 128 rows x 64 bf16 = 16 KB
    static constexpr int kABytes = 2 * kAtom;                    // a stage holds 128 K elements
    static constexpr int kBBytes = 2 * kAtom;
    static constexpr int kSaBytes = 128 * 8 * 4;                 // s_A: 128 rows x up to 8 blocks
    static constexpr int kSbBytes = 8 * kF32sBN * 4;             // s_B: up to 8 blocks x 128 columns
    static constexpr int kOffB = kF32sStages * kABytes;
    static constexpr int kOffSa = kOffB + kF32sStages * kBBytes;
    static constexpr int kOffSb = kOffSa + kF32sStages * kSaBytes;
    static constexpr int kOffBars = kOffSb + kF32sStages * kSbBytes;
    static constexpr int kNumBars = 2 * kF32sStages + 2 * kF32sPBufs;
    static constexpr int kSmem = kOffBars + 8 * kNumBars + 16 + 1024;
    static_assert(kSmem <= 232448, "shared memory overflow");
};

struct F32sKParams {
    int M, N, k_tiles, kb_per_tile;  // k_tiles: 128-element K tiles; blocks per K tile (8 or 4)
    int m_tiles, n_tiles;
    int kb_pad;                       // s_A row length (floats) in the workspace
    float* D;
    int64_t ldd;
    uint32_t idesc;                   // kind::f16, bf16 x bf16 -> fp32, M = 128, N = 128
    int mmas_per_block;               // 1 (16-element blocks) or 2 (32)
};

__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
        ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}

__global__ void __launch_bounds__(kF32sThreads, 1)
gemm_f32s_kernel(const __grid_constant__ CUtensorMap tmap_a, const __grid_constant__ CUtensorMap tmap_b,
                 const __grid_constant__ CUtensorMap tmap_sa, const __grid_constant__ CUtensorMap tmap_sb,
                 const F32sKParams p) {
    using C = F32sCfg;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - raw);
    const uint32_t bars = base + C::kOffBars;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kF32sStages + s); };
    auto pfull_bar = [&](int b) { return bars + 8u * (2 * kF32sStages + b); };
    auto pempty_bar = [&](int b) { return bars + 8u * (2 * kF32sStages + kF32sPBufs + b); };
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kOffBars + 8 * C::kNumBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::kOffBars + 8 * C::kNumBars + 4);
    auto stage_a = [&](int s) { return base + s * C::kABytes; };
    auto stage_b = [&](int s) { return base + C::kOffB + s * C::kBBytes; };
    const float* sa_s = reinterpret_cast<const float*>(gbase + C::kOffSa);
    const float* sb_s = reinterpret_cast<const float*>(gbase + C::kOffSb);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int num_tiles = p.m_tiles * p.n_tiles;
    const int kb = p.kb_per_tile;
    constexpr int kRescalers = 16;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kF32sStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1 + kRescalers);  // the MMA commit and every rescaler warp
        }
        for (int b = 0; b < kF32sPBufs; ++b) {
            mbar_init(pfull_bar(b), 1);
            mbar_init(pempty_bar(b), kRescalers);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    griddep_wait();
    griddep_launch();

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------- TMA producer
        int s = 0;
        uint32_t ph = 0;
        const uint64_t keep = policy_evict_last();
        for (int tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
            const int mb = tile % p.m_tiles, nb = tile / p.m_tiles;
            for (int kt = 0; kt < p.k_tiles; ++kt) {
                if (!mbar_wait(empty_bar(s), ph ^ 1u)) {
                    *abort_flag = 1;
                    break;
                }
                mbar_expect_tx(full_bar(s), C::kABytes + C::kBBytes + 128 * kb * 4 + kb * kF32sBN * 4);
                for (int j = 0; j < 2; ++j) {
                    tma_load_2d(stage_a(s) + j * C::kAtom, &tmap_a, (2 * kt + j) * kBKBytes, mb * kBM, full_bar(s),
                                keep);
                    tma_load_2d(stage_b(s) + j * C::kAtom, &tmap_b, (2 * kt + j) * kBKBytes, nb * kF32sBN,
                                full_bar(s), keep);
                }
                tma_load_2d(base + C::kOffSa + s * C::kSaBytes, &tmap_sa, kt * kb, mb * kBM, full_bar(s), keep);
                tma_load_2d(base + C::kOffSb + s * C::kSbBytes, &tmap_sb, 0, nb * p.k_tiles * kb + kt * kb,
                            full_bar(s), keep);
                if (++s == kF32sStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ----------------------------------------------------- MMA issuer
        int s = 0, pb = 0;
        uint32_t ph = 0, pph = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
            for (int kt = 0; kt < p.k_tiles && ok; ++kt) {
                if (!mbar_wait(full_bar(s), ph) || *abort_flag) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int j = 0; j < kb; ++j) {
                    if (!mbar_wait(pempty_bar(pb), pph ^ 1u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // block j covers 16 * mmas_per_block K elements: 32-byte steps inside 128-byte atoms
                    for (int q = 0; q < p.mmas_per_block; ++q) {
                        const int step = j * p.mmas_per_block + q;  // 16-element step within the stage
                        const uint64_t da = sw128_desc(stage_a(s) + (step >> 2) * C::kAtom) + 2 * (step & 3);
                        const uint64_t db = sw128_desc(stage_b(s) + (step >> 2) * C::kAtom) + 2 * (step & 3);
                        mma_f16(tmem + pb * kF32sBN, da, db, p.idesc, q > 0 ? 1u : 0u);
                    }
                    tc_commit(pfull_bar(pb));
                    if (++pb == kF32sPBufs) {
                        pb = 0;
                        pph ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(empty_bar(s));  // the operand tiles may be refilled once these MMAs are done
                if (++s == kF32sStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp >= 4) {
        // -------------------------------------------------------- rescalers
        const int q = warp & 3;               // tensor-memory lane quadrant (rows 32q .. 32q+31)
        const int grp = (warp - 4) >> 2;       // columns 32 grp .. +31
        const int row_in_tile = q * 32 + lane;
        int s = 0, pb = 0;
        uint32_t ph = 0, pph = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            const int mb = tile % p.m_tiles, nb = tile / p.m_tiles;
            float acc[32];
#pragma unroll
            for (int c = 0; c < 32; ++c) acc[c] = 0.0f;
            bool ok = true;
            for (int kt = 0; kt < p.k_tiles && ok; ++kt) {
                if (!__all_sync(0xFFFFFFFFu, mbar_wait(full_bar(s), ph)) || *abort_flag) {
                    ok = false;
                    break;
                }
                const float* sa = sa_s + s * (C::kSaBytes / 4) + row_in_tile * kb;  // this row's block scales
                const float* sb = sb_s + s * (C::kSbBytes / 4);                      // [block][128 columns]
                for (int j = 0; j < kb; ++j) {
                    if (!__all_sync(0xFFFFFFFFu, mbar_wait(pfull_bar(pb), pph))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t r[32];
                    tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + pb * kF32sBN + grp * 32, r);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(pempty_bar(pb));  // the partial buffer may be refilled
                    if (++pb == kF32sPBufs) {
                        pb = 0;
                        pph ^= 1u;
                    }
                    const float a = sa[j];
                    const float4* sbv = reinterpret_cast<const float4*>(sb + j * kF32sBN + grp * 32);
#pragma unroll
                    for (int c4 = 0; c4 < 8; ++c4) {
                        const float4 b = sbv[c4];
                        acc[4 * c4 + 0] = __fmaf_rn(__fmul_rn(__uint_as_float(r[4 * c4 + 0]), b.x), a, acc[4 * c4 + 0]);
                        acc[4 * c4 + 1] = __fmaf_rn(__fmul_rn(__uint_as_float(r[4 * c4 + 1]), b.y), a, acc[4 * c4 + 1]);
                        acc[4 * c4 + 2] = __fmaf_rn(__fmul_rn(__uint_as_float(r[4 * c4 + 2]), b.z), a, acc[4 * c4 + 2]);
                        acc[4 * c4 + 3] = __fmaf_rn(__fmul_rn(__uint_as_float(r[4 * c4 + 3]), b.w), a, acc[4 * c4 + 3]);
                    }
                }
                if (!ok) break;
                // this stage's scales have been read: release it (with the MMA's commit)
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));
                if (++s == kF32sStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
            if (!ok) break;
            const int row = mb * kBM + row_in_tile;
            const int n0 = nb * kF32sBN + grp * 32;
            if (row < p.M) {
                float* dst = p.D + (int64_t)row * p.ldd + n0;
                if (n0 + 32 <= p.N) {
#pragma unroll
                    for (int c = 0; c < 32; c += 4)
                        *reinterpret_cast<float4*>(dst + c) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
                } else {
                    for (int c = 0; c < 32; ++c)
                        if (n0 + c < p.N) dst[c] = acc[c];
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
    }
}

// ------------------------------------------------------------- prep kernels

// One operand of the prep launch.
struct PrepSide {
    const uint8_t* codes;
    const uint8_t* scales;
    int64_t codes_ld, scales_ld;
    int rows;          // rows of the operand
    int rows_cover;    // chunk rows written: rows rounded up to whole GEMM tiles
    int tile_rows;     // rows of one GEMM tile of this operand (128 for A, BN for B)
    uint8_t* out_fp8;  // rows x K bytes (E1M2/INT4 only)
    uint8_t* out_chunks;
    int K;             // elements along K
    int chunks_k;      // chunk cells along K per 128 rows
};

// Up to kPairGroups GEMMs (both operands of each) in one prep launch:
// blockIdx.z picks the side, 2 g + (0 for A, 1 for B).
constexpr int kPairGroups = 8;
struct PrepParams {
    PrepSide side[2 * kPairGroups];
    int grid;          // codebook
    int lbr, lbc;      // log2 of the block rows and columns
    int lhw;           // log2 of the hardware scale block: 4 (E2M1 1x16) or 5
    int copies;        // stored copies of each chunk (4: replicated)
};

// Replicated scale chunks of the CTA-pair kernel.  Chunk g along K (g = K
// tile * chunks per K tile + c) of the 128-row part h of GEMM tile t
// (tile_rows rows) is stored four times, at
// ((((t * chunks_k + g) * parts + h) * 4 + copy) * 512, with row w of the part
// and scale cell byte j at (w % 32) * 16 + (w / 32) * 4 + j in each copy
// (the tcgen05.cp 32x128b chunk layout).

// Widen E1M2 / INT4 codes into FP8 E5M2 with one UE8M0 hardware scale per 32
// elements (replicated chunk layout above).  A CTA is 32 x 8 threads and
// covers, in one 128-row part of a GEMM tile, the rows w = 32 q + 2 j + e
// (q = 0..3, e = 0..1; warp 2 q + e) for its j = blockIdx.x % 16: the rows
// whose chunk cells make up two whole 16-byte lines of every chunk.  Each warp
// owns its row, each lane two adjacent 32-element groups of it (32 code bytes
// in, 64 FP8 bytes out, contiguous across the warp); the scale bytes are
// gathered in shared memory and leave as whole 32-byte sectors, four copies
// per chunk.  blockIdx.x: (part, j), blockIdx.y: 64-group slab along K,
// blockIdx.z: operand (of one of the GEMMs of the launch).
__global__ void __launch_bounds__(256) prep_widen_kernel(const PrepParams p) {
    __shared__ __align__(16) uint8_t cells[16][32];  // per chunk of the slab: lines 2 j and 2 j + 1
    griddep_wait();
    griddep_launch();
    const PrepSide& s = p.side[blockIdx.z];
    const int parts = (s.tile_rows + 127) >> 7;
    const int part = blockIdx.x >> 4, jj = blockIdx.x & 15;
    if (part >= (s.rows_cover / s.tile_rows) * parts) return;  // whole CTAs
    const int t = part / parts, h = part - t * parts;
    const int part_rows = min(128, s.tile_rows - h * 128);
    const int y = threadIdx.y, lane = threadIdx.x;
    const int w = 32 * (y >> 1) + 2 * jj + (y & 1);
    const bool has_row = w < part_rows;            // rows past a 224-row tile's end do not exist
    const int row = t * s.tile_rows + h * 128 + w;
    const bool live = has_row && row < s.rows;     // rows up to rows_cover get zero cells
    const int g0 = blockIdx.y * 64 + 2 * lane;     // groups g0, g0 + 1 along K
    const int step_log2 = p.grid == 0 ? -2 : 0;    // E1M2 levels are k/4, INT4 levels k
    const uint8_t* srow = s.scales + (int64_t)(row >> p.lbr) * s.scales_ld;
    uint4 cw[2];
    int e0[2] = {0, 0}, e1[2] = {0, 0};
    bool ok[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        ok[q] = live && (g0 + q) * 32 < s.K;
        cw[q] = make_uint4(0u, 0u, 0u, 0u);
        if (ok[q]) cw[q] = *reinterpret_cast<const uint4*>(s.codes + (int64_t)row * s.codes_ld + (g0 + q) * 16);
    }
    // the scale bytes of both groups: one aligned word (1 x 16) or half word (1 x 32) where possible
    const uintptr_t sa = reinterpret_cast<uintptr_t>(srow);
    if (ok[1] && p.lbc == 4 && (sa & 3) == 0) {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(srow + 2 * g0);
        e0[0] = v & 0xFF; e1[0] = (v >> 8) & 0xFF; e0[1] = (v >> 16) & 0xFF; e1[1] = v >> 24;
    } else if (ok[1] && p.lbc == 5 && (sa & 1) == 0) {
        const uint32_t v = *reinterpret_cast<const uint16_t*>(srow + g0);
        e0[0] = e1[0] = v & 0xFF; e0[1] = e1[1] = v >> 8;
    } else {
#pragma unroll
        for (int q = 0; q < 2; ++q)
            if (ok[q]) {
                const int k0 = (g0 + q) * 32;
                e0[q] = srow[k0 >> p.lbc];
                e1[q] = p.lbc == 4 ? srow[(k0 >> 4) + 1] : e0[q];
            }
    }
    int hw[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        hw[q] = ok[q] ? max(max(e0[q], e1[q]) + step_log2, 0) : 0;
        if (!ok[q]) continue;
        const int d0 = hw[q] - step_log2 - e0[q], d1 = hw[q] - step_log2 - e1[q];  // >= 0
        uint32_t words[4] = {cw[q].x, cw[q].y, cw[q].z, cw[q].w};
        if (p.grid == 1)
#pragma unroll
            for (int k = 0; k < 4; ++k) words[k] = twos_to_signmag8(words[k]);
        // elements 0-15: the first 16-element block, 16-31: the second
        const uint4 lo16 = widen16_e5m2(words[0], words[1], d0);
        const uint4 hi16 = widen16_e5m2(words[2], words[3], d1);
        const uint32_t outw[8] = {lo16.x, lo16.y, lo16.z, lo16.w, hi16.x, hi16.y, hi16.z, hi16.w};
        uint4* dst = reinterpret_cast<uint4*>(s.out_fp8 + (int64_t)row * s.K + (g0 + q) * 32);
        dst[0] = make_uint4(outw[0], outw[1], outw[2], outw[3]);
        dst[1] = make_uint4(outw[4], outw[5], outw[6], outw[7]);
    }
    // the cell of row w in chunk c: bytes (w % 32) * 16 + (w / 32) * 4 + (group % 4) of each copy;
    // here line e = w % 2 of the CTA's two, bytes (w / 32) * 4 + 2 (lane % 2) + {0, 1}
    *reinterpret_cast<uint16_t*>(&cells[lane >> 1][(y & 1) * 16 + (y >> 1) * 4 + 2 * (lane & 1)]) =
        (uint16_t)(hw[0] | (hw[1] << 8));
    __syncthreads();
    const int tid = y * 32 + lane;
    if (tid < 128) {
        const int c = tid >> 3, copy = (tid >> 1) & 3, e = tid & 1;
        const int g = blockIdx.y * 16 + c;  // chunk along K
        if (g < s.chunks_k) {
            const int64_t off =
                ((((int64_t)t * s.chunks_k + g) * parts + h) * 4 + copy) * kChunkBytes + (2 * jj + e) * 16;
            *reinterpret_cast<uint4*>(s.out_chunks + off) = *reinterpret_cast<const uint4*>(&cells[c][e * 16]);
        }
    }
}

// E2M1 and MXFP8: only the scales move, into the chunk layout of the pair kernel
// (hardware blocks of 16 or 32 elements, one scale byte each: UE8M0, or E4M3
// for the two-level format), replicated or not as pair_replicated says.  A
// warp writes one chunk: lane i builds the chunk's 16-byte line i (cells of
// rows i, i + 32, i + 64, i + 96 of the part) and stores it into each copy,
// so every store of the warp covers 512 contiguous bytes.  blockIdx.x: 8 chunks (one per warp), blockIdx.z: operand.
__global__ void __launch_bounds__(256) prep_scales_kernel(const PrepParams p) {
    griddep_wait();
    griddep_launch();
    const PrepSide& s = p.side[blockIdx.z];
    const int parts = (s.tile_rows + 127) >> 7;
    const int64_t blocks = (int64_t)(s.rows_cover / s.tile_rows) * parts;  // 128-row parts
    const int64_t item = (int64_t)blockIdx.x * 8 + threadIdx.y;            // (part block, chunk) pair
    if (item >= blocks * s.chunks_k) return;                               // whole warps
    const int g = (int)(item % s.chunks_k);
    const int64_t pb = item / s.chunks_k;
    const int t = (int)(pb / parts), h = (int)(pb % parts);
    const int i = threadIdx.x;
    uint32_t cell[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const int rr = h * 128 + i + 32 * c;  // row within the tile
        const int row = t * s.tile_rows + rr;
        uint32_t v = 0;
        if (rr < s.tile_rows && row < s.rows) {
            const uint8_t* srow = s.scales + (int64_t)(row >> p.lbr) * s.scales_ld;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int k0 = (g * 4 + j) << p.lhw;
                if (k0 < s.K) v |= (uint32_t)srow[k0 >> p.lbc] << (8 * j);
            }
        }
        cell[c] = v;
    }
    const uint4 line = make_uint4(cell[0], cell[1], cell[2], cell[3]);
    const int copies = p.copies;
    uint8_t* dst = s.out_chunks + ((((int64_t)t * s.chunks_k + g) * parts + h) * copies) * kChunkBytes + i * 16;
#pragma unroll
    for (int copy = 0; copy < copies; ++copy) *reinterpret_cast<uint4*>(dst + copy * kChunkBytes) = line;
}

// Level value of a 4-bit code (E1M2 k/4, INT4 two's complement k, E2M1 codes
// for grids 2 and 3).
__device__ __forceinline__ float decode_level_gemm(int grid, uint32_t nib) {
    if (grid == 1) return (float)((nib & 8u) ? (int)nib - 16 : (int)nib);
    const uint32_t k = nib & 7u;
    float v;
    if (grid == 0) v = (float)k * 0.25f;
    else v = k < 4 ? (float)k * 0.5f : (k == 4 ? 2.0f : (k == 5 ? 3.0f : (k == 6 ? 4.0f : 6.0f)));
    return (nib & 8u) ? -v : v;
}

// fp32 block scales: bf16 copies of the levels (exact) and the scales in the
// two-scale kernel's layout (A: [row][block]; B: [tile][block][128 columns]).
// One thread: one row, one 16-element chunk.
struct F32sSide {
    const uint8_t* codes;
    const float* scales;
    int64_t codes_ld, scales_ld;
    int rows, rows_cover, tile_rows, transposed;
    uint16_t* levels;
    float* scales_out;
};
struct F32sPrep {
    F32sSide side[2];
    int K, bc, grid;
};

__global__ void __launch_bounds__(256) prep_f32s_kernel(const F32sPrep p) {
    griddep_wait();
    griddep_launch();
    const F32sSide& s = p.side[blockIdx.z];
    const int64_t cpr = p.K / 16;
    const int64_t idx = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (idx >= (int64_t)s.rows_cover * cpr) return;
    const int row = (int)(idx / cpr);
    const int ch = (int)(idx - (int64_t)row * cpr);
    const bool live = row < s.rows;
    if (live) {
        const uint2 code = *reinterpret_cast<const uint2*>(s.codes + (int64_t)row * s.codes_ld + ch * 8);
        uint32_t out[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t word = i < 4 ? code.x : code.y;
            const float lo = decode_level_gemm(p.grid, (word >> (8 * (i & 3))) & 0xFu);
            const float hi = decode_level_gemm(p.grid, (word >> (8 * (i & 3) + 4)) & 0xFu);
            out[i] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
                     ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
        }
        uint4* dst = reinterpret_cast<uint4*>(s.levels + (int64_t)row * p.K + ch * 16);
        dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
        dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
    }
    if ((ch * 16) % p.bc == 0) {  // the first chunk of a block moves its scale (0 on padding rows)
        const int64_t kbt = p.K / p.bc;
        const int b = ch * 16 / p.bc;
        const float v = live ? s.scales[(int64_t)row * s.scales_ld + b] : 0.0f;
        if (s.transposed) {
            const int t = row / s.tile_rows, c = row - t * s.tile_rows;
            s.scales_out[((int64_t)t * kbt + b) * s.tile_rows + c] = v;
        } else {
            s.scales_out[(int64_t)row * kbt + b] = v;
        }
    }
}

// ------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeTiledFn)f;
    }
    return fn;
}

// 2-D byte tensor (rows x row_bytes, pitch bytes) read in boxes of 128 bytes x box_rows, 128B swizzle.
bool make_map(CUtensorMap* map, const void* ptr, int64_t rows, int64_t row_bytes, int64_t pitch, int box_rows) {
    return encode_map_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, ptr, (uint64_t)row_bytes, (uint64_t)rows,
                         (uint64_t)pitch, (uint32_t)kBKBytes, (uint32_t)box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

struct Plan {
    int kind;          // 0 fp8, 1 fp4 2X, 2 fp4 4X, 3 fp32 block scales (bf16 partials rescaled), 4 fp4 4X wide tiles
    bool native;       // kind 0 on MXFP8 codes: E4M3 operands used in place (no widening)
    int bn;            // B tile rows (output tile columns)
    int64_t k_bytes;   // bytes of K per row in the MMA operand
    int64_t k_tiles;
    int64_t chunks_k;  // scale chunks along K per 128 rows (multiple of chunks per stage)
    size_t fp8_a, fp8_b, sfa, sfb;  // workspace offsets
    size_t total;
};

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

float grid_qmax_host(int grid) { return grid == 0 ? 1.75f : (grid == 1 ? 7.0f : (grid == 2 ? 6.0f : 2.0f)); }

int ilog2(int v) {  // v a power of two
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}



Plan make_plan(int64_t M, int64_t N, int64_t K, int grid, int br, int bc, int sf) {
    Plan pl{};
    (void)br;
    if (sf == 0) {
        // fp32 block scales: bf16 level copies and the scales, laid out for the two-scale kernel
        pl.kind = 3;
        pl.bn = kF32sBN;
        pl.k_bytes = K * 2;
        pl.k_tiles = K / 128;
        const int64_t kbt = K / bc;  // blocks along K
        const int64_t mt = (M + kBM - 1) / kBM, nt = (N + kF32sBN - 1) / kF32sBN;
        size_t off = 0;
        pl.fp8_a = off;  // bf16 levels of A
        off = align256(off + (size_t)M * K * 2);
        pl.fp8_b = off;  // bf16 levels of B
        off = align256(off + (size_t)N * K * 2);
        pl.sfa = off;    // s_A [mt * 128][kbt]
        off = align256(off + (size_t)mt * kBM * kbt * 4);
        pl.sfb = off;    // s_B [nt][kbt][128]
        off = align256(off + (size_t)nt * kbt * kF32sBN * 4);
        pl.total = off;
        return pl;
    }
    pl.kind = (grid == 2 || grid == 3) ? (bc == 16 ? 2 : 1) : 0;  // E2M1 codes (grids 2, 3): native FP4
    if (pl.kind == 2 && (K / 2 + kBKBytes - 1) / kBKBytes >= kWideFp4MinKTiles) pl.kind = 4;
    pl.native = grid == 4;                                          // MXFP8: E4M3 bytes
    pl.bn = pair_bn(pl.kind);
    pl.k_bytes = (grid == 2 || grid == 3) ? K / 2 : K;
    pl.k_tiles = (pl.k_bytes + kBKBytes - 1) / kBKBytes;
    const int cps = pl.kind == 0 ? 1 : (pl.kind == 1 ? 2 : 4);
    pl.chunks_k = pl.k_tiles * cps;
    const int64_t mb = (M + 127) / 128;
    const int64_t nb = (N + pl.bn - 1) / pl.bn * ((pl.bn + 127) / 128);  // chunk blocks of B
    size_t off = 0;
    if (pl.kind == 0 && !pl.native) {
        pl.fp8_a = off;
        off = align256(off + (size_t)M * K);
        pl.fp8_b = off;
        off = align256(off + (size_t)N * K);
    }
    const size_t copies = pair_replicated(pl.kind) ? 4 : 1;
    pl.sfa = off;
    off = align256(off + (size_t)mb * pl.chunks_k * kChunkBytes * copies);
    pl.sfb = off;
    off = align256(off + (size_t)nb * pl.chunks_k * kChunkBytes * copies);
    pl.total = off;
    return pl;
}

// Co-resident two-CTA clusters of the pair kernel on this device (cached).
template <int KIND, int STAGES, int KPS, int G>
int pair_clusters(const cudaLaunchConfig_t& cfg) {
    static int cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<KIND, STAGES, KPS, G>, &cfg) != cudaSuccess) return 0;
    cached[dev] = n;
    return n;
}

template <int KIND, int STAGES, int KPS, int G>
cudaError_t run_gemm_pair(const PairMaps<G>& maps, const PairKParams<G>& kp, cudaStream_t st) {
    using C = PairCfg<KIND, STAGES, KPS>;
    auto k = gemm_pair_kernel<KIND, STAGES, KPS, G>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int max_clusters = pair_clusters<KIND, STAGES, KPS, G>(cfg);
    if (max_clusters <= 0) return cudaErrorLaunchOutOfResources;
    const int tiles = kp.num_tiles;
    cfg.gridDim = dim3(2 * (tiles < max_clusters ? tiles : max_clusters));  // persistent: one pair per two SMs
    cfg.numAttrs = st ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, k, maps, kp);
}

}  // namespace

bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr, uint64_t inner, uint64_t outer,
                   uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
    const cuuint64_t strides[1] = {(cuuint64_t)pitch_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int grid, int br, int bc, int sf) {
    return make_plan(M, N, K, grid, br, bc, sf).total;
}

// ------------------------------------------------ pair-kernel launches
// Shape checks and the plan of one GEMM of the pair kernel (kinds 0-2).
cudaError_t pair_plan(const GemmArgs& g, Plan& pl) {
    const bool fp4 = g.grid == 2 || g.grid == 3;
    if (g.K % 32 && !(fp4 && g.bc == 16)) return cudaErrorNotSupported;
    if (g.K % 64 && fp4) return cudaErrorNotSupported;  // FP4 rows must be 32-byte multiples
    pl = make_plan(g.M, g.N, g.K, g.grid, g.br, g.bc, g.sf);
    if (g.workspace_bytes < pl.total) return cudaErrorInvalidValue;
    return cudaSuccess;
}

cudaError_t gemm_prep_targets(const GemmArgs& g, PrepTarget out[2]) {
    Plan pl{};
    const cudaError_t e = pair_plan(g, pl);
    if (e != cudaSuccess) return e;
    if (pl.kind != 0 || pl.native) return cudaErrorNotSupported;
    // the quantizer zeroes the cells past a tile's short last part from that
    // part's first rows, so that part must hold at least half of its 128
    if (pl.bn % 128 != 0 && pl.bn % 128 < 64) return cudaErrorNotSupported;
    uint8_t* ws = (uint8_t*)g.workspace;
    for (int side = 0; side < 2; ++side) {
        PrepTarget& t = out[side];
        const int64_t rows = side ? g.N : g.M;
        t.fp8 = ws + (side ? pl.fp8_b : pl.fp8_a);
        t.chunks = ws + (side ? pl.sfb : pl.sfa);
        t.K = g.K;
        t.tile_rows = side ? pl.bn : kBM;
        t.parts = (t.tile_rows + 127) / 128;
        t.chunks_k = (int)pl.chunks_k;
        t.rows_cover = (int)((rows + t.tile_rows - 1) / t.tile_rows) * t.tile_rows;
    }
    return cudaSuccess;
}

// Operand prep of n <= kPairGroups GEMMs sharing the kind, in one launch:
// FP8 widening of E1M2 / INT4 (with the folded scale chunks), or the scale
// chunks alone for FP4 and MXFP8.
cudaError_t launch_prep_pair(const GemmArgs* gs, int n, cudaStream_t st) {
    if (n < 1 || n > kPairGroups) return cudaErrorInvalidValue;
    PrepParams pp{};
    int row_blocks = 0;
    int64_t kslabs = 0, items = 0;
    Plan pl{};
    for (int i = 0; i < n; ++i) {
        const GemmArgs& g = gs[i];
        const cudaError_t e = pair_plan(g, pl);
        if (e != cudaSuccess) return e;
        uint8_t* ws = (uint8_t*)g.workspace;
        for (int side = 0; side < 2; ++side) {
            const GemmOperand& op = side ? g.b : g.a;
            PrepSide& ps = pp.side[2 * i + side];
            ps.codes = op.codes;
            ps.scales = op.scales;
            ps.codes_ld = op.codes_ld;
            ps.scales_ld = op.scales_ld;
            ps.rows = (int)op.rows;
            ps.tile_rows = side ? pl.bn : kBM;
            ps.rows_cover = (int)((op.rows + ps.tile_rows - 1) / ps.tile_rows) * ps.tile_rows;  // whole output tiles
            ps.out_fp8 = (pl.kind == 0 && !pl.native) ? ws + (side ? pl.fp8_b : pl.fp8_a) : nullptr;
            ps.out_chunks = ws + (side ? pl.sfb : pl.sfa);
            ps.K = (int)g.K;
            ps.chunks_k = (int)pl.chunks_k;
            row_blocks = std::max(row_blocks, 16 * (ps.rows_cover / ps.tile_rows) * ((ps.tile_rows + 127) / 128));
            kslabs = std::max(kslabs, (pl.chunks_k * 4 + 63) / 64);
            items = std::max(items, (int64_t)(ps.rows_cover / ps.tile_rows) * ((ps.tile_rows + 127) / 128) *
                                        pl.chunks_k);
        }
    }
    // every GEMM of the launch has the same kind (same descriptor)
    pp.grid = gs[0].grid;
    pp.lbr = ilog2(gs[0].br);
    pp.lbc = ilog2(gs[0].bc);
    pp.lhw = (pl.kind == 2 || pl.kind == 4) ? 4 : 5;
    pp.copies = pair_replicated(pl.kind) ? 4 : 1;
    if (pl.kind == 0 && !pl.native) {
        // 64 groups of 32 elements per CTA along K; 16 CTAs per 128-row part of a GEMM tile
        if (kslabs > 65535) return cudaErrorNotSupported;  // grid y limit
        return launch_pdl(prep_widen_kernel, dim3((unsigned)row_blocks, (unsigned)kslabs, 2 * n), dim3(32, 8), 0,
                          st, pp);
    }
    // FP4 and MXFP8: only the scales move, one warp per (128-row part, chunk)
    const int64_t blocks = (items + 7) / 8;
    if (blocks > 0x7FFFFFFF) return cudaErrorNotSupported;
    return launch_pdl(prep_scales_kernel, dim3((unsigned)blocks, 1, 2 * n), dim3(32, 8), 0, st, pp);
}

// Tensor maps and parameters of one GEMM of a pair launch.
cudaError_t fill_pair_group(const GemmArgs& g, const Plan& pl, CUtensorMap* maps, PairGroup& pg) {
    uint8_t* ws = (uint8_t*)g.workspace;
    // E1M2 / INT4 read the widened copies in the workspace; FP4 and MXFP8
    // the codes themselves.
    const bool widened = pl.kind == 0 && !pl.native;
    const void* a_ptr = widened ? (const void*)(ws + pl.fp8_a) : (const void*)g.a.codes;
    const void* b_ptr = widened ? (const void*)(ws + pl.fp8_b) : (const void*)g.b.codes;
    const int64_t a_pitch = widened ? g.K : g.a.codes_ld;
    const int64_t b_pitch = widened ? g.K : g.b.codes_ld;
    // CTA pairs, 256 x bn tiles: A 128 rows per CTA, B bn/2 rows per CTA
    if (!make_map(&maps[0], a_ptr, g.M, pl.k_bytes, a_pitch, kBM)) return cudaErrorInvalidValue;
    if (!make_map(&maps[1], b_ptr, g.N, pl.k_bytes, b_pitch, pl.bn / 2)) return cudaErrorInvalidValue;
    // scale chunks as rows of 128 x 32-bit words (one 512-byte copy of a chunk
    // per row); boxes: one stage's chunks, rpc rows per chunk for A, 2 rpc for B
    const int cpk = pl.kind == 0 ? 1 : (pl.kind == 1 ? 2 : 4);
    const int kps = pl.kind == 0 ? kPairKps : 1;
    const int rpc = pair_replicated(pl.kind) ? 4 : 1;  // 512-byte rows per chunk
    const int64_t a_blocks = (g.M + kBM - 1) / kBM;
    const int64_t b_blocks = (g.N + pl.bn - 1) / pl.bn * 2;
    if (!encode_map_2d(&maps[2], CU_TENSOR_MAP_DATA_TYPE_UINT32, ws + pl.sfa, 128,
                       (uint64_t)(a_blocks * pl.chunks_k * rpc), kChunkBytes, 128, (uint32_t)(rpc * kps * cpk),
                       CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (!encode_map_2d(&maps[3], CU_TENSOR_MAP_DATA_TYPE_UINT32, ws + pl.sfb, 128,
                       (uint64_t)(b_blocks * pl.chunks_k * rpc), kChunkBytes, 128, (uint32_t)(2 * rpc * kps * cpk),
                       CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    pg.M = (int)g.M;
    pg.N = (int)g.N;
    pg.k_tiles = (int)pl.k_tiles;
    pg.m_pairs = (int)((g.M + 2 * kBM - 1) / (2 * kBM));
    pg.group_m = std::min(pg.m_pairs, kPairGroupM);
    pg.n_tiles = (int)((g.N + pl.bn - 1) / pl.bn);
    pg.sf_chunks_k = pl.chunks_k;
    pg.D = g.D;
    pg.ldd = g.ldd;
    pg.vec8 = ((uintptr_t)g.D % 32 == 0) && (g.ldd % 8 == 0);
    pg.amax_a = g.amax_a;
    pg.amax_b = g.amax_b;
    return cudaSuccess;
}

template <int G>
cudaError_t launch_main_pair_g(const GemmArgs* gs, int n, cudaStream_t st) {
    PairMaps<G> maps;
    std::memset(&maps, 0, sizeof(maps));
    PairKParams<G> kp;
    std::memset(&kp, 0, sizeof(kp));
    Plan pl{};
    int tiles = 0;
    for (int i = 0; i < n; ++i) {
        cudaError_t e = pair_plan(gs[i], pl);
        if (e != cudaSuccess) return e;
        e = fill_pair_group(gs[i], pl, maps.m[i], kp.g[i]);
        if (e != cudaSuccess) return e;
        kp.g[i].tile0 = tiles;
        tiles += kp.g[i].m_pairs * kp.g[i].n_tiles;
    }
    kp.ngroups = n;
    kp.num_tiles = tiles;
    if (tiles == 0) return cudaSuccess;
    const GemmArgs& g = gs[0];  // kind, grid and scale format are shared
    if (pl.kind == 0) {
        // E5M2 x E5M2 (format 1) for the widened codes, E4M3 x E4M3 (format 0) for MXFP8; M = 256
        const int fmt = pl.native ? 0 : 1;
        for (int j = 0; j < 4; ++j) kp.idesc[j] = make_idesc(fmt, fmt, 2 * kBM, kBnFp8, j);
        return run_gemm_pair<0, kPairStages, kPairKps, G>(maps, kp, st);
    }
    if (pl.kind == 1) {
        for (int j = 0; j < 4; ++j) kp.idesc[j] = make_idesc(1, 1, 2 * kBM, kBnFp4x2, (j % 2) * 2);  // E2M1
        return run_gemm_pair<1, kPairStagesFp4x2, 1, G>(maps, kp, st);
    }
    // scale_vec::4X: UE8M0 scales, or E4M3 ones (scale type bit 0) for the two-level format
    const bool two_level = g.sf == 2;
    for (int j = 0; j < 4; ++j) kp.idesc[j] = make_idesc(1, 1, 2 * kBM, pair_bn(pl.kind), 0, !two_level);
    kp.two_level = two_level;
    kp.den = grid_qmax_host(g.grid) * 448.0f;
    if (pl.kind == 4) return run_gemm_pair<4, kPairStagesFp4x4, 1, G>(maps, kp, st);
    return run_gemm_pair<2, kPairStagesFp4x4, 1, G>(maps, kp, st);
}

// The tensor-core kernel over one GEMM.  The kernel can walk the tiles of
// several GEMMs in one launch (G > 1, one set of tensor maps per GEMM in its
// parameters), but such launches stalled for minutes when they followed
// other GEMMs on a stream (a timing-dependent stall, not seen when run alone
// or with eager module loading), so every GEMM gets its own launch.
cudaError_t launch_main_pair(const GemmArgs* gs, int n, cudaStream_t st) {
    for (int i = 0; i < n; ++i) {
        const cudaError_t e = launch_main_pair_g<1>(&gs[i], 1, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Operand preparation: FP8 widening (E1M2/INT4) and scale chunks into the workspace.
cudaError_t launch_gemm_prep(const GemmArgs& g, cudaStream_t st) {
    if (g.sf == 0) {
        if (g.K % 128) return cudaErrorNotSupported;
        const Plan pl = make_plan(g.M, g.N, g.K, g.grid, g.br, g.bc, g.sf);
        if (g.workspace_bytes < pl.total) return cudaErrorInvalidValue;
        uint8_t* ws = (uint8_t*)g.workspace;
        F32sPrep pp{};
        pp.K = (int)g.K;
        pp.bc = g.bc;
        pp.grid = g.grid;
        for (int side = 0; side < 2; ++side) {
            const GemmOperand& op = side ? g.b : g.a;
            F32sSide& ps = pp.side[side];
            ps.codes = op.codes;
            ps.scales = reinterpret_cast<const float*>(op.scales);
            ps.codes_ld = op.codes_ld;
            ps.scales_ld = op.scales_ld;
            ps.rows = (int)op.rows;
            ps.tile_rows = side ? kF32sBN : kBM;
            ps.rows_cover = (int)((op.rows + ps.tile_rows - 1) / ps.tile_rows) * ps.tile_rows;
            ps.levels = reinterpret_cast<uint16_t*>(ws + (side ? pl.fp8_b : pl.fp8_a));
            ps.scales_out = reinterpret_cast<float*>(ws + (side ? pl.sfb : pl.sfa));
            ps.transposed = side;
        }
        const int64_t chunks = (int64_t)std::max(pp.side[0].rows_cover, pp.side[1].rows_cover) * (g.K / 16);
        const int64_t blocks = (chunks + 255) / 256;
        if (blocks > 0x7FFFFFFF) return cudaErrorNotSupported;
        return launch_pdl(prep_f32s_kernel, dim3((unsigned)blocks, 1, 2), dim3(256), 0, st, pp);
    }
    return launch_prep_pair(&g, 1, st);
}

// The tensor-core kernel on a workspace filled by launch_gemm_prep for the same arguments.
cudaError_t launch_gemm_main(const GemmArgs& g, int num_sms, cudaStream_t st) {
    if (g.sf == 0) {
        if (g.K % 128) return cudaErrorNotSupported;
        const Plan pl = make_plan(g.M, g.N, g.K, g.grid, g.br, g.bc, g.sf);
        if (g.workspace_bytes < pl.total) return cudaErrorInvalidValue;
        uint8_t* ws = (uint8_t*)g.workspace;
        const int64_t kbt = g.K / g.bc;
        const int kb = (int)(128 / g.bc);
        const int64_t mt = (g.M + kBM - 1) / kBM, nt = (g.N + kF32sBN - 1) / kF32sBN;
        CUtensorMap ma, mb, msa, msb;
        if (!make_map(&ma, ws + pl.fp8_a, g.M, g.K * 2, g.K * 2, kBM)) return cudaErrorInvalidValue;
        if (!make_map(&mb, ws + pl.fp8_b, g.N, g.K * 2, g.K * 2, kF32sBN)) return cudaErrorInvalidValue;
        if (!encode_map_2d(&msa, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ws + pl.sfa, (uint64_t)kbt, (uint64_t)(mt * kBM),
                           (uint64_t)kbt * 4, (uint32_t)kb, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        if (!encode_map_2d(&msb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, ws + pl.sfb, kF32sBN, (uint64_t)(nt * kbt),
                           kF32sBN * 4, kF32sBN, (uint32_t)kb, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
        F32sKParams kp{};
        kp.M = (int)g.M;
        kp.N = (int)g.N;
        kp.k_tiles = (int)(g.K / 128);
        kp.kb_per_tile = kb;
        kp.m_tiles = (int)mt;
        kp.n_tiles = (int)nt;
        kp.kb_pad = (int)kbt;
        kp.D = g.D;
        kp.ldd = g.ldd;
        kp.idesc = make_idesc_f16(kBM, kF32sBN);
        kp.mmas_per_block = g.bc / 16;
        auto k = gemm_f32s_kernel;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, F32sCfg::kSmem);
        if (e != cudaSuccess) return e;
        const int tiles = kp.m_tiles * kp.n_tiles;
        const int grid = tiles < num_sms ? tiles : num_sms;
        return launch_pdl(k, dim3(grid), dim3(kF32sThreads), (size_t)F32sCfg::kSmem, st, ma, mb, msa, msb, kp);
    }
    (void)num_sms;
    return launch_main_pair(&g, 1, st);
}

// One group of a grouped call: operand prep and tensor-core launch, or
// D = 0 for K = 0.
static cudaError_t launch_one_group(const GemmArgs& g, int num_sms, cudaStream_t st) {
    if (g.K == 0)
        return cudaMemset2DAsync(g.D, (size_t)g.ldd * sizeof(float), 0, (size_t)g.N * sizeof(float), (size_t)g.M, st);
    return launch_gemm(g, num_sms, st);
}

// Two streams per device that grouped calls spread their groups over, with
// the caller's stream; created on first use and kept for the process.
constexpr int kLanes = 2;
struct GroupLanes {
    cudaStream_t s[kLanes];
    bool ready;
};
static std::mutex g_lanes_mu;
static GroupLanes g_lanes[64];

// GEMMs sharing a descriptor, each with its own workspace region.  Every
// group on its own is a small GEMM whose last wave of tiles leaves much of the
// GPU idle, so the groups are dealt round-robin to the caller's stream and
// two internal streams: an event recorded on the caller's stream orders them
// after the caller's earlier work, and the caller's stream waits for events
// recorded on the internal streams after their last group.  The kernels of
// different groups never wait on one another; the whole fork, launch and join
// sequence of a call is enqueued under one lock, so every wait refers to work
// already enqueued.  Empty products are skipped and K = 0 gives D = 0.
// (Launching several GEMMs from one persistent grid was tried; it stalled for
// minutes when it followed other GEMMs with lazily loaded modules.)
cudaError_t launch_gemm_groups(const GemmArgs* gs, int n, int num_sms, cudaStream_t st) {
    int live = 0;
    for (int i = 0; i < n; ++i) live += gs[i].M > 0 && gs[i].N > 0;
    int dev = 0;
    if (live < 2 || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        for (int i = 0; i < n; ++i) {
            if (gs[i].M == 0 || gs[i].N == 0) continue;
            const cudaError_t e = launch_one_group(gs[i], num_sms, st);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    std::lock_guard<std::mutex> lock(g_lanes_mu);
    GroupLanes& L = g_lanes[dev];
    if (!L.ready) {
        for (int j = 0; j < kLanes; ++j) {
            const cudaError_t e = cudaStreamCreateWithFlags(&L.s[j], cudaStreamNonBlocking);
            if (e != cudaSuccess) {
                for (int k = 0; k < j; ++k) cudaStreamDestroy(L.s[k]);
                return e;
            }
        }
        L.ready = true;
    }
    cudaEvent_t fork = nullptr, join[kLanes] = {};
    cudaError_t e = cudaEventCreateWithFlags(&fork, cudaEventDisableTiming);
    for (int j = 0; j < kLanes && e == cudaSuccess; ++j) e = cudaEventCreateWithFlags(&join[j], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(fork, st);
    for (int j = 0; j < kLanes && e == cudaSuccess; ++j) e = cudaStreamWaitEvent(L.s[j], fork, 0);
    if (e == cudaSuccess) {
        const cudaStream_t lanes[kLanes + 1] = {st, L.s[0], L.s[1]};
        int k = 0;
        for (int i = 0; i < n && e == cudaSuccess; ++i) {
            if (gs[i].M == 0 || gs[i].N == 0) continue;
            e = launch_one_group(gs[i], num_sms, lanes[k++ % (kLanes + 1)]);
        }
        // join even after a failed launch, so that the caller's stream stays ordered after the lanes
        for (int j = 0; j < kLanes; ++j) {
            cudaError_t r = cudaEventRecord(join[j], L.s[j]);
            if (r == cudaSuccess) r = cudaStreamWaitEvent(st, join[j], 0);
            if (e == cudaSuccess) e = r;
        }
    }
    if (fork) cudaEventDestroy(fork);  // released once the recorded work completes
    for (int j = 0; j < kLanes; ++j)
        if (join[j]) cudaEventDestroy(join[j]);
    return e;
}

cudaError_t preload_gemm_kernels() {
    cudaFuncAttributes a;
    cudaFuncGetAttributes(&a, gemm_pair_kernel<0, kPairStages, kPairKps, 1>);
    cudaFuncGetAttributes(&a, gemm_pair_kernel<1, kPairStagesFp4x2, 1, 1>);
    cudaFuncGetAttributes(&a, gemm_pair_kernel<2, kPairStagesFp4x4, 1, 1>);
    cudaFuncGetAttributes(&a, gemm_pair_kernel<4, kPairStagesFp4x4, 1, 1>);
    cudaFuncGetAttributes(&a, gemm_f32s_kernel);
    cudaFuncGetAttributes(&a, prep_widen_kernel);
    cudaFuncGetAttributes(&a, prep_scales_kernel);
    return cudaFuncGetAttributes(&a, prep_f32s_kernel);
}

cudaError_t launch_gemm(const GemmArgs& g, int num_sms, cudaStream_t st) {
    const cudaError_t e = launch_gemm_prep(g, st);
    if (e != cudaSuccess) return e;
    return launch_gemm_main(g, num_sms, st);
}

}  // namespace ufp4

extern "C" ufp4_status ufp4_device_error(int32_t* code) {
    if (!code) return UFP4_ERR_INVALID_ARG;
    int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return UFP4_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, ufp4::g_device_error, sizeof(int)) != cudaSuccess) return UFP4_ERR_CUDA;
    const int zero = 0;
    if (v && cudaMemcpyToSymbol(ufp4::g_device_error, &zero, sizeof(int)) != cudaSuccess) return UFP4_ERR_CUDA;
    int q = 0;
    if (ufp4::quant_error_read_clear(&q) != cudaSuccess) return UFP4_ERR_CUDA;
    *code = v ? v : q;
    return *code ? UFP4_ERR_TIMEOUT : UFP4_OK;
}
