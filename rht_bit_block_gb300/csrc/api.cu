// C ABI of the UFP4 library (declared in include/ufp4.h): host-side argument
// validation, the sign vector, and dispatch to the kernels.  Nothing here
// allocates device memory; the only host state kept between calls is the
// per-device kernels-loaded flag below.
#include <algorithm>
#include <cmath>
#include <mutex>
#include <new>
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "../../include/ufp4.h"
#include "internal.h"

using namespace ufp4;

namespace {

// Host Philox4x32-10 (Salmon et al., SC'11) for the sign vector.
void philox_host(const uint32_t ctr[4], uint32_t k0, uint32_t k1, uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    for (int i = 0; i < 10; ++i) {
        if (i) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        const uint64_t p0 = (uint64_t)0xD2511F53u * c0;
        const uint64_t p1 = (uint64_t)0xCD9E8D57u * c2;
        const uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0;
        const uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1;
        c1 = (uint32_t)p1;
        c3 = (uint32_t)p0;
        c0 = n0;
        c2 = n2;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

// eps_i = 1 - 2 * (bit (i % 32) of word (i % 128) / 32 of Philox(sign_seed, (i/128, 0, 2, 0))).
int sign_bit(uint64_t seed, int i) {
    const uint32_t ctr[4] = {(uint32_t)(i / 128), 0u, 2u, 0u};
    uint32_t w[4];
    philox_host(ctr, (uint32_t)seed, (uint32_t)(seed >> 32), w);
    return (int)((w[(i % 128) / 32] >> (i % 32)) & 1u);
}

// Bit i (0..255) set <=> eps_{i mod n} = -1.  n = 1 switches the transform off.
void make_sign_bits(uint64_t seed, int n, uint32_t bits[8]) {
    std::memset(bits, 0, 8 * sizeof(uint32_t));
    if (n <= 1) return;
    int base[256];
    for (int i = 0; i < n; ++i) base[i] = sign_bit(seed, i);
    for (int i = 0; i < 256; ++i)
        if (base[i % n]) bits[i / 32] |= 1u << (i % 32);
}

// The ten round keys of Philox4x32-10 (Salmon et al., SC'11) for a seed.
SrKeys sr_round_keys(uint64_t seed) {
    SrKeys k;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
    for (int i = 0; i < 10; ++i) {
        k.k[2 * i] = k0;
        k.k[2 * i + 1] = k1;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return k;
}

bool is_pow2(int64_t v) { return v >= 1 && (v & (v - 1)) == 0; }

float inv_sqrt_n(int n) { return (float)(1.0 / std::sqrt((double)n)); }

// Loads every kernel of the library on the current device, once, before the
// library's first launch there (see the preload functions).
void ensure_loaded() {
    static std::mutex mu;
    static bool done[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return;
    preload_quantize_kernels();
    preload_gemm_kernels();
    preload_dequant_kernels();
    preload_stats_kernels();
    preload_round_levels_kernels();
    cudaGetLastError();  // a failed query shows up again at the launch
    done[dev] = true;
}

// SM count of the current device; every launch path asks for it right before
// launching, so it also makes sure the kernels are loaded.
int num_sms_current() {
    ensure_loaded();
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p % a) == 0; }

struct BlockShape {
    bool is2d;
    int b2d;   // side of 2-D blocks
    int bw;    // width along the quantized dimension
};

ufp4_status check_desc(const ufp4_quant_desc* d, BlockShape* bs) {
    if (!d) return UFP4_ERR_INVALID_ARG;
    if (d->grid < 0 || d->grid > 4 || d->round < 0 || d->round > 1 || d->scale_fmt < 0 || d->scale_fmt > 2)
        return UFP4_ERR_INVALID_ARG;
    if (!is_pow2(d->hadamard_n) || d->hadamard_n > 256) return UFP4_ERR_INVALID_ARG;
    // MXFP8: 1 x 32 blocks with E8M0 scales, rounded to nearest
    if (d->grid == UFP4_GRID_MXFP8 && (d->block_rows != 1 || d->block_cols != 32 ||
                                       d->scale_fmt != UFP4_SCALE_UE8M0 || d->round != UFP4_ROUND_RTNE))
        return UFP4_ERR_UNSUPPORTED;
    if (d->block_rows == 1 && (d->block_cols == 16 || d->block_cols == 32)) {
        *bs = {false, 0, d->block_cols};
    } else if (d->block_rows == d->block_cols &&
               (d->block_rows == 8 || d->block_rows == 16 || d->block_rows == 32 || d->block_rows == 64)) {
        if (d->scale_fmt != UFP4_SCALE_UE8M0) return UFP4_ERR_INVALID_ARG;  // 2-D blocks: power-of-two scale
        *bs = {true, d->block_rows, d->block_rows};
    } else {
        return UFP4_ERR_INVALID_ARG;
    }
    return UFP4_OK;
}

ufp4_status check_out(const ufp4_qtensor* q, int64_t rows, int64_t cols, const BlockShape& bs,
                      int scale_fmt, bool grouped, int grid) {
    if (!q || !q->codes || !q->scales) return UFP4_ERR_INVALID_ARG;
    if (q->rows != rows || q->cols != cols) return UFP4_ERR_INVALID_ARG;
    if (!aligned(q->codes, 16)) return UFP4_ERR_ALIGNMENT;
    if (!aligned(q->scales, scale_fmt == UFP4_SCALE_FP32 ? 4 : 1)) return UFP4_ERR_ALIGNMENT;
    if (scale_fmt == UFP4_SCALE_E4M3 && !q->tensor_amax) return UFP4_ERR_INVALID_ARG;
    if (scale_fmt == UFP4_SCALE_E4M3 && !aligned(q->tensor_amax, 4)) return UFP4_ERR_ALIGNMENT;
    if (grouped) return UFP4_OK;
    const bool bytes = grid == UFP4_GRID_MXFP8;  // one byte per code
    if (q->codes_ld % (bytes ? 16 : 8)) return UFP4_ERR_ALIGNMENT;
    if (q->codes_ld < (bytes ? cols : cols / 2)) return UFP4_ERR_INVALID_ARG;
    const int64_t sc_cols = cols / bs.bw;
    if (q->scales_ld < sc_cols) return UFP4_ERR_INVALID_ARG;
    return UFP4_OK;
}

ufp4_status cuda_status(cudaError_t e) { return e == cudaSuccess ? UFP4_OK : UFP4_ERR_CUDA; }

// Shared body of the plain and grouped quantizer calls.
// Row-wise quantization of `count` tensors in one launch of the lean kernel
// (arguments already validated).
// prep (optional, one per tensor): also write each tensor's prepared GEMM
// operand there; its tiles then run over the rows of whole GEMM tiles.
ufp4_status quantize_rows_batch(int count, const void* const* x, const int64_t* rows, const int64_t* cols,
                                const int64_t* ld, const ufp4_quant_desc* desc, const BlockShape& bs,
                                const ufp4_qtensor* rowwise, cudaStream_t stream,
                                const PrepTarget* prep = nullptr) {
    RowsParams p;
    std::memset(&p, 0, sizeof(p));
    auto ilog2 = [](int v) { int l = 0; while ((1 << l) < v) ++l; return l; };
    const int n = desc->hadamard_n;
    // tile columns and rows: 16 K elements, or 8 K (one row pair per thread) with 2-D blocks in the
    // row kernel; n = 64 and n = 256 run the segment kernel, 16 K-element tiles either way
    const bool seg = n == 64 || n == 256;
    const int tc = n == 256 ? 256 : 128, tr = bs.is2d && !seg ? 2 * (256 / (tc / 16)) : 16384 / tc;
    int64_t tiles = 0;
    int k = 0;
    for (int i = 0; i < count; ++i) {
        if (rows[i] == 0 || cols[i] == 0) continue;  // empty tensors take no tiles
        RowsTensor& T = p.t[k++];
        T.x = (const uint16_t*)x[i];
        T.ld = ld[i];
        T.codes = (uint8_t*)rowwise[i].codes;
        T.scales = (uint8_t*)rowwise[i].scales;
        T.codes_ld = rowwise[i].codes_ld;
        T.scales_ld = rowwise[i].scales_ld;
        T.rows = (int)rows[i];
        T.cols = (int)cols[i];
        T.col_tiles = (int)((cols[i] + tc - 1) / tc);
        T.row_tiles = (int)((rows[i] + tr - 1) / tr);
        if (prep) {
            T.prep = prep[i];
            T.row_tiles = (int)((std::max<int64_t>(rows[i], prep[i].rows_cover) + tr - 1) / tr);
        }
        T.tile0 = (int)tiles;
        T.amax = rowwise[i].tensor_amax;
        tiles += (int64_t)T.col_tiles * T.row_tiles;
    }
    if (k == 0) return UFP4_OK;
    if (tiles > 0x7FFFFFFF) return UFP4_ERR_UNSUPPORTED;
    p.count = k;
    p.num_tiles = (int)tiles;
    p.tc = tc;
    p.tr = tr;
    p.lb2d = 0;
    if (bs.is2d)
        while ((1 << p.lb2d) < bs.b2d) ++p.lb2d;
    p.n = n;
    p.lbw = ilog2(bs.bw);
    p.log4n = 0;
    while ((1 << (2 * p.log4n)) < n) ++p.log4n;
    p.pow4 = (1 << (2 * p.log4n)) == n;
    p.stages = 0;  // set by the launcher (the ring depth depends on the kernel it picks)
    p.inv_sqrt_n = inv_sqrt_n(n);
    make_sign_bits(desc->sign_seed, n, p.sign_bits);
    for (int j = 0; j < 64; ++j) p.smask[j] = ((p.sign_bits[j / 32] >> (j % 32)) & 1u) << 31;
    p.sr_seed = desc->round == UFP4_ROUND_SR ? desc->sr_seed : 0;
    p.sr_keys = sr_round_keys(p.sr_seed);
    p.group = desc->group;
    p.prep = prep ? 1 : 0;
    if (desc->scale_fmt == UFP4_SCALE_E4M3)  // two-level: the tensor amax pre-pass first
        for (int i = 0; i < k; ++i) {
            const RowsTensor& T = p.t[i];
            const cudaError_t e = launch_tensor_amax(T.x, T.rows, T.cols, T.ld, n, p.inv_sqrt_n, p.sign_bits,
                                                     const_cast<float*>(T.amax), num_sms_current(), stream);
            if (e != cudaSuccess) return UFP4_ERR_CUDA;
        }
    return cuda_status(launch_quantize_rows(p, desc->grid, desc->round == UFP4_ROUND_SR, desc->scale_fmt,
                                            num_sms_current(), stream));
}

ufp4_status quantize_common(const void* x, int64_t cols, int64_t ld, const int64_t* offsets, int ngroups,
                            bool grouped, const ufp4_quant_desc* desc, const ufp4_qtensor* rowwise,
                            const ufp4_qtensor* colwise, cudaStream_t stream) {
    BlockShape bs;
    ufp4_status st = check_desc(desc, &bs);
    if (st != UFP4_OK) return st;
    if (cols < 0 || ngroups < 1 || ngroups > kMaxGroups) return UFP4_ERR_INVALID_ARG;
    if (desc->out_mask < 1 || desc->out_mask > 3) return UFP4_ERR_INVALID_ARG;
    if (offsets[ngroups] == 0 || cols == 0) return UFP4_OK;  // empty input: nothing to do (pointers, ld unused)
    if (ld < cols) return UFP4_ERR_INVALID_ARG;
    if (!x) return UFP4_ERR_INVALID_ARG;
    const bool do_row = desc->out_mask & UFP4_OUT_ROWWISE;
    const bool do_col = desc->out_mask & UFP4_OUT_COLWISE;
    const int n = desc->hadamard_n;
    if (grouped && bs.is2d) return UFP4_ERR_UNSUPPORTED;
    if (do_col && n > 128) return UFP4_ERR_UNSUPPORTED;  // column pass keeps n <= 128
    if (!aligned(x, 16) || ld % 8) return UFP4_ERR_ALIGNMENT;
    const int64_t total_rows = offsets[ngroups];
    if (offsets[0] != 0 || total_rows < 0) return UFP4_ERR_INVALID_ARG;
    for (int g = 0; g < ngroups; ++g)
        if (offsets[g + 1] < offsets[g]) return UFP4_ERR_INVALID_ARG;
    // shape rules
    if (cols % 16) return UFP4_ERR_INVALID_ARG;
    if (do_row && (cols % n || cols % bs.bw)) return UFP4_ERR_INVALID_ARG;
    if (bs.is2d && (total_rows % bs.b2d || cols % bs.b2d)) return UFP4_ERR_INVALID_ARG;
    const int64_t unit = grouped ? (int64_t)std::max<int>(std::max(n, bs.bw), 64) : 1;
    int64_t padded_total = 0;
    int64_t pad0[kMaxGroups + 1];
    pad0[0] = 0;
    for (int g = 0; g < ngroups; ++g) {
        const int64_t c = offsets[g + 1] - offsets[g];
        const int64_t pc = grouped ? ((c + unit - 1) / unit) * unit : c;
        pad0[g + 1] = pad0[g] + pc;
    }
    padded_total = pad0[ngroups];
    if (do_col && !grouped && (total_rows % 16 || total_rows % n || total_rows % bs.bw))
        return UFP4_ERR_INVALID_ARG;
    if (do_row) {
        st = check_out(rowwise, total_rows, cols, bs, desc->scale_fmt, false, desc->grid);
        if (st != UFP4_OK) return st;
    }
    if (do_col) {
        st = check_out(colwise, cols, padded_total, bs, desc->scale_fmt, grouped, desc->grid);
        if (st != UFP4_OK) return st;
    }
    if (total_rows == 0 || cols == 0) return UFP4_OK;

    if ((desc->scale_fmt == UFP4_SCALE_E4M3 || desc->grid == UFP4_GRID_MXFP8) &&
        (do_col || grouped || bs.is2d || n > 128 || total_rows >= (1LL << 31) || cols >= (1LL << 31)))
        return UFP4_ERR_UNSUPPORTED;  // two-level scale and MXFP8: row-wise, 1-D blocks, n <= 128
    // the row kernels: row-wise, not grouped; 1-D blocks, or b x b blocks with b = 16, 32 or 64
    const bool rows_2d = bs.is2d && bs.b2d >= 16;
    if (do_row && !do_col && (!bs.is2d || rows_2d) && !grouped && total_rows < (1LL << 31) &&
        cols < (1LL << 31)) {
        const ufp4_qtensor* rw = rowwise;
        return quantize_rows_batch(1, &x, &total_rows, &cols, &ld, desc, bs, rw, stream);
    }

    QuantParams p;
    std::memset(&p, 0, sizeof(p));
    const int tc = (n == 256) ? 256 : 128;
    const int seg_lanes = (bs.is2d ? std::max(n, 16) : std::max(std::max(n, bs.bw), 16)) / 16;
    // row-only work takes 128-row tiles (more elements per thread per tile);
    // the column pass takes 64-row tiles unless a segment spans 8 row chunks
    // 2-D blocks take 64-row tiles where they can: one row pair (and one
    // column task) per thread, whose values stay in registers across the
    // block-amax barrier
    int tr = (do_col && seg_lanes < 8) ? 64 : ((n == 256 || (bs.is2d && !do_col)) ? 64 : 128);
    if (do_col && seg_lanes < 8 && !bs.is2d) {
        // 1-D blocks: 128-row tiles give each warp two column tasks per tile
        // (more work per tile barrier) where the walk still has about four
        // waves of tiles for the three CTAs per SM; small tensors keep 64
        int64_t t128 = 0;
        for (int g = 0; g < ngroups; ++g) t128 += (pad0[g + 1] - pad0[g] + 127) / 128;
        if (t128 * ((cols + tc - 1) / tc) >= 12LL * num_sms_current()) tr = 128;
    }
    p.x = (const uint16_t*)x;
    p.cols = cols;
    p.ld = ld;
    p.n = n;
    p.inv_sqrt_n = inv_sqrt_n(n);
    make_sign_bits(desc->sign_seed, n, p.sign_bits);
    for (int j = 0; j < 16; ++j) p.smask16[j] = ((p.sign_bits[0] >> j) & 1u) << 31;
    p.is2d = bs.is2d;
    p.b2d = bs.b2d;
    p.bw_row = bs.bw;
    p.bw_col = bs.bw;
    p.col_seg_lanes = seg_lanes;
    p.amax_slots = bs.is2d ? (tr / bs.b2d) * (tc / bs.b2d) : 0;
    p.tile_rows = tr;
    p.stages = 0;  // set by the launcher (the ring depth depends on the block shape)
    auto ilog2 = [](int v) { int l = 0; while ((1 << l) < v) ++l; return l; };
    p.lbw_row = ilog2(bs.bw);
    p.lbw_col = ilog2(bs.bw);
    p.lb2d = bs.is2d ? ilog2(bs.b2d) : 0;
    p.lseg = ilog2(seg_lanes);
    p.log4n = 0;
    while ((1 << (2 * p.log4n)) < n) ++p.log4n;
    p.pow4 = (1 << (2 * p.log4n)) == n;
    p.sr_seed = desc->round == UFP4_ROUND_SR ? desc->sr_seed : 0;
    p.sr_keys = sr_round_keys(p.sr_seed);
    p.do_row = do_row;
    p.do_col = do_col;
    p.vec256 = aligned(x, 32) && (ld % 16 == 0);
    p.col_grouped = grouped;
    if (do_row) p.row = {rowwise->codes, rowwise->scales, rowwise->codes_ld, rowwise->scales_ld};
    if (do_col) p.col = {colwise->codes, colwise->scales, colwise->codes_ld, colwise->scales_ld};
    p.col_tiles = (int)((cols + tc - 1) / tc);
    p.num_groups = ngroups;
    int64_t tiles = 0;
    for (int g = 0; g <= ngroups; ++g) {
        p.grp_row0[g] = offsets[g];
        p.grp_pad0[g] = pad0[g];
        p.grp_tile0[g] = (int)tiles;
        if (g < ngroups) {
            // the tile walk covers the padded rows when the column pass needs them
            const int64_t len = do_col ? pad0[g + 1] - pad0[g] : offsets[g + 1] - offsets[g];
            tiles += (len + tr - 1) / tr;
        }
    }
    const int64_t num_tiles = tiles * p.col_tiles;
    if (num_tiles == 0) return UFP4_OK;
    if (num_tiles > 0x7FFFFFFF) return UFP4_ERR_UNSUPPORTED;
    p.group_base = grouped ? 0 : desc->group;
    return cuda_status(launch_quantize(p, desc->grid, desc->round == UFP4_ROUND_SR,
                                       desc->scale_fmt == UFP4_SCALE_UE8M0, tc, tr, (int)num_tiles, total_rows,
                                       num_sms_current(), stream));
}

// Checks one GEMM call and fills its launch arguments (nothing is launched).
ufp4_status prepare_gemm(const ufp4_qtensor* A, const ufp4_qtensor* B, const ufp4_quant_desc* desc, float* D,
                         int64_t ldd, void* workspace, size_t workspace_bytes, GemmArgs* out) {
    BlockShape bs;
    ufp4_status st = check_desc(desc, &bs);
    if (st != UFP4_OK) return st;
    if (!A || !B) return UFP4_ERR_INVALID_ARG;
    const bool two_level = desc->scale_fmt == UFP4_SCALE_E4M3;
    // UE8M0 block scales; the two-level scale only for E2M1 codes in 1 x 16 blocks (native FP4 with E4M3 scales)
    const bool fp32_scales = desc->scale_fmt == UFP4_SCALE_FP32;  // 1-D blocks only (check_desc)
    if (desc->scale_fmt != UFP4_SCALE_UE8M0 && !fp32_scales &&
        !(two_level && desc->grid >= UFP4_GRID_E2M1 && !bs.is2d && bs.bw == 16))
        return UFP4_ERR_UNSUPPORTED;
    if (fp32_scales && A->cols % 128) return UFP4_ERR_UNSUPPORTED;  // the fp32-scale path walks 128-element K tiles
    if (bs.is2d && bs.b2d != 32) return UFP4_ERR_UNSUPPORTED;
    const int64_t M = A->rows, N = B->rows, K = A->cols;
    if (B->cols != K || M < 0 || N < 0 || K < 0 || ldd < N) return UFP4_ERR_INVALID_ARG;
    if (M > (1LL << 30) || N > (1LL << 30) || K > (1LL << 30)) return UFP4_ERR_UNSUPPORTED;  // 32-bit indexing
    if (M > 0 && N > 0 && !D) return UFP4_ERR_INVALID_ARG;
    if (K % 32 && !(bs.bw == 16 && K % 16 == 0)) return UFP4_ERR_INVALID_ARG;
    std::memset(out, 0, sizeof(*out));
    out->M = M;
    out->N = N;
    out->K = K;
    out->D = D;
    out->ldd = ldd;
    if (M == 0 || N == 0) return UFP4_OK;  // nothing to compute
    if (!aligned(D, 16) || ldd % 4) return UFP4_ERR_ALIGNMENT;
    if (K == 0) return UFP4_OK;  // D = 0 (written by run_prepared_gemm)
    st = check_out(A, M, K, bs, desc->scale_fmt, false, desc->grid);
    if (st != UFP4_OK) return st;
    st = check_out(B, N, K, bs, desc->scale_fmt, false, desc->grid);
    if (st != UFP4_OK) return st;
    if (A->codes_ld % 16 || B->codes_ld % 16) return UFP4_ERR_ALIGNMENT;  // TMA row pitch
    const size_t need = gemm_workspace_bytes(M, N, K, desc->grid, bs.is2d ? bs.b2d : 1, bs.bw, desc->scale_fmt);
    if (workspace_bytes < need || (need && !workspace)) return UFP4_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return UFP4_ERR_ALIGNMENT;
    out->a = {(const uint8_t*)A->codes, (const uint8_t*)A->scales, M, A->codes_ld, A->scales_ld};
    out->b = {(const uint8_t*)B->codes, (const uint8_t*)B->scales, N, B->codes_ld, B->scales_ld};
    out->grid = desc->grid;
    out->br = bs.is2d ? bs.b2d : 1;
    out->bc = bs.bw;
    out->sf = desc->scale_fmt;
    out->amax_a = A->tensor_amax;
    out->amax_b = B->tensor_amax;
    out->workspace = workspace;
    out->workspace_bytes = workspace_bytes;
    return UFP4_OK;
}

ufp4_status run_prepared_gemm(const GemmArgs& g, cudaStream_t stream) {
    if (g.M == 0 || g.N == 0) return UFP4_OK;
    if (g.K == 0)  // an empty sum: D = 0
        return cuda_status(cudaMemset2DAsync(g.D, (size_t)g.ldd * sizeof(float), 0, (size_t)g.N * sizeof(float),
                                             (size_t)g.M, stream));
    const cudaError_t e = launch_gemm(g, num_sms_current(), stream);
    if (e == cudaErrorNotSupported) return UFP4_ERR_UNSUPPORTED;
    return cuda_status(e);
}

}  // namespace

extern "C" {

const char* ufp4_status_string(ufp4_status s) {
    switch (s) {
        case UFP4_OK: return "UFP4_OK";
        case UFP4_ERR_INVALID_ARG: return "UFP4_ERR_INVALID_ARG";
        case UFP4_ERR_UNSUPPORTED: return "UFP4_ERR_UNSUPPORTED";
        case UFP4_ERR_ALIGNMENT: return "UFP4_ERR_ALIGNMENT";
        case UFP4_ERR_CUDA: return "UFP4_ERR_CUDA";
        case UFP4_ERR_TIMEOUT: return "UFP4_ERR_TIMEOUT";
    }
    return "UFP4_ERR_UNKNOWN";
}

ufp4_status ufp4_set_quantize_wait_limit(int64_t polls) {
    if (polls > (int64_t)0xFFFFFFFF) return UFP4_ERR_INVALID_ARG;
    ensure_loaded();
    if (cudaDeviceSynchronize() != cudaSuccess) return UFP4_ERR_CUDA;
    return cuda_status(set_quant_wait_limit(polls < 0 ? quant_wait_limit_default() : (uint32_t)polls));
}

ufp4_status ufp4_sign_vector(uint64_t sign_seed, int32_t n, int8_t* out_host) {
    if (!out_host || !is_pow2(n) || n > 256) return UFP4_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) out_host[i] = (n == 1) ? 1 : (int8_t)(1 - 2 * sign_bit(sign_seed, i));
    return UFP4_OK;
}

ufp4_status ufp4_round_levels(int32_t grid, int32_t rounding, int32_t scale_fmt, const float* t,
                              const uint16_t* u16, int64_t count, uint8_t* codes, cudaStream_t stream) {
    if (grid < UFP4_GRID_E1M2 || grid > UFP4_GRID_E2M1_R2) return UFP4_ERR_INVALID_ARG;
    if (rounding != UFP4_ROUND_RTNE && rounding != UFP4_ROUND_SR) return UFP4_ERR_INVALID_ARG;
    if (scale_fmt != UFP4_SCALE_FP32 && scale_fmt != UFP4_SCALE_UE8M0) return UFP4_ERR_INVALID_ARG;
    if (count < 0 || count % 32 != 0) return UFP4_ERR_INVALID_ARG;
    if (count == 0) return UFP4_OK;
    const bool sr = rounding == UFP4_ROUND_SR;
    if (!t || !codes || (sr && !u16)) return UFP4_ERR_INVALID_ARG;
    if ((uintptr_t)t % 16 || (uintptr_t)codes % 8 || (sr && (uintptr_t)u16 % 4)) return UFP4_ERR_ALIGNMENT;
    ensure_loaded();
    return cuda_status(launch_round_levels(grid, sr, scale_fmt, t, sr ? u16 : nullptr, count, codes, stream));
}

ufp4_status ufp4_rht_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, const ufp4_quant_desc* desc,
                              const ufp4_qtensor* rowwise, const ufp4_qtensor* colwise, cudaStream_t stream) {
    if (rows < 0 || !desc) return UFP4_ERR_INVALID_ARG;
    if (desc->group < 0) return UFP4_ERR_INVALID_ARG;
    const int64_t offsets[2] = {0, rows};
    return quantize_common(x, cols, ld, offsets, 1, false, desc, rowwise, colwise, stream);
}

extern "C" ufp4_status ufp4_rht_quantize_batch(int32_t count, const void* const* x, const int64_t* rows,
                                               const int64_t* cols, const int64_t* ld, const ufp4_quant_desc* desc,
                                               const ufp4_qtensor* rowwise, cudaStream_t stream) {
    BlockShape bs;
    ufp4_status st = check_desc(desc, &bs);
    if (st != UFP4_OK) return st;
    if (count < 0 || count > UFP4_MAX_BATCH) return UFP4_ERR_INVALID_ARG;
    if (count == 0) return UFP4_OK;
    if (!x || !rows || !cols || !ld || !rowwise) return UFP4_ERR_INVALID_ARG;
    if (desc->out_mask != UFP4_OUT_ROWWISE) return UFP4_ERR_INVALID_ARG;
    if (bs.is2d) return UFP4_ERR_UNSUPPORTED;
    if (desc->hadamard_n > 128 && (desc->scale_fmt == UFP4_SCALE_E4M3 || desc->grid == UFP4_GRID_MXFP8))
        return UFP4_ERR_UNSUPPORTED;  // two-level scale and MXFP8: n <= 128
    const int n = desc->hadamard_n;
    for (int i = 0; i < count; ++i) {
        if (rows[i] < 0 || cols[i] < 0) return UFP4_ERR_INVALID_ARG;
        if (rows[i] >= (1LL << 31) || cols[i] >= (1LL << 31)) return UFP4_ERR_UNSUPPORTED;
        if (rows[i] == 0 || cols[i] == 0) continue;  // empty: its pointers and leading dimension are not used
        if (ld[i] < cols[i]) return UFP4_ERR_INVALID_ARG;
        if (!x[i]) return UFP4_ERR_INVALID_ARG;
        if (!aligned(x[i], 16) || ld[i] % 8) return UFP4_ERR_ALIGNMENT;
        if (cols[i] % 16 || cols[i] % n || cols[i] % bs.bw) return UFP4_ERR_INVALID_ARG;
        st = check_out(&rowwise[i], rows[i], cols[i], bs, desc->scale_fmt, false, desc->grid);
        if (st != UFP4_OK) return st;
    }
    return quantize_rows_batch(count, x, rows, cols, ld, desc, bs, rowwise, stream);
}

extern "C" ufp4_status ufp4_rht_quantize_prepare(const void* a, int64_t lda, const void* b, int64_t ldb,
                                                 const ufp4_quant_desc* desc, const ufp4_qtensor* A,
                                                 const ufp4_qtensor* B, void* workspace, size_t workspace_bytes,
                                                 cudaStream_t stream) {
    BlockShape bs;
    ufp4_status st = check_desc(desc, &bs);
    if (st != UFP4_OK) return st;
    if (!A || !B) return UFP4_ERR_INVALID_ARG;
    if (desc->out_mask != UFP4_OUT_ROWWISE) return UFP4_ERR_INVALID_ARG;
    if ((desc->grid != UFP4_GRID_E1M2 && desc->grid != UFP4_GRID_INT4) || desc->scale_fmt != UFP4_SCALE_UE8M0 ||
        bs.is2d || desc->hadamard_n != 16)
        return UFP4_ERR_UNSUPPORTED;
    // the GEMM's rules (shapes, alignment, workspace); D is not touched here
    GemmArgs g;
    float dummy_d[4] __attribute__((aligned(16)));
    st = prepare_gemm(A, B, desc, dummy_d, B->rows, workspace, workspace_bytes, &g);
    if (st != UFP4_OK) return st;
    // the quantizer's rules, as ufp4_rht_quantize_batch checks them
    const void* const xs[2] = {a, b};
    const int64_t rows[2] = {A->rows, B->rows}, cols[2] = {A->cols, B->cols}, lds[2] = {lda, ldb};
    const ufp4_qtensor outs[2] = {*A, *B};
    for (int i = 0; i < 2; ++i) {
        if (rows[i] == 0 || cols[i] == 0) continue;
        if (lds[i] < cols[i] || !xs[i]) return UFP4_ERR_INVALID_ARG;
        if (!aligned(xs[i], 16) || lds[i] % 8) return UFP4_ERR_ALIGNMENT;
        if (cols[i] % 16 || cols[i] % bs.bw) return UFP4_ERR_INVALID_ARG;
    }
    if (g.M == 0 || g.N == 0 || g.K == 0)  // no GEMM operand to prepare
        return quantize_rows_batch(2, xs, rows, cols, lds, desc, bs, outs, stream);
    PrepTarget targets[2];
    const cudaError_t e = gemm_prep_targets(g, targets);
    if (e == cudaErrorNotSupported) return UFP4_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return UFP4_ERR_INVALID_ARG;
    return quantize_rows_batch(2, xs, rows, cols, lds, desc, bs, outs, stream, targets);
}

int64_t ufp4_grouped_padded_rows(int64_t rows, const ufp4_quant_desc* desc) {
    if (!desc || rows < 0) return -1;
    int bw = desc->block_rows == 1 ? desc->block_cols : desc->block_rows;
    const int64_t unit = std::max<int64_t>(std::max<int64_t>(desc->hadamard_n, bw), 64);
    return ((rows + unit - 1) / unit) * unit;
}

ufp4_status ufp4_rht_quantize_grouped(const void* x, int64_t cols, int64_t ld, const int64_t* offsets,
                                      int32_t num_groups, const ufp4_quant_desc* desc,
                                      const ufp4_qtensor* rowwise, const ufp4_qtensor* colwise,
                                      cudaStream_t stream) {
    if (!offsets || num_groups < 1) return UFP4_ERR_INVALID_ARG;
    return quantize_common(x, cols, ld, offsets, num_groups, true, desc, rowwise, colwise, stream);
}

ufp4_status ufp4_rht_transform(const void* x, int64_t rows, int64_t cols, int64_t ld, int32_t n,
                               uint64_t sign_seed, float* z, int64_t ldz, cudaStream_t stream) {
    if (!x || !z || rows < 0 || cols < 0 || ld < cols || ldz < cols) return UFP4_ERR_INVALID_ARG;
    if (!is_pow2(n) || n > 256 || cols % 16 || cols % n) return UFP4_ERR_INVALID_ARG;
    if (!aligned(x, 16) || ld % 8 || !aligned(z, 16) || ldz % 4) return UFP4_ERR_ALIGNMENT;
    if (rows == 0 || cols == 0) return UFP4_OK;
    SignBits sb;
    make_sign_bits(sign_seed, n, sb.bits);
    return cuda_status(launch_rht((const uint16_t*)x, rows, cols, ld, n, inv_sqrt_n(n), sb, z, ldz,
                                  num_sms_current(), stream));
}

ufp4_status ufp4_dequantize(const ufp4_qtensor* q, const ufp4_quant_desc* desc, int32_t inverse_rht, float* out,
                            int64_t ld_out, cudaStream_t stream) {
    BlockShape bs;
    ufp4_status st = check_desc(desc, &bs);
    if (st != UFP4_OK) return st;
    if (!q || !out || q->rows < 0 || q->cols < 0 || ld_out < q->cols) return UFP4_ERR_INVALID_ARG;
    if (q->cols % 16 || q->cols % bs.bw || (bs.is2d && q->rows % bs.b2d)) return UFP4_ERR_INVALID_ARG;
    if (inverse_rht && q->cols % desc->hadamard_n) return UFP4_ERR_INVALID_ARG;
    st = check_out(q, q->rows, q->cols, bs, desc->scale_fmt, false, desc->grid);
    if (st != UFP4_OK) return st;
    if (q->rows == 0 || q->cols == 0) return UFP4_OK;
    DequantParams p;
    std::memset(&p, 0, sizeof(p));
    p.codes = (const uint8_t*)q->codes;
    p.scales = q->scales;
    p.rows = q->rows;
    p.cols = q->cols;
    p.codes_ld = q->codes_ld;
    p.scales_ld = q->scales_ld;
    p.grid = desc->grid;
    p.br = bs.is2d ? bs.b2d : 1;
    p.bc = bs.bw;
    p.sf = desc->scale_fmt;
    p.amax = q->tensor_amax;
    p.n = desc->hadamard_n;
    p.inverse = inverse_rht ? 1 : 0;
    p.inv_sqrt_n = inv_sqrt_n(desc->hadamard_n);
    make_sign_bits(desc->sign_seed, desc->hadamard_n, p.sign_bits);
    p.out = out;
    p.ld_out = ld_out;
    return cuda_status(launch_dequantize(p, num_sms_current(), stream));
}

ufp4_status ufp4_quant_error_stats(const void* x, int64_t rows, int64_t cols, int64_t ld, const ufp4_quant_desc* desc,
                                   const ufp4_qtensor* rowwise, double* stats, cudaStream_t stream) {
    BlockShape bs;
    ufp4_status st = check_desc(desc, &bs);
    if (st != UFP4_OK) return st;
    if (!rowwise || !stats || rows < 0 || cols < 0) return UFP4_ERR_INVALID_ARG;
    if (!aligned(stats, 8)) return UFP4_ERR_ALIGNMENT;
    if (desc->grid == UFP4_GRID_MXFP8) return UFP4_ERR_UNSUPPORTED;  // the statistics decode 4-bit codes
    const int n = desc->hadamard_n;
    if (cols % 16 || cols % n || cols % bs.bw || (bs.is2d && rows % bs.b2d)) return UFP4_ERR_INVALID_ARG;
    st = check_out(rowwise, rows, cols, bs, desc->scale_fmt, false, desc->grid);
    if (st != UFP4_OK) return st;
    if (rows > 0 && cols > 0) {
        if (!x || ld < cols) return UFP4_ERR_INVALID_ARG;
        if (!aligned(x, 16) || ld % 8) return UFP4_ERR_ALIGNMENT;
    }
    QStatsParams p;
    std::memset(&p, 0, sizeof(p));
    p.x = (const uint16_t*)x;
    p.ld = ld;
    p.rows = rows;
    p.cols = cols;
    p.codes = (const uint8_t*)rowwise->codes;
    p.scales = rowwise->scales;
    p.codes_ld = rowwise->codes_ld;
    p.scales_ld = rowwise->scales_ld;
    p.grid = desc->grid;
    p.br = bs.is2d ? bs.b2d : 1;
    p.bc = bs.bw;
    p.sf = desc->scale_fmt;
    p.amax = rowwise->tensor_amax;
    p.n = n;
    p.inv_sqrt_n = inv_sqrt_n(n);
    make_sign_bits(desc->sign_seed, n, p.sign_bits);
    p.stats = stats;
    return cuda_status(launch_qstats(p, num_sms_current(), stream));
}

ufp4_status ufp4_error_stats(const float* ref, int64_t ld_ref, const float* approx, int64_t ld_approx, int64_t rows,
                             int64_t cols, double* stats, cudaStream_t stream) {
    if (!stats || rows < 0 || cols < 0) return UFP4_ERR_INVALID_ARG;
    if (!aligned(stats, 8)) return UFP4_ERR_ALIGNMENT;
    if (rows > 0 && cols > 0 && (!ref || !approx || ld_ref < cols || ld_approx < cols)) return UFP4_ERR_INVALID_ARG;
    return cuda_status(launch_dstats(ref, ld_ref, approx, ld_approx, rows, cols, stats, num_sms_current(), stream));
}

ufp4_status ufp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K, const ufp4_quant_desc* desc, size_t* bytes) {
    BlockShape bs;
    ufp4_status st = check_desc(desc, &bs);
    if (st != UFP4_OK) return st;
    if (!bytes || M < 0 || N < 0 || K < 0) return UFP4_ERR_INVALID_ARG;
    *bytes = gemm_workspace_bytes(M, N, K, desc->grid, bs.is2d ? bs.b2d : 1, bs.bw, desc->scale_fmt);
    return UFP4_OK;
}

ufp4_status ufp4_gemm(const ufp4_qtensor* A, const ufp4_qtensor* B, const ufp4_quant_desc* desc, float* D,
                      int64_t ldd, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    GemmArgs g;
    const ufp4_status st = prepare_gemm(A, B, desc, D, ldd, workspace, workspace_bytes, &g);
    if (st != UFP4_OK) return st;
    return run_prepared_gemm(g, stream);
}

ufp4_status ufp4_gemm_prepare(const ufp4_qtensor* A, const ufp4_qtensor* B, const ufp4_quant_desc* desc,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    GemmArgs g;
    float dummy_d[4] __attribute__((aligned(16)));  // shape checks only; D is not touched here
    const ufp4_status st = prepare_gemm(A, B, desc, dummy_d, B ? B->rows : 0, workspace, workspace_bytes, &g);
    if (st != UFP4_OK) return st;
    if (g.M == 0 || g.N == 0 || g.K == 0) return UFP4_OK;
    ensure_loaded();
    const cudaError_t e = launch_gemm_prep(g, stream);
    if (e == cudaErrorNotSupported) return UFP4_ERR_UNSUPPORTED;
    return cuda_status(e);
}

ufp4_status ufp4_gemm_prepared(const ufp4_qtensor* A, const ufp4_qtensor* B, const ufp4_quant_desc* desc, float* D,
                               int64_t ldd, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    GemmArgs g;
    const ufp4_status st = prepare_gemm(A, B, desc, D, ldd, workspace, workspace_bytes, &g);
    if (st != UFP4_OK) return st;
    if (g.M == 0 || g.N == 0) return UFP4_OK;
    if (g.K == 0) return run_prepared_gemm(g, stream);
    const cudaError_t e = launch_gemm_main(g, num_sms_current(), stream);
    if (e == cudaErrorNotSupported) return UFP4_ERR_UNSUPPORTED;
    return cuda_status(e);
}

ufp4_status ufp4_gemm_grouped_workspace_size(int32_t num_groups, const ufp4_qtensor* A, const ufp4_qtensor* B,
                                             const ufp4_quant_desc* desc, size_t* bytes) {
    if (num_groups < 0 || (num_groups && (!A || !B)) || !bytes) return UFP4_ERR_INVALID_ARG;
    // each group its own 256-byte aligned region (the groups of one launch run together)
    size_t need = 0;
    for (int32_t i = 0; i < num_groups; ++i) {
        size_t b = 0;
        const ufp4_status st = ufp4_gemm_workspace_size(A[i].rows, B[i].rows, A[i].cols, desc, &b);
        if (st != UFP4_OK) return st;
        if (A[i].rows == 0 || B[i].rows == 0 || A[i].cols == 0) b = 0;  // an empty product needs none
        need += (b + 255) & ~(size_t)255;
    }
    *bytes = need;
    return UFP4_OK;
}

ufp4_status ufp4_gemm_grouped(int32_t num_groups, const ufp4_qtensor* A, const ufp4_qtensor* B,
                              const ufp4_quant_desc* desc, float* const* D, const int64_t* ldd, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
    if (num_groups < 0 || (num_groups && (!A || !B || !D || !ldd))) return UFP4_ERR_INVALID_ARG;
    if (workspace && !aligned(workspace, 256)) return UFP4_ERR_ALIGNMENT;
    // every group is checked before anything is launched; group i takes the
    // workspace region after those of groups 0..i-1
    GemmArgs* args = new (std::nothrow) GemmArgs[num_groups > 0 ? num_groups : 1];
    if (!args) return UFP4_ERR_INVALID_ARG;
    size_t off = 0;
    for (int32_t i = 0; i < num_groups; ++i) {
        size_t need = 0;
        ufp4_status st = ufp4_gemm_workspace_size(A[i].rows, B[i].rows, A[i].cols, desc, &need);
        if (A[i].rows == 0 || B[i].rows == 0 || A[i].cols == 0) need = 0;  // an empty product needs none
        if (st == UFP4_OK && off + need > workspace_bytes) st = UFP4_ERR_INVALID_ARG;
        if (st == UFP4_OK)
            st = prepare_gemm(&A[i], &B[i], desc, D[i], ldd[i], need ? (uint8_t*)workspace + off : nullptr, need,
                              &args[i]);
        if (st != UFP4_OK) {
            delete[] args;
            return st;
        }
        off += (need + 255) & ~(size_t)255;
    }
    const cudaError_t e = launch_gemm_groups(args, num_groups, num_sms_current(), stream);
    delete[] args;
    if (e == cudaErrorNotSupported) return UFP4_ERR_UNSUPPORTED;
    return cuda_status(e);
}

}  // extern "C"
