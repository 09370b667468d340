// Internal launch interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace ufp4 {

constexpr int kMaxGroups = 64;

// Programmatic dependent launch.  Kernels launched through launch_pdl may
// start while the previous kernel of the stream is still running; each of
// them executes griddep_wait() before it touches global memory that the
// previous kernel may write or read (the wait returns once that kernel has
// completed and its writes are visible), and griddep_launch() to let the
// next kernel start early.  Without the launch attribute both are no-ops.
#ifdef __CUDACC__
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif

// The attribute is set on non-default streams only; launches on the legacy
// default stream stay plain.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = st ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

struct SignBits {
    uint32_t bits[8];  // bit i set <=> eps_{i mod n} = -1, for i in 0..255
};

// Round keys of Philox4x32-10 for one SR seed, computed on the host:
// k[2i] = seed lo + i * 0x9E3779B9, k[2i + 1] = seed hi + i * 0xBB67AE85
// (i = 0..9).  As kernel parameters they sit in the constant bank, where the
// XOR of each round reads them directly.
struct SrKeys {
    uint32_t k[20];
};

struct QOut {
    void* codes;
    void* scales;
    int64_t codes_ld;   // bytes
    int64_t scales_ld;  // elements
};

// Everything one quantizer launch needs (passed by value as the kernel parameter).
struct QuantParams {
    const uint16_t* x;
    int64_t cols, ld;
    int n;
    float inv_sqrt_n;
    uint32_t sign_bits[8];
    uint32_t smask16[16];  // n = 16: sign bit of element j of a segment (0x80000000 when eps_j = -1)
    int is2d, b2d;      // 2-D square blocks of side b2d
    int bw_row, bw_col; // 1-D block widths (or b2d)
    int col_seg_lanes;  // lanes sharing one column segment in the column pass
    int amax_slots;     // 2-D block amax slots per tile (0 for 1-D blocks)
    int tile_rows;      // rows per tile: 64, or 128 when the column pass needs 8 lanes per segment
    int stages;         // TMA ring depth
    int lbw_row, lbw_col, lb2d, lseg;  // log2 of block widths, 2-D side and col_seg_lanes
    int pow4, log4n;    // n = 4^log4n: 1/sqrt(n) is a power of two
    uint64_t sr_seed;
    SrKeys sr_keys;
    int do_row, do_col, vec256, col_grouped;
    QOut row, col;
    int col_tiles;
    int group_base;  // SR counter group id of group 0 (the caller's id when not grouped)
    int num_groups;
    int64_t grp_row0[kMaxGroups + 1];  // input row offsets
    int64_t grp_pad0[kMaxGroups + 1];  // padded row offsets (column-wise output)
    int grp_tile0[kMaxGroups + 1];     // first row tile of each group
};

cudaError_t launch_quantize(const QuantParams& p, int grid, bool sr, bool po2, int tc, int tr, int num_tiles,
                            int64_t total_rows, int num_sms, cudaStream_t st);

// The prepared form of one FP8-path GEMM operand (E1M2 / INT4, UE8M0, 1-D
// blocks) in the GEMM workspace: E5M2 copies of the levels with one hardware
// scale per 32 elements, and those scales in the replicated chunk layout of
// the CTA-pair kernel (widen_e5m2.cuh).
struct PrepTarget {
    uint8_t* fp8;     // rows x K bytes, row pitch K
    uint8_t* chunks;  // replicated scale chunks
    int64_t K;
    int tile_rows;    // rows of one GEMM tile of the operand (128 for A, the tile width for B)
    int parts;        // 128-row parts of a GEMM tile
    int chunks_k;     // chunks along K per 128 rows
    int rows_cover;   // rows with scale cells: rows rounded up to whole GEMM tiles
};

// Row-wise only, 1-D blocks (or b x b blocks, b = 16, 32, 64), n <= 256: the lean kernel, over up to
// kMaxBatch independent tensors in one launch.
constexpr int kMaxBatch = 4;
struct RowsTensor {
    const uint16_t* x;  // host side only (the kernel reads through its tensor map)
    int64_t ld;         // elements
    uint8_t* codes;
    uint8_t* scales;
    int64_t codes_ld;   // bytes
    int64_t scales_ld;  // elements
    int rows, cols;
    int col_tiles, row_tiles;
    int tile0;          // first tile of this tensor in the launch
    const float* amax;  // two-level scale: the tensor amax T (device)
    PrepTarget prep;    // with RowsParams::prep: where the prepared GEMM operand goes
};
struct RowsParams {
    RowsTensor t[kMaxBatch];
    int count, num_tiles;
    int tc, tr;         // tile columns (128, or 256 for n = 256) and rows
    int lb2d;           // log2 b of b x b blocks, 0 for 1-D blocks
    int n, lbw, pow4, log4n, stages;
    float inv_sqrt_n;
    uint32_t sign_bits[8];
    uint32_t smask[64];  // n = 64: sign bit of element j of a segment (0x80000000 when eps_j = -1)
    uint64_t sr_seed;
    SrKeys sr_keys;
    int group;
    int prep;           // also write each tensor's prepared GEMM operand (n = 16, E1M2 / INT4, UE8M0, 1-D)
};
cudaError_t launch_quantize_rows(RowsParams& p, int grid, bool sr, int sf, int num_sms, cudaStream_t st);
// Two-level scale pre-pass: *amax = max |RHT(x)| over the tensor (zeroed first).
cudaError_t launch_tensor_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int n, float inv_sqrt_n,
                               const uint32_t sign_bits[8], float* amax, int num_sms, cudaStream_t st);
cudaError_t quant_error_read_clear(int* value);
// Polls of a tile barrier before the quantizer kernels give up (device-wide;
// the default is restored by passing quant_wait_limit_default()).
cudaError_t set_quant_wait_limit(uint32_t polls);
uint32_t quant_wait_limit_default();
// The row kernel's unit (quantize_rows.cu) keeps its own error word and wait
// limit; the two functions above read and set every quantizer unit's.
cudaError_t rows_error_read_clear(int* value);
cudaError_t set_rows_wait_limit(uint32_t polls);
cudaError_t preload_rows_kernels();
// The general kernel's SR instantiations (quantize_sr.cu), with their own
// error word and wait limit.
cudaError_t launch_quantize_sr(const CUtensorMap& map, const QuantParams& p, int grid, bool po2, int tc,
                               int num_tiles, int num_sms, cudaStream_t st);
cudaError_t sr_error_read_clear(int* value);
cudaError_t set_sr_wait_limit(uint32_t polls);
cudaError_t preload_quantize_sr_kernels();

// 2-D tiled tensor map (TMA) over a row-major matrix: inner x outer elements,
// pitch bytes between rows, boxes of box_inner x box_outer elements.
bool encode_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* ptr, uint64_t inner, uint64_t outer,
                   uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);
cudaError_t launch_rht(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int n,
                       float inv_sqrt_n, const SignBits& sb, float* z, int64_t ldz, int num_sms,
                       cudaStream_t st);

struct DequantParams {
    const uint8_t* codes;
    const void* scales;
    int64_t rows, cols, codes_ld, scales_ld;
    int grid, br, bc;
    int sf;             // scale format: 0 fp32, 1 UE8M0, 2 two-level E4M3
    const float* amax;  // two-level: tensor amax T
    int n, inverse;
    float inv_sqrt_n;
    uint32_t sign_bits[8];
    float* out;
    int64_t ld_out;
};
cudaError_t launch_dequantize(const DequantParams& p, int num_sms, cudaStream_t st);

// Diagnostics (stats.cu): fp64 sums over a row-wise quantization and its input,
// and over two fp32 matrices.
struct QStatsParams {
    const uint16_t* x;
    int64_t ld, rows, cols;
    const uint8_t* codes;
    const void* scales;
    int64_t codes_ld, scales_ld;
    int grid, br, bc, sf, n;  // sf: 0 fp32, 1 UE8M0, 2 two-level E4M3
    const float* amax;        // two-level: tensor amax T
    float inv_sqrt_n;
    uint32_t sign_bits[8];
    double* stats;  // device, 4 doubles
};
cudaError_t launch_qstats(const QStatsParams& p, int num_sms, cudaStream_t st);
cudaError_t launch_dstats(const float* a, int64_t lda, const float* b, int64_t ldb, int64_t rows, int64_t cols,
                          double* stats, int num_sms, cudaStream_t st);

// ---------------------------------------------------------------- GEMM
struct GemmOperand {
    const uint8_t* codes;
    const uint8_t* scales;  // UE8M0
    int64_t rows, codes_ld, scales_ld;
};
struct GemmArgs {
    GemmOperand a, b;
    int64_t M, N, K;
    int grid, br, bc;
    int sf;                              // 0 fp32 block scales, 1 UE8M0, 2 two-level (E4M3 x tensor scale)
    const float* amax_a;                 // two-level: tensor amax of A and of B
    const float* amax_b;
    float* D;
    int64_t ldd;
    void* workspace;
    size_t workspace_bytes;
};
size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int grid, int br, int bc, int sf);
// The workspace targets of A (out[0]) and B (out[1]) for ufp4_gemm_prepared;
// cudaErrorNotSupported unless the GEMM takes the widened FP8 path.
cudaError_t gemm_prep_targets(const GemmArgs& g, PrepTarget out[2]);
cudaError_t launch_gemm(const GemmArgs& g, int num_sms, cudaStream_t st);
cudaError_t launch_gemm_prep(const GemmArgs& g, cudaStream_t st);
cudaError_t launch_gemm_main(const GemmArgs& g, int num_sms, cudaStream_t st);
// Load every kernel of each unit.  The library does it once per device
// before its first launch: with lazy module loading, loading a kernel while
// earlier kernels of the library are in flight (programmatic dependent
// launches waiting on one another) stalled the stream for minutes.
cudaError_t preload_quantize_kernels();
cudaError_t preload_gemm_kernels();
cudaError_t preload_dequant_kernels();
cudaError_t preload_stats_kernels();
cudaError_t preload_round_levels_kernels();
// The quantizer's rounding and packing step on count given scaled values
// (count a multiple of 32; u16: SR draws), round_levels.cu.
cudaError_t launch_round_levels(int grid, bool sr, int sf, const float* t, const uint16_t* u16, int64_t count,
                                uint8_t* codes, cudaStream_t st);
// n GEMMs sharing a descriptor, each with its own workspace (the grouped call)
cudaError_t launch_gemm_groups(const GemmArgs* gs, int n, int num_sms, cudaStream_t st);

}  // namespace ufp4
