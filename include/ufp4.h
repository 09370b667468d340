/*
 * ufp4.h -- C ABI of the GB300 (sm_103a) library for the UFP4 recipe's
 * data-parallel hot path: the fused Random Hadamard Transform (RHT) + block
 * scaled 4-bit quantizer that prepares the operands of the three training
 * GEMMs, and the quantized GEMM that consumes them.
 *
 * Sources, cited as page + section/equation:
 *  [UFP4-data]   UFP4 summary (hyper.ai, arXiv 2606.20381), section 数据集:
 *                codebooks G (E2M1, E1M2, INT4), contiguous blocks, block scale
 *                s_B = block amax / largest level, RTNE and SR rounding, and
 *                Q_G(T) meaning the dequantized tensor.
 *  [UFP4-method] same page, section 方法: Eq. H_2n (Sylvester recursion),
 *                H'_n = S_n H_n, Eq. Y = XW^T = (XH')(WH')^T, Eq. of the
 *                quantized GEMM Y^ = Q_G(XH') Q_G(WH')^T, RHT on FPROP, DGRAD
 *                and WGRAD, SR on dY only, free choice of the scale hierarchy.
 *  [2D-block]    "Stable FP4 Training via Transposition-Invariant Block
 *                Quantization" tutorial: b x b square blocks (Eq. S(B)=S(B^T)),
 *                truncation-free scale S = 2^ceil(log2(2M/(Qp-Qn))), and the
 *                transposes in dX = dY W, dW = dY^T X.
 *
 * General rules
 *  - Ownership: the caller allocates and owns every buffer.  Only the entry
 *    points documented as such read or write host memory; all other pointers
 *    are device pointers on the current CUDA device.
 *  - Asynchrony: device work is enqueued on `stream` and the call returns
 *    without waiting.  Argument errors are detected on the host before any
 *    launch and return an error code; nothing is launched then.
 *  - Layouts are row-major.  A matrix of `rows x cols` elements with leading
 *    dimension `ld` holds element (r, c) at offset r*ld + c.  Byte matrices
 *    of codes hold two 4-bit codes per byte, the lower column index in the low
 *    nibble.
 *  - Inputs are bf16 bit patterns.  Non-finite inputs, and blocks whose
 *    absolute maximum after the RHT is nonzero but below 2^-120 or above
 *    2^120, are outside the contract (outputs are then unspecified but the
 *    call stays memory-safe).
 *  - Host state: calls may be made from several threads on different
 *    streams.  The library keeps a little process-lifetime state per device,
 *    set up on first use and guarded by locks: a flag that its kernels have
 *    been loaded (done once, before its first launch on the device), the
 *    cached co-residency figures of the GEMM launch, the two internal streams
 *    of ufp4_gemm_grouped (created on its first call with two or more
 *    groups) and the device address of the ufp4_gemm_noalloc scratch.  After
 *    cudaDeviceReset that state is stale: do not call the library on that
 *    device again in the same process.
 */
#ifndef UFP4_H_
#define UFP4_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    UFP4_OK = 0,
    UFP4_ERR_INVALID_ARG = 1, /* a null pointer, a bad size or an inconsistent shape */
    UFP4_ERR_UNSUPPORTED = 2, /* a valid combination this library does not implement */
    UFP4_ERR_ALIGNMENT = 3,   /* a pointer or leading dimension breaks the alignment rule */
    UFP4_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed */
    UFP4_ERR_TIMEOUT = 5      /* a bounded device-side wait gave up (see ufp4_device_error) */
} ufp4_status;

/* Codebooks [UFP4-data].  Levels (non-negative magnitudes, 3-bit index 0..7):
 *   E1M2: 0, 0.25, 0.5, ..., 1.75 (uniform, largest level 1.75)
 *   INT4: 0, 1, ..., 7            (uniform, signed range -7..7, -8 unused)
 *   E2M1: 0, 0.5, 1, 1.5, 2, 3, 4, 6 (non-uniform, largest level 6)
 * Nibble encodings: E1M2 and E2M1 are sign << 3 | index (a zero level is
 * always written as 0x0); INT4 is the two's complement of the signed level. */
/* UFP4_GRID_E2M1_R2: range-limited E2M1 -- blocks scaled so that amax maps to
 * 2 and rounded to E2M1's uniform levels 0, 0.5, 1, 1.5, 2 only; the codes
 * are E2M1 codes, so the GEMM runs on the native FP4 path (a reading of the
 * UFP4 summary, section 实验: a uniform grid cannot simply be substituted on
 * FP4 hardware). */
/* UFP4_GRID_MXFP8: the format the 2D-block page keeps for the Query and Key
 * projections (section on mixed precision: more precision and a wider
 * dynamic range than FP4), read as the OCP Microscaling MXFP8 format with
 * E4M3 elements.  Codes are E4M3 bytes, ONE BYTE PER ELEMENT (codes_ld >=
 * cols bytes, a multiple of 16); blocks are 1 x 32 with an E8M0 scale byte
 * e + 127, e = floor(log2 M) - 8 clamped to [-127, 127] (M the block amax of
 * the RHT output; 8 is the exponent of E4M3's largest normal 448), and each
 * element is z * 2^-e rounded to E4M3, nearest even, saturated at 448; a
 * zero code is written as +0.  Requires block 1 x 32, UFP4_SCALE_UE8M0 (the
 * E8M0 byte; the rule above replaces the truncation-free one), RTNE and the
 * row-wise output; the GEMM runs it on the FP8 tensor cores in place. */
typedef enum {
    UFP4_GRID_E1M2 = 0,
    UFP4_GRID_INT4 = 1,
    UFP4_GRID_E2M1 = 2,
    UFP4_GRID_E2M1_R2 = 3,
    UFP4_GRID_MXFP8 = 4
} ufp4_grid;

/* Rounding [UFP4-data; UFP4-method: RTNE for X and W, SR for dY]:
 *   RTNE: nearest level, exact ties to the even index.
 *   SR:   with lo <= |t| <= hi the neighbouring levels and p = (|t|-lo)/(hi-lo),
 *         the magnitude rounds up iff u < p * 65536, u a 16-bit Philox4x32-10
 *         draw: key = sr_seed, counter = (g lo32, g hi32, stream, group) with
 *         g = (row-major linear index of the element in the output tensor) / 8,
 *         stream 0 for the row-wise output and 1 for the column-wise one;
 *         element j = index % 8 takes the low 16 bits of word j/2 when j is
 *         even and the high 16 bits when j is odd. */
typedef enum { UFP4_ROUND_RTNE = 0, UFP4_ROUND_SR = 1 } ufp4_round;

/* Scale formats.
 *   FP32:  s = fp32(M / qmax) [UFP4-data]; elements are scaled as
 *          t = z * fp32(1/s) (an all-zero block has s = 0 and t = 0).
 *          Only for 1-D blocks.
 *   UE8M0: S = 2^e with e the smallest integer such that M <= qmax * 2^e
 *          [2D-block, truncation-free scale, with Qp = -Qn = qmax], clamped
 *          to [-127, 127]; stored as the byte e + 127.  Required for b x b
 *          blocks and for GEMM operands.
 *   E4M3:  two-level [UFP4-method: the scale hierarchy is free to follow the
 *          hardware]: a per-tensor fp32 scale g = fp32(T / fp32(qmax * 448)),
 *          T = amax of the whole RHT output, times a per-block E4M3 byte
 *          b = E4M3 round-to-nearest-even, saturated at 448, of
 *          fp32(fp32(M / qmax) / g) (0 when g = 0); elements are scaled by
 *          fp32(1/s), s = fp32(e4m3(b) * g) (0 when s = 0).  T is stored in
 *          the qtensor's tensor_amax.  Row-wise only, 1-D blocks, n <= 128;
 *          the GEMM takes it for E2M1 codes with 1 x 16 blocks (native
 *          block-scaled FP4 with E4M3 scales, g_A * g_B applied to D). */
typedef enum { UFP4_SCALE_FP32 = 0, UFP4_SCALE_UE8M0 = 1, UFP4_SCALE_E4M3 = 2 } ufp4_scale_fmt;

/* Output selection bits for ufp4_rht_quantize. */
enum { UFP4_OUT_ROWWISE = 1, UFP4_OUT_COLWISE = 2 };

/* What to compute.
 *   grid        ufp4_grid
 *   block_rows, block_cols
 *               1 x 16 or 1 x 32 (1-D blocks along the quantized dimension),
 *               or b x b with b in {8, 16, 32, 64} (2-D square blocks,
 *               [2D-block]); for the column-wise output the block shape applies
 *               to the transposed tensor.
 *   hadamard_n  n = 2^k in {1, 2, ..., 256}; the RHT acts on each length-n
 *               segment of the quantized dimension with the same signs
 *               [UFP4-method].  n = 1 switches the transform off.
 *   sign_seed   eps_i = 1 - 2 b_i, b_i = bit (i % 32) of word (i % 128) / 32 of
 *               Philox4x32-10(key = sign_seed, counter = (i/128, 0, 2, 0)).
 *   round, sr_seed   see ufp4_round.
 *   scale_fmt   ufp4_scale_fmt.
 *   out_mask    UFP4_OUT_ROWWISE | UFP4_OUT_COLWISE.
 *   group       fourth Philox counter word of SR draws (the expert id in the
 *               grouped calls, which set it themselves; 0 otherwise). */
typedef struct {
    int32_t grid;
    int32_t block_rows;
    int32_t block_cols;
    int32_t hadamard_n;
    uint64_t sign_seed;
    int32_t round;
    int32_t scale_fmt;
    uint64_t sr_seed;
    int32_t out_mask;
    int32_t group;
} ufp4_quant_desc;

/* A quantized matrix in device memory, described in its own layout: the
 * row-wise output of an R x C input has rows = R, cols = C; the column-wise
 * output (the quantization of the transpose) has rows = C, cols = R.
 *   codes      rows x cols/2 bytes (rows x cols for UFP4_GRID_MXFP8),
 *              leading dimension codes_ld bytes (multiple of 8; of 16 for
 *              GEMM operands and for MXFP8; the pointer 16-byte aligned)
 *   scales     (rows/block_rows) x (cols/block_cols) elements, float for FP32
 *              scales and uint8 for UE8M0 and E4M3, leading dimension
 *              scales_ld elements (the pointer 4-byte aligned for float)
 *   tensor_amax  device float: T of the two-level scale (UFP4_SCALE_E4M3),
 *              written by the quantizer, read by dequantize, the GEMM and the
 *              diagnostics; unused (may be NULL) for the other formats */
typedef struct {
    void* codes;
    void* scales;
    int64_t rows;
    int64_t cols;
    int64_t codes_ld;
    int64_t scales_ld;
    float* tensor_amax;
} ufp4_qtensor;

/* ufp4_rht_quantize -- fused RHT + block-scaled 4-bit quantization.
 * [UFP4-data] blocks, scale, rounding; [UFP4-method] z = x S_n H_n along the
 * GEMM's shared dimension; [2D-block] square blocks and the transposed copy.
 *   x        device bf16 [rows x cols], leading dimension ld elements
 *            (ld >= cols, ld multiple of 8, x 16-byte aligned)
 *   rowwise  written when out_mask has UFP4_OUT_ROWWISE: quantization of each
 *            row (RHT and blocks along cols); rows x cols
 *   colwise  written when out_mask has UFP4_OUT_COLWISE: quantization of x^T
 *            (RHT and blocks along rows); cols x rows
 * Both outputs come from one read of x.  Requirements: cols divisible by n
 * and by the block width for the row-wise output, rows divisible by n and by
 * the block width for the column-wise one (2-D blocks: both dimensions by b).
 * The qtensor's rows/cols must equal the shapes above.  On a non-default
 * stream the kernel is launched as a programmatic dependent of the previous
 * kernel; it waits for that kernel to finish before it reads or writes. */
ufp4_status ufp4_rht_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld,
                              const ufp4_quant_desc* desc, const ufp4_qtensor* rowwise,
                              const ufp4_qtensor* colwise, cudaStream_t stream);

/* ufp4_rht_quantize_batch -- the row-wise ufp4_rht_quantize of `count`
 * independent tensors that share one descriptor, in a single launch, e.g. the
 * X and W operands of one FPROP GEMM [UFP4-method, quantized GEMM Y^ =
 * Q_G(XH') Q_G(WH')^T: both operands are quantized along K].  Element i of
 * each host array describes tensor i exactly as the arguments of
 * ufp4_rht_quantize do (x: device bf16 rows[i] x cols[i], leading dimension
 * ld[i]; rowwise[i]: its row-wise output).  Requirements: 0 <= count <=
 * UFP4_MAX_BATCH, desc->out_mask == UFP4_OUT_ROWWISE, 1-D blocks, and
 * hadamard_n <= 128 for the two-level scale and MXFP8 (UFP4_ERR_UNSUPPORTED
 * otherwise), and per tensor the shape and
 * alignment rules of ufp4_rht_quantize.  The results are bit-identical to
 * `count` separate ufp4_rht_quantize calls.  Nothing is written when any
 * argument is rejected. */
#define UFP4_MAX_BATCH 4
ufp4_status ufp4_rht_quantize_batch(int32_t count, const void* const* x, const int64_t* rows, const int64_t* cols,
                                    const int64_t* ld, const ufp4_quant_desc* desc, const ufp4_qtensor* rowwise,
                                    cudaStream_t stream);

/* ufp4_rht_quantize_grouped -- the same for a stack of groups (MoE experts).
 *   x             device bf16 [total_rows x cols], leading dimension ld, the
 *                 rows of group g being offsets[g] .. offsets[g+1]-1
 *   offsets       HOST int64 array of num_groups + 1 nondecreasing row offsets,
 *                 offsets[0] = 0, offsets[num_groups] = total_rows
 *   rowwise       total_rows x cols: each group's row-wise quantization in its
 *                 own rows; SR draws use the group's id and the row index
 *                 within the group
 *   colwise       the column-wise quantization of each group, stacked: group g
 *                 has padded length P_g = round_up(c_g, max(n, block width, 64))
 *                 (missing rows read as zero; 64 makes P_g a valid GEMM K for
 *                 WGRAD), and occupies a cols x P_g
 *                 row-major matrix starting at codes + cols * (Poff_g / 2)
 *                 bytes and scales + cols * Poff_g / block_width elements,
 *                 Poff_g = P_0 + ... + P_{g-1}; its qtensor has rows = cols
 *                 and cols = sum of P_g, its *_ld fields are ignored.
 *   desc->group   ignored (each group uses its index)
 * 1-D blocks only. */
ufp4_status ufp4_rht_quantize_grouped(const void* x, int64_t cols, int64_t ld,
                                      const int64_t* offsets, int32_t num_groups,
                                      const ufp4_quant_desc* desc, const ufp4_qtensor* rowwise,
                                      const ufp4_qtensor* colwise, cudaStream_t stream);

/* Padded length P_g used by the grouped column-wise output (host helper). */
int64_t ufp4_grouped_padded_rows(int64_t rows, const ufp4_quant_desc* desc);

/* ufp4_rht_transform -- the RHT alone: z = fp32 result of x S_n H_n on each
 * length-n segment of every row [UFP4-method], with exactly the arithmetic of
 * the quantizer (signs, butterfly strides 1..n/2, one multiply by
 * fp32(1/sqrt n)).
 *   x  device bf16 [rows x cols], ld elements; z device float [rows x cols], ldz */
ufp4_status ufp4_rht_transform(const void* x, int64_t rows, int64_t cols, int64_t ld,
                               int32_t hadamard_n, uint64_t sign_seed, float* z, int64_t ldz,
                               cudaStream_t stream);

/* ufp4_dequantize -- Q_G(T) = level(code) * scale as fp32 [UFP4-data], in the
 * qtensor's own layout (rows x cols, leading dimension ld_out elements).
 * With inverse_rht != 0 the rotation is undone on each length-n segment of a
 * row: x = z H'^T = (z H) S, same butterfly, then the signs.
 * desc supplies grid, block shape, scale format, hadamard_n and sign_seed. */
ufp4_status ufp4_dequantize(const ufp4_qtensor* q, const ufp4_quant_desc* desc,
                            int32_t inverse_rht, float* out, int64_t ld_out, cudaStream_t stream);

/* ufp4_quant_error_stats -- diagnostics of one row-wise quantization
 * [UFP4-data: Q_G(T) is the dequantized tensor; UFP4-method: RTNE on a
 * non-uniform grid shrinks values bin by bin].  From x (device bf16 rows x
 * cols, ld elements) and its row-wise quantization `rowwise` made with desc,
 * the library recomputes z = RHT(x) with the quantizer's arithmetic and q =
 * level * scale, and writes to stats (device, 4 doubles, 8-byte aligned):
 *   stats[0] = sum z^2, stats[1] = sum (q - z)^2, stats[2] = sum q z,
 *   stats[3] = sum q^2, accumulated in fp64 over 16-element fp32 partial
 * sums (relative difference from an exact sum of order 1e-6; the order of
 * the additions is unspecified).  SQNR = stats[0] / stats[1]; the shrinkage factor
 * E[Q(t) t] / E[t^2] = stats[2] / stats[0]. */
ufp4_status ufp4_quant_error_stats(const void* x, int64_t rows, int64_t cols, int64_t ld, const ufp4_quant_desc* desc,
                                   const ufp4_qtensor* rowwise, double* stats, cudaStream_t stream);

/* ufp4_error_stats -- the same four fp64 sums for two device fp32 matrices
 * (rows x cols): stats[0] = sum ref^2, stats[1] = sum (approx - ref)^2,
 * stats[2] = sum ref * approx, stats[3] = sum approx^2; e.g. a quantized GEMM
 * output against a reference product. */
ufp4_status ufp4_error_stats(const float* ref, int64_t ld_ref, const float* approx, int64_t ld_approx, int64_t rows,
                             int64_t cols, double* stats, cudaStream_t stream);

/* ufp4_gemm_workspace_size -- device scratch bytes ufp4_gemm needs for
 * operands A (M x K) and B (N x K) quantized with desc. */
ufp4_status ufp4_gemm_workspace_size(int64_t M, int64_t N, int64_t K, const ufp4_quant_desc* desc,
                                     size_t* bytes);

/* ufp4_gemm -- the quantized GEMM consumer [UFP4-method, Eq. Y^ = Q_G(XH')
 * Q_G(WH')^T]: D[M x N] = Q(A) Q(B)^T in fp32 with fp32 accumulation, A and B
 * both quantized along K (K-major): A = the M x K qtensor, B = the N x K
 * qtensor, same desc (UE8M0 scales; 1 x 16, 1 x 32 or 32 x 32 blocks).
 * FPROP uses (X rowwise, W rowwise); DGRAD (dY rowwise, W colwise); WGRAD
 * (dY colwise, X colwise).  E2M1 runs on the native block-scaled FP4 tensor
 * path; E1M2 and INT4 levels are integers times a power of two and are
 * widened exactly into FP8 (E5M2) in the workspace first.
 *   D          device float, leading dimension ldd (multiple of 4, D 16-byte aligned)
 *   workspace  device scratch of at least ufp4_gemm_workspace_size bytes,
 *              256-byte aligned; contents on entry are ignored.
 * M, N and K up to 2^30 (UFP4_ERR_UNSUPPORTED beyond).  On a non-default
 * stream the kernels are launched as programmatic dependents: each one waits
 * for the previous kernel of the stream to finish before it touches memory,
 * so stream order is kept exactly as with plain launches. */
ufp4_status ufp4_gemm(const ufp4_qtensor* A, const ufp4_qtensor* B, const ufp4_quant_desc* desc,
                      float* D, int64_t ldd, void* workspace, size_t workspace_bytes,
                      cudaStream_t stream);

/* ufp4_gemm_prepare / ufp4_gemm_prepared -- the two stages of ufp4_gemm,
 * for callers that reuse prepared operands or time the stages apart.
 * ufp4_gemm_prepare writes the tensor-core form of A and B into the workspace
 * (E1M2/INT4: FP8 E5M2 copies with one UE8M0 scale per 32 elements; all
 * grids: the scales in the tensor-memory copy layout).  ufp4_gemm_prepared
 * then computes D from that workspace; it must get the same A, B (shapes and
 * scales), desc and workspace as the ufp4_gemm_prepare call before it on the
 * stream.  ufp4_gemm(...) == ufp4_gemm_prepare(...) + ufp4_gemm_prepared(...). */
ufp4_status ufp4_gemm_prepare(const ufp4_qtensor* A, const ufp4_qtensor* B, const ufp4_quant_desc* desc,
                              void* workspace, size_t workspace_bytes, cudaStream_t stream);
ufp4_status ufp4_gemm_prepared(const ufp4_qtensor* A, const ufp4_qtensor* B, const ufp4_quant_desc* desc, float* D,
                               int64_t ldd, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ufp4_rht_quantize_prepare -- the two operands of one FPROP-style GEMM
 * quantized and prepared in one launch: ufp4_rht_quantize_batch of a (the
 * A operand, A->rows x A->cols) and b (B->rows x B->cols) fused with
 * ufp4_gemm_prepare(A, B, desc, workspace) [UFP4-method: both operands of the
 * quantized GEMM Y^ = Q_G(XH') Q_G(WH')^T are quantized along K, and E1M2 /
 * INT4 levels widen exactly into FP8 for the tensor cores].  A and B receive
 * exactly what ufp4_rht_quantize_batch writes, and the workspace exactly what
 * ufp4_gemm_prepare writes, so ufp4_gemm_prepared(A, B, desc, D, ...) follows
 * directly, with no separate prep pass over the codes.
 *   a, b     device bf16, leading dimensions lda, ldb elements (the rules of
 *            ufp4_rht_quantize)
 *   A, B     their row-wise outputs; A->cols == B->cols == K
 *   workspace, workspace_bytes  as for ufp4_gemm_prepare
 * Requirements: desc->out_mask == UFP4_OUT_ROWWISE, grid E1M2 or INT4,
 * UFP4_SCALE_UE8M0, 1 x 16 or 1 x 32 blocks and hadamard_n == 16
 * (UFP4_ERR_UNSUPPORTED otherwise), and the rules of ufp4_rht_quantize_batch
 * and ufp4_gemm_prepare.  Nothing is written when any argument is rejected. */
ufp4_status ufp4_rht_quantize_prepare(const void* a, int64_t lda, const void* b, int64_t ldb,
                                      const ufp4_quant_desc* desc, const ufp4_qtensor* A, const ufp4_qtensor* B,
                                      void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ufp4_gemm_grouped_workspace_size -- scratch bytes ufp4_gemm_grouped needs:
 * the sum over the groups of ufp4_gemm_workspace_size, each rounded up to 256
 * bytes (0 for a group with an empty product); A, B: HOST arrays of
 * num_groups qtensors. */
ufp4_status ufp4_gemm_grouped_workspace_size(int32_t num_groups, const ufp4_qtensor* A, const ufp4_qtensor* B,
                                             const ufp4_quant_desc* desc, size_t* bytes);

/* ufp4_gemm_grouped -- the quantized GEMM over a set of independent groups
 * (MoE experts) [UFP4-method: the same quantized GEMM on every expert's
 * linear layer]: D_g = Q(A_g) Q(B_g)^T for g = 0 .. num_groups-1, each group
 * with its own shapes, as in ufp4_gemm.
 *   A, B   HOST arrays of num_groups qtensors describing device buffers.  The
 *          grouped quantizer's outputs slot in directly: FPROP uses the
 *          row-wise X slab of expert g and W_g; DGRAD the row-wise dY slab and
 *          W_g column-wise; WGRAD the column-wise dY_g and X_g (K = P_g, the
 *          padded token count).
 *   D, ldd HOST arrays of num_groups device output pointers and leading
 *          dimensions.
 *   workspace  device scratch of at least ufp4_gemm_grouped_workspace_size
 *          bytes; group g uses its own region of it (after those of groups
 *          0 .. g-1).
 * A group with no rows (M_g = 0 or N_g = 0) is skipped; a group with K_g = 0
 * writes D_g = 0.  Every group is checked before anything is launched.
 * Streams: with two or more non-empty groups, the groups are dealt
 * round-robin to `stream` and two internal non-blocking streams of the
 * current device (created on the first such call, kept for the process), so
 * that small groups run side by side.  The internal streams start after the
 * work already enqueued on `stream`, and `stream` waits for them before any
 * later work, so the call is ordered on `stream` like a single launch.  The
 * enqueue sequence is serialized by a lock (safe from several host threads). */
ufp4_status ufp4_gemm_grouped(int32_t num_groups, const ufp4_qtensor* A, const ufp4_qtensor* B,
                              const ufp4_quant_desc* desc, float* const* D, const int64_t* ldd, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* Size of the fixed device scratch behind ufp4_gemm_noalloc: 32 MiB. */
#define UFP4_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

/* ufp4_gemm_noalloc -- ufp4_gemm for callers that must not allocate device
 * memory (no counterpart in the pages: it is an interface convenience).
 * Some callers cannot call cudaMalloc at all: plugins or custom ops whose
 * host framework owns every device allocation and hands out none for
 * scratch, and latency-critical loops where an allocation may synchronize
 * the device.  This entry point takes the same A, B, desc, D and ldd as
 * ufp4_gemm but no workspace: it uses one scratch array of
 * UFP4_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU that
 * loads the library keeps until the process exits.
 *   - It allocates nothing and calls no allocating routine.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.
 *   - Returns UFP4_ERR_UNSUPPORTED when ufp4_gemm_workspace_size for these
 *     shapes exceeds UFP4_NOALLOC_SCRATCH_BYTES (E1M2/INT4 need about
 *     (M + N) * K bytes; E2M1 needs only its scale chunks).
 *   - All calls share the one array and it keeps the last call's contents
 *     (nothing in it has to start at zero).  Calls whose GPU work overlaps,
 *     for example on two streams at once, race on the array: serialize them. */
ufp4_status ufp4_gemm_noalloc(const ufp4_qtensor* A, const ufp4_qtensor* B, const ufp4_quant_desc* desc,
                              float* D, int64_t ldd, cudaStream_t stream);

/* ufp4_sign_vector -- the n signs eps_i of the RHT (HOST output, int8 +-1),
 * for consumers that apply the rotation themselves. */
ufp4_status ufp4_sign_vector(uint64_t sign_seed, int32_t n, int8_t* out_host);

/* ufp4_round_levels -- the rounding and packing step of ufp4_rht_quantize on
 * given scaled values, for checking it against a reference on any fp32 input
 * (UFP4 summary, section 数据集: RTNE and SR to the codebook levels and the
 * 4-bit encodings; 2D-block tutorial, 2D 方块量化: E[roundS(x)] = x).
 * It runs the quantizer's own code on blocks whose amax is the grid's largest
 * level qmax (n = 1), so the block reciprocal is 1 and each value t is
 * rounded as the quantizer rounds t = z * r.
 *   grid       UFP4_GRID_E1M2 .. UFP4_GRID_E2M1_R2 (not MXFP8).
 *   rounding   UFP4_ROUND_RTNE or UFP4_ROUND_SR.
 *   scale_fmt  UFP4_SCALE_FP32 or UFP4_SCALE_UE8M0: which of the quantizer's
 *              two arithmetic paths rounds (they agree wherever both apply).
 *   t          DEVICE, count fp32 values, |t| <= qmax (the values a block
 *              can hold; larger ones are outside the quantizer's domain),
 *              16-byte aligned.
 *   u16        DEVICE, count 16-bit draws for SR (element i uses u16[i]), 4-byte
 *              aligned; ignored (may be NULL) for RTNE.
 *   count      a multiple of 32 (0 does nothing).
 *   codes      DEVICE, count / 2 bytes, 8-byte aligned: packed as the
 *              quantizer packs them (element i in the low nibble of byte i/2
 *              when i is even), a zero level as +0.
 * Errors: UFP4_ERR_INVALID_ARG (enum values, count, NULL pointers),
 * UFP4_ERR_ALIGNMENT, UFP4_ERR_CUDA (launch). */
ufp4_status ufp4_round_levels(int32_t grid, int32_t rounding, int32_t scale_fmt, const float* t, const uint16_t* u16,
                              int64_t count, uint8_t* codes, cudaStream_t stream);

/* ufp4_device_error -- reads and clears the library's device error words on
 * the current device (synchronizes the device first).  Every device-side wait
 * of the library is bounded: a kernel whose wait gives up records the event,
 * lets its copies in flight land, releases what it holds and returns, leaving
 * its outputs unspecified.  Returns UFP4_ERR_TIMEOUT, with *code = 1, when
 * such a wait has given up since the last call, and UFP4_OK with *code = 0
 * otherwise (UFP4_ERR_CUDA if the device cannot be read).  The library does
 * not check the words on its other calls, which never synchronize. */
ufp4_status ufp4_device_error(int32_t* code);

/* ufp4_set_quantize_wait_limit -- failure-detection hook (no counterpart in
 * the pages).  Sets how many times the quantizer kernels poll for a tile's
 * arrival before they give up, on the current device, for later launches;
 * polls < 0 restores the default (2^24 polls, seconds).  With polls = 0 the
 * first wait of every quantizer CTA gives up at once: the kernel records the
 * timeout, waits (with the default limit) for the copies it has started and
 * returns, so tests can exercise the timeout path without hanging or faulting
 * the GPU; ufp4_device_error then returns UFP4_ERR_TIMEOUT.  Synchronizes the
 * device; do not call it while quantizer work is in flight on another
 * thread. */
ufp4_status ufp4_set_quantize_wait_limit(int64_t polls);

/* ufp4_status_string -- static, human-readable name of a status code. */
const char* ufp4_status_string(ufp4_status status);

#ifdef __cplusplus
}
#endif

#endif /* UFP4_H_ */
