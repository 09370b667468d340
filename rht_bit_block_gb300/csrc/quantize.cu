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
// Row-wise calls with 1-D blocks take the leaner kernel of quantize_rows.cu;
// the steps both share are in quantize_common.cuh.  The general kernel's
// template is in quantize_general.cuh: this unit instantiates its RTNE
// kernels and holds the RHT-only kernel and the host side; quantize_sr.cu
// instantiates the SR kernels.
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "quantize_general.cuh"

namespace ufp4 {

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

cudaError_t launch_quantize(const QuantParams& p, int grid, bool sr, bool po2, int tc, int tr, int num_tiles,
                            int64_t total_rows, int num_sms, cudaStream_t st) {
    CUtensorMap map;
    if (!encode_map_2d(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, p.x, (uint64_t)p.cols, (uint64_t)total_rows,
                       (uint64_t)p.ld * 2, (uint32_t)tc, (uint32_t)tr, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (sr) return launch_quantize_sr(map, p, grid, po2, tc, num_tiles, num_sms, st);
    return launch_general<false>(map, p, grid, po2, tc, num_tiles, num_sms, st);
}

uint32_t quant_wait_limit_default() { return kWaitLimit; }

cudaError_t set_quant_wait_limit(uint32_t polls) {
    cudaError_t e = general_set_wait_limit(polls);
    if (e == cudaSuccess) e = set_sr_wait_limit(polls);
    return e != cudaSuccess ? e : set_rows_wait_limit(polls);
}

// The first nonzero error word of the three quantizer units (each is cleared).
cudaError_t quant_error_read_clear(int* value) {
    int v = 0, w = 0, r = 0;
    cudaError_t e = general_error_read_clear(&v);
    if (e == cudaSuccess) e = sr_error_read_clear(&w);
    if (e == cudaSuccess) e = rows_error_read_clear(&r);
    *value = v ? v : (w ? w : r);
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

cudaError_t preload_quantize_kernels() {
    preload_general<false>();
    preload_quantize_sr_kernels();
    preload_rows_kernels();
    cudaFuncAttributes a;
    return cudaFuncGetAttributes(&a, rht_kernel);
}

}  // namespace ufp4
