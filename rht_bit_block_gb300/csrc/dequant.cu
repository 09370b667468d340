// Dequantization Q_G(T) = level(code) * scale (UFP4 summary, section 数据集:
// inside arithmetic the quantized tensor stands for its dequantized values),
// with an optional inverse RHT x = (z H) S (H'_n = S_n H_n is orthogonal,
// section 方法).  MXFP8 codes are E4M3 bytes, one per element.  A check and
// diagnostics path, off the hot path.
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ufp4_device.cuh"

namespace ufp4 {


__global__ void __launch_bounds__(256) dequant_kernel(const DequantParams p) {
    // two-level scale: g = fp32(T / fp32(qmax * 448))
    const float g = p.sf == 2 ? __fdiv_rn(*p.amax, grid_qmax(p.grid) * 448.0f) : 0.0f;
    const int64_t cpr = p.cols / kChunk;
    const int64_t total = p.rows * cpr;
    for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < total; base += (int64_t)gridDim.x * blockDim.x) {
        const int64_t q = base + threadIdx.x;
        const bool valid = q < total;
        const int64_t r = valid ? q / cpr : 0;
        const int64_t cc = valid ? q % cpr : 0;
        const int64_t c = cc * kChunk;
        float v[16];
        const bool bytes = p.grid == 4;  // MXFP8: one E4M3 byte per element
        uint4 code = make_uint4(0u, 0u, 0u, 0u);
        if (valid && bytes) code = *reinterpret_cast<const uint4*>(p.codes + r * p.codes_ld + c);
        if (valid && !bytes) {
            const uint2 c2 = *reinterpret_cast<const uint2*>(p.codes + r * p.codes_ld + c / 2);
            code.x = c2.x;
            code.y = c2.y;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint32_t word = i < 8 ? code.x : code.y;
            const uint32_t nib = (word >> (4 * (i & 7))) & 0xFu;
            const uint32_t w4 = i < 4 ? code.x : (i < 8 ? code.y : (i < 12 ? code.z : code.w));
            const uint32_t byte = (w4 >> (8 * (i & 3))) & 0xFFu;
            float s = 0.0f;
            if (valid) {
                const int64_t si = (r / p.br) * p.scales_ld + (c + i) / p.bc;
                if (p.sf == 1) {
                    const int e = (int)((const uint8_t*)p.scales)[si] - 127;
                    s = (e >= -126) ? __uint_as_float((uint32_t)(e + 127) << 23)
                                    : __uint_as_float(0x00400000u >> (-127 - e));
                } else if (p.sf == 2) {
                    s = __fmul_rn(e4m3_value(((const uint8_t*)p.scales)[si]), g);
                } else {
                    s = ((const float*)p.scales)[si];
                }
            }
            const float lv = bytes ? ((byte & 0x80u) ? -e4m3_value(byte & 0x7Fu) : e4m3_value(byte))
                                   : decode_level(p.grid, nib);
            v[i] = __fmul_rn(lv, s);
        }
        if (p.inverse && p.n > 1) {
            const int seg_lane = (int)((c % (p.n > kChunk ? p.n : kChunk)) / kChunk);
            fwht16(v, p.n, seg_lane);
            const int pos = (int)(c % 256);
            const uint32_t sgn = (p.sign_bits[pos >> 5] >> (pos & 31)) & 0xFFFFu;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float t = __fmul_rn(v[i], p.inv_sqrt_n);
                v[i] = __uint_as_float(__float_as_uint(t) ^ (((sgn >> i) & 1u) << 31));
            }
        }
        if (valid) {
            float* dst = p.out + r * p.ld_out + c;
#pragma unroll
            for (int i = 0; i < 16; ++i) dst[i] = v[i];
        }
    }
}

cudaError_t launch_dequantize(const DequantParams& p, int num_sms, cudaStream_t st) {
    const int64_t total = p.rows * (p.cols / kChunk);
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    if (blocks < 1) blocks = 1;
    dequant_kernel<<<(unsigned)blocks, 256, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t preload_dequant_kernels() {
    cudaFuncAttributes a;
    return cudaFuncGetAttributes(&a, dequant_kernel);
}

}  // namespace ufp4
