// Quantization diagnostics (the single-tensor and GEMM-output error figures
// of the UFP4 summary, sections 数据集 and 方法: Q_G(T) stands for the
// dequantized tensor, and RTNE on a non-uniform grid shrinks values toward
// zero bin by bin, a bias that multiplies over layers).
//
//  * quant error stats: from x and its row-wise quantization, recompute z =
//    RHT(x) with the quantizer's arithmetic, dequantize q = level * scale, and
//    accumulate sum z^2, sum (q - z)^2, sum q z, sum q^2 in fp64.  SQNR =
//    sum z^2 / sum (q - z)^2; the shrinkage factor E[Q(t) t] / E[t^2] =
//    sum q z / sum z^2.
//  * error stats of two fp32 matrices (e.g. a quantized GEMM output against a
//    reference): sum a^2, sum (b - a)^2, sum a b, sum b^2.
// The quantizer sums go through 16-element fp32 partial sums (fused
// multiply-adds) before fp64 accumulation: a relative difference of order
// 1e-6 from an exact fp64 sum, plenty for SQNR and shrinkage figures.
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "ufp4_device.cuh"

namespace ufp4 {

namespace {

constexpr int kStatThreads = 256;

// Block-wide reduction of four fp64 sums, then one atomic add each.
__device__ __forceinline__ void reduce_add4(double v[4], double* out) {
    __shared__ double part[kStatThreads / 32][4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_down_sync(0xFFFFFFFFu, v[k], o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0)
        for (int k = 0; k < 4; ++k) part[warp][k] = v[k];
    __syncthreads();
    if (warp == 0) {
        for (int k = 0; k < 4; ++k) v[k] = lane < kStatThreads / 32 ? part[lane][k] : 0.0;
#pragma unroll
        for (int k = 0; k < 4; ++k)
            for (int o = 16; o > 0; o >>= 1) v[k] += __shfl_down_sync(0xFFFFFFFFu, v[k], o);
        if (lane == 0)
            for (int k = 0; k < 4; ++k) atomicAdd(out + k, v[k]);
    }
}

__global__ void __launch_bounds__(kStatThreads) qstats_kernel(const QStatsParams p) {
    const float g = p.sf == 2 ? __fdiv_rn(*p.amax, grid_qmax(p.grid) * 448.0f) : 0.0f;
    const int64_t cpr = p.cols / kChunk;
    const int64_t total = p.rows * cpr;
    double acc[4] = {0.0, 0.0, 0.0, 0.0};
    // grid-stride over whole warps so that the butterfly's shuffles see full warps
    for (int64_t base = (int64_t)blockIdx.x * kStatThreads; base < total;
         base += (int64_t)gridDim.x * kStatThreads) {
        const int64_t qi = base + threadIdx.x;
        const bool valid = qi < total;
        const int64_t r = valid ? qi / cpr : 0;
        const int64_t cc = valid ? qi % cpr : 0;
        uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        uint2 code = make_uint2(0u, 0u);
        if (valid) {
            const uint4* src = reinterpret_cast<const uint4*>(p.x + r * p.ld + cc * kChunk);
            const uint4 a = __ldg(src), b = __ldg(src + 1);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
            w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
            code = *reinterpret_cast<const uint2*>(p.codes + r * p.codes_ld + cc * (kChunk / 2));
        }
        const int pos = (int)((cc * kChunk) % 256);
        const uint32_t sgn = (p.sign_bits[pos / 32] >> (pos % 32)) & 0xFFFFu;
        const int seg_lane = (int)((cc * kChunk) % (p.n > kChunk ? p.n : kChunk)) / kChunk;
        float z[16];
        widen16(w, sgn, z);
        fwht16(z, p.n, seg_lane);
#pragma unroll
        for (int k = 0; k < 16; ++k) z[k] = __fmul_rn(z[k], p.inv_sqrt_n);
        if (valid) {
            // 16-element partial sums in fp32 (fp64 throughput is low on this
            // part), then one fp64 addition per sum and chunk
            float part[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int64_t c = cc * kChunk + i;
                const int64_t sidx = (r / p.br) * p.scales_ld + c / p.bc;
                float s;
                if (p.sf == 1) {
                    const int b = reinterpret_cast<const uint8_t*>(p.scales)[sidx];
                    s = b >= 1 ? __uint_as_float((uint32_t)b << 23) : __uint_as_float(0x00400000u);
                } else if (p.sf == 2) {
                    s = __fmul_rn(e4m3_value(reinterpret_cast<const uint8_t*>(p.scales)[sidx]), g);
                } else {
                    s = reinterpret_cast<const float*>(p.scales)[sidx];
                }
                const uint32_t word = i < 8 ? code.x : code.y;
                const float q = __fmul_rn(decode_level(p.grid, (word >> (4 * (i & 7))) & 0xFu), s);
                const float d = __fsub_rn(q, z[i]);
                part[0] = __fmaf_rn(z[i], z[i], part[0]);
                part[1] = __fmaf_rn(d, d, part[1]);
                part[2] = __fmaf_rn(q, z[i], part[2]);
                part[3] = __fmaf_rn(q, q, part[3]);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) acc[k] += (double)part[k];
        }
    }
    reduce_add4(acc, p.stats);
}

__global__ void __launch_bounds__(kStatThreads) dstats_kernel(const float* a, int64_t lda, const float* b, int64_t ldb,
                                                              int64_t rows, int64_t cols, double* stats) {
    double acc[4] = {0.0, 0.0, 0.0, 0.0};
    const int64_t total = rows * cols;
    for (int64_t i = (int64_t)blockIdx.x * kStatThreads + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * kStatThreads) {
        const int64_t r = i / cols, c = i - r * cols;
        const float x = a[r * lda + c], y = b[r * ldb + c];
        const double d = (double)y - (double)x;  // exact
        acc[0] += (double)__fmul_rn(x, x);
        acc[1] += d * d;
        acc[2] += (double)__fmul_rn(x, y);
        acc[3] += (double)__fmul_rn(y, y);
    }
    reduce_add4(acc, stats);
}

// Two-level scale pre-pass: T = max |z| over the tensor, z = RHT(x) with the
// quantizer's arithmetic (non-negative floats order like their bits, so the
// maximum is an integer atomicMax on the bit patterns).
__global__ void __launch_bounds__(kStatThreads) amax_kernel(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld,
                                                            int n, float inv_sqrt_n, SignBits sb, float* amax) {
    __shared__ unsigned int part[kStatThreads / 32];
    const int64_t cpr = cols / kChunk;
    const int64_t total = rows * cpr;
    float m = 0.0f;
    for (int64_t base = (int64_t)blockIdx.x * kStatThreads; base < total;
         base += (int64_t)gridDim.x * kStatThreads) {
        const int64_t qi = base + threadIdx.x;
        const bool valid = qi < total;
        const int64_t r = valid ? qi / cpr : 0;
        const int64_t cc = valid ? qi % cpr : 0;
        uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (valid) {
            const uint4* src = reinterpret_cast<const uint4*>(x + r * ld + cc * kChunk);
            const uint4 a = __ldg(src), b = __ldg(src + 1);
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
            w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        }
        const int pos = (int)((cc * kChunk) % 256);
        const uint32_t sgn = (sb.bits[pos / 32] >> (pos % 32)) & 0xFFFFu;
        const int seg_lane = (int)((cc * kChunk) % (n > kChunk ? n : kChunk)) / kChunk;
        float z[16];
        widen16(w, sgn, z);
        fwht16(z, n, seg_lane);
        if (valid)
#pragma unroll
            for (int k = 0; k < 16; ++k) m = fmaxf(m, fabsf(__fmul_rn(z[k], inv_sqrt_n)));
    }
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) part[warp] = __float_as_uint(m);
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int v = 0;
        for (int i = 0; i < kStatThreads / 32; ++i) v = v > part[i] ? v : part[i];
        atomicMax(reinterpret_cast<unsigned int*>(amax), v);
    }
}

}  // namespace

cudaError_t launch_tensor_amax(const uint16_t* x, int64_t rows, int64_t cols, int64_t ld, int n, float inv_sqrt_n,
                               const uint32_t sign_bits[8], float* amax, int num_sms, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float), st);
    if (e != cudaSuccess) return e;
    SignBits sb;
    for (int i = 0; i < 8; ++i) sb.bits[i] = sign_bits[i];
    const int64_t total = rows * (cols / kChunk);
    int64_t blocks = (total + kStatThreads - 1) / kStatThreads;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    if (blocks < 1) blocks = 1;
    amax_kernel<<<(unsigned)blocks, kStatThreads, 0, st>>>(x, rows, cols, ld, n, inv_sqrt_n, sb, amax);
    return cudaGetLastError();
}

cudaError_t launch_qstats(const QStatsParams& p, int num_sms, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(p.stats, 0, 4 * sizeof(double), st);
    if (e != cudaSuccess) return e;
    const int64_t total = p.rows * (p.cols / kChunk);
    int64_t blocks = (total + kStatThreads - 1) / kStatThreads;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    if (blocks < 1) blocks = 1;
    qstats_kernel<<<(unsigned)blocks, kStatThreads, 0, st>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_dstats(const float* a, int64_t lda, const float* b, int64_t ldb, int64_t rows, int64_t cols,
                          double* stats, int num_sms, cudaStream_t st) {
    cudaError_t e = cudaMemsetAsync(stats, 0, 4 * sizeof(double), st);
    if (e != cudaSuccess) return e;
    const int64_t total = rows * cols;
    int64_t blocks = (total + kStatThreads - 1) / kStatThreads;
    if (blocks > (int64_t)num_sms * 8) blocks = (int64_t)num_sms * 8;
    if (blocks < 1) blocks = 1;
    dstats_kernel<<<(unsigned)blocks, kStatThreads, 0, st>>>(a, lda, b, ldb, rows, cols, stats);
    return cudaGetLastError();
}

cudaError_t preload_stats_kernels() {
    cudaFuncAttributes a;
    cudaFuncGetAttributes(&a, qstats_kernel);
    cudaFuncGetAttributes(&a, dstats_kernel);
    return cudaFuncGetAttributes(&a, amax_kernel);
}

}  // namespace ufp4
