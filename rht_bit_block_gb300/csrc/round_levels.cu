// The quantizer's rounding and packing step on given scaled values, so that it
// can be checked against a reference on every fp32 value a block can hold
// (UFP4 summary, section 数据集: RTNE and SR to the codebook levels, the
// 4-bit encodings; 2D-block tutorial: E[roundS(x)] = x).
//
// A thread takes 32 values and passes them through emit_pair, the quantizer's
// own scale-round-pack code, as the two 16-element vectors of one block whose
// amax is qmax, with n = 1.  The block's reciprocal is then exactly 1 before
// the power-of-two factor each path folds in (fp32 scales: s = qmax / qmax;
// UE8M0: exponent 0), so the step sees the values themselves.
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "quantize_common.cuh"
#include "ufp4_device.cuh"

namespace ufp4 {

template <int GRID, bool SR, int SF>
__global__ void __launch_bounds__(256) round_levels_kernel(const float* __restrict__ t,
                                                           const uint16_t* __restrict__ u16, int64_t groups,
                                                           uint8_t* __restrict__ codes) {
    const int64_t gi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (gi >= groups) return;
    const float4* tv = reinterpret_cast<const float4*>(t + gi * 32);
    float v[32];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float4 q = tv[k];
        v[4 * k] = q.x; v[4 * k + 1] = q.y; v[4 * k + 2] = q.z; v[4 * k + 3] = q.w;
    }
    uint64_t e[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) e[i] = pk2(v[i], v[16 + i]);
    Fold fd;
    fd.g = 0.0f;
    fd.inv_s = 1.0f;
    fd.pow4 = true;
    fd.j = 0;
    Dest A, B;
    A.codes = codes + gi * 16;
    B.codes = A.codes + 8;
    A.s0 = A.s1 = B.s0 = B.s1 = nullptr;  // no scale is written (w0 = w1 = false)
    A.valid = B.valid = true;
    A.w0 = A.w1 = B.w0 = B.w1 = false;
    A.lin0 = B.lin0 = 0;
    SrDraws dr{};
    if (SR) {
        // draw of element i: word i / 2, low half for even i (the quantizer's layout)
        const uint32_t* w = reinterpret_cast<const uint32_t*>(u16 + gi * 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            dr.a[k] = w[k];
            dr.b[k] = w[8 + k];
        }
    }
    constexpr float q = grid_qmax(GRID);
    emit_pair<GRID, SR, SF>(e, q, q, q, q, false, fd, A, B, dr);
}

namespace {
template <int GRID, bool SR>
cudaError_t launch_sf(int sf, const float* t, const uint16_t* u16, int64_t groups, uint8_t* codes, cudaStream_t st) {
    const unsigned blocks = (unsigned)((groups + 255) / 256);
    if (sf == 0)
        round_levels_kernel<GRID, SR, 0><<<blocks, 256, 0, st>>>(t, u16, groups, codes);
    else
        round_levels_kernel<GRID, SR, 1><<<blocks, 256, 0, st>>>(t, u16, groups, codes);
    return cudaGetLastError();
}
template <int GRID>
cudaError_t launch_grid(bool sr, int sf, const float* t, const uint16_t* u16, int64_t groups, uint8_t* codes,
                        cudaStream_t st) {
    return sr ? launch_sf<GRID, true>(sf, t, u16, groups, codes, st)
              : launch_sf<GRID, false>(sf, t, u16, groups, codes, st);
}
}  // namespace

cudaError_t launch_round_levels(int grid, bool sr, int sf, const float* t, const uint16_t* u16, int64_t count,
                                uint8_t* codes, cudaStream_t st) {
    const int64_t groups = count / 32;
    if (groups == 0) return cudaSuccess;
    if (groups > (int64_t)0x7FFFFFFF * 256) return cudaErrorInvalidValue;
    switch (grid) {
        case 0: return launch_grid<0>(sr, sf, t, u16, groups, codes, st);
        case 1: return launch_grid<1>(sr, sf, t, u16, groups, codes, st);
        case 2: return launch_grid<2>(sr, sf, t, u16, groups, codes, st);
        case 3: return launch_grid<3>(sr, sf, t, u16, groups, codes, st);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t preload_round_levels_kernels() {
    cudaFuncAttributes a;
    cudaFuncGetAttributes(&a, round_levels_kernel<0, false, 0>);
    cudaFuncGetAttributes(&a, round_levels_kernel<0, false, 1>);
    cudaFuncGetAttributes(&a, round_levels_kernel<0, true, 0>);
    cudaFuncGetAttributes(&a, round_levels_kernel<0, true, 1>);
    cudaFuncGetAttributes(&a, round_levels_kernel<1, false, 0>);
    cudaFuncGetAttributes(&a, round_levels_kernel<1, false, 1>);
    cudaFuncGetAttributes(&a, round_levels_kernel<1, true, 0>);
    cudaFuncGetAttributes(&a, round_levels_kernel<1, true, 1>);
    cudaFuncGetAttributes(&a, round_levels_kernel<2, false, 0>);
    cudaFuncGetAttributes(&a, round_levels_kernel<2, false, 1>);
    cudaFuncGetAttributes(&a, round_levels_kernel<2, true, 0>);
    cudaFuncGetAttributes(&a, round_levels_kernel<2, true, 1>);
    cudaFuncGetAttributes(&a, round_levels_kernel<3, false, 0>);
    cudaFuncGetAttributes(&a, round_levels_kernel<3, false, 1>);
    cudaFuncGetAttributes(&a, round_levels_kernel<3, true, 0>);
    return cudaFuncGetAttributes(&a, round_levels_kernel<3, true, 1>);
}

}  // namespace ufp4
