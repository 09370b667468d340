// ufp4_gemm_noalloc: the quantized GEMM for callers that may not allocate
// device memory.  Instead of a caller-supplied workspace it uses one fixed
// scratch array that lives in this library's device image.
//
// Who needs it: code that runs where cudaMalloc is off limits -- inside a
// plugin or custom op whose host framework owns every allocation and hands
// out none for scratch, or in a latency-critical loop where an allocation
// (which can synchronize the whole device) is not acceptable.
// Such callers still own and pass A, B and D; only the scratch moves here.
#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

#include "../../include/ufp4.h"
#include "internal.h"

namespace {

// The scratch array: every GPU that loads this library holds it until the
// process exits.  In host code `g_noalloc_scratch` is only a host-side
// handle, never a device address; its device address comes from
// cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) uint8_t g_noalloc_scratch[UFP4_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call on that device).  Returns nullptr on failure.
void* scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" ufp4_status ufp4_gemm_noalloc(const ufp4_qtensor* A, const ufp4_qtensor* B,
                                         const ufp4_quant_desc* desc, float* D, int64_t ldd,
                                         cudaStream_t stream) {
    if (!A || !B || !desc) return UFP4_ERR_INVALID_ARG;
    size_t need = 0;
    const ufp4_status st = ufp4_gemm_workspace_size(A->rows, B->rows, A->cols, desc, &need);
    if (st != UFP4_OK) return st;
    if (need > (size_t)UFP4_NOALLOC_SCRATCH_BYTES) return UFP4_ERR_UNSUPPORTED;  // beyond the fixed scratch
    void* scratch = scratch_on_current_device();
    if (!scratch) return UFP4_ERR_CUDA;
    // Nothing in the scratch has to start at zero: the operand preparation
    // writes every byte the GEMM kernel later reads.
    return ufp4_gemm(A, B, desc, D, ldd, scratch, (size_t)UFP4_NOALLOC_SCRATCH_BYTES, stream);
}
