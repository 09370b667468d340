// The general quantizer kernel's SR instantiations (the kernel template is in
// quantize_general.cuh; quantize.cu holds the RTNE ones), compiled as a unit
// of their own so that the two compile in parallel.
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "quantize_general.cuh"

namespace ufp4 {

cudaError_t launch_quantize_sr(const CUtensorMap& map, const QuantParams& p, int grid, bool po2, int tc,
                               int num_tiles, int num_sms, cudaStream_t st) {
    return launch_general<true>(map, p, grid, po2, tc, num_tiles, num_sms, st);
}

cudaError_t sr_error_read_clear(int* value) { return general_error_read_clear(value); }

cudaError_t set_sr_wait_limit(uint32_t polls) { return general_set_wait_limit(polls); }

cudaError_t preload_quantize_sr_kernels() { return preload_general<true>(); }

}  // namespace ufp4
