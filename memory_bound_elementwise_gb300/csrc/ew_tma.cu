// ew_tma.cu -- bulk-copy staging variant and the device error word.
#include "ew_internal.h"

namespace ew {

// Written by a kernel whose bounded wait gave up (the value names the wait
// site); read and cleared by the host through ew_device_error.
__device__ int32_t g_device_error = 0;

cudaError_t read_and_clear_device_error(cudaStream_t s, int32_t *code) {
    int32_t v = 0;
    const int32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_device_error, sizeof(v), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess && v != 0)
        e = cudaMemcpyToSymbolAsync(g_device_error, &zero, sizeof(zero), 0,
                                    cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    *code = v;
    return e;
}

const TmaEntry *tma_entry(int, int) { return nullptr; }

}  // namespace ew
