// Test hook: the objective's phase function on its own (accuracy test of fast_atan2).
#include "../../include/ssb_debug.h"
#include "ssb_device.cuh"
#include "ssb_internal.h"

namespace ssb {

__global__ void k_atan2(const float *__restrict__ y, const float *__restrict__ x, size_t n,
                        float *__restrict__ out) {
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        out[i] = fast_atan2(y[i], x[i]);
}

}  // namespace ssb

extern "C" ssb_status ssb_debug_atan2(const float *y_device, const float *x_device, size_t n,
                                      float *out_device, void *cuda_stream) {
    ssb::set_last_error("");
    if (n == 0) return SSB_OK;
    if (!y_device || !x_device || !out_device) {
        ssb::set_last_error("NULL argument");
        return SSB_ERR_ARG;
    }
    cudaStream_t s = (cudaStream_t)cuda_stream;
    const size_t blocks = (n + 255) / 256;
    ssb::k_atan2<<<(unsigned)(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(y_device, x_device, n,
                                                                           out_device);
    ssb::count_launch();
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        ssb::set_last_error(cudaGetErrorString(e));
        return SSB_ERR_CUDA;
    }
    return SSB_OK;
}
