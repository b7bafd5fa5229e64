// fp16-input / fp32-accumulate GEMM on the tcgen05 tensor cores of sm_103a.
#include <cuda_runtime.h>

#include "gemm_internal.h"

namespace gemm {

// Error word raised by kernels whose bounded barrier waits expire (0 = no error).
__device__ unsigned int g_device_status = 0;

gemm_status_t launch_hgemm(const DeviceInfo &, int, int, int64_t, int64_t, int64_t, float,
                           const uint16_t *, int64_t, const uint16_t *, int64_t, float, float *,
                           int64_t, cudaStream_t)
{
    return GEMM_ERR_UNSUPPORTED;
}

gemm_status_t read_and_clear_device_status(cudaStream_t stream)
{
    unsigned int word = 0;
    const unsigned int zero = 0;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_LAUNCH;
    if (cudaMemcpyFromSymbol(&word, g_device_status, sizeof(word)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_device_status, &zero, sizeof(zero)) != cudaSuccess)
        return GEMM_ERR_LAUNCH;
    return word ? GEMM_ERR_DEVICE_TIMEOUT : GEMM_OK;
}

}  // namespace gemm
