// SGEMM kernels of one tile configuration: 128 x 256 tiles (all loader modes).
#include "sgemm_kernel.cuh"

namespace gemm {
namespace sg {

cudaError_t launch_X(int dev_id, int a_mode, int b_mode, const SgemmParams &p, cudaStream_t s)
{
    return launch_ab<CfgX, false>(dev_id, a_mode, b_mode, p, s);
}

}  // namespace sg
}  // namespace gemm
