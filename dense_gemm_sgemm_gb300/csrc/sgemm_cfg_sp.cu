// SGEMM kernels of one tile configuration: 64 x 64 tiles, every tile split in two K halves
// that form a two-CTA cluster and hand off through distributed shared memory (all loader
// modes).
#include "sgemm_kernel.cuh"

namespace gemm {
namespace sg {

cudaError_t launch_SP(int dev_id, int a_mode, int b_mode, const SgemmParams &p, cudaStream_t s)
{
    return launch_ab<CfgS, true, true>(dev_id, a_mode, b_mode, p, s);
}

}  // namespace sg
}  // namespace gemm
