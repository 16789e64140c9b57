// Backward attention on sm_103a tensor cores (placeholder entry: routes to the SIMT kernels
// until the tensor-core kernels land).
#include "fa_common.cuh"

namespace fa {
cudaError_t launch_bwd_simt(int d, int is_f32, const BwdParams& p, cudaStream_t st);

cudaError_t launch_bwd_tc(int d, const CUtensorMap* maps, const BwdParams& p, cudaStream_t st)
{
    (void)maps;
    return launch_bwd_simt(d, 0, p, st);
}
}  // namespace fa
