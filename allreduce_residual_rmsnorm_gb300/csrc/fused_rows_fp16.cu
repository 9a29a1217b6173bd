// fp16 instantiations of the register-resident row kernels.
#include "fused_rows_impl.cuh"

namespace arf {
cudaError_t launch_fused_rows_fp16(int variant, const FusedArgs& a, const LaunchCfg& c)
{
    return launch_fused_rows_t<Fp16>(variant, a, c);
}
}  // namespace arf
