// bf16 instantiations of the register-resident row kernels.
#include "fused_rows_impl.cuh"

namespace arf {
cudaError_t launch_fused_rows_bf16(int variant, const FusedArgs& a, const LaunchCfg& c)
{
    return launch_fused_rows_t<Bf16>(variant, a, c);
}
}  // namespace arf
