// fp32 instantiations of the register-resident row kernels (the 4-byte
// exchange type of FlashInfer's use_fp32_lamport workspaces).
#include "fused_rows_impl.cuh"

namespace arf {
cudaError_t launch_fused_rows_fp32(int variant, const FusedArgs& a, const LaunchCfg& c)
{
    return launch_fused_rows_t<F32>(variant, a, c);
}
}  // namespace arf
