// Bulk-copy pipelined fused epilogue (persistent blocks).  Not built yet.
#include "ar_internal.h"

namespace arf {
bool fused_pipe_supported(int, int, int) { return false; }
cudaError_t launch_fused_pipe(int, const FusedArgs&, const LaunchCfg&) { return cudaErrorNotSupported; }
}  // namespace arf
