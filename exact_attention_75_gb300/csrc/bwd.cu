#include "bwd.cuh"
namespace attn {
cudaError_t launch_bwd(const BwdLaunch&) { return cudaErrorNotSupported; }
}  // namespace attn
