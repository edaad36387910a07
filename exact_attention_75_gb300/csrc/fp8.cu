#include "fp8.cuh"
namespace attn {
cudaError_t launch_quantize(const QuantLaunch&) { return cudaErrorNotSupported; }
cudaError_t launch_fwd_fp8(const Fp8FwdLaunch&) { return cudaErrorNotSupported; }
}  // namespace attn
