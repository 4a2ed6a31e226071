// Forward kernel instantiation for head dim 64 (one translation unit per head
// dim so the three compile in parallel).
#include "fa_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d64(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<64>(p, grid, stream);
}
cudaError_t launch_fwd_d64_dual(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<64, false, true>(p, grid, stream);
}
cudaError_t launch_fwd_d64_rows64(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<64, false, false, false, true>(p, grid, stream);
}
cudaError_t launch_fwd_d64_persist(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<64, false, false, true>(p, grid, stream);
}
}  // namespace fa
