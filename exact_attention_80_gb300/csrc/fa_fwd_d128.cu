// Forward kernel instantiation for head dim 128 (one translation unit per head
// dim so the three compile in parallel).
#include "fa_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_d128(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<128>(p, grid, stream);
}
cudaError_t launch_fwd_d128_dual(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<128, false, true>(p, grid, stream);
}
cudaError_t launch_fwd_d128_rows64(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<128, false, false, false, true>(p, grid, stream);
}
cudaError_t launch_fwd_d128_persist(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<128, false, false, true>(p, grid, stream);
}
}  // namespace fa
