// Forward kernel instantiations for e4m3 Q, K, V at head dims 64, 128 and 256.
#include "fa_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_f8_d64(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<64, true>(p, grid, stream);
}
cudaError_t launch_fwd_f8_d64_dual(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<64, true, true>(p, grid, stream);
}
cudaError_t launch_fwd_f8_d64_persist(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<64, true, false, true>(p, grid, stream);
}
cudaError_t launch_fwd_f8_d128_persist(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<128, true, false, true>(p, grid, stream);
}
cudaError_t launch_fwd_f8_d128(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<128, true>(p, grid, stream);
}
cudaError_t launch_fwd_f8_d128_dual(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<128, true, true>(p, grid, stream);
}
cudaError_t launch_fwd_f8_d256(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    return launch_fwd<256, true>(p, grid, stream);
}
}  // namespace fa
