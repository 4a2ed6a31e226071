// fa_noalloc.cu — fa_fwd_splitkv_static: the split-KV forward and merge with
// their partial states in a library-owned static device buffer, for callers
// that cannot allocate device memory themselves (see include/fa.h).
#include <mutex>

#include "fa.h"

namespace fa {
namespace {

// The partial-state scratch shared by every call on a device. In host code
// this name is only a stand-in for the device object: kernels get the device
// address looked up below, never this symbol.
static __device__ __align__(256) float g_static_scratch[FA_STATIC_SCRATCH_BYTES / sizeof(float)];

std::mutex g_scratch_mutex;
float* g_scratch_ptr[64] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
cudaError_t static_scratch(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool valid_head_dim(int d) { return d == 64 || d == 128 || d == 256; }

}  // namespace
}  // namespace fa

extern "C" fa_status fa_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o,
                                           float* lse, int B, int H, int Nq, int Nk, int d,
                                           float scale, int causal, int num_splits,
                                           cudaStream_t stream) {
    // Everything checkable on the host is checked before the size test and
    // before any CUDA call; the calls below repeat the full validation.
    if (!q || !k || !v || !o || !lse) return FA_ERR_NULL;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_SHAPE;
    if (!fa::valid_head_dim(d)) return FA_ERR_HEADDIM;
    if (num_splits < 1 || num_splits > FA_MAX_SPLITS) return FA_ERR_SPLITS;
    const size_t need = fa_splitkv_workspace_bytes(B, H, Nq, d, num_splits);
    if (need == 0) return FA_ERR_SHAPE;
    if (need > FA_STATIC_SCRATCH_BYTES) return FA_ERR_SCRATCH;
    float* scratch = nullptr;
    if (fa::static_scratch(&scratch) != cudaSuccess) return FA_ERR_CUDA;
    const fa_status s = fa_fwd_splitkv(q, k, v, scratch, B, H, Nq, Nk, d, scale, causal,
                                       num_splits, stream);
    if (s != FA_OK) return s;
    return fa_combine(scratch, o, lse, B, H, Nq, d, num_splits, stream);
}
