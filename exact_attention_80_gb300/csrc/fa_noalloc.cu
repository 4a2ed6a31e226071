// fa_noalloc.cu — fa_fwd_splitkv_static: the split-KV forward and merge with
// their partial states in a library-owned static device buffer, for callers
// that cannot allocate device memory themselves (see include/fa.h).
#include "fa.h"
#include "fa_internal.h"

namespace fa {
namespace {

// The partial-state scratch shared by every call on a device. In host code
// this name is only a stand-in for the device object: kernels get the device
// address looked up below, never this symbol.
static __device__ __align__(256) float g_static_scratch[FA_STATIC_SCRATCH_BYTES / sizeof(float)];

// Device address of the scratch on the current device, looked up with that
// device current (cudaGetSymbolAddress) on the first call in each CUDA context
// and cached; a new context (after cudaDeviceReset) gets a fresh lookup.
cudaError_t static_scratch(float** out) {
    static ContextCache<float*> cache;
    return cache.get(out, [](float** ptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        *ptr = static_cast<float*>(p);
        return e;
    });
}

}  // namespace
}  // namespace fa

extern "C" fa_status fa_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o,
                                           float* lse, int B, int H, int Nq, int Nk, int d,
                                           float scale, int causal, int num_splits,
                                           cudaStream_t stream) {
    // Everything checkable on the host (pointers, alignment, shapes, scale,
    // mask, split count) is checked before the size test and before any CUDA
    // call, so a refused call has queued no work; the calls below repeat it.
    const fa_status s0 = fa::check_common(q, k, v, B, H, Nq, Nk, d, scale);
    if (s0 != FA_OK) return s0;
    if (!fa::valid_causal(causal)) return FA_ERR_CAUSAL;
    if (!o || !lse) return FA_ERR_NULL;
    if (!fa::aligned(o, 16) || !fa::aligned(lse, 4)) return FA_ERR_ALIGN;
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
