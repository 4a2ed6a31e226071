// fa_combine.cu — merge of split-KV partial states, one warp per query row.
//
// Merge operator ("AI 大模型之 FlashAttention_02", section "工程实操 沿键切分的
// 归约与沿查询切分的区别", steps 2-3): with M = max_s m_s and w_s = exp(m_s - M),
//   L = sum_s w_s l_s,   O = (sum_s w_s O_s) / L,   LSE = M + ln L.
// Splits with m_s = -inf (empty, or every key masked) get weight 0.
// HBM-bound: each row reads num_splits * (d + 2) floats and writes d bf16 + 1
// float; a warp reads one split's d floats as one contiguous 4*d-byte segment.
#include <cuda_bf16.h>

#include "fa_internal.h"

namespace fa {

constexpr int kCombineWarps = 8;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int D>
__global__ void __launch_bounds__(kCombineWarps * 32)
    fa_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_m,
                      const float* __restrict__ ws_l, __nv_bfloat16* __restrict__ o,
                      float* __restrict__ lse, long long rows, int num_splits) {
    constexpr int PER = D / 32;  // output elements per lane: 2, 4 or 8
    const long long row = static_cast<long long>(blockIdx.x) * kCombineWarps + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;

    float big_m = -INFINITY;
    for (int s = lane; s < num_splits; s += 32) big_m = fmaxf(big_m, ws_m[s * rows + row]);
    big_m = warp_max(big_m);
    const float ref = (big_m == -INFINITY) ? 0.f : big_m;

    float big_l = 0.f;
    for (int s = lane; s < num_splits; s += 32) {
        const float ms = ws_m[s * rows + row];
        if (ms != -INFINITY) big_l += expf(ms - ref) * ws_l[s * rows + row];
    }
    big_l = warp_sum(big_l);

    float acc[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
#pragma unroll 4
    for (int s = 0; s < num_splits; ++s) {
        const float ms = ws_m[s * rows + row];  // same address in every lane: one broadcast
        if (ms == -INFINITY) continue;
        const float w = expf(ms - ref);
        const float* src = ws_o + (static_cast<size_t>(s) * rows + row) * D + lane * PER;
        if constexpr (PER == 2) {
            const float2 x = *reinterpret_cast<const float2*>(src);
            acc[0] = fmaf(w, x.x, acc[0]);
            acc[1] = fmaf(w, x.y, acc[1]);
        } else {
#pragma unroll
            for (int i = 0; i < PER; i += 4) {
                const float4 x = *reinterpret_cast<const float4*>(src + i);
                acc[i + 0] = fmaf(w, x.x, acc[i + 0]);
                acc[i + 1] = fmaf(w, x.y, acc[i + 1]);
                acc[i + 2] = fmaf(w, x.z, acc[i + 2]);
                acc[i + 3] = fmaf(w, x.w, acc[i + 3]);
            }
        }
    }
    const float inv = (big_l > 0.f) ? 1.f / big_l : 0.f;
    __nv_bfloat162 packed[PER / 2];
#pragma unroll
    for (int i = 0; i < PER / 2; ++i)
        packed[i] = __floats2bfloat162_rn(acc[2 * i] * inv, acc[2 * i + 1] * inv);
    __nv_bfloat16* dst = o + static_cast<size_t>(row) * D + lane * PER;
    if constexpr (PER == 2) {
        *reinterpret_cast<__nv_bfloat162*>(dst) = packed[0];
    } else if constexpr (PER == 4) {
        *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(packed);
    } else {
        *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(packed);
    }
    if (lane == 0) lse[row] = (big_l > 0.f) ? ref + logf(big_l) : -INFINITY;
}

cudaError_t launch_combine(const float* ws_o, const float* ws_m, const float* ws_l, void* o,
                           float* lse, long long rows, int num_splits, int d,
                           cudaStream_t stream) {
    const long long blocks = (rows + kCombineWarps - 1) / kCombineWarps;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(kCombineWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    auto* out = static_cast<__nv_bfloat16*>(o);
    switch (d) {
        case 64:
            return cudaLaunchKernelEx(&cfg, fa_combine_kernel<64>, ws_o, ws_m, ws_l, out, lse, rows,
                                      num_splits);
        case 128:
            return cudaLaunchKernelEx(&cfg, fa_combine_kernel<128>, ws_o, ws_m, ws_l, out, lse,
                                      rows, num_splits);
        case 256:
            return cudaLaunchKernelEx(&cfg, fa_combine_kernel<256>, ws_o, ws_m, ws_l, out, lse,
                                      rows, num_splits);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace fa
