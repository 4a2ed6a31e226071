// fa_combine.cu — merge of split-KV partial states.
//
// Merge operator ("AI 大模型之 FlashAttention_02", section "工程实操 沿键切分的
// 归约与沿查询切分的区别", steps 2-3): with M = max_s m_s and w_s = exp(m_s - M),
//   L = sum_s w_s l_s,   O = (sum_s w_s O_s) / L,   LSE = M + ln L.
// Splits with m_s = -inf (empty, or every key masked) get weight 0.
//
// HBM-bound and short: at decode shapes the whole workspace is a few tens of
// MB, more than the register file of the GPU can hold in flight, so a warp
// must stream: W warps share a row (W = 1, 2, 4 or 8, from the split count);
// warp w takes splits w, w + W, ... in batches of partial rows (64 floats per
// lane per batch), and the loads of its next batch are in flight while it sums
// the current one (two register buffers). Each lane owns d/32 consecutive
// columns, so a warp reads a split's row as one contiguous 4d-byte segment with
// vector loads. Before it waits for anything a warp has its first two batches
// and the row's m and l of every split (lane-strided) in flight; it then forms
// M, the weights w_s = exp(m_s - M) (each by the lane that loaded m_s, kept in
// shared memory for the whole warp) and L = sum_s w_s l_s. With W > 1 the
// warps' sums meet in shared memory; every warp computes the same M and L, so
// no rescaling is needed there.
#include <atomic>
#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

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
struct CombineShape {
    static constexpr int PER = D / 32;                     // columns per lane: 2, 4, 8
    static constexpr int BATCH = 32 / PER;                 // partial rows per batch (32 floats a lane)
    static constexpr int MAX_WARPS = 8;                    // warps per row, at most
    static constexpr int MREGS = FA_MAX_SPLITS / 32;       // m (and l) values per lane
};

// One lane's PER consecutive floats of a partial row.
template <int PER>
__device__ __forceinline__ void load_cols(float* x, const float* src) {
    if constexpr (PER == 2) {
        const float2 a = *reinterpret_cast<const float2*>(src);
        x[0] = a.x;
        x[1] = a.y;
    } else {
#pragma unroll
        for (int i = 0; i < PER; i += 4) {
            const float4 a = *reinterpret_cast<const float4*>(src + i);
            x[i] = a.x;
            x[i + 1] = a.y;
            x[i + 2] = a.z;
            x[i + 3] = a.w;
        }
    }
}

// Block: rows_per_block rows x W warps; warp = r * W + wi.
template <int D>
__global__ void __launch_bounds__(256)
    fa_combine_kernel(const float* __restrict__ ws_o, const float* __restrict__ ws_m,
                      const float* __restrict__ ws_l, __nv_bfloat16* __restrict__ o,
                      float* __restrict__ lse, long long rows, int num_splits, int W) {
    using Sh = CombineShape<D>;
    constexpr int PER = Sh::PER, BATCH = Sh::BATCH;
    __shared__ float part[Sh::MAX_WARPS][D];
    __shared__ float wsh[Sh::MAX_WARPS][FA_MAX_SPLITS];

    // Launched with programmatic stream serialization after the split-KV
    // kernel: nothing here reads the workspace before that grid has completed.
    // A forward launched next may be scheduled once every CTA here has started.
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();
    const int S = num_splits;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rows_per_block = (blockDim.x >> 5) / W;
    const int r = warp / W, wi = warp % W;
    const long long row = static_cast<long long>(blockIdx.x) * rows_per_block + r;
    const bool live = row < rows;
    // Splits of this warp: s = wi + W * i, i < n.
    const int n = (live && wi < S) ? (S - wi + W - 1) / W : 0;
    const float* col = ws_o + static_cast<size_t>(live ? row : 0) * D + lane * PER;
    const size_t split_stride = static_cast<size_t>(rows) * D;

    float xa[BATCH][PER], xb[BATCH][PER];
    auto load_batch = [&](float (&x)[BATCH][PER], int b0) {
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            if (b0 + i < n) {
                load_cols<PER>(x[i], col + static_cast<size_t>(wi + W * (b0 + i)) * split_stride);
            } else {
#pragma unroll
                for (int e = 0; e < PER; ++e) x[i][e] = 0.f;
            }
        }
    };
    load_batch(xa, 0);
    load_batch(xb, BATCH);

    // m and l of split lane + 32 k, then M, the weights and L.
    float mv[Sh::MREGS], lv[Sh::MREGS];
    float mx = -INFINITY;
#pragma unroll
    for (int k = 0; k < Sh::MREGS; ++k) {
        const int sp = lane + 32 * k;
        const bool ok = live && sp < S;
        const size_t idx = static_cast<size_t>(ok ? sp : 0) * rows + (live ? row : 0);
        mv[k] = ok ? ws_m[idx] : -INFINITY;
        lv[k] = ok ? ws_l[idx] : 0.f;
        mx = fmaxf(mx, mv[k]);
    }
    mx = warp_max(mx);
    const float ref = (mx == -INFINITY) ? 0.f : mx;
    float lsum = 0.f;
#pragma unroll
    for (int k = 0; k < Sh::MREGS; ++k) {
        const int sp = lane + 32 * k;
        const float wk = (mv[k] == -INFINITY) ? 0.f : expf(mv[k] - ref);
        lsum = fmaf(wk, lv[k], lsum);
        if (sp < S) wsh[warp][sp] = wk;
    }
    lsum = warp_sum(lsum);
    __syncwarp();

    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    auto sum_batch = [&](const float (&x)[BATCH][PER], int b0) {
#pragma unroll
        for (int i = 0; i < BATCH; ++i) {
            if (b0 + i < n) {
                const float w = wsh[warp][wi + W * (b0 + i)];
#pragma unroll
                for (int e = 0; e < PER; ++e) acc[e] = fmaf(w, x[i][e], acc[e]);
            }
        }
    };
    // Two batches per trip: while one buffer is summed, the other's loads fly.
    for (int b0 = 0; b0 < n; b0 += 2 * BATCH) {
        sum_batch(xa, b0);
        if (b0 + 2 * BATCH < n) load_batch(xa, b0 + 2 * BATCH);
        if (b0 + BATCH < n) sum_batch(xb, b0 + BATCH);
        if (b0 + 3 * BATCH < n) load_batch(xb, b0 + 3 * BATCH);
    }

    if (W > 1) {  // the same for every thread of the launch
#pragma unroll
        for (int e = 0; e < PER; ++e) part[warp][lane * PER + e] = acc[e];
        __syncthreads();
        if (wi == 0) {
            for (int k = 1; k < W; ++k) {
#pragma unroll
                for (int e = 0; e < PER; ++e) acc[e] += part[warp + k][lane * PER + e];
            }
        }
    }
    if (wi == 0 && live) {
        const float inv = (lsum > 0.f) ? 1.f / lsum : 0.f;
        __nv_bfloat162 packed[PER / 2];
#pragma unroll
        for (int e = 0; e < PER / 2; ++e)
            packed[e] = __floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv);
        __nv_bfloat16* dst = o + static_cast<size_t>(row) * D + lane * PER;
        if constexpr (PER == 2) {
            *reinterpret_cast<__nv_bfloat162*>(dst) = packed[0];
        } else if constexpr (PER == 4) {
            *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(packed);
        } else {
            *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(packed);
        }
        if (lane == 0) lse[row] = (lsum > 0.f) ? ref + logf(lsum) : -INFINITY;
    }
}

// Blocks of this kernel the whole GPU holds at once at `threads` threads per
// block (per-SM occupancy x SMs), queried once per device and block size.
// Concurrent first calls may both query; they store the same value through an
// atomic, so the cache is race-free.
template <int D>
int combine_resident_blocks(int threads) {
    static std::atomic<int> cache[64][2];  // [device][threads == 256]
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
    std::atomic<int>& slot = cache[dev][threads == 256 ? 1 : 0];
    int value = slot.load(std::memory_order_relaxed);
    if (value == 0) {
        int per_sm = 0, sms = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fa_combine_kernel<D>, threads, 0) !=
                cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return 1;
        value = (per_sm > 0 ? per_sm : 1) * (sms > 0 ? sms : 1);
        slot.store(value, std::memory_order_relaxed);
    }
    return value;
}

// Warps per row W (1, 2, 4 or 8): enough for two batches per warp (one trip of
// the streaming loop), reduced while the grid would not fit on the GPU in one
// wave; then each warp streams more batches. Blocks hold four warps (four rows
// at W = 1) or, at W = 8, eight.
template <int D>
cudaError_t launch_combine_d(const float* ws_o, const float* ws_m, const float* ws_l,
                             __nv_bfloat16* o, float* lse, long long rows, int num_splits,
                             cudaStream_t stream) {
    using Sh = CombineShape<D>;
    const int trips = (num_splits + 2 * Sh::BATCH - 1) / (2 * Sh::BATCH);
    int W = 1;
    while (W < trips && W < Sh::MAX_WARPS) W <<= 1;
    auto blocks_for = [rows](int w) {
        const int per_block = (w > 4 ? w : 4) / w;
        return (rows + per_block - 1) / per_block;
    };
    while (W > 1 && blocks_for(W) > combine_resident_blocks<D>(W > 4 ? W * 32 : 128)) W >>= 1;
    const int warps = W > 4 ? W : 4;
    const long long blocks = blocks_for(W);
    if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(warps * 32), 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    // Programmatic dependent launch: the merge may be scheduled while the
    // split-KV grid before it in the stream finishes (the kernel waits for that
    // grid's completion before its first read), which hides the launch gap.
    cudaLaunchAttribute attr = {};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, fa_combine_kernel<D>, ws_o, ws_m, ws_l, o, lse, rows,
                              num_splits, W);
}

cudaError_t launch_combine(const float* ws_o, const float* ws_m, const float* ws_l, void* o,
                           float* lse, long long rows, int num_splits, int d,
                           cudaStream_t stream) {
    auto* out = static_cast<__nv_bfloat16*>(o);
    switch (d) {
        case 64:
            return launch_combine_d<64>(ws_o, ws_m, ws_l, out, lse, rows, num_splits, stream);
        case 128:
            return launch_combine_d<128>(ws_o, ws_m, ws_l, out, lse, rows, num_splits, stream);
        case 256:
            return launch_combine_d<256>(ws_o, ws_m, ws_l, out, lse, rows, num_splits, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace fa
