// fa_fwd_kernel.cuh — selects the forward kernel design per head dim and
// launches it.
//   d = 64, 128: fa_fwd_tm.cuh — two 128-row query tiles per CTA, BN = 128,
//                P handed to the PV MMA in TMEM over its S columns, the two
//                tiles alternating on the tensor core.
//   d = 256:     fa_fwd_tp.cuh — one query tile per CTA (O takes half of TMEM),
//                BN = 96, S double-buffered in TMEM with P packed over it.
//   e4m3 inputs: the same kernels instantiated for 8-bit operands (d = 64,
//                128: fa_fwd_tm.cuh; d = 256: fa_fwd_tp.cuh).
//   Plain launches of at least four waves of units at d = 64, 128 run the
//   two-tile kernel's persistent form (one CTA per SM).
#pragma once

#include <type_traits>

#include "fa_fwd_tm.cuh"
#include "fa_fwd_tp.cuh"

namespace fa {

template <int D>
using FwdLayout = std::conditional_t<D == 256, LayoutTP<D>, LayoutTM<D>>;

// F8: e4m3 inputs. DUAL: dual-range split-KV CTAs (one query tile). PERSIST:
// persistent CTAs (plain mode). All are forms of the two-tile kernel
// (d = 64 or 128), but for e4m3 at d = 256.
// M64: one 64-row query tile per CTA (bf16, d = 64 or 128).
template <int D, bool F8 = false, bool DUAL = false, bool PERSIST = false, bool M64 = false>
cudaError_t launch_fwd(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    using L = std::conditional_t<
        PERSIST, LayoutTM<D, F8, true>,
        std::conditional_t<F8, std::conditional_t<D == 256, LayoutTP<D, true>, LayoutTM<D, true>>, FwdLayout<D>>>;
    constexpr auto kernel = [] {
        if constexpr (M64) return fa_fwd_tm64_kernel<D>;
        else if constexpr (PERSIST && F8) return fa_fwd_tmp8_kernel<D>;
        else if constexpr (PERSIST) return fa_fwd_tmp_kernel<D>;
        else if constexpr (F8 && DUAL) return fa_fwd_tm8d_kernel<D>;
        else if constexpr (F8 && D == 256) return fa_fwd_tp8_kernel<D>;
        else if constexpr (F8) return fa_fwd_tm8_kernel<D>;
        else if constexpr (DUAL) return fa_fwd_tmd_kernel<D>;
        else if constexpr (D == 256) return fa_fwd_tp_kernel<D>;
        else return fa_fwd_tm_kernel<D>;
    }();
    // Kernel attributes belong to the context: set once per device and context.
    static ContextCache<int> attr_set;
    int done = 0;
    cudaError_t e = attr_set.get(&done, [kernel](int* out) {
        if constexpr (L::REG_SPLIT) {
            // The setmaxnreg split is sized for exactly LAUNCH_REGS per thread.
            cudaFuncAttributes a;
            cudaError_t err = cudaFuncGetAttributes(&a, kernel);
            if (err != cudaSuccess) return err;
            if (a.numRegs != L::LAUNCH_REGS) return cudaErrorInvalidKernelImage;
        }
        *out = 1;
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(L::ALLOC_BYTES));
    });
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(L::THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::ALLOC_BYTES;
    cfg.stream = stream;
    // Programmatic dependent launch: the kernels wait for the previous grid in
    // the stream before touching global memory, so their launch and start-up
    // may overlap its end.
    cudaLaunchAttribute attr = {};
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace fa
