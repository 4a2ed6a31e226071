// fa_api.cu — the C ABI declared in include/fa.h (the backward's entry points
// live beside its kernels in fa_bwd.cu): argument validation, TMA tensor-map
// encoding, work partition and kernel dispatch. Host code only, apart from the
// device status word defined here.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <atomic>
#include <mutex>

#include <cudaTypedefs.h>

#include "fa.h"
#include "fa_fwd_kernel.cuh"
#include "fa_internal.h"

namespace fa {

// Error word raised by kernels whose bounded waits give up (bits: fa_internal.h).
__device__ unsigned g_fa_device_status = 0u;

unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa = cudaDriverEntryPointSymbolNotFound;
        cudaDriverEntryPointQueryResult qb = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) ==
                cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
                cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<GetCurrent>(a);
            get_id = reinterpret_cast<GetId>(b);
        }
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    return get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

cudaError_t device_status_ptr(unsigned** ptr) {
    static ContextCache<unsigned*> cache;
    return cache.get(ptr, [](unsigned** out) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_fa_device_status);
        *out = static_cast<unsigned*>(p);
        return e;
    });
}

FwdConfig fwd_config(int d) {
    FwdConfig c = {};
    switch (d) {
        case 64:
            c = {FwdLayout<64>::Q_TILES, FwdLayout<64>::BN, FwdLayout<64>::STAGES,
                 FwdLayout<64>::THREADS, FwdLayout<64>::ALLOC_BYTES};
            break;
        case 128:
            c = {FwdLayout<128>::Q_TILES, FwdLayout<128>::BN, FwdLayout<128>::STAGES,
                 FwdLayout<128>::THREADS, FwdLayout<128>::ALLOC_BYTES};
            break;
        case 256:
            c = {FwdLayout<256>::Q_TILES, FwdLayout<256>::BN, FwdLayout<256>::STAGES,
                 FwdLayout<256>::THREADS, FwdLayout<256>::ALLOC_BYTES};
            break;
        default:
            break;
    }
    return c;
}

namespace {

cudaError_t sm_count(int* out) {
    static std::atomic<int> cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) {
            *out = c;
            return cudaSuccess;
        }
    }
    e = cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess && dev >= 0 && dev < 64) cache[dev].store(*out, std::memory_order_relaxed);
    return e;
}

}  // namespace

// Argument checks and tensor maps shared with the backward's entry points
// (declared in fa_internal.h).
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool valid_d(int d) { return d == 64 || d == 128 || d == 256; }

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// bf16 [BH][N][d] viewed as a 3-D tensor (d, N, BH); box = 64 columns x rows,
// 128-byte swizzle; rows past N read as zeros.
// 3-D bf16 map (d, rows, heads) with the given row and head strides in bytes,
// box {64, box_rows, 1}, 128-byte swizzle.
// Elements are bf16, or single bytes (e4m3) when `bytes`; the box is one
// 128-byte swizzle row wide (64 bf16 or 128 bytes), except for 64-byte e4m3
// rows (d = 64), which take a 64-byte box and the 64-byte swizzle.
bool encode_map(CUtensorMap* map, const void* base, int d, long long rows, long long heads,
                unsigned long long row_stride, unsigned long long head_stride, int box_rows,
                bool bytes = false) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(heads)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_stride),
                                   static_cast<cuuint64_t>(head_stride)};
    const bool row64 = bytes && d == 64;
    const cuuint32_t box[3] = {bytes ? (row64 ? 64u : 128u) : 64u, static_cast<cuuint32_t>(box_rows), 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r =
        enc(map, bytes ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, row64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Dense [BH][N][d]: rows d*2 bytes apart, heads N*d*2.
bool encode_rows_map(CUtensorMap* map, const void* base, int d, int N, int BH, int box_rows) {
    return encode_map(map, base, d, N, BH, static_cast<unsigned long long>(d) * 2,
                      static_cast<unsigned long long>(N) * d * 2, box_rows);
}

// Dense e4m3 [BH][N][d]: rows d bytes apart, heads N*d.
bool encode_rows_map8(CUtensorMap* map, const void* base, int d, int N, int BH, int box_rows) {
    return encode_map(map, base, d, N, BH, static_cast<unsigned long long>(d),
                      static_cast<unsigned long long>(N) * d, box_rows, true);
}

// Token-major packed [total][H][d] (variable-length batches): tokens H*d*2 bytes
// apart, heads d*2.
bool encode_tokens_map(CUtensorMap* map, const void* base, int d, int total, int H, int box_rows) {
    return encode_map(map, base, d, total, H, static_cast<unsigned long long>(H) * d * 2,
                      static_cast<unsigned long long>(d) * 2, box_rows);
}

bool valid_causal(int causal) {
    return causal == FA_CAUSAL_NONE || causal == FA_CAUSAL_TOP_LEFT || causal == FA_CAUSAL_BOTTOM_RIGHT;
}

fa_status check_common(const void* q, const void* k, const void* v, int B, int H, int Nq, int Nk,
                       int d, float scale) {
    if (!q || !k || !v) return FA_ERR_NULL;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_SHAPE;
    const long long bh = static_cast<long long>(B) * H;
    if (bh > 0x7fffffffll) return FA_ERR_SHAPE;
    if (!valid_d(d)) return FA_ERR_HEADDIM;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_SCALE;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16)) return FA_ERR_ALIGN;
    return FA_OK;
}

namespace {

long long grid_ctas(int B, int H, int Nq, int d, int num_splits, int tiles_per_cta = 0,
                    bool bm64 = false) {
    const FwdConfig c = fwd_config(d);
    const long long rows_per_cta = bm64 ? 64ll : 128ll * (tiles_per_cta > 0 ? tiles_per_cta : c.q_tiles);
    const long long units = (Nq + rows_per_cta - 1) / rows_per_cta;
    return static_cast<long long>(B) * H * units * num_splits;
}

// Variable-length batch description (device cu arrays; see include/fa.h).
struct Varlen {
    const int* cu_q;
    const int* cu_k;
    int total_q, total_k;
};

// Dense: Q [B][H][Nq][d], K/V [B][H][Nk][d]. Varlen (vl != nullptr): token-major
// packed sequences, Nq = max_seqlen_q, Nk = total_k, one work row per (b, h).
fa_status launch_forward(const void* q, const void* k, const void* v, void* o, float* lse,
                         float* ws, int B, int H, int Nq, int Nk, int d, float scale, int causal,
                         int num_splits, int split_mode, cudaStream_t stream,
                         long long wait_limit = kDefaultWaitLimit, int withhold_q = 0,
                         const Varlen* vl = nullptr, const float* f8_descale = nullptr,
                         int tiles_per_cta = 0, bool bm64 = false) {
    const FwdConfig c = fwd_config(d);
    // Persistent CTAs for the plain dense forward of the two-tile kernel
    // when its units fill at least four waves of CTAs and are short: the saved
    // CTA start-up and Q latency are per unit, the persistent control code's
    // slower key steps per step, and its static schedule balances long causal
    // units worse than the hardware does. Measured crossover (one unit per CTA
    // against persistent): persistent wins up to 16 key tiles of 128 (Nk <=
    // 2048), and non-causal d = 128 up to 32; beyond, one unit per CTA is as
    // fast or faster (up to 24 % on long causal sequences). fa_fwd_rows, which
    // fixes the rows per CTA, keeps one unit per CTA.
    const bool row_choice = tiles_per_cta > 0;
    if (tiles_per_cta <= 0) tiles_per_cta = c.q_tiles;
    const long long ctas = grid_ctas(B, H, Nq, d, num_splits, tiles_per_cta, bm64);
    if (ctas < 1 || ctas > 0x7fffffffll) return FA_ERR_SHAPE;
    const bool dual = use_dual(Nq, d, num_splits, split_mode, vl != nullptr);

    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    const int BH = B * H;
    if (vl) {
        if (!encode_tokens_map(&p.tm_q, q, d, vl->total_q, H, 128) ||
            !encode_tokens_map(&p.tm_k, k, d, vl->total_k, H, c.bn) ||
            !encode_tokens_map(&p.tm_v, v, d, vl->total_k, H, c.bn))
            return FA_ERR_CUDA;
        p.varlen = 1;
        p.H = H;
        p.total_q = vl->total_q;
        p.cu_q = vl->cu_q;
        p.cu_k = vl->cu_k;
    } else if (f8_descale) {
        // e4m3 Q, K, V; bf16 O in plain mode.
        if (!encode_rows_map8(&p.tm_q, q, d, Nq, BH, 128) ||
            !encode_rows_map8(&p.tm_k, k, d, Nk, BH, c.bn) ||
            !encode_rows_map8(&p.tm_v, v, d, Nk, BH, c.bn))
            return FA_ERR_CUDA;
        if (!split_mode && !encode_rows_map(&p.tm_o, o, d, Nq, BH, d == 256 ? 128 : 32)) return FA_ERR_CUDA;
    } else {
        if (!encode_rows_map(&p.tm_q, q, d, Nq, BH, 128) ||
            !encode_rows_map(&p.tm_k, k, d, Nk, BH, c.bn) ||
            !encode_rows_map(&p.tm_v, v, d, Nk, BH, c.bn))
            return FA_ERR_CUDA;
        if (!split_mode && !encode_rows_map(&p.tm_o, o, d, Nq, BH, d == 256 ? 128 : 32)) return FA_ERR_CUDA;
    }
    p.o = o;
    p.lse = lse;
    if (split_mode) {
        const size_t rows = static_cast<size_t>(BH) * Nq;
        p.ws_o = ws;
        p.ws_m = ws + static_cast<size_t>(num_splits) * rows * d;
        p.ws_l = p.ws_m + static_cast<size_t>(num_splits) * rows;
    }
    p.BH = BH;
    p.Nq = Nq;
    p.Nk = Nk;
    p.causal = causal ? 1 : 0;
    // Bottom-right: key j visible to query row i iff j <= i + Nk - Nq of the
    // sequence (the kernels take the offset per sequence).
    p.causal_br = (causal == FA_CAUSAL_BOTTOM_RIGHT) ? 1 : 0;
    p.num_splits = num_splits;
    p.split_mode = split_mode;
    p.n_units = static_cast<int>(ctas / (static_cast<long long>(BH) * num_splits));
    p.tiles_per_cta = tiles_per_cta;
    p.bm64 = bm64 ? 1 : 0;
    const int kv_tiles = (Nk + c.bn - 1) / c.bn;
    // (Varlen: one split; every sequence's key tiles fit in ceil(total_k / BN).)
    p.kv_tiles_per_split = (kv_tiles + num_splits - 1) / num_splits;
    // Heads per scheduling group: about one wave of CTAs (one CTA per SM).
    int sms = 0;
    if (sm_count(&sms) != cudaSuccess) return FA_ERR_CUDA;
    const long long ctas_per_head = static_cast<long long>(p.n_units) * num_splits;
    p.head_group = static_cast<int>(std::max<long long>(1, std::min<long long>(BH, sms / ctas_per_head)));
    p.scale_log2 = scale * 1.4426950408889634f;
    p.o_scale = 1.f;
    if (f8_descale) {
        p.scale_log2 *= f8_descale[0] * f8_descale[1];
        p.o_scale = f8_descale[2];
    }
    p.wait_limit = wait_limit;
    p.test_withhold_q = withhold_q;
    if (device_status_ptr(&p.status) != cudaSuccess) return FA_ERR_CUDA;

    cudaError_t e = cudaErrorInvalidValue;
    p.dual = dual ? 1 : 0;
    const int key_tiles = (Nk + 127) / 128;
    const bool short_units = key_tiles <= 16 || (d == 128 && !causal && key_tiles <= 32);
    const bool persist =
        !row_choice && !vl && !split_mode && (d == 64 || d == 128) && short_units && ctas >= 4ll * sms;
    p.total_units = ctas;
    const unsigned grid = static_cast<unsigned>(
        dual ? static_cast<long long>(BH) * ((num_splits + 1) / 2) : (persist ? sms : ctas));
    if (persist) {
        if (f8_descale)
            e = d == 64 ? launch_fwd_f8_d64_persist(p, grid, stream) : launch_fwd_f8_d128_persist(p, grid, stream);
        else
            e = d == 64 ? launch_fwd_d64_persist(p, grid, stream) : launch_fwd_d128_persist(p, grid, stream);
        return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
    if (f8_descale) {
        if (d == 64) e = dual ? launch_fwd_f8_d64_dual(p, grid, stream) : launch_fwd_f8_d64(p, grid, stream);
        else if (d == 128) e = dual ? launch_fwd_f8_d128_dual(p, grid, stream) : launch_fwd_f8_d128(p, grid, stream);
        else if (d == 256) e = launch_fwd_f8_d256(p, grid, stream);
        return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
    if (bm64) {
        e = d == 64 ? launch_fwd_d64_rows64(p, grid, stream) : launch_fwd_d128_rows64(p, grid, stream);
        return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
    }
    switch (d) {
        case 64: e = dual ? launch_fwd_d64_dual(p, grid, stream) : launch_fwd_d64(p, grid, stream); break;
        case 128: e = dual ? launch_fwd_d128_dual(p, grid, stream) : launch_fwd_d128(p, grid, stream); break;
        case 256: e = launch_fwd_d256(p, grid, stream); break;
        default: break;
    }
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace
}  // namespace fa

extern "C" {

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                 int Nq, int Nk, int d, float scale, int causal, cudaStream_t stream) {
    fa_status s = fa::check_common(q, k, v, B, H, Nq, Nk, d, scale);
    if (s != FA_OK) return s;
    if (!fa::valid_causal(causal)) return FA_ERR_CAUSAL;
    if (!o || !lse) return FA_ERR_NULL;
    if (!fa::aligned(o, 16) || !fa::aligned(lse, 4)) return FA_ERR_ALIGN;
    return fa::launch_forward(q, k, v, o, lse, nullptr, B, H, Nq, Nk, d, scale, causal, 1, 0,
                              stream);
}

fa_status fa_fwd_rows(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, float scale, int causal, int rows_per_cta,
                      cudaStream_t stream) {
    fa_status s = fa::check_common(q, k, v, B, H, Nq, Nk, d, scale);
    if (s != FA_OK) return s;
    if (!fa::valid_causal(causal)) return FA_ERR_CAUSAL;
    if (!o || !lse) return FA_ERR_NULL;
    if (!fa::aligned(o, 16) || !fa::aligned(lse, 4)) return FA_ERR_ALIGN;
    const int slots = fa::fwd_config(d).q_tiles;
    // 64 rows: one M = 64 tile per CTA, at d = 64 and 128 (the two-tile kernel).
    if (rows_per_cta == 64 && slots >= 2)
        return fa::launch_forward(q, k, v, o, lse, nullptr, B, H, Nq, Nk, d, scale, causal, 1, 0,
                                  stream, fa::kDefaultWaitLimit, 0, nullptr, nullptr, 1, true);
    if (rows_per_cta % 128 != 0 || rows_per_cta < 128 || rows_per_cta / 128 > slots) return FA_ERR_TILE;
    return fa::launch_forward(q, k, v, o, lse, nullptr, B, H, Nq, Nk, d, scale, causal, 1, 0,
                              stream, fa::kDefaultWaitLimit, 0, nullptr, nullptr, rows_per_cta / 128);
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, float q_descale,
                     float k_descale, float v_descale, void* o, float* lse, int B, int H, int Nq,
                     int Nk, int d, float scale, int causal, cudaStream_t stream) {
    fa_status s = fa::check_common(q, k, v, B, H, Nq, Nk, d, scale);
    if (s != FA_OK) return s;
    if (d != 64 && d != 128 && d != 256) return FA_ERR_HEADDIM;
    if (!fa::valid_causal(causal)) return FA_ERR_CAUSAL;
    const float ds[3] = {q_descale, k_descale, v_descale};
    for (float x : ds)
        if (!std::isfinite(x) || !(x > 0.f)) return FA_ERR_SCALE;
    const float s_eff = scale * q_descale * k_descale;
    if (!std::isfinite(s_eff) || !(s_eff > 0.f)) return FA_ERR_SCALE;
    if (!o || !lse) return FA_ERR_NULL;
    if (!fa::aligned(o, 16) || !fa::aligned(lse, 4)) return FA_ERR_ALIGN;
    return fa::launch_forward(q, k, v, o, lse, nullptr, B, H, Nq, Nk, d, scale, causal, 1, 0,
                              stream, fa::kDefaultWaitLimit, 0, nullptr, ds);
}

fa_status fa_fwd_fp8_splitkv(const void* q, const void* k, const void* v, float q_descale,
                             float k_descale, float v_descale, void* workspace, int B, int H,
                             int Nq, int Nk, int d, float scale, int causal, int num_splits,
                             cudaStream_t stream) {
    fa_status s = fa::check_common(q, k, v, B, H, Nq, Nk, d, scale);
    if (s != FA_OK) return s;
    if (d != 64 && d != 128 && d != 256) return FA_ERR_HEADDIM;
    if (!fa::valid_causal(causal)) return FA_ERR_CAUSAL;
    const float ds[3] = {q_descale, k_descale, v_descale};
    for (float x : ds)
        if (!std::isfinite(x) || !(x > 0.f)) return FA_ERR_SCALE;
    const float s_eff = scale * q_descale * k_descale;
    if (!std::isfinite(s_eff) || !(s_eff > 0.f)) return FA_ERR_SCALE;
    if (num_splits < 1 || num_splits > FA_MAX_SPLITS) return FA_ERR_SPLITS;
    if (!workspace || !fa::aligned(workspace, 16)) return FA_ERR_WORKSPACE;
    return fa::launch_forward(q, k, v, nullptr, nullptr, static_cast<float*>(workspace), B, H, Nq,
                              Nk, d, scale, causal, num_splits, 1, stream, fa::kDefaultWaitLimit, 0,
                              nullptr, ds);
}

size_t fa_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits) {
    if (B < 1 || H < 1 || Nq < 1 || !fa::valid_d(d) || num_splits < 1 ||
        num_splits > FA_MAX_SPLITS)
        return 0;
    const size_t rows = static_cast<size_t>(B) * H * Nq;
    return static_cast<size_t>(num_splits) * rows * (static_cast<size_t>(d) + 2) * sizeof(float);
}

fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                        int total_q, int total_k, int max_seqlen_q, int d, float scale,
                        int causal, cudaStream_t stream) {
    fa_status s = fa::check_common(q, k, v, B, H, total_q, total_k, d, scale);
    if (s != FA_OK) return s;
    if (!fa::valid_causal(causal)) return FA_ERR_CAUSAL;
    if (!o || !lse || !cu_seqlens_q || !cu_seqlens_k) return FA_ERR_NULL;
    if (!fa::aligned(o, 16) || !fa::aligned(lse, 4) || !fa::aligned(cu_seqlens_q, 4) ||
        !fa::aligned(cu_seqlens_k, 4))
        return FA_ERR_ALIGN;
    if (max_seqlen_q < 1 || max_seqlen_q > total_q) return FA_ERR_SHAPE;
    if (static_cast<long long>(total_q) * H * d > 0x7fffffffffffll ||
        static_cast<long long>(total_k) * H * d > 0x7fffffffffffll)
        return FA_ERR_SHAPE;
    const fa::Varlen vl = {cu_seqlens_q, cu_seqlens_k, total_q, total_k};
    return fa::launch_forward(q, k, v, o, lse, nullptr, B, H, max_seqlen_q, total_k, d, scale,
                              causal, 1, 0, stream, fa::kDefaultWaitLimit, 0, &vl);
}

fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* workspace, int B,
                         int H, int Nq, int Nk, int d, float scale, int causal, int num_splits,
                         cudaStream_t stream) {
    fa_status s = fa::check_common(q, k, v, B, H, Nq, Nk, d, scale);
    if (s != FA_OK) return s;
    if (!fa::valid_causal(causal)) return FA_ERR_CAUSAL;
    if (num_splits < 1 || num_splits > FA_MAX_SPLITS) return FA_ERR_SPLITS;
    if (!workspace || !fa::aligned(workspace, 16)) return FA_ERR_WORKSPACE;
    return fa::launch_forward(q, k, v, nullptr, nullptr, static_cast<float*>(workspace), B, H, Nq,
                              Nk, d, scale, causal, num_splits, 1, stream);
}

fa_status fa_combine(const void* workspace, void* o, float* lse, int B, int H, int Nq, int d,
                     int num_splits, cudaStream_t stream) {
    if (!o || !lse) return FA_ERR_NULL;
    if (B < 1 || H < 1 || Nq < 1) return FA_ERR_SHAPE;
    if (static_cast<long long>(B) * H > 0x7fffffffll) return FA_ERR_SHAPE;
    if (!fa::valid_d(d)) return FA_ERR_HEADDIM;
    if (num_splits < 1 || num_splits > FA_MAX_SPLITS) return FA_ERR_SPLITS;
    if (!workspace || !fa::aligned(workspace, 16)) return FA_ERR_WORKSPACE;
    if (!fa::aligned(o, 16) || !fa::aligned(lse, 4)) return FA_ERR_ALIGN;
    const long long rows = static_cast<long long>(B) * H * Nq;
    const float* ws = static_cast<const float*>(workspace);
    const float* ws_m = ws + static_cast<size_t>(num_splits) * rows * d;
    const float* ws_l = ws_m + static_cast<size_t>(num_splits) * rows;
    const cudaError_t e = fa::launch_combine(ws, ws_m, ws_l, o, lse, rows, num_splits, d, stream);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

fa_status fa_test_fwd_withheld_q(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int Nq, int Nk, int d, long long wait_limit_cycles,
                                 cudaStream_t stream) {
    fa_status s = fa::check_common(q, k, v, B, H, Nq, Nk, d, 1.0f);
    if (s != FA_OK) return s;
    if (!o || !lse) return FA_ERR_NULL;
    if (!fa::aligned(o, 16) || !fa::aligned(lse, 4)) return FA_ERR_ALIGN;
    if (wait_limit_cycles < (1ll << 16) || wait_limit_cycles > fa::kDefaultWaitLimit)
        return FA_ERR_SHAPE;
    return fa::launch_forward(q, k, v, o, lse, nullptr, B, H, Nq, Nk, d, 1.0f, 0, 1, 0, stream,
                              wait_limit_cycles, 1);
}

long long fa_fwd_grid_ctas(int B, int H, int Nq, int d, int num_splits) {
    if (B < 1 || H < 1 || Nq < 1 || !fa::valid_d(d) || num_splits < 1 ||
        num_splits > FA_MAX_SPLITS)
        return -1;
    if (fa::use_dual(Nq, d, num_splits, num_splits > 1, false))
        return static_cast<long long>(B) * H * ((num_splits + 1) / 2);
    return fa::grid_ctas(B, H, Nq, d, num_splits);
}

fa_status fa_device_status(cudaStream_t stream, int clear) {
    unsigned* ptr = nullptr;
    if (fa::device_status_ptr(&ptr) != cudaSuccess) return FA_ERR_CUDA;
    unsigned host = 0;
    if (cudaMemcpyAsync(&host, ptr, sizeof(host), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return FA_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    if (clear && host) {
        const unsigned zero = 0;
        if (cudaMemcpyAsync(ptr, &zero, sizeof(zero), cudaMemcpyHostToDevice, stream) != cudaSuccess)
            return FA_ERR_CUDA;
        if (cudaStreamSynchronize(stream) != cudaSuccess) return FA_ERR_CUDA;
    }
    // Bounded waits that gave up take precedence; otherwise a rejected
    // variable-length partition.
    if (host & ~fa::kStatusBadSeqlens) return FA_ERR_TIMEOUT;
    return host ? FA_ERR_SEQLENS : FA_OK;
}

const char* fa_status_string(fa_status status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_NULL: return "FA_ERR_NULL: a required pointer is NULL";
        case FA_ERR_ALIGN: return "FA_ERR_ALIGN: a pointer is not 16-byte (lse: 4-byte) aligned";
        case FA_ERR_SHAPE: return "FA_ERR_SHAPE: B, H, Nq or Nk out of range";
        case FA_ERR_HEADDIM: return "FA_ERR_HEADDIM: head dim must be 64, 128 or 256";
        case FA_ERR_SPLITS: return "FA_ERR_SPLITS: num_splits must be in [1, FA_MAX_SPLITS]";
        case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace NULL or not 16-byte aligned";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA runtime or driver call failed";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel gave up on a bounded wait";
        case FA_ERR_SCALE: return "FA_ERR_SCALE: scale must be finite and > 0";
        case FA_ERR_SCRATCH:
            return "FA_ERR_SCRATCH: partial states exceed the library's static scratch buffer";
        case FA_ERR_CAUSAL:
            return "FA_ERR_CAUSAL: causal must be FA_CAUSAL_NONE, _TOP_LEFT or _BOTTOM_RIGHT";
        case FA_ERR_SEQLENS:
            return "FA_ERR_SEQLENS: cu_seqlens are not a valid partition (see fa_fwd_varlen)";
        case FA_ERR_TILE:
            return "FA_ERR_TILE: rows_per_cta is not offered for this head dim (see fa_fwd_rows)";
    }
    return "unknown fa_status";
}

}  // extern "C"
