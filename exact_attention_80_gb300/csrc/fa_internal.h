// fa_internal.h — parameters and launchers shared by the host API (fa_api.cu)
// and the kernel translation units. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime_api.h>

#include "fa.h"

namespace fa {

// Bits of the device status word (one per kind of bounded wait that gave up).
enum : unsigned {
    kStatusWaitQ = 1u << 0,
    kStatusWaitKvFull = 1u << 1,
    kStatusWaitKvEmpty = 1u << 2,
    kStatusWaitS = 1u << 3,
    kStatusWaitP = 1u << 4,
    kStatusWaitO = 1u << 5,
    kStatusWaitDrain = 1u << 6,
    // Not a wait: variable-length offsets that are not a valid partition
    // (decreasing, past the token count, or longer than max_seqlen_q).
    kStatusBadSeqlens = 1u << 7,
};

// Default bound of one wait, in SM clock cycles (~1 s at 2 GHz). Legitimate
// waits in these kernels last microseconds.
constexpr long long kDefaultWaitLimit = 1ll << 31;

struct FwdParams {
    CUtensorMap tm_q;  // bf16 [B*H][Nq][d], box {64, 128, 1}, 128B swizzle
    CUtensorMap tm_k;  // bf16 [B*H][Nk][d], box {64, BN, 1}
    CUtensorMap tm_v;  // same as tm_k
    CUtensorMap tm_o;  // bf16 [B*H][Nq][d], box {64, 32 (d <= 128) or 128 (d = 256), 1},
                       // 128B swizzle (plain mode)
    void* o;           // bf16 [B*H][Nq][d]      (plain mode)
    float* lse;        // fp32 [B*H][Nq]         (plain mode)
    float* ws_o;       // fp32 [S][B*H][Nq][d]   (split mode)
    float* ws_m;       // fp32 [S][B*H][Nq]
    float* ws_l;       // fp32 [S][B*H][Nq]
    int BH, Nq, Nk;
    int causal;              // 1: causal mask
    int causal_br;           // 1: bottom-right alignment (key j visible to query i iff
                             //    j <= i + Nk - Nq of the sequence), 0: top-left
    // Variable-length batches (varlen = 1): Q, K, V, O token-major [total][H][d]
    // with sequence b at tokens cu_q[b] .. cu_q[b+1]-1 (keys: cu_k); LSE
    // [H][total_q]. BH = B * H work rows; Nq = max_seqlen_q; Nk = total_k.
    int varlen;
    int H;
    int total_q;
    const int* cu_q;         // device int32 [B + 1]
    const int* cu_k;
    int num_splits;          // 1 in plain mode
    int split_mode;          // 0: write O/LSE, 1: write partial (O, m, l)
    int n_units;             // query units of (tiles_per_cta * 128) rows per head
    int tiles_per_cta;       // 128-row query tiles a CTA owns (up to the kernel's tile slots)
    int bm64;                // 1: one 64-row query tile per CTA (M = 64 MMAs; fa_fwd_rows)
    int kv_tiles_per_split;  // ceil(ceil(Nk/BN) / num_splits)
    int head_group;          // heads per scheduling group (CTA order)
    int dual;                // 1: dual-range split CTAs (split mode, Nq <= 128, d <= 128)
    long long total_units;   // persistent launches: work units in the launch (CTAs walk them)
    float scale_log2;        // scale * log2(e) (8-bit inputs: times the Q and K descales)
    float o_scale;           // 8-bit inputs: the V descale, applied to O at the end
    long long wait_limit;    // cycles
    int test_withhold_q;     // failure-detection test hook: 1 = never load Q
    unsigned* status;        // device status word
};

// Backward (d = 128): one CTA per (head, 128-key tile).
struct FwdConfig {
    int q_tiles;  // 128-row query tiles per CTA
    int bn;       // keys per KV tile
    int stages;   // K/V ring slots
    int threads;
    size_t smem;  // dynamic shared memory bytes
};

FwdConfig fwd_config(int d);

cudaError_t launch_fwd_d64(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_d64_rows64(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_d128(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_d128_rows64(const FwdParams& p, unsigned grid, cudaStream_t stream);
// Persistent two-tile kernels (plain mode, dense bf16 or e4m3): grid min(units, SMs).
cudaError_t launch_fwd_d64_persist(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_d128_persist(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_f8_d64_persist(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_f8_d128_persist(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_d256(const FwdParams& p, unsigned grid, cudaStream_t stream);
// e4m3 Q, K, V (tm_q/tm_k/tm_v are byte maps, box {128, rows, 1}, or {64,
// rows, 1} with the 64-byte swizzle at d = 64); d = 64, 128, 256.
cudaError_t launch_fwd_f8_d64(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_f8_d128(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_f8_d256(const FwdParams& p, unsigned grid, cudaStream_t stream);
// Dual-range split-KV CTAs (p.dual = 1): grid B*H*ceil(num_splits / 2).
cudaError_t launch_fwd_d64_dual(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_d128_dual(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_f8_d64_dual(const FwdParams& p, unsigned grid, cudaStream_t stream);
cudaError_t launch_fwd_f8_d128_dual(const FwdParams& p, unsigned grid, cudaStream_t stream);

// Split-KV launches with one query tile per head (Nq <= 128, d <= 128, dense)
// run dual-range CTAs: two splits per CTA.
inline bool use_dual(int Nq, int d, int num_splits, int split_mode, bool varlen) {
    return split_mode && !varlen && num_splits >= 2 && Nq <= 128 && d <= 128;
}

cudaError_t launch_combine(const float* ws_o, const float* ws_m, const float* ws_l, void* o,
                           float* lse, long long rows, int num_splits, int d,
                           cudaStream_t stream);

// Address of the device status word on the current device (cached per device
// and context).
cudaError_t device_status_ptr(unsigned** ptr);

// Unique identifier of the calling thread's current CUDA context (cuCtxGetId),
// or 0 when there is none or the driver does not provide the call.
unsigned long long current_context_id();

// A value bound to a device's CUDA context: a device symbol's address, or the
// fact that a kernel attribute has been set. Cached per device; derived again
// when the device's current context is not the one it was derived in (after
// cudaDeviceReset, or when the primary context was released and re-created), so
// no stale address is ever handed to a kernel. Safe to call from several host
// threads at once.
template <typename T>
class ContextCache {
  public:
    // `derive(T*)` computes the value with the device current; its error is returned.
    template <typename F>
    cudaError_t get(T* out, F&& derive) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        const unsigned long long ctx = current_context_id();
        std::lock_guard<std::mutex> lock(mutex_);
        Entry& en = entries_[dev];
        if (en.valid && ctx != 0 && en.ctx == ctx) {
            *out = en.value;
            return cudaSuccess;
        }
        T value{};
        e = derive(&value);
        if (e != cudaSuccess) return e;
        en.value = value;
        en.ctx = current_context_id();  // the derivation may have created the context
        en.valid = true;
        *out = value;
        return cudaSuccess;
    }

  private:
    static constexpr int kMaxDevices = 64;
    struct Entry {
        unsigned long long ctx = 0;
        T value{};
        bool valid = false;
    };
    std::mutex mutex_;
    Entry entries_[kMaxDevices];
};

// Host-side argument checks and tensor maps (fa_api.cu), shared by the
// forward and backward entry points.
bool aligned(const void* p, uintptr_t a);
bool valid_causal(int causal);
// Non-null q, k, v; B, H, Nq, Nk >= 1 with B * H in int; d in {64, 128, 256};
// finite scale > 0; q, k, v 16-byte aligned.
fa_status check_common(const void* q, const void* k, const void* v, int B, int H, int Nq, int Nk,
                       int d, float scale);
// bf16 [BH][N][d] as a 3-D TMA map, box {64, box_rows, 1}, 128-byte swizzle.
bool encode_rows_map(CUtensorMap* map, const void* base, int d, int N, int BH, int box_rows);

}  // namespace fa
