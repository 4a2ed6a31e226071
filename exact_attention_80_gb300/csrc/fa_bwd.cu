// fa_bwd.cu — attention backward for head dims 64, 128 and 256: dQ, dK, dV. Holds the
// backward's kernels and its C entry points (fa_bwd_workspace_bytes, fa_bwd).
//
// What is computed (the plain definition of the forward differentiated; the
// FA-2 page, "AI 大模型之 FlashAttention_02", sections "warp之间怎样减少通信" and
// "训练与部署 切分与归约的反向一致性": the training backward needs dQ, dK, dV,
// with dK and dV accumulated across query rows):
//   P = exp(scale Q K^T - LSE) (the forward's row LSE; masked entries 0)
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_c dO_ic O_ic,  dS = P * (dP - D)
//   dQ = scale dS K,  dK = scale dS^T Q.
//
// Responsibilities and accumulation (the page asks that they be written down):
//   * fa_bwd_pre_kernel: per query row (rows padded to whole 128-row tiles),
//     -LSE log2(e) and -D_i in fp32 (D_i from bf16 dO and O; padded rows and
//     rows that saw no key get -inf and 0); zeroes the fp32 dQ accumulator.
//   * fa_bwd_kernel: one CTA per (head, 128-key tile). It owns dK and dV of its
//     keys and accumulates them over every query tile in TMEM (fp32), so they
//     need no cross-CTA reduction. Its dQ contribution, dS K for its keys, is
//     added to the fp32 accumulator with atomic adds: dQ is the one quantity
//     summed across CTAs (across key tiles).
//   * fa_bwd_dq_kernel: dQ = scale * accumulator, to bf16.
//
// fa_bwd_kernel steps over the queries 64 at a time. Roles: warp 0 loads K
// and V once and, per step, Q, dO and the step's -LSE log2e and -D into a ring
// of three slots (TMA); warp 1 issues tcgen05 MMAs; warps 4-11 are the compute
// group, two warps per TMEM lane quarter, one per 32-query chunk of a step
// (thread = TMEM lane = key row); warps 12-15 read dQ^T out (lane = head dim).
// TMEM holds two step buffers of 128 columns beside dV and dK. Per step h
// (buffer h & 1):
//   S^T = K Q_h^T and dP^T = V dO_h^T (lanes = keys, 64 query columns each);
//   the compute group forms P^T = exp2(S^T scale log2e - LSE log2e) and
//   dS^T = P^T (dP^T - D), writes both as bf16 into TMEM over the first half
//   of each chunk's own columns, and dS^T into shared memory (128-byte
//   swizzle);
//   dV += P^T dO_h and dK += dS^T Q_h (A from TMEM, B = dO_h / Q_h MN-major);
//   dQ_h^T = K^T dS^T (A = K MN-major, B = dS^T from shared memory) over the
//   buffer's S^T columns; the readout group takes it out of TMEM, releases the
//   buffer and adds it to the fp32 accumulator, 32 consecutive floats per warp
//   instruction.
// The issuer runs the MMAs in pairs of steps, S^T and dP^T of two steps then
// dV, dK and dQ^T of the same two, so that each of the three groups (tensor
// core, compute, readout) always has the other step's work to overlap.
// Every mbarrier wait is bounded, as in the forward kernels.
//
// Head dim 64: the same steps with half-width K, V, Q and dO tiles and 64
// TMEM columns each for dV and dK. dQ^T keeps M = 128 (head-dim lanes): its A
// operand, K read MN-major, has a second 64-dim chunk of zeros that the CTA
// writes once, so lanes 64-127 of dQ^T are zero and only the readout warps of
// lanes 0-63 take it out.
//
// Head dim 256: dV and dK of 128 keys at d = 256 would take all 512 TMEM
// columns, so each key tile has two CTAs, one per 128-column half of the head
// dim. Both compute the whole S^T and dP^T (the contraction runs over all 256
// columns); each accumulates its half of dV and dK in TMEM and adds its half
// of dQ. K and V stay resident (64 KB each), which leaves shared memory for one
// Q/dO stage: the issuer then runs the steps one after another (S^T and dP^T
// of step h + 1 once step h's dV and dK have read the stage and its load has
// landed) instead of in pairs.
#include <cuda_bf16.h>

#include <cstring>

#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// Kernel parameters, filled by fa_bwd below.
struct BwdParams {
    CUtensorMap tm_q;   // bf16 [B*H][Nq][d], box {64, 64, 1} (64 head-dim columns)
    CUtensorMap tm_k;   // bf16 [B*H][Nk][d], box {64, 128, 1}
    CUtensorMap tm_v;   // same as tm_k
    CUtensorMap tm_do;  // same as tm_q (dO)
    const float* nlse2; // fp32 [B*H][Nq_pad]: -LSE log2(e); -inf past Nq or with no key
    const float* ndd;   // fp32 [B*H][Nq_pad]: -D_i = -sum_c dO_ic O_ic; 0 past Nq
    float* dq_acc;      // fp32 [B*H][Nq_pad][d], zeroed, unscaled dS K accumulated
    void* dk;           // bf16 [B*H][Nk][d]
    void* dv;           // bf16 [B*H][Nk][d]
    int BH, Nq, Nk;
    int Nq_pad;         // Nq rounded up to whole 128-row query tiles
    int causal, causal_br;
    int k_tiles;        // ceil(Nk / 128)
    int pair_tiles;     // 1: a CTA takes key tiles kt and k_tiles - 1 - kt (causal)
    int tile_units;     // key-tile units per head: k_tiles, or ceil(k_tiles / 2) when paired
    float scale;
    float scale_log2;   // scale * log2(e)
    long long wait_limit;
    unsigned* status;
};

namespace {

constexpr int kBwdKeys = 128;   // keys per CTA (TMEM lanes of S^T, dP^T, dV, dK)
constexpr int kBwdHalf = 64;    // queries per step
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct LayoutBwd {
    static_assert(D == 64 || D == 128 || D == 256, "head dim 64, 128 or 256");
    static constexpr int DH = D < 128 ? D : 128;        // head-dim columns of dV, dK, dQ a CTA owns
    static constexpr int HALVES = D / DH;               // CTAs per key tile
    static constexpr int STAGES = D == 256 ? 1 : 3;     // Q/dO (+ -LSE log2e, -D) ring slots
    // warp 0 producer, warp 1 issuer, warps 2-3 idle, warps 4-11 compute (two
    // per TMEM lane quarter, one per 32-query chunk of a step), warps 12-15
    // dQ readout (one per lane quarter; at D = 64 the first two only).
    static constexpr int COMPUTE_WARPS = 8;
    static constexpr int READOUT_WARPS = 4;
    static constexpr int READOUT_ACTIVE = DH / 32;                  // lane quarters holding dQ^T
    static constexpr int CHUNKS = D / 64;                           // 64-column chunks of a row
    static constexpr int DH_CHUNKS = DH / 64;                       // chunks of the CTA's head-dim part
    static constexpr int THREADS = 128 + 32 * (COMPUTE_WARPS + READOUT_WARPS);
    static constexpr uint32_t KV_CHUNK = kBwdKeys * 128;            // 16 KB: 64 columns of K or V
    // K spans at least two chunks: dQ^T reads it as an M = 128 operand, and at
    // D = 64 the second chunk is zeros.
    static constexpr uint32_t K_BYTES = (CHUNKS < 2 ? 2 : CHUNKS) * KV_CHUNK;
    static constexpr uint32_t V_BYTES = CHUNKS * KV_CHUNK;
    static constexpr uint32_t QH_CHUNK = kBwdHalf * 128;            // 8 KB: 64 columns of a step's Q or dO
    static constexpr uint32_t QH_BYTES = CHUNKS * QH_CHUNK;
    static constexpr uint32_t ROWS_BYTES = kBwdHalf * 4;            // 256 B of -LSE log2e (or -D)
    static constexpr uint32_t STAGE_BYTES = 2 * QH_BYTES;           // Q and dO of a step
    static constexpr uint32_t DS_BYTES = kBwdKeys * kBwdHalf * 2;   // 16 KB: dS^T bf16 [keys][64 queries]
    // Swizzled tiles start on 1024-byte boundaries (the MMA descriptors'
    // base offset is 0); the per-row arrays need 16 bytes.
    static constexpr uint32_t K_OFF = 0;
    static constexpr uint32_t V_OFF = K_OFF + K_BYTES;
    static constexpr uint32_t STAGE_OFF = V_OFF + V_BYTES;           // [stage]: Q, dO
    static constexpr uint32_t Q_IN = 0, DO_IN = QH_BYTES;
    static constexpr uint32_t DS_OFF = STAGE_OFF + STAGES * STAGE_BYTES;  // [buffer]
    static constexpr uint32_t ROWS_OFF = DS_OFF + 2 * DS_BYTES;     // [stage]: -LSE log2e, -D
    static constexpr uint32_t NL_IN = 0, ND_IN = ROWS_BYTES;
    static constexpr uint32_t BAR_OFF = ROWS_OFF + STAGES * 2 * ROWS_BYTES;
    static_assert(STAGE_OFF % 1024 == 0 && STAGE_BYTES % 1024 == 0 && QH_CHUNK % 1024 == 0 &&
                      DS_OFF % 1024 == 0 && DS_BYTES % 1024 == 0, "swizzle atoms must be 1024-aligned");
    static constexpr int BAR_KV = 0;
    static constexpr int BAR_QFULL = 1;                    // [stage]
    static constexpr int BAR_QEMPTY = BAR_QFULL + STAGES;   // [stage]
    static constexpr int BAR_SFULL = BAR_QEMPTY + STAGES;   // [buffer] S^T, dP^T done
    static constexpr int BAR_PREADY = BAR_SFULL + 2;    // [buffer] P^T, dS^T written (one arrival per compute warp)
    static constexpr int BAR_DQFULL = BAR_PREADY + 2;   // [buffer] dQ^T done (and every earlier MMA)
    static constexpr int BAR_DQREAD = BAR_DQFULL + 2;   // [buffer] dQ^T read (one arrival per readout warp)
    static constexpr int BAR_KVFREE = BAR_DQREAD + 2;   // the first of two key tiles' MMAs done
    static constexpr int BAR_ACCFREE = BAR_KVFREE + 1;  // its dK, dV read out of TMEM (one arrival per compute warp)
    static constexpr int BAR_DRAIN = BAR_ACCFREE + 1;
    static constexpr int NUM_BARS = BAR_DRAIN + 1;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr uint32_t BYTES = MISC_OFF + 16;
    static constexpr size_t ALLOC_BYTES = BYTES + 1024;
    // TMEM columns. Buffer b (b = step & 1) at 128 b: S^T in its first 64
    // columns (then P^T packed over their first halves, then dQ^T), dP^T in
    // the next 64 (then dS^T packed over their first halves). dV and dK last
    // (D columns each).
    __host__ __device__ static constexpr uint32_t BUF_COL(int b) { return 128u * static_cast<uint32_t>(b); }
    static constexpr uint32_t DP_IN = 64, DV_COL = 256, DK_COL = 384;
    static_assert(ALLOC_BYTES <= 232448, "shared memory over the 227 KB per-CTA limit");
    static_assert(THREADS * 128 <= 65536, "registers: 128 per thread at most");
};

__device__ __forceinline__ bool bwd_wait(uint32_t bar, uint32_t parity, const BwdParams& p,
                                         volatile uint32_t* abort_flag, unsigned what,
                                         bool honor_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long start = clock64();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (honor_abort && *abort_flag) return false;
        if (clock64() - start > p.wait_limit) {
            *abort_flag = 1u;
            atomicOr(p.status, what);
            return false;
        }
    }
}

// The 64-query steps a key tile sees: all of them, or (causal) those with a
// row at or after the tile's first key minus the alignment offset.
__device__ __forceinline__ void bwd_steps(const BwdParams& p, int kt, int& h0, int& n) {
    const int steps = (p.Nq + kBwdHalf - 1) / kBwdHalf;
    h0 = 0;
    if (p.causal) {
        const int off = p.causal_br ? p.Nk - p.Nq : 0;
        const int first_row = kt * kBwdKeys - off;  // key k is visible to rows >= k - off
        h0 = first_row <= 0 ? 0 : first_row / kBwdHalf;
    }
    n = max(0, steps - h0);
}

// P^T and dS^T of one 32-query chunk for this thread's key row: s and dp are
// the chunk's S^T and dP^T columns, nl and nd the chunk's -LSE log2e and -D in
// shared memory (the same addresses for every lane: broadcast loads). MASK:
// `lim` is the first visible chunk column (causal) and `key_ok` whether the
// key exists; without MASK every entry is visible.
template <bool MASK>
__device__ __forceinline__ void bwd_chunk(const uint32_t (&s)[32], const uint32_t (&dp)[32], uint32_t nl,
                                          uint32_t nd, float sl2, int lim, bool key_ok, uint32_t (&pk)[16],
                                          uint32_t (&dk)[16]) {
    const uint64_t sl2x2 = f2pack(sl2, sl2);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        float l4[4], d4[4];
        ld_shared_v4f(nl + 16 * u, l4);
        ld_shared_v4f(nd + 16 * u, d4);
        const uint64_t x01 = ffma2(f2pack(__uint_as_float(s[4 * u]), __uint_as_float(s[4 * u + 1])), sl2x2,
                                   f2pack(l4[0], l4[1]));
        const uint64_t x23 = ffma2(f2pack(__uint_as_float(s[4 * u + 2]), __uint_as_float(s[4 * u + 3])), sl2x2,
                                   f2pack(l4[2], l4[3]));
        float x[4];
        f2unpack(x01, x[0], x[1]);
        f2unpack(x23, x[2], x[3]);
        float pv[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            // The exponential runs for every element and the mask selects after
            // it (x is finite or -inf: no NaN), so there are no branches.
            const float ex = ex2(x[h]);
            pv[h] = MASK ? ((key_ok && 4 * u + h >= lim) ? ex : 0.f) : ex;
        }
        const uint64_t g01 = fadd2(f2pack(__uint_as_float(dp[4 * u]), __uint_as_float(dp[4 * u + 1])),
                                   f2pack(d4[0], d4[1]));
        const uint64_t g23 = fadd2(f2pack(__uint_as_float(dp[4 * u + 2]), __uint_as_float(dp[4 * u + 3])),
                                   f2pack(d4[2], d4[3]));
        float ds[4];
        f2unpack(fmul2(f2pack(pv[0], pv[1]), g01), ds[0], ds[1]);
        f2unpack(fmul2(f2pack(pv[2], pv[3]), g23), ds[2], ds[3]);
        pk[2 * u] = pack_bf16x2(pv[0], pv[1]);
        pk[2 * u + 1] = pack_bf16x2(pv[2], pv[3]);
        dk[2 * u] = pack_bf16x2(ds[0], ds[1]);
        dk[2 * u + 1] = pack_bf16x2(ds[2], ds[3]);
    }
}

// One CTA per (head, key-tile unit, head-dim part), stepping over the queries
// 64 at a time. A unit is one 128-key tile, or under a causal mask the pair of
// tiles kt and k_tiles - 1 - kt, run one after the other: the steps of a tile
// fall with its index, so every pair has about the same number of steps and no
// CTA is left with the few steps of a last tile alone. The two tiles share the
// step sequence: global step G (over both tiles) uses TMEM buffer G & 1 and
// ring slot G % STAGES. Between the tiles K and V are reloaded once the first
// tile's MMAs are done (KVFREE) and the first MMA into dV and dK waits until
// the compute group has read the first tile's out of TMEM (ACCFREE).
//   The issuer runs each tile's MMAs in pairs of steps: S^T and dP^T of steps
// 2k+2 and 2k+3 (each needs its buffer's dQ^T of two steps back read out),
// then dV, dK and dQ^T of steps 2k+2 and 2k+3 (each needs its P^T and dS^T).
// While the tensor core runs one step's MMAs, the compute group forms P^T and
// dS^T of the other and the readout group adds the previous dQ^T to the
// accumulator. With one ring slot (d = 256) the steps run in order.
template <int D>
__global__ void __launch_bounds__(LayoutBwd<D>::THREADS, 1) fa_bwd_kernel(const __grid_constant__ BwdParams p) {
    using L = LayoutBwd<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
    volatile uint32_t* abort_flag = misc + 1;
    auto bar = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8u * i; };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // CTA = (head, key-tile unit, head-dim part), the part fastest.
    const int hd = static_cast<int>(blockIdx.x % L::HALVES);
    const int unit_lin = static_cast<int>(blockIdx.x / L::HALVES);
    const int bh = unit_lin / p.tile_units;
    const int ui = unit_lin % p.tile_units;
    int kts[2], h0s[2], ns[2];
    int nt = 1;
    kts[0] = ui;
    if (p.pair_tiles && p.k_tiles - 1 - ui != ui) {
        kts[1] = p.k_tiles - 1 - ui;
        nt = 2;
    } else {
        kts[1] = ui;
    }
    bwd_steps(p, kts[0], h0s[0], ns[0]);
    if (nt == 2) bwd_steps(p, kts[1], h0s[1], ns[1]);
    else ns[1] = 0, h0s[1] = 0;
    const int n_all = ns[0] + ns[1];
    // The second tile reuses K/V, dV and dK only if both tiles have steps.
    const bool handoff = nt == 2 && ns[0] > 0 && ns[1] > 0;
    const size_t row0 = static_cast<size_t>(bh) * p.Nq_pad;

    if (threadIdx.x == 0) {
        mbar_init(bar(L::BAR_KV), 1);
        mbar_init(bar(L::BAR_KVFREE), 1);
        mbar_init(bar(L::BAR_ACCFREE), L::COMPUTE_WARPS);
        for (int st = 0; st < L::STAGES; ++st) {
            mbar_init(bar(L::BAR_QFULL + st), 1);
            mbar_init(bar(L::BAR_QEMPTY + st), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::BAR_SFULL + b), 1);
            mbar_init(bar(L::BAR_PREADY + b), L::COMPUTE_WARPS);
            mbar_init(bar(L::BAR_DQFULL + b), 1);
            mbar_init(bar(L::BAR_DQREAD + b), L::READOUT_ACTIVE);
        }
        mbar_init(bar(L::BAR_DRAIN), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
        tma_prefetch_desc(&p.tm_do);
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::MISC_OFF, 512);
        tmem_relinquish();
    }
    if constexpr (D == 64) {
        // The zero second chunk of K (head dims 64-127 of dQ^T's A operand),
        // written through the generic proxy and fenced for the MMAs. Only the
        // first chunk is ever loaded.
        const uint32_t z = sbase + L::K_OFF + L::KV_CHUNK + 32u * threadIdx.x;
        static_assert(L::THREADS * 32 == L::KV_CHUNK, "one 32-byte piece per thread");
        st_shared_v4(z, 0u, 0u, 0u, 0u);
        st_shared_v4(z + 16, 0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0 && n_all > 0) {
        // ------------------------------------------------------------ producer
        const bool leader = elect_one();
        bool ok = true;
        int issued = 0;    // global steps whose Q/dO loads were issued
        int kv_loads = 0;
        for (int tt = 0; tt < nt && ok; ++tt) {
            const int n = ns[tt];
            if (n == 0) continue;
            if (kv_loads > 0)  // the previous tile's MMAs are done with K and V
                ok = __all_sync(0xffffffffu, bwd_wait(bar(L::BAR_KVFREE), (kv_loads - 1) & 1, p, abort_flag,
                                                      kStatusWaitKvEmpty));
            if (!ok) break;
            if (leader) {
                const int k0 = kts[tt] * kBwdKeys;
                mbar_arrive_expect_tx(bar(L::BAR_KV), 2 * L::V_BYTES);
                for (int c = 0; c < L::CHUNKS; ++c) {
                    tma_load_3d(sbase + L::K_OFF + c * L::KV_CHUNK, &p.tm_k, bar(L::BAR_KV), 64 * c, k0, bh);
                    tma_load_3d(sbase + L::V_OFF + c * L::KV_CHUNK, &p.tm_v, bar(L::BAR_KV), 64 * c, k0, bh);
                }
            }
            ++kv_loads;
            for (int h = 0; h < n && ok; ++h) {
                const int G = issued;
                const int st = G % L::STAGES;
                if (G >= L::STAGES)
                    ok = __all_sync(0xffffffffu, bwd_wait(bar(L::BAR_QEMPTY + st), ((G / L::STAGES) - 1) & 1, p,
                                                          abort_flag, kStatusWaitKvEmpty));
                if (!ok) break;
                if (leader) {
                    const int q0 = (h0s[tt] + h) * kBwdHalf;
                    const uint32_t sb = sbase + L::STAGE_OFF + st * L::STAGE_BYTES;
                    const uint32_t rb = sbase + L::ROWS_OFF + st * 2 * L::ROWS_BYTES;
                    mbar_arrive_expect_tx(bar(L::BAR_QFULL + st), L::STAGE_BYTES + 2 * L::ROWS_BYTES);
                    for (int c = 0; c < L::CHUNKS; ++c) {
                        tma_load_3d(sb + L::Q_IN + c * L::QH_CHUNK, &p.tm_q, bar(L::BAR_QFULL + st), 64 * c, q0, bh);
                        tma_load_3d(sb + L::DO_IN + c * L::QH_CHUNK, &p.tm_do, bar(L::BAR_QFULL + st), 64 * c, q0,
                                    bh);
                    }
                    bulk_load(rb + L::NL_IN, p.nlse2 + row0 + q0, L::ROWS_BYTES, bar(L::BAR_QFULL + st));
                    bulk_load(rb + L::ND_IN, p.ndd + row0 + q0, L::ROWS_BYTES, bar(L::BAR_QFULL + st));
                }
                issued = G + 1;
            }
        }
        if (ok) {
            // The issuer's last slot releases: no commit arrival may still be in
            // flight when the CTA exits.
            for (int G = max(0, n_all - L::STAGES); G < n_all && ok; ++G)
                ok = __all_sync(0xffffffffu, bwd_wait(bar(L::BAR_QEMPTY + G % L::STAGES), (G / L::STAGES) & 1, p,
                                                      abort_flag, kStatusWaitKvEmpty));
        } else {
            if (kv_loads > 0) bwd_wait(bar(L::BAR_KV), (kv_loads - 1) & 1, p, abort_flag, kStatusWaitDrain, false);
            for (int G = max(0, issued - L::STAGES); G < issued; ++G)
                bwd_wait(bar(L::BAR_QFULL + G % L::STAGES), (G / L::STAGES) & 1, p, abort_flag,
                         kStatusWaitDrain, false);
        }
    } else if (warp == 1 && n_all > 0) {
        // ------------------------------------------------------------ MMA issuer
        const bool leader = elect_one();
        auto wait_all = [&](uint32_t b, uint32_t parity, unsigned what) {
            return __all_sync(0xffffffffu, bwd_wait(b, parity, p, abort_flag, what));
        };
        constexpr uint32_t IDESC_S = make_idesc_bf16(128, kBwdHalf, false, false);  // S^T, dP^T
        constexpr uint32_t IDESC_ACC = make_idesc_bf16(128, L::DH, false, true);    // dV, dK (this CTA's part)
        constexpr uint32_t IDESC_DQ = make_idesc_bf16(128, kBwdHalf, true, true);   // dQ^T
        // K-major operands (8-row groups 1024 bytes apart); MN-major ones with
        // their 64-element chunks KV_CHUNK (K as A of dQ^T) or QH_CHUNK (Q, dO
        // as B of dK, dV) apart; dS^T is one 64-query chunk.
        const uint64_t kmaj0 = make_sdesc_sw128(sbase, 16, 1024);
        const uint64_t kmn0 = make_sdesc_sw128(sbase, L::KV_CHUNK, 1024);
        const uint64_t qmn0 = make_sdesc_sw128(sbase, L::QH_CHUNK, 1024);
        const uint32_t kmaj_lo = static_cast<uint32_t>(kmaj0), kmaj_hi = static_cast<uint32_t>(kmaj0 >> 32);
        const uint32_t kmn_lo = static_cast<uint32_t>(kmn0), kmn_hi = static_cast<uint32_t>(kmn0 >> 32);
        const uint32_t qmn_lo = static_cast<uint32_t>(qmn0), qmn_hi = static_cast<uint32_t>(qmn0 >> 32);
        auto desc = [](uint32_t lo, uint32_t hi, uint32_t off) -> uint64_t {
            return (static_cast<uint64_t>(hi) << 32) | (lo + (off >> 4));
        };
        // S^T_G = K Q_G^T and dP^T_G = V dO_G^T into buffer G & 1 (lanes = keys,
        // 64 query columns each), reading ring slot G % STAGES; first, from
        // G = 2 on, the readout group must have taken that buffer's dQ^T of two
        // steps back out.
        auto issue_sdp = [&](int G) -> bool {
            if (G >= 2) {
                if (!wait_all(bar(L::BAR_DQREAD + (G & 1)), ((G - 2) >> 1) & 1, kStatusWaitO)) return false;
            }
            const int st = G % L::STAGES;
            if (!wait_all(bar(L::BAR_QFULL + st), (G / L::STAGES) & 1, kStatusWaitQ)) return false;
            tc_fence_after();
            const uint32_t sb = L::STAGE_OFF + st * L::STAGE_BYTES;
            const uint32_t col = L::BUF_COL(G & 1);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t in_a = (kk & 3) * 32 + (kk >> 2) * L::KV_CHUNK;
                const uint32_t in_b = (kk & 3) * 32 + (kk >> 2) * L::QH_CHUNK;
                const uint64_t ak = desc(kmaj_lo, kmaj_hi, L::K_OFF + in_a);
                const uint64_t av = desc(kmaj_lo, kmaj_hi, L::V_OFF + in_a);
                const uint64_t bq = desc(kmaj_lo, kmaj_hi, sb + L::Q_IN + in_b);
                const uint64_t bdo = desc(kmaj_lo, kmaj_hi, sb + L::DO_IN + in_b);
                if (leader) {
                    umma_ss(tmem + col, ak, bq, IDESC_S, kk > 0 ? 1u : 0u);
                    umma_ss(tmem + col + L::DP_IN, av, bdo, IDESC_S, kk > 0 ? 1u : 0u);
                }
            }
            if (leader) umma_commit(bar(L::BAR_SFULL + (G & 1)));
            return true;
        };
        // dV += P^T_G dO_G, dK += dS^T_G Q_G (A from TMEM: 16 queries = 8 packed
        // columns, each 32-query chunk packed into the first 16 of its own 32;
        // B MN-major, 16 query rows = 2048 bytes), then dQ^T_G = K^T dS^T_G
        // over buffer G & 1's S^T columns (after the dV MMAs that read P^T
        // there, in issue order): A = K MN-major (M = head dim), B = dS^T
        // MN-major (N = queries), 16 keys = 2048 bytes per MMA. `first`: the
        // tile's first step, which starts dV and dK.
        auto issue_vkq = [&](int G, bool first) -> bool {
            const int b = G & 1;
            if (!wait_all(bar(L::BAR_PREADY + b), (G >> 1) & 1, kStatusWaitP)) return false;
            tc_fence_after();
            const int st = G % L::STAGES;
            // B of dV and dK: this CTA's head-dim part of dO_G and Q_G.
            const uint32_t sb = L::STAGE_OFF + st * L::STAGE_BYTES + hd * L::DH_CHUNKS * L::QH_CHUNK;
            const uint32_t col = L::BUF_COL(b);
#pragma unroll
            for (int kk = 0; kk < kBwdHalf / 16; ++kk) {
                const uint32_t acc = (!first || kk > 0) ? 1u : 0u;
                const uint32_t pcol = col + 32 * (kk >> 1) + 8 * (kk & 1);
                const uint64_t bdo = desc(qmn_lo, qmn_hi, sb + L::DO_IN + kk * 2048);
                const uint64_t bq = desc(qmn_lo, qmn_hi, sb + L::Q_IN + kk * 2048);
                if (leader) {
                    umma_ts(tmem + L::DV_COL, tmem + pcol, bdo, IDESC_ACC, acc);
                    umma_ts(tmem + L::DK_COL, tmem + pcol + L::DP_IN, bq, IDESC_ACC, acc);
                }
            }
            if (leader) umma_commit(bar(L::BAR_QEMPTY + st));
            const uint32_t dsb = L::DS_OFF + b * L::DS_BYTES;
#pragma unroll
            for (int kk = 0; kk < kBwdKeys / 16; ++kk) {
                // A: this CTA's head-dim part of K (M = 128 head dims).
                const uint64_t a = desc(kmn_lo, kmn_hi, L::K_OFF + hd * L::DH_CHUNKS * L::KV_CHUNK + kk * 2048);
                const uint64_t bds = desc(qmn_lo, qmn_hi, dsb + kk * 2048);
                if (leader) umma_ss(tmem + col, a, bds, IDESC_DQ, kk > 0 ? 1u : 0u);
            }
            if (leader) umma_commit(bar(L::BAR_DQFULL + b));
            return true;
        };
        bool ok = true;
        int gb = 0;        // global index of the tile's first step
        int kv_loads = 0;
        for (int tt = 0; tt < nt && ok; ++tt) {
            const int n = ns[tt];
            if (n == 0) continue;
            ok = wait_all(bar(L::BAR_KV), kv_loads & 1, kStatusWaitKvFull);
            ++kv_loads;
            if (!ok) break;
            tc_fence_after();
            // The tile's first MMA into dV and dK waits until the compute group
            // has read the previous tile's out of TMEM.
            auto first_vkq = [&](int G) -> bool {
                if (tt > 0 && handoff) {
                    if (!wait_all(bar(L::BAR_ACCFREE), 0, kStatusWaitO)) return false;
                    tc_fence_after();
                }
                return issue_vkq(G, true);
            };
            if constexpr (L::STAGES >= 3) {
                if (ok) ok = issue_sdp(gb);
                if (ok && n > 1) ok = issue_sdp(gb + 1);
                for (int a = 0; a < n && ok; a += 2) {
                    ok = a == 0 ? first_vkq(gb) : issue_vkq(gb + a, false);
                    if (ok && a + 1 < n) ok = issue_vkq(gb + a + 1, false);
                    // The next pair's S^T and dP^T.
                    for (int h = a + 2; h < a + 4 && h < n && ok; ++h) ok = issue_sdp(gb + h);
                }
            } else {
                // One stage: step G + 1's Q and dO load once step G's dV and dK
                // MMAs have read the stage, so its S^T and dP^T follow step G's
                // MMAs.
                if (ok) ok = issue_sdp(gb);
                for (int h = 0; h < n && ok; ++h) {
                    ok = h == 0 ? first_vkq(gb) : issue_vkq(gb + h, false);
                    if (ok && h + 1 < n) ok = issue_sdp(gb + h + 1);
                }
            }
            // K and V free for the next tile once every MMA so far is done.
            if (ok && tt == 0 && handoff && leader) umma_commit(bar(L::BAR_KVFREE));
            gb += n;
        }
        if (leader) umma_commit(bar(L::BAR_DRAIN));
        bwd_wait(bar(L::BAR_DRAIN), 0, p, abort_flag, kStatusWaitDrain, false);
    } else if (warp >= 4 && warp < 4 + L::COMPUTE_WARPS) {
        // ------------------------------------------------------------ compute group
        const int quarter = warp & 3;
        const int g = (warp - 4) >> 2;       // 32-query chunk of each step
        const int r = quarter * 32 + lane;   // TMEM lane: key row
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        const int off = p.causal_br ? p.Nk - p.Nq : 0;
        const float sl2 = p.scale_log2;
        bool ok = true;
        int gb = 0;
        for (int tt = 0; tt < nt && ok; ++tt) {
            const int n = ns[tt];
            const int h0 = h0s[tt];
            const int k0 = kts[tt] * kBwdKeys;
            const int key = k0 + r;
            const bool key_ok = key < p.Nk;
            const bool key_tail = k0 + kBwdKeys > p.Nk;
            for (int h = 0; h < n && ok; ++h) {
                const int G = gb + h;
                const int b = G & 1;
                const int q0 = (h0 + h) * kBwdHalf;
                // Every entry of the step is visible unless the tile holds missing
                // keys or (causal) crosses the diagonal; padded query rows carry
                // -inf as -LSE log2e, so their P is 0 either way.
                const bool masked = key_tail || (p.causal && k0 + kBwdKeys - 1 > q0 + off);
                ok = __all_sync(0xffffffffu, bwd_wait(bar(L::BAR_SFULL + b), (G >> 1) & 1, p, abort_flag, kStatusWaitS));
                if (!ok) break;
                tc_fence_after();
                const uint32_t col = L::BUF_COL(b) + 32 * g;
                uint32_t sraw[32], draw[32];
                tmem_ld32(tmem + lane_field + col, sraw);
                tmem_ld32(tmem + lane_field + col + L::DP_IN, draw);
                tmem_wait_ld();
                // The slot's -LSE log2e and -D for this chunk's 32 queries (the S^T
                // commit implies the slot's loads landed: the issuer waited for them).
                const uint32_t rb = sbase + L::ROWS_OFF + (G % L::STAGES) * 2 * L::ROWS_BYTES;
                const uint32_t nl = rb + L::NL_IN + 128 * g;
                const uint32_t nd = rb + L::ND_IN + 128 * g;
                uint32_t pk[16], dk[16];
                if (masked) {
                    // Key row `key` is visible to query q iff key <= q + off.
                    const int lim = p.causal ? key - off - q0 - 32 * g : -1;
                    bwd_chunk<true>(sraw, draw, nl, nd, sl2, lim, key_ok, pk, dk);
                } else {
                    bwd_chunk<false>(sraw, draw, nl, nd, sl2, 0, true, pk, dk);
                }
                // P^T and dS^T over the first 16 of the chunk's own 32 columns (no
                // other warp reads or writes them).
                tmem_st16(tmem + lane_field + col, pk);
                tmem_st16(tmem + lane_field + col + L::DP_IN, dk);
                // dS^T into shared memory: row r, queries 32 g .. 32 g + 31 of the
                // step's 128-byte row (128-byte swizzle).
                const uint32_t line = sbase + L::DS_OFF + b * L::DS_BYTES + r * 128;
                const uint32_t swz = static_cast<uint32_t>(r & 7);
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    const uint32_t u = static_cast<uint32_t>(g * 4 + uu);
                    st_shared_v4(line + ((u ^ swz) << 4), dk[4 * uu], dk[4 * uu + 1], dk[4 * uu + 2], dk[4 * uu + 3]);
                }
                fence_proxy_async_smem();
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::BAR_PREADY + b));
            }
            // dK (scaled) and dV of this key row, columns DH/2 g .. DH/2 g + DH/2 - 1 of
            // the CTA's head-dim part, once every MMA of the tile has finished (its
            // last dQ^T commit covers them all); zero when no query step sees the
            // key tile. tcgen05.ld is warp-collective: the loads run for the whole
            // warp (`ok` is warp-uniform), and only the stores check that the key
            // exists. After the first of two tiles the TMEM reads are handed back
            // (ACCFREE) before the stores.
            if (ok && n > 0) {
                const int G = gb + n - 1;
                ok = __all_sync(0xffffffffu, bwd_wait(bar(L::BAR_DQFULL + (G & 1)), (G >> 1) & 1, p, abort_flag,
                                                      kStatusWaitO));
                if (ok) tc_fence_after();
            }
            if (ok) {
                // This CTA's head-dim part of the key row's dK and dV.
                __nv_bfloat16* dkp =
                    static_cast<__nv_bfloat16*>(p.dk) + (static_cast<size_t>(bh) * p.Nk + key) * D + hd * L::DH;
                __nv_bfloat16* dvp =
                    static_cast<__nv_bfloat16*>(p.dv) + (static_cast<size_t>(bh) * p.Nk + key) * D + hd * L::DH;
#pragma unroll 1
                for (int j = 0; j < L::DH_CHUNKS; ++j) {
                    const int cc = L::DH_CHUNKS * g + j;
                    uint32_t kr[32], vr[32];
                    if (n > 0) {
                        tmem_ld32(tmem + lane_field + L::DK_COL + cc * 32, kr);
                        tmem_ld32(tmem + lane_field + L::DV_COL + cc * 32, vr);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) kr[e] = vr[e] = 0u;
                    }
                    if (j == L::DH_CHUNKS - 1 && tt == 0 && handoff) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(bar(L::BAR_ACCFREE));
                    }
                    uint32_t kp[16], vp[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        kp[e] = pack_bf16x2(__uint_as_float(kr[2 * e]) * p.scale, __uint_as_float(kr[2 * e + 1]) * p.scale);
                        vp[e] = pack_bf16x2(__uint_as_float(vr[2 * e]), __uint_as_float(vr[2 * e + 1]));
                    }
                    if (key_ok) {
                        uint4* dk4 = reinterpret_cast<uint4*>(dkp + cc * 32);
                        uint4* dv4 = reinterpret_cast<uint4*>(dvp + cc * 32);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            dk4[e] = make_uint4(kp[4 * e], kp[4 * e + 1], kp[4 * e + 2], kp[4 * e + 3]);
                            dv4[e] = make_uint4(vp[4 * e], vp[4 * e + 1], vp[4 * e + 2], vp[4 * e + 3]);
                        }
                    }
                }
            }
            gb += n;
        }
    } else if (warp >= 4 + L::COMPUTE_WARPS && (warp & 3) < L::READOUT_ACTIVE && n_all > 0) {
        // ------------------------------------------------------------ dQ readout
        // Lane r = head dim r; columns = the step's 64 queries. The TMEM loads
        // finish before the buffer is released; the atomic adds follow. The
        // accumulator has rows for whole 128-row tiles, so every add is in
        // bounds. (Warps 12-15 cover lane quarters 0-3: warp & 3 is the
        // quarter.)
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        bool ok = true;
        int gb = 0;
        for (int tt = 0; tt < nt && ok; ++tt) {
            const int n = ns[tt];
            for (int h = 0; h < n && ok; ++h) {
                const int G = gb + h;
                const int b = G & 1;
                ok = __all_sync(0xffffffffu, bwd_wait(bar(L::BAR_DQFULL + b), (G >> 1) & 1, p, abort_flag, kStatusWaitO));
                if (!ok) break;
                tc_fence_after();
                uint32_t lo[32], hi[32];
                tmem_ld32(tmem + lane_field + L::BUF_COL(b), lo);
                tmem_ld32(tmem + lane_field + L::BUF_COL(b) + 32, hi);
                tmem_wait_ld();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::BAR_DQREAD + b));
                float* dst = p.dq_acc + (row0 + static_cast<size_t>(h0s[tt] + h) * kBwdHalf) * D + hd * L::DH + r;
#pragma unroll
                for (int e = 0; e < 32; ++e) atomicAdd(dst + e * D, __uint_as_float(lo[e]));
#pragma unroll
                for (int e = 0; e < 32; ++e) atomicAdd(dst + (32 + e) * D, __uint_as_float(hi[e]));
            }
            gb += n;
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// Per padded query row (one warp per row, D / 32 columns per lane): -D_i =
// -sum_c dO_ic O_ic (fp32 from bf16), -LSE log2e, and a zeroed dQ accumulator
// row. Rows past Nq get -inf and 0; so do rows whose LSE is -inf (no key).
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_pre_kernel(const __nv_bfloat16* __restrict__ o,
                                                         const __nv_bfloat16* __restrict__ dout,
                                                         const float* __restrict__ lse,
                                                         float* __restrict__ nlse2, float* __restrict__ ndd,
                                                         float* __restrict__ dq_acc, long long rows_pad,
                                                         int Nq, int Nq_pad) {
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows_pad) return;
    const long long bh = row / Nq_pad;
    const int q = static_cast<int>(row - bh * Nq_pad);
    float s = 0.f, nl = -INFINITY;
    if (q < Nq) {
        const size_t src_row = static_cast<size_t>(bh) * Nq + q;
        const size_t base = src_row * D + lane * (D / 32);
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(o + base);
        const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(dout + base);
#pragma unroll
        for (int e = 0; e < D / 64; ++e) {
            const float2 a = __bfloat1622float2(o2[e]);
            const float2 b = __bfloat1622float2(d2[e]);
            s = fmaf(a.x, b.x, s);
            s = fmaf(a.y, b.y, s);
        }
        for (int w = 16; w > 0; w >>= 1) s += __shfl_xor_sync(0xffffffffu, s, w);
        const float l = lse[src_row];
        nl = (l == -INFINITY) ? -INFINITY : -(l * kLog2e);
    }
    if (lane == 0) {
        ndd[row] = -s;
        nlse2[row] = nl;
    }
    float* z = dq_acc + static_cast<size_t>(row) * D + lane * (D / 32);
    if constexpr (D >= 128) {
#pragma unroll
        for (int e = 0; e < D / 128; ++e) reinterpret_cast<float4*>(z)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
        *reinterpret_cast<float2*>(z) = make_float2(0.f, 0.f);
    }
}

// dQ = scale * accumulator, to bf16: one warp per query row, D / 32 columns
// per lane, reading the accumulator's padded rows.
template <int D>
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float* __restrict__ acc,
                                                        __nv_bfloat16* __restrict__ dq, long long rows,
                                                        int Nq, int Nq_pad, float scale) {
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const long long bh = row / Nq;
    const long long arow = bh * Nq_pad + (row - bh * Nq);
    const float* src = acc + static_cast<size_t>(arow) * D + lane * (D / 32);
    __nv_bfloat16* dst = dq + static_cast<size_t>(row) * D + lane * (D / 32);
    if constexpr (D >= 128) {
#pragma unroll
        for (int e = 0; e < D / 128; ++e) {
            const float4 a = reinterpret_cast<const float4*>(src)[e];
            __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * scale, a.y * scale);
            __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * scale, a.w * scale);
            uint2 out;
            out.x = *reinterpret_cast<uint32_t*>(&lo);
            out.y = *reinterpret_cast<uint32_t*>(&hi);
            reinterpret_cast<uint2*>(dst)[e] = out;
        }
    } else {
        const float2 a = *reinterpret_cast<const float2*>(src);
        *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(a.x * scale, a.y * scale);
    }
}

}  // namespace

template <int D>
cudaError_t launch_bwd_pre(const void* o, const void* dout, const float* lse, float* nlse2, float* ndd,
                           float* dq_acc, int BH, int Nq, int Nq_pad, cudaStream_t stream) {
    const long long rows_pad = static_cast<long long>(BH) * Nq_pad;
    const long long blocks = (rows_pad + 7) / 8;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    fa_bwd_pre_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, nlse2, ndd,
        dq_acc, rows_pad, Nq, Nq_pad);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_main(const BwdParams& p, cudaStream_t stream) {
    using L = LayoutBwd<D>;
    // Kernel attributes belong to the context: set once per device and context.
    static ContextCache<int> attr_set;
    int done = 0;
    const cudaError_t e = attr_set.get(&done, [](int* out) {
        *out = 1;
        return cudaFuncSetAttribute(fa_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(L::ALLOC_BYTES));
    });
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.BH) * p.tile_units * L::HALVES;
    if (ctas < 1 || ctas > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    fa_bwd_kernel<D><<<static_cast<unsigned>(ctas), L::THREADS, L::ALLOC_BYTES, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_bwd_dq(const float* dq_acc, void* dq, int BH, int Nq, int Nq_pad, float scale,
                          cudaStream_t stream) {
    const long long rows = static_cast<long long>(BH) * Nq;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    fa_bwd_dq_kernel<D><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        dq_acc, static_cast<__nv_bfloat16*>(dq), rows, Nq, Nq_pad, scale);
    return cudaGetLastError();
}

// The three launches of one backward call at head dim D.
template <int D>
cudaError_t launch_bwd(const BwdParams& p, const void* o, const void* dout, const float* lse, void* dq,
                       cudaStream_t stream) {
    cudaError_t e = launch_bwd_pre<D>(o, dout, lse, const_cast<float*>(p.nlse2), const_cast<float*>(p.ndd),
                                      p.dq_acc, p.BH, p.Nq, p.Nq_pad, stream);
    if (e == cudaSuccess) e = launch_bwd_main<D>(p, stream);
    if (e == cudaSuccess) e = launch_bwd_dq<D>(p.dq_acc, dq, p.BH, p.Nq, p.Nq_pad, p.scale, stream);
    return e;
}

}  // namespace fa

extern "C" {

size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int d) {
    if (B < 1 || H < 1 || Nq < 1 || (d != 64 && d != 128 && d != 256)) return 0;
    const size_t rows_pad = static_cast<size_t>(B) * H * ((static_cast<size_t>(Nq) + 127) / 128 * 128);
    return rows_pad * (static_cast<size_t>(d) + 2) * sizeof(float);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace, int B, int H,
                 int Nq, int Nk, int d, float scale, int causal, cudaStream_t stream) {
    fa_status s = fa::check_common(q, k, v, B, H, Nq, Nk, d, scale);
    if (s != FA_OK) return s;
    // Query rows are padded to whole 128-row tiles and key tiles counted in
    // int: both lengths must leave room for that rounding.
    if (Nq > 0x7fffffff - 127 || Nk > 0x7fffffff - 127) return FA_ERR_SHAPE;
    if (d != 64 && d != 128 && d != 256) return FA_ERR_HEADDIM;
    if (!fa::valid_causal(causal)) return FA_ERR_CAUSAL;
    if (!o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_NULL;
    if (!fa::aligned(o, 16) || !fa::aligned(dout, 16) || !fa::aligned(lse, 4) ||
        !fa::aligned(dq, 16) || !fa::aligned(dk, 16) || !fa::aligned(dv, 16))
        return FA_ERR_ALIGN;
    if (!workspace || !fa::aligned(workspace, 16)) return FA_ERR_WORKSPACE;
    const int BH = B * H;
    const int Nq_pad = (Nq + 127) / 128 * 128;
    const size_t rows_pad = static_cast<size_t>(BH) * Nq_pad;
    float* dq_acc = static_cast<float*>(workspace);
    float* nlse2 = dq_acc + rows_pad * d;
    float* ndd = nlse2 + rows_pad;
    fa::BwdParams p;
    std::memset(&p, 0, sizeof(p));
    if (!fa::encode_rows_map(&p.tm_q, q, d, Nq, BH, 64) ||
        !fa::encode_rows_map(&p.tm_k, k, d, Nk, BH, 128) ||
        !fa::encode_rows_map(&p.tm_v, v, d, Nk, BH, 128) ||
        !fa::encode_rows_map(&p.tm_do, dout, d, Nq, BH, 64))
        return FA_ERR_CUDA;
    p.nlse2 = nlse2;
    p.ndd = ndd;
    p.dq_acc = dq_acc;
    p.dk = dk;
    p.dv = dv;
    p.BH = BH;
    p.Nq = Nq;
    p.Nk = Nk;
    p.Nq_pad = Nq_pad;
    p.causal = causal ? 1 : 0;
    p.causal_br = (causal == FA_CAUSAL_BOTTOM_RIGHT) ? 1 : 0;
    p.k_tiles = (Nk + 127) / 128;
    // Under a causal mask a key tile's query steps fall with its index: pairs
    // of tiles from both ends give every CTA about the same work (measured on
    // the C2 shape: 1-2.5 % faster at d = 64 and 128; at d = 256, whose single
    // Q/dO stage leaves the hand-over between the tiles exposed, 2 % slower).
    p.pair_tiles = (causal && d <= 128) ? 1 : 0;
    p.tile_units = p.pair_tiles ? (p.k_tiles + 1) / 2 : p.k_tiles;
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_limit = fa::kDefaultWaitLimit;
    if (fa::device_status_ptr(&p.status) != cudaSuccess) return FA_ERR_CUDA;
    const cudaError_t e = d == 64    ? fa::launch_bwd<64>(p, o, dout, lse, dq, stream)
                          : d == 128 ? fa::launch_bwd<128>(p, o, dout, lse, dq, stream)
                                     : fa::launch_bwd<256>(p, o, dout, lse, dq, stream);
    return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
