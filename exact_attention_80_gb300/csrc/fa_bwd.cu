// fa_bwd.cu — attention backward for head dim 128: dQ, dK, dV. Holds the
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
// fa_bwd_kernel roles: warp 0 loads K and V once and (Q_i, dO_i) per query
// tile into two buffers (TMA); warp 1 issues tcgen05 MMAs; warps 4-11 are the
// compute group, two warps per TMEM lane quarter, each owning two 32-query
// chunks (thread = TMEM lane = key row). Per query tile i:
//   S^T = K Q_i^T and dP^T = V dO_i^T (lanes = keys, columns = queries);
//   the compute group forms P^T = exp2(S^T scale log2e - LSE log2e) and
//   dS^T = P^T (dP^T - D), writes both as bf16 into TMEM over the first half
//   of each chunk's own columns, and dS^T into shared memory (128-byte
//   swizzle);
//   dV += P^T dO_i and dK += dS^T Q_i (A from TMEM, B = dO_i / Q_i MN-major);
//   dQ_i^T = K^T dS^T (A = K MN-major, B = dS^T from shared memory) into the
//   dP^T columns, so S^T of the next tile can be computed while the compute
//   group (lane = head dim) adds dQ_i^T to the fp32 accumulator, 32
//   consecutive floats per warp instruction.
// Every mbarrier wait is bounded, as in the forward kernels.
#include <cuda_bf16.h>

#include <cstring>

#include "fa.h"
#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

// Kernel parameters, filled by fa_bwd below.
struct BwdParams {
    CUtensorMap tm_q;   // bf16 [B*H][Nq][d], box {64, 128, 1}
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
    float scale;
    float scale_log2;   // scale * log2(e)
    long long wait_limit;
    unsigned* status;
};

namespace {

constexpr int kBwdD = 128;
constexpr int kBwdTile = 128;   // keys per CTA, queries per step
constexpr int kBwdGroups = 2;   // compute warps per TMEM lane quarter
constexpr int kBwdChunks = (kBwdTile / 32) / kBwdGroups;  // 32-query chunks per compute warp
constexpr float kLog2e = 1.4426950408889634f;

struct LayoutBwd {
    static constexpr int COMPUTE_WARPS = 4 * kBwdGroups;
    static constexpr int THREADS = 128 + 32 * COMPUTE_WARPS;
    static constexpr uint32_t TILE_BYTES = kBwdTile * kBwdD * 2;  // 32 KB, two 64-column chunks
    static constexpr uint32_t CHUNK_BYTES = kBwdTile * 128;       // one 64-column chunk
    static constexpr uint32_t K_OFF = 0;
    static constexpr uint32_t V_OFF = K_OFF + TILE_BYTES;
    static constexpr uint32_t Q_OFF = V_OFF + TILE_BYTES;        // [2]
    static constexpr uint32_t DO_OFF = Q_OFF + 2 * TILE_BYTES;   // [2]
    static constexpr uint32_t DS_OFF = DO_OFF + 2 * TILE_BYTES;  // dS^T, bf16 [keys][queries]
    static constexpr uint32_t BAR_OFF = DS_OFF + TILE_BYTES;
    static constexpr int BAR_KV = 0;
    static constexpr int BAR_QFULL = 1;    // [2]
    static constexpr int BAR_QEMPTY = 3;   // [2]
    static constexpr int BAR_SFULL = 5;    // S^T and dP^T done
    static constexpr int BAR_PREADY = 6;   // P^T, dS^T written (one arrival per compute warp)
    static constexpr int BAR_DQFULL = 7;   // dQ^T done (and every earlier MMA)
    static constexpr int BAR_DQREAD = 8;   // dQ^T read out (one arrival per compute warp)
    static constexpr int BAR_DRAIN = 9;
    static constexpr int NUM_BARS = 10;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;
    static constexpr uint32_t BYTES = MISC_OFF + 16;
    static constexpr size_t ALLOC_BYTES = BYTES + 1024;
    // TMEM columns: S^T (then P^T), dP^T (then dS^T, then dQ^T), dV, dK.
    static constexpr uint32_t ST_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 384;
    static_assert(ALLOC_BYTES <= 232448, "shared memory over the 227 KB per-CTA limit");
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

// Query tiles a key tile sees: all of them, or (causal) those with a row at or
// after the tile's first key minus the alignment offset.
__device__ __forceinline__ void bwd_steps(const BwdParams& p, int kt, int& i0, int& n) {
    const int q_tiles = (p.Nq + kBwdTile - 1) / kBwdTile;
    i0 = 0;
    if (p.causal) {
        const int off = p.causal_br ? p.Nk - p.Nq : 0;
        const int first_row = kt * kBwdTile - off;  // key k is visible to rows >= k - off
        i0 = first_row <= 0 ? 0 : first_row / kBwdTile;
    }
    n = max(0, q_tiles - i0);
}

// P^T and dS^T of one 32-query chunk for this thread's key row: s and dp are
// the chunk's S^T and dP^T columns, nl and nd point at the chunk's -LSE log2e
// and -D (the same addresses for every lane: one broadcast load per four
// queries). MASK: `lim` is the first visible chunk column (causal) and
// `key_ok` whether the key exists; without MASK every entry is visible.
template <bool MASK>
__device__ __forceinline__ void bwd_chunk(const uint32_t (&s)[32], const uint32_t (&dp)[32],
                                          const float* __restrict__ nl, const float* __restrict__ nd,
                                          float sl2, int lim, bool key_ok, uint32_t (&pk)[16],
                                          uint32_t (&dk)[16]) {
    const uint64_t sl2x2 = f2pack(sl2, sl2);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const float4 l4 = __ldg(reinterpret_cast<const float4*>(nl) + u);
        const float4 d4 = __ldg(reinterpret_cast<const float4*>(nd) + u);
        const uint64_t x01 = ffma2(f2pack(__uint_as_float(s[4 * u]), __uint_as_float(s[4 * u + 1])), sl2x2,
                                   f2pack(l4.x, l4.y));
        const uint64_t x23 = ffma2(f2pack(__uint_as_float(s[4 * u + 2]), __uint_as_float(s[4 * u + 3])), sl2x2,
                                   f2pack(l4.z, l4.w));
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
                                   f2pack(d4.x, d4.y));
        const uint64_t g23 = fadd2(f2pack(__uint_as_float(dp[4 * u + 2]), __uint_as_float(dp[4 * u + 3])),
                                   f2pack(d4.z, d4.w));
        float ds[4];
        f2unpack(fmul2(f2pack(pv[0], pv[1]), g01), ds[0], ds[1]);
        f2unpack(fmul2(f2pack(pv[2], pv[3]), g23), ds[2], ds[3]);
        pk[2 * u] = pack_bf16x2(pv[0], pv[1]);
        pk[2 * u + 1] = pack_bf16x2(pv[2], pv[3]);
        dk[2 * u] = pack_bf16x2(ds[0], ds[1]);
        dk[2 * u + 1] = pack_bf16x2(ds[2], ds[3]);
    }
}

__global__ void __launch_bounds__(LayoutBwd::THREADS, 1) fa_bwd_kernel(const __grid_constant__ BwdParams p) {
    using L = LayoutBwd;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
    volatile uint32_t* abort_flag = misc + 1;
    auto bar = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8u * i; };
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const int bh = blockIdx.x / p.k_tiles;
    const int kt = blockIdx.x % p.k_tiles;
    const int k0 = kt * kBwdTile;
    int i0, n;
    bwd_steps(p, kt, i0, n);

    if (threadIdx.x == 0) {
        mbar_init(bar(L::BAR_KV), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::BAR_QFULL + b), 1);
            mbar_init(bar(L::BAR_QEMPTY + b), 1);
        }
        mbar_init(bar(L::BAR_SFULL), 1);
        mbar_init(bar(L::BAR_PREADY), L::COMPUTE_WARPS);
        mbar_init(bar(L::BAR_DQFULL), 1);
        mbar_init(bar(L::BAR_DQREAD), L::COMPUTE_WARPS);
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
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0 && n > 0) {
        // ------------------------------------------------------------ producer
        const bool leader = elect_one();
        if (leader) {
            mbar_arrive_expect_tx(bar(L::BAR_KV), 2 * L::TILE_BYTES);
            for (int c = 0; c < 2; ++c) {
                tma_load_3d(sbase + L::K_OFF + c * L::CHUNK_BYTES, &p.tm_k, bar(L::BAR_KV), 64 * c, k0, bh);
                tma_load_3d(sbase + L::V_OFF + c * L::CHUNK_BYTES, &p.tm_v, bar(L::BAR_KV), 64 * c, k0, bh);
            }
        }
        bool ok = true;
        int issued = 0;
        for (int i = 0; i < n && ok; ++i) {
            const int b = i & 1;
            if (i >= 2)
                ok = __all_sync(0xffffffffu, bwd_wait(bar(L::BAR_QEMPTY + b), ((i >> 1) - 1) & 1, p,
                                                      abort_flag, kStatusWaitKvEmpty));
            if (!ok) break;
            if (leader) {
                const int q0 = (i0 + i) * kBwdTile;
                mbar_arrive_expect_tx(bar(L::BAR_QFULL + b), 2 * L::TILE_BYTES);
                for (int c = 0; c < 2; ++c) {
                    tma_load_3d(sbase + L::Q_OFF + b * L::TILE_BYTES + c * L::CHUNK_BYTES, &p.tm_q,
                                bar(L::BAR_QFULL + b), 64 * c, q0, bh);
                    tma_load_3d(sbase + L::DO_OFF + b * L::TILE_BYTES + c * L::CHUNK_BYTES, &p.tm_do,
                                bar(L::BAR_QFULL + b), 64 * c, q0, bh);
                }
            }
            issued = i + 1;
        }
        if (ok) {
            // The issuer's last buffer releases: no commit arrival may still be in
            // flight when the CTA exits.
            for (int i = max(0, n - 2); i < n && ok; ++i)
                ok = __all_sync(0xffffffffu, bwd_wait(bar(L::BAR_QEMPTY + (i & 1)), (i >> 1) & 1, p, abort_flag,
                                                      kStatusWaitKvEmpty));
        } else {
            bwd_wait(bar(L::BAR_KV), 0, p, abort_flag, kStatusWaitDrain, false);
            for (int i = max(0, issued - 2); i < issued; ++i)
                bwd_wait(bar(L::BAR_QFULL + (i & 1)), (i >> 1) & 1, p, abort_flag, kStatusWaitDrain, false);
        }
    } else if (warp == 1 && n > 0) {
        // ------------------------------------------------------------ MMA issuer
        const bool leader = elect_one();
        auto wait_all = [&](uint32_t b, uint32_t parity, unsigned what) {
            return __all_sync(0xffffffffu, bwd_wait(b, parity, p, abort_flag, what));
        };
        constexpr uint32_t IDESC_T = make_idesc_bf16(128, 128, false, false);  // S^T, dP^T
        constexpr uint32_t IDESC_ACC = make_idesc_bf16(128, 128, false, true);  // dV, dK
        constexpr uint32_t IDESC_DQ = make_idesc_bf16(128, 128, true, true);    // dQ^T
        const uint64_t kmaj0 = make_sdesc_sw128(sbase, 16, 1024);
        const uint64_t mn0 = make_sdesc_sw128(sbase, L::CHUNK_BYTES, 1024);
        const uint32_t kmaj_lo = static_cast<uint32_t>(kmaj0), kmaj_hi = static_cast<uint32_t>(kmaj0 >> 32);
        const uint32_t mn_lo = static_cast<uint32_t>(mn0), mn_hi = static_cast<uint32_t>(mn0 >> 32);
        auto desc = [](uint32_t lo, uint32_t hi, uint32_t off) -> uint64_t {
            return (static_cast<uint64_t>(hi) << 32) | (lo + (off >> 4));
        };
        // D(lanes = rows of a) = a b^T over the head dim, both K-major tiles.
        auto mma_t = [&](uint32_t d_col, uint32_t a_off, uint32_t b_off) {
#pragma unroll
            for (int kk = 0; kk < kBwdD / 16; ++kk) {
                const uint32_t in_row = (kk & 3) * 32 + (kk >> 2) * L::CHUNK_BYTES;
                const uint64_t a = desc(kmaj_lo, kmaj_hi, a_off + in_row);
                const uint64_t b = desc(kmaj_lo, kmaj_hi, b_off + in_row);
                if (leader) umma_ss(tmem + d_col, a, b, IDESC_T, kk > 0 ? 1u : 0u);
            }
        };
        bool ok = wait_all(bar(L::BAR_KV), 0, kStatusWaitKvFull);
        for (int i = 0; i < n && ok; ++i) {
            const int b = i & 1;
            ok = wait_all(bar(L::BAR_QFULL + b), (i >> 1) & 1, kStatusWaitQ);
            if (!ok) break;
            tc_fence_after();
            const uint32_t qb = L::Q_OFF + b * L::TILE_BYTES;
            const uint32_t dob = L::DO_OFF + b * L::TILE_BYTES;
            // S^T = K Q^T. The S^T columns last held P^T of the previous tile,
            // which its dV MMAs (issued earlier, run in order) have consumed.
            mma_t(L::ST_COL, L::K_OFF, qb);
            // dQ^T of the previous tile sits in the dP^T columns until read out.
            if (i > 0) {
                ok = wait_all(bar(L::BAR_DQREAD), (i - 1) & 1, kStatusWaitO);
                if (!ok) break;
                tc_fence_after();
            }
            mma_t(L::DP_COL, L::V_OFF, dob);  // dP^T = V dO^T
            if (leader) umma_commit(bar(L::BAR_SFULL));
            ok = wait_all(bar(L::BAR_PREADY), i & 1, kStatusWaitP);
            if (!ok) break;
            tc_fence_after();
            // dV += P^T dO and dK += dS^T Q: A from TMEM (16 queries = 8 packed
            // columns, each 32-query chunk packed into the first 16 columns of its
            // own 32), B MN-major (16 query rows = 2048 bytes).
#pragma unroll
            for (int kk = 0; kk < kBwdTile / 16; ++kk) {
                const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
                const uint32_t pcol = 32 * (kk >> 1) + 8 * (kk & 1);
                const uint64_t bdo = desc(mn_lo, mn_hi, dob + kk * 2048);
                const uint64_t bq = desc(mn_lo, mn_hi, qb + kk * 2048);
                if (leader) {
                    umma_ts(tmem + L::DV_COL, tmem + L::ST_COL + pcol, bdo, IDESC_ACC, acc);
                    umma_ts(tmem + L::DK_COL, tmem + L::DP_COL + pcol, bq, IDESC_ACC, acc);
                }
            }
            if (leader) umma_commit(bar(L::BAR_QEMPTY + b));
            // dQ^T = K^T dS^T into the dP^T columns (after the dK MMAs that read
            // dS^T there, in issue order): A = K MN-major (M = head dim), B = dS^T
            // MN-major (N = queries), 16 keys = 2048 bytes per step.
#pragma unroll
            for (int kk = 0; kk < kBwdTile / 16; ++kk) {
                const uint64_t a = desc(mn_lo, mn_hi, L::K_OFF + kk * 2048);
                const uint64_t bds = desc(mn_lo, mn_hi, L::DS_OFF + kk * 2048);
                if (leader) umma_ss(tmem + L::DP_COL, a, bds, IDESC_DQ, kk > 0 ? 1u : 0u);
            }
            if (leader) umma_commit(bar(L::BAR_DQFULL));
        }
        if (leader) umma_commit(bar(L::BAR_DRAIN));
        bwd_wait(bar(L::BAR_DRAIN), 0, p, abort_flag, kStatusWaitDrain, false);
    } else if (warp >= 4) {
        // ------------------------------------------------------------ compute group
        const int quarter = warp & 3;
        const int grp = (warp - 4) >> 2;
        const int r = quarter * 32 + lane;   // TMEM lane: key row, or head dim for dQ^T
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        const int key = k0 + r;
        const bool key_ok = key < p.Nk;
        const bool key_tail = k0 + kBwdTile > p.Nk;
        const int off = p.causal_br ? p.Nk - p.Nq : 0;
        const float sl2 = p.scale_log2;
        const size_t row0 = static_cast<size_t>(bh) * p.Nq_pad;
        bool ok = true;
        for (int i = 0; i < n && ok; ++i) {
            const int q0 = (i0 + i) * kBwdTile;
            // Every entry of the tile is visible unless the tile holds missing
            // keys or (causal) crosses the diagonal; padded query rows carry
            // -inf as -LSE log2e, so their P is 0 either way.
            const bool masked = key_tail || (p.causal && k0 + kBwdTile - 1 > q0 + off);
            ok = __all_sync(0xffffffffu, bwd_wait(bar(L::BAR_SFULL), i & 1, p, abort_flag, kStatusWaitS));
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int j = 0; j < kBwdChunks; ++j) {
                const int cc = grp * kBwdChunks + j;
                uint32_t sraw[32], draw[32];
                tmem_ld32(tmem + lane_field + L::ST_COL + cc * 32, sraw);
                tmem_ld32(tmem + lane_field + L::DP_COL + cc * 32, draw);
                tmem_wait_ld();
                const float* nl = p.nlse2 + row0 + q0 + cc * 32;
                const float* nd = p.ndd + row0 + q0 + cc * 32;
                uint32_t pk[16], dk[16];
                if (masked) {
                    // Key row `key` is visible to query q iff key <= q + off.
                    const int lim = p.causal ? key - off - q0 - cc * 32 : -1;
                    bwd_chunk<true>(sraw, draw, nl, nd, sl2, lim, key_ok, pk, dk);
                } else {
                    bwd_chunk<false>(sraw, draw, nl, nd, sl2, 0, true, pk, dk);
                }
                // P^T and dS^T over the first 16 of the chunk's own 32 columns
                // (no other warp reads or writes them).
                tmem_st16(tmem + lane_field + L::ST_COL + cc * 32, pk);
                tmem_st16(tmem + lane_field + L::DP_COL + cc * 32, dk);
                // dS^T into shared memory: row r, queries 32 cc .. 32 cc + 31.
                const uint32_t line = sbase + L::DS_OFF + (cc >> 1) * L::CHUNK_BYTES + r * 128;
                const uint32_t swz = static_cast<uint32_t>(r & 7);
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    const uint32_t u = static_cast<uint32_t>((cc & 1) * 4 + uu);
                    st_shared_v4(line + ((u ^ swz) << 4), dk[4 * uu], dk[4 * uu + 1], dk[4 * uu + 2], dk[4 * uu + 3]);
                }
            }
            fence_proxy_async_smem();
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::BAR_PREADY));
            // dQ^T: lane r = head dim r, columns = this tile's queries. The
            // accumulator has rows for whole tiles, so every add is in bounds.
            ok = __all_sync(0xffffffffu, bwd_wait(bar(L::BAR_DQFULL), i & 1, p, abort_flag, kStatusWaitO));
            if (!ok) break;
            tc_fence_after();
#pragma unroll 1
            for (int j = 0; j < kBwdChunks; ++j) {
                const int cc = grp * kBwdChunks + j;
                uint32_t raw[32];
                tmem_ld32(tmem + lane_field + L::DP_COL + cc * 32, raw);
                tmem_wait_ld();
                float* dst = p.dq_acc + (row0 + q0 + cc * 32) * kBwdD + r;
#pragma unroll
                for (int e = 0; e < 32; ++e) atomicAdd(dst + e * kBwdD, __uint_as_float(raw[e]));
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::BAR_DQREAD));
        }
        // dK (scaled) and dV of this key row, 32 head-dim columns per chunk;
        // zero when no query tile sees it. tcgen05.ld is warp-collective: the
        // loads run for the whole warp (`ok` is warp-uniform), and only the
        // stores check that the key exists.
        if (ok) {
            __nv_bfloat16* dkp = static_cast<__nv_bfloat16*>(p.dk) + (static_cast<size_t>(bh) * p.Nk + key) * kBwdD;
            __nv_bfloat16* dvp = static_cast<__nv_bfloat16*>(p.dv) + (static_cast<size_t>(bh) * p.Nk + key) * kBwdD;
#pragma unroll 1
            for (int j = 0; j < kBwdChunks; ++j) {
                const int cc = grp * kBwdChunks + j;
                uint32_t kr[32], vr[32];
                if (n > 0) {
                    tmem_ld32(tmem + lane_field + L::DK_COL + cc * 32, kr);
                    tmem_ld32(tmem + lane_field + L::DV_COL + cc * 32, vr);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) kr[e] = vr[e] = 0u;
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
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// Per padded query row (one warp per row, four columns per lane): -D_i =
// -sum_c dO_ic O_ic (fp32 from bf16), -LSE log2e, and a zeroed dQ accumulator
// row. Rows past Nq get -inf and 0; so do rows whose LSE is -inf (no key).
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
        const size_t base = src_row * kBwdD + lane * 4;
        const uint2 ov = *reinterpret_cast<const uint2*>(o + base);
        const uint2 dv = *reinterpret_cast<const uint2*>(dout + base);
        const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov);
        const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dv);
        for (int e = 0; e < 2; ++e) {
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
    *reinterpret_cast<float4*>(dq_acc + static_cast<size_t>(row) * kBwdD + lane * 4) =
        make_float4(0.f, 0.f, 0.f, 0.f);
}

// dQ = scale * accumulator, to bf16: one warp per query row, four columns per
// lane, reading the accumulator's padded rows.
__global__ void __launch_bounds__(256) fa_bwd_dq_kernel(const float* __restrict__ acc,
                                                        __nv_bfloat16* __restrict__ dq, long long rows,
                                                        int Nq, int Nq_pad, float scale) {
    const long long row = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const long long bh = row / Nq;
    const long long arow = bh * Nq_pad + (row - bh * Nq);
    const float4 a = *reinterpret_cast<const float4*>(acc + static_cast<size_t>(arow) * kBwdD + lane * 4);
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * scale, a.y * scale);
    __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * scale, a.w * scale);
    uint2 out;
    out.x = *reinterpret_cast<uint32_t*>(&lo);
    out.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dq + static_cast<size_t>(row) * kBwdD + lane * 4) = out;
}

}  // namespace

cudaError_t launch_bwd_pre(const void* o, const void* dout, const float* lse, float* nlse2, float* ndd,
                           float* dq_acc, int BH, int Nq, int Nq_pad, cudaStream_t stream) {
    const long long rows_pad = static_cast<long long>(BH) * Nq_pad;
    const long long blocks = (rows_pad + 7) / 8;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    fa_bwd_pre_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dout), lse, nlse2, ndd,
        dq_acc, rows_pad, Nq, Nq_pad);
    return cudaGetLastError();
}

cudaError_t launch_bwd_main(const BwdParams& p, cudaStream_t stream) {
    // Kernel attributes belong to the context: set once per device and context.
    static ContextCache<int> attr_set;
    int done = 0;
    const cudaError_t e = attr_set.get(&done, [](int* out) {
        *out = 1;
        return cudaFuncSetAttribute(fa_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(LayoutBwd::ALLOC_BYTES));
    });
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>(p.BH) * p.k_tiles;
    if (ctas < 1 || ctas > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    fa_bwd_kernel<<<static_cast<unsigned>(ctas), LayoutBwd::THREADS, LayoutBwd::ALLOC_BYTES, stream>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq(const float* dq_acc, void* dq, int BH, int Nq, int Nq_pad, float scale,
                          cudaStream_t stream) {
    const long long rows = static_cast<long long>(BH) * Nq;
    const long long blocks = (rows + 7) / 8;
    if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    fa_bwd_dq_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        dq_acc, static_cast<__nv_bfloat16*>(dq), rows, Nq, Nq_pad, scale);
    return cudaGetLastError();
}

}  // namespace fa

extern "C" {

size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int d) {
    if (B < 1 || H < 1 || Nq < 1 || d != 128) return 0;
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
    if (d != 128) return FA_ERR_HEADDIM;
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
    if (!fa::encode_rows_map(&p.tm_q, q, d, Nq, BH, 128) ||
        !fa::encode_rows_map(&p.tm_k, k, d, Nk, BH, 128) ||
        !fa::encode_rows_map(&p.tm_v, v, d, Nk, BH, 128) ||
        !fa::encode_rows_map(&p.tm_do, dout, d, Nq, BH, 128))
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
    p.scale = scale;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.wait_limit = fa::kDefaultWaitLimit;
    if (fa::device_status_ptr(&p.status) != cudaSuccess) return FA_ERR_CUDA;
    if (fa::launch_bwd_pre(o, dout, lse, nlse2, ndd, dq_acc, BH, Nq, Nq_pad, stream) != cudaSuccess)
        return FA_ERR_CUDA;
    if (fa::launch_bwd_main(p, stream) != cudaSuccess) return FA_ERR_CUDA;
    if (fa::launch_bwd_dq(dq_acc, dq, BH, Nq, Nq_pad, scale, stream) != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

}  // extern "C"
