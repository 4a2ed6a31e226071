// fa_fwd_kernel.cuh — fused exact attention forward for sm_103a.
//
// One CTA owns Q_TILES query tiles of 128 rows of one (batch, head) and
// sweeps the keys those rows need (all of them, or one key range in split
// mode). Roles, by warp:
//   warp 0      TMA producer: Q tiles once, then K_j, V_j into a ring of
//               STAGES shared-memory slots (full/empty mbarriers).
//   warp 1      tcgen05 issuer (one thread): S_t = Q_t K_j^T into TMEM, and
//               O_t += P_t V_j with P_t read from TMEM; owns TMEM alloc.
//   warps 2-3   idle.
//   warps 4..   one 128-thread softmax group per query tile t: thread = row
//               = TMEM lane. Online softmax on S_t, P_t (bf16) written back
//               into TMEM over S_t, O_t rescaled in TMEM when the running max
//               moves, deferred 1/l and LSE at the end.
// With two query tiles the tensor core works on one tile while the other
// tile's softmax runs (the tensor/vector overlap the FlashAttention-T page
// asks for, section "工程落地：参数、监控与未来演进", "Wavefront 调度").
//
// The recurrence is the FA-3 page's (section 二): per key tile x_j,
//   m_j = max(m_{j-1}, rowmax x_j), l_j = e^{m_{j-1}-m_j} l_{j-1} + rowsum e^{x_j-m_j},
//   O_j = e^{m_{j-1}-m_j} O_{j-1} + e^{x_j-m_j} V_j,
// evaluated in base 2 with log2(e) folded into the scale (x = scale*log2e*s).
//
// Every mbarrier wait is bounded: past `wait_limit` cycles the waiting role
// sets a shared abort flag and a bit in the device status word, the others
// leave at their next wait, in-flight TMA copies and MMAs are waited for
// (again bounded), TMEM is freed and the CTA exits.
#pragma once

#include <cuda_bf16.h>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {

constexpr int kBM = 128;  // query rows per tile = TMEM lanes
// How far (base-2 units) a row's max may rise above the exponent reference
// before the reference moves and O, l are rescaled: p <= 2^8 = 256 is exact
// in bf16's exponent range and far from fp32 overflow.
constexpr float kRescaleSlack = 8.0f;

template <int D>
struct FwdCfg;
template <>
struct FwdCfg<64> {
    static constexpr int Q_TILES = 2, BN = 128, STAGES = 8;
};
template <>
struct FwdCfg<128> {
    static constexpr int Q_TILES = 2, BN = 128, STAGES = 4;
};
template <>
struct FwdCfg<256> {
    static constexpr int Q_TILES = 1, BN = 64, STAGES = 4;
};

template <int D>
struct FwdLayout {
    static constexpr int Q_TILES = FwdCfg<D>::Q_TILES;
    static constexpr int BN = FwdCfg<D>::BN;
    static constexpr int STAGES = FwdCfg<D>::STAGES;
    static constexpr int THREADS = (4 + 4 * Q_TILES) * 32;
    static constexpr int CHUNKS = D / 64;  // 64-element (128-byte) column chunks

    // shared memory (offsets from a 1024-aligned base)
    static constexpr uint32_t Q_TILE_BYTES = kBM * D * 2;
    static constexpr uint32_t SLOT_BYTES = BN * D * 2;
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t SLOT_OFF = Q_OFF + Q_TILES * Q_TILE_BYTES;
    static constexpr uint32_t BAR_OFF = SLOT_OFF + STAGES * SLOT_BYTES;
    static constexpr int BAR_QFULL = 0;
    static constexpr int BAR_KVFULL = 1;
    static constexpr int BAR_KVEMPTY = BAR_KVFULL + STAGES;
    static constexpr int BAR_SFULL = BAR_KVEMPTY + STAGES;
    static constexpr int P_CHUNKS = BN / 64;  // P is written to TMEM in 64-key chunks
    static constexpr int HANDOFFS = 1;  // ... and handed to the MMA in this many parts (one measured best)
    static constexpr int BAR_PFULL = BAR_SFULL + Q_TILES;  // [tile][handoff]
    static constexpr int BAR_OFULL = BAR_PFULL + Q_TILES * HANDOFFS;
    static constexpr int BAR_DRAIN = BAR_OFULL + Q_TILES;
    static constexpr int NUM_BARS = BAR_DRAIN + 1;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;  // [0] tmem base, [1] abort
    static constexpr uint32_t BYTES = MISC_OFF + 16;
    static constexpr size_t ALLOC_BYTES = BYTES + 1024;  // slack for 1024 alignment

    // tensor memory columns (32-bit each; 512 allocated)
    static constexpr uint32_t TMEM_COLS = 512;
    __host__ __device__ static constexpr uint32_t S_COL(int t) { return t * BN; }  // P_t packed over S_t's first BN/2
    __host__ __device__ static constexpr uint32_t O_COL(int t) { return 256 + t * D; }

    static_assert(Q_TILES * BN <= 256, "S/P region overflows its half of TMEM");
    static_assert(256 + Q_TILES * D <= 512, "O region overflows TMEM");
    static_assert(ALLOC_BYTES <= 232448, "shared memory over the 227 KB per-CTA limit");
    static_assert(ALLOC_BYTES > 232448 / 2, "two CTAs per SM would contend for TMEM");
    static_assert(BN % 32 == 0 && D % 64 == 0, "tile shape");

    // Register split (two query tiles): the kernel is compiled for LAUNCH_REGS
    // per thread; the control warpgroup gives registers back and the two
    // softmax warpgroups take them. setmaxnreg.inc waits until the pool has the
    // registers, so the split must add up to exactly the launch allocation;
    // the host refuses to launch if the compiled count differs.
    static constexpr bool REG_SPLIT = (Q_TILES == 2);
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int CTRL_REGS = 72;
    static constexpr int SOFTMAX_REGS = 216;
    static_assert(!REG_SPLIT || 128 * CTRL_REGS + 256 * SOFTMAX_REGS == THREADS * LAUNCH_REGS,
                  "register split must equal the launch allocation");
    static_assert(65536 / THREADS >= LAUNCH_REGS || !REG_SPLIT, "launch registers");
};

// Work owned by one CTA.
template <int Q_TILES>
struct Work {
    int bh;        // batch * H + head
    int q0;        // first query row of the unit
    int split;     // key split index (0 in plain mode)
    int kv_tile0;  // first key tile of the split
    int kv_end;    // exclusive key bound of the split (for masking)
    int n[Q_TILES];  // key tiles each query tile visits
    int nmax;
};

template <int D>
__device__ __forceinline__ void compute_work(const FwdParams& p, Work<FwdCfg<D>::Q_TILES>& w) {
    using L = FwdLayout<D>;
    // CTA order: key splits fastest; then heads in groups of p.head_group
    // (sized so one group is about one wave of CTAs), and within a group the
    // query units heaviest first (last rows first under a causal mask) across
    // the group's heads. CTAs running together share a few heads' K/V in L2,
    // and long causal units start before short ones.
    long long lin = blockIdx.x;
    w.split = static_cast<int>(lin % p.num_splits);
    lin /= p.num_splits;
    const long long per_group = static_cast<long long>(p.head_group) * p.n_units;
    const int group = static_cast<int>(lin / per_group);
    const int r = static_cast<int>(lin % per_group);
    const int heads_here = min(p.head_group, p.BH - group * p.head_group);
    const int unit = p.n_units - 1 - r / heads_here;
    w.bh = group * p.head_group + r % heads_here;
    w.q0 = unit * L::Q_TILES * kBM;
    const int total_tiles = (p.Nk + L::BN - 1) / L::BN;
    const int t0 = min(w.split * p.kv_tiles_per_split, total_tiles);
    const int t1 = min(t0 + p.kv_tiles_per_split, total_tiles);
    w.kv_tile0 = t0;
    w.kv_end = min(p.Nk, t1 * L::BN);
    w.nmax = 0;
#pragma unroll
    for (int t = 0; t < L::Q_TILES; ++t) {
        const int row0 = w.q0 + t * kBM;
        int n = 0;
        if (row0 < p.Nq) {
            int end = t1;
            if (p.causal) {
                const int last_row = min(row0 + kBM - 1, p.Nq - 1);
                end = min(end, last_row / L::BN + 1);
            }
            n = max(0, end - t0);
        }
        w.n[t] = n;
        w.nmax = max(w.nmax, n);
    }
}

// Bounded wait on an mbarrier phase. Returns false if this CTA is aborting
// (honor_abort) or the wait ran past the limit (then raises the abort).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const FwdParams& p,
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

template <int D>
__global__ void __launch_bounds__(FwdLayout<D>::THREADS, 1)
    fa_fwd_kernel(const __grid_constant__ FwdParams p) {
    using L = FwdLayout<D>;
    constexpr int QT = L::Q_TILES;
    constexpr int BN = L::BN;
    constexpr int ST = L::STAGES;

    extern __shared__ uint8_t smem_raw[];
    // Swizzle atoms need 1024-byte alignment in the shared window itself.
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    uint32_t* misc = reinterpret_cast<uint32_t*>(smem + L::MISC_OFF);
    volatile uint32_t* abort_flag = misc + 1;
    auto bar = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8u * i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    Work<QT> w;
    compute_work<D>(p, w);

    if (threadIdx.x == 0) {
        mbar_init(bar(L::BAR_QFULL), 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar(L::BAR_KVFULL + s), 1);
            mbar_init(bar(L::BAR_KVEMPTY + s), 1);
        }
        for (int t = 0; t < QT; ++t) {
            mbar_init(bar(L::BAR_SFULL + t), 1);
            for (int h = 0; h < L::HANDOFFS; ++h) mbar_init(bar(L::BAR_PFULL + t * L::HANDOFFS + h), kBM);
            mbar_init(bar(L::BAR_OFULL + t), 1);
        }
        mbar_init(bar(L::BAR_DRAIN), 1);
        *abort_flag = 0u;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&p.tm_q);
        tma_prefetch_desc(&p.tm_k);
        tma_prefetch_desc(&p.tm_v);
    }
    if (warp == 1) {
        tmem_alloc(sbase + L::MISC_OFF, L::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp < 4) {
      // Control warpgroup. setmaxnreg sits inside each role's branch so that
      // the register allocator sees one limit per code path.
      if constexpr (L::REG_SPLIT) setmaxnreg_dec<L::CTRL_REGS>();
      if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && w.nmax > 0) {
            int nvalid = 0;
#pragma unroll
            for (int t = 0; t < QT; ++t) nvalid += (w.n[t] > 0) ? 1 : 0;
            mbar_arrive_expect_tx(bar(L::BAR_QFULL), nvalid * L::Q_TILE_BYTES);
#pragma unroll
            for (int t = 0; t < QT; ++t) {
                if (w.n[t] > 0) {
#pragma unroll
                    for (int c = 0; c < L::CHUNKS; ++c)
                        tma_load_3d(sbase + L::Q_OFF + t * L::Q_TILE_BYTES + c * (kBM * 128),
                                    &p.tm_q, bar(L::BAR_QFULL), 64 * c, w.q0 + t * kBM, w.bh);
                }
            }
            const int total = 2 * w.nmax;  // K_0, V_0, K_1, V_1, ...
            int issued = 0;
            bool ok = true;
            for (int seq = 0; seq < total; ++seq) {
                const int slot = seq % ST;
                const int use = seq / ST;
                if (use > 0) {
                    ok = wait_phase(bar(L::BAR_KVEMPTY + slot), (use - 1) & 1, p, abort_flag,
                                    kStatusWaitKvEmpty);
                    if (!ok) break;
                }
                mbar_arrive_expect_tx(bar(L::BAR_KVFULL + slot), L::SLOT_BYTES);
                const CUtensorMap* map = (seq & 1) ? &p.tm_v : &p.tm_k;
                const int row = (w.kv_tile0 + (seq >> 1)) * BN;
#pragma unroll
                for (int c = 0; c < L::CHUNKS; ++c)
                    tma_load_3d(sbase + L::SLOT_OFF + slot * L::SLOT_BYTES + c * (BN * 128), map,
                                bar(L::BAR_KVFULL + slot), 64 * c, row, w.bh);
                issued = seq + 1;
            }
            if (ok) {
                // Producer tail: wait until the issuer has released the last use
                // of every slot, so no tcgen05.commit arrival is still in flight
                // towards this CTA's shared memory when it exits.
                for (int seq = max(0, total - ST); seq < total && ok; ++seq)
                    ok = wait_phase(bar(L::BAR_KVEMPTY + seq % ST), (seq / ST) & 1, p, abort_flag,
                                    kStatusWaitKvEmpty);
            }
            if (!ok) {
                // Let every copy already issued land before the CTA goes away.
                wait_phase(bar(L::BAR_QFULL), 0, p, abort_flag, kStatusWaitDrain, false);
                for (int seq = max(0, issued - ST); seq < issued; ++seq)
                    wait_phase(bar(L::BAR_KVFULL + seq % ST), (seq / ST) & 1, p, abort_flag,
                               kStatusWaitDrain, false);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0 && w.nmax > 0) {
            constexpr uint32_t IDESC_S = make_idesc_bf16(kBM, BN, false, false);
            constexpr uint32_t IDESC_O = make_idesc_bf16(kBM, D, false, true);
            auto issue_s = [&](int t, int slot) {
                const uint32_t qa = sbase + L::Q_OFF + t * L::Q_TILE_BYTES;
                const uint32_t kb = sbase + L::SLOT_OFF + slot * L::SLOT_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t in_row = (kk & 3) * 32;  // 16 bf16 = 32 bytes of a 128-byte row
                    const uint64_t a = make_sdesc_sw128(qa + (kk >> 2) * (kBM * 128) + in_row, 16, 1024);
                    const uint64_t b = make_sdesc_sw128(kb + (kk >> 2) * (BN * 128) + in_row, 16, 1024);
                    umma_ss(tmem + L::S_COL(t), a, b, IDESC_S, kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int slot, int part, bool accumulate) {
                const uint32_t vb = sbase + L::SLOT_OFF + slot * L::SLOT_BYTES;
                constexpr int KK = BN / 16 / L::HANDOFFS;  // MMAs (16 keys each) per hand-off
#pragma unroll
                for (int kk = part * KK; kk < part * KK + KK; ++kk) {
                    // V is MN-major: 16 keys = two 8-row swizzle atoms (2048 bytes);
                    // 64-column chunks of d are BN*128 bytes apart.
                    const uint64_t b = make_sdesc_sw128(vb + kk * 2048, BN * 128, 1024);
                    umma_ts(tmem + L::O_COL(t), tmem + L::S_COL(t) + kk * 8, b, IDESC_O,
                            (accumulate || kk > 0) ? 1u : 0u);
                }
            };

            bool ok = wait_phase(bar(L::BAR_QFULL), 0, p, abort_flag, kStatusWaitQ);
            int seq = 0;
            if (ok) ok = wait_phase(bar(L::BAR_KVFULL + 0), 0, p, abort_flag, kStatusWaitKvFull);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < QT; ++t) {
                    if (w.n[t] > 0) {
                        issue_s(t, 0);
                        umma_commit(bar(L::BAR_SFULL + t));
                    }
                }
                umma_commit(bar(L::BAR_KVEMPTY + 0));
                seq = 1;
                for (int j = 0; j < w.nmax && ok; ++j) {
                    const int slot_v = seq % ST;
                    ok = wait_phase(bar(L::BAR_KVFULL + slot_v), (seq / ST) & 1, p, abort_flag,
                                    kStatusWaitKvFull);
                    if (!ok) break;
                    ++seq;
                    const bool k_next = (j + 1 < w.nmax);
                    int slot_k = 0;
                    if (k_next) {
                        slot_k = seq % ST;
                        ok = wait_phase(bar(L::BAR_KVFULL + slot_k), (seq / ST) & 1, p, abort_flag,
                                        kStatusWaitKvFull);
                        if (!ok) break;
                        ++seq;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int t = 0; t < QT; ++t) {
                        if (ok && j < w.n[t]) {
                            // O_t += P_t V_j chunk by chunk, each as soon as the
                            // softmax has written that chunk of P_t.
#pragma unroll
                            for (int h = 0; h < L::HANDOFFS; ++h) {
                                ok = wait_phase(bar(L::BAR_PFULL + t * L::HANDOFFS + h), j & 1, p,
                                                abort_flag, kStatusWaitP);
                                if (!ok) break;
                                tc_fence_after();
                                issue_pv(t, slot_v, h, j > 0);
                            }
                            if (!ok) break;
                            if (j + 1 < w.n[t]) {
                                issue_s(t, slot_k);
                                umma_commit(bar(L::BAR_SFULL + t));
                            } else {
                                umma_commit(bar(L::BAR_OFULL + t));
                            }
                        }
                    }
                    if (!ok) break;
                    umma_commit(bar(L::BAR_KVEMPTY + slot_v));
                    if (k_next) umma_commit(bar(L::BAR_KVEMPTY + slot_k));
                }
            }
            if (!ok) {
                // Wait for every MMA already issued before TMEM is released.
                umma_commit(bar(L::BAR_DRAIN));
                wait_phase(bar(L::BAR_DRAIN), 0, p, abort_flag, kStatusWaitDrain, false);
            }
        }
      }
    } else {
        // ------------------------------------------------------------ softmax
        if constexpr (L::REG_SPLIT) setmaxnreg_inc<L::SOFTMAX_REGS>();
        const int t = (warp - 4) >> 2;
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int r = quarter * 32 + lane;
        const int q_row = w.q0 + t * kBM + r;
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_field + L::S_COL(t);
        const uint32_t tO = tmem + lane_field + L::O_COL(t);
        const float sl2 = p.scale_log2;
        int n = w.n[0];
#pragma unroll
        for (int i = 1; i < QT; ++i)
            if (t == i) n = w.n[i];

        float m = -INFINITY;       // exponent reference (base-2 units of scale*log2e*s)
        float m_true = -INFINITY;  // true running row max, same units
        float l = 0.f;             // running sum relative to m
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            ok = wait_phase(bar(L::BAR_SFULL + t), j & 1, p, abort_flag, kStatusWaitS);
            // tcgen05.ld/st are warp-collective: the whole warp leaves together.
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            tc_fence_after();

            float s[BN];
#pragma unroll
            for (int cc = 0; cc < BN / 32; ++cc) {
                uint32_t raw[32];
                tmem_ld32(tS + cc * 32, raw);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[cc * 32 + i] = __uint_as_float(raw[i]);
            }
            tmem_wait_ld();

            // Mask: keys past the split / sequence end, and (causal) keys after
            // this row. TMA zero-fills keys >= Nk, so they must become -inf.
            const int kv0 = (w.kv_tile0 + j) * BN;
            int valid = w.kv_end - kv0;
            if (p.causal) valid = min(valid, q_row - kv0 + 1);
            if (valid < BN) {
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (c >= valid) s[c] = -INFINITY;
            }
            __syncwarp();

            // Row max: four independent three-input max chains.
            float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; c += 8) {
                a0 = max3f(a0, s[c + 0], s[c + 1]);
                a1 = max3f(a1, s[c + 2], s[c + 3]);
                a2 = max3f(a2, s[c + 4], s[c + 5]);
                a3 = max3f(a3, s[c + 6], s[c + 7]);
            }
            const float m_tile = max3f(a0, a1, fmaxf(a2, a3)) * sl2;  // base-2 units
            m_true = fmaxf(m_true, m_tile);
            // The exponent reference m only moves when this tile's max exceeds it
            // by more than kRescaleSlack; otherwise every p = 2^(x - m) <= 2^slack
            // and the old reference is kept, so O and l need no rescale. The
            // result is the same: O/l and m + log2(l) do not depend on which
            // reference is used, only rounding does.
            const bool move = m_tile > m + kRescaleSlack;
            const float m_new = move ? m_tile : m;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // all masked so far
            const float alpha = move ? ex2(m - m_use) : 1.f;
            const float neg = -m_use;

            // Rescale the accumulator before any of this tile's PV MMAs run.
            // PV_{j-1} has completed: the commit that signalled S_j came after it.
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                const uint64_t ax2 = f2pack(alpha, alpha);
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tO + cc * 32, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float x0, x1;
                        f2unpack(fmul2(f2pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), ax2),
                                 x0, x1);
                        o[2 * i] = __float_as_uint(x0);
                        o[2 * i + 1] = __float_as_uint(x1);
                    }
                    tmem_st32(tO + cc * 32, o);
                }
            }

            float part[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // partial row sums
#pragma unroll
            for (int cc = 0; cc < L::P_CHUNKS; ++cc) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float e0 = ex2(fmaf(s[cc * 64 + 2 * i], sl2, neg));
                    const float e1 = ex2(fmaf(s[cc * 64 + 2 * i + 1], sl2, neg));
                    part[(2 * i) & 7] += e0;
                    part[(2 * i + 1) & 7] += e1;
                    pk[i] = pack_bf16x2(e0, e1);
                }
                tmem_st32(tS + cc * 32, pk);  // P chunk over S's columns [32cc, 32cc+32)
                constexpr int PER_HANDOFF = L::P_CHUNKS / L::HANDOFFS;
                if ((cc + 1) % PER_HANDOFF == 0) {
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(bar(L::BAR_PFULL + t * L::HANDOFFS + cc / PER_HANDOFF));
                }
            }
            const float sum = ((part[0] + part[1]) + (part[2] + part[3])) +
                              ((part[4] + part[5]) + (part[6] + part[7]));
            l = l * alpha + sum;
            m = m_new;
        }

        if (ok && n > 0) {
            ok = wait_phase(bar(L::BAR_OFULL + t), 0, p, abort_flag, kStatusWaitO);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) tc_fence_after();
        }
        if (ok) {
            const bool row_ok = q_row < p.Nq;
            const size_t row_idx = static_cast<size_t>(w.bh) * p.Nq + q_row;
            if (!p.split_mode) {
                // Deferred normalisation: one division per row, at the write.
                const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
                __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.o) + row_idx * D;
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    if (n > 0) {
                        tmem_ld32(tO + cc * 32, o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0u;
                    }
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv_l,
                                            __uint_as_float(o[2 * i + 1]) * inv_l);
                    if (row_ok) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                    }
                }
                if (row_ok)
                    p.lse[row_idx] = (l > 0.f) ? (m + lg2(l)) * 0.69314718055994530942f : -INFINITY;
            } else {
                const size_t part_idx =
                    (static_cast<size_t>(w.split) * p.BH + w.bh) * p.Nq + q_row;
                float* orow = p.ws_o + part_idx * D;
                // Partial states are stated relative to the split's true row max:
                // move l and O from the lazy reference m to m_true.
                const float rebase = (l > 0.f && m != m_true) ? ex2(m - m_true) : 1.f;
                const uint64_t rb2 = f2pack(rebase, rebase);
#pragma unroll 1
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    if (n > 0) {
                        tmem_ld32(tO + cc * 32, o);
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] = 0u;
                    }
                    if (rebase != 1.f) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            float x0, x1;
                            f2unpack(fmul2(f2pack(__uint_as_float(o[2 * i]),
                                                  __uint_as_float(o[2 * i + 1])), rb2), x0, x1);
                            o[2 * i] = __float_as_uint(x0);
                            o[2 * i + 1] = __float_as_uint(x1);
                        }
                    }
                    if (row_ok) {
                        uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
                    }
                }
                if (row_ok) {
                    p.ws_m[part_idx] = (l > 0.f) ? m_true * 0.69314718055994530942f : -INFINITY;
                    p.ws_l[part_idx] = l * rebase;
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::TMEM_COLS);
}

template <int D>
cudaError_t launch_fwd(const FwdParams& p, unsigned grid, cudaStream_t stream) {
    using L = FwdLayout<D>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        if constexpr (L::REG_SPLIT) {
            // The setmaxnreg split is sized for exactly LAUNCH_REGS per thread.
            cudaFuncAttributes a;
            e = cudaFuncGetAttributes(&a, fa_fwd_kernel<D>);
            if (e != cudaSuccess) return e;
            if (a.numRegs != L::LAUNCH_REGS) return cudaErrorInvalidKernelImage;
        }
        e = cudaFuncSetAttribute(fa_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(L::ALLOC_BYTES));
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(L::THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::ALLOC_BYTES;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, fa_fwd_kernel<D>, p);
}

}  // namespace fa
