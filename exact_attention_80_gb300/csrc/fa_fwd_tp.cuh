// fa_fwd_tp.cuh — fused exact attention forward, P kept in tensor memory.
//
// Used for head dim 256 (one query tile per CTA). One CTA owns Q_TILES query
// tiles of 128 rows of one (batch, head) and sweeps the keys those rows need
// (all of them, or one key range in split mode) in key tiles of BN = 96.
// Roles, by warp:
//   warp 0      TMA producer: Q tiles once, then K and V tiles into a ring of
//               STAGES shared-memory slots (full/empty mbarriers), in the order
//               the issuer consumes them: K_0, then per step j: K_{j+1}, V_j.
//   warp 1      tcgen05 issuer (a warp-uniform loop, one elected lane
//               issues), owns the TMEM allocation. Step j:
//               S_t(j+1) = Q_t K_{j+1}^T for every tile, then O_t += P_t(j) V_j
//               as each tile's P arrives. S is double-buffered per tile in
//               TMEM, so the next S is computed while the softmax works on
//               the current one and the tensor core never waits for a softmax
//               to finish before it has the next S to compute.
//   warps 2-3   idle.
//   warps 4..   one 128-thread softmax group per query tile t: thread = row
//               = TMEM lane. Online softmax on S_t(j); P_t(j) (bf16) written
//               into TMEM over the S buffer it came from; O_t rescaled in TMEM
//               when the exponent reference moves; deferred 1/l and LSE.
// The tensor/vector overlap is the one the FlashAttention-T page asks for
// (section "工程落地：参数、监控与未来演进", "Wavefront 调度").
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

#include "fa_fwd_common.cuh"

namespace fa {

template <int D>
struct TpCfg;
template <>
struct TpCfg<64> {
    static constexpr int Q_TILES = 2, BN = 64, STAGES = 16;
};
template <>
struct TpCfg<128> {
    static constexpr int Q_TILES = 2, BN = 64, STAGES = 8;
};
template <>
struct TpCfg<256> {
    // BN = 96: an N = 96 MMA runs at 86 % of the per-instruction rate (48 of 56
    // cycles) against 67 % for N = 64; two S buffers (192 columns) and O (256)
    // fit TMEM, and three 48 KB K/V slots fit shared memory next to Q.
    static constexpr int Q_TILES = 1, BN = 96, STAGES = 3;
};

// F8: e4m3 Q, K, V (one byte per element) and kind::f8f6f4 MMAs; otherwise
// bf16 and kind::f16.
template <int D, bool F8 = false>
struct LayoutTP {
    static constexpr int Q_TILES = TpCfg<D>::Q_TILES;
    static constexpr int BN = TpCfg<D>::BN;
    // 8-bit K/V slots are half the size: six of them fit beside the Q tile.
    static constexpr int STAGES = F8 ? 6 : TpCfg<D>::STAGES;
    static constexpr int EB = F8 ? 1 : 2;              // input bytes per element
    static constexpr int CHUNK_ELEMS = 128 / EB;       // elements per 128-byte swizzle row
    static constexpr int K_MMA = 32 / EB;              // K elements per MMA instruction
    // Warps: 0-3 control, then one softmax warpgroup per query tile, then one
    // correction warpgroup per query tile (rescales O when the exponent
    // reference moves, off the softmax's path).
    static constexpr int SOFTMAX_WARP0 = 4;
    static constexpr int CORR_WARP0 = SOFTMAX_WARP0 + 4 * Q_TILES;
    static constexpr int THREADS = (CORR_WARP0 + 4 * Q_TILES) * 32;
    static constexpr int CHUNKS = D / CHUNK_ELEMS;  // 128-byte column chunks of a row

    // shared memory (offsets from a 1024-aligned base)
    static constexpr uint32_t Q_TILE_BYTES = kBM * D * EB;
    static constexpr uint32_t SLOT_BYTES = BN * D * EB;
    // bf16 O is staged for its TMA store in the tile's Q memory when that holds
    // a bf16 tile; with 8-bit inputs in the K/V slots, which are all free once
    // the last PV has finished (every load was consumed).
    static_assert(!F8 || STAGES * BN * D * EB >= kBM * D * 2, "O staging fits the K/V slots");
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t SLOT_OFF = Q_OFF + Q_TILES * Q_TILE_BYTES;
    // Per-row rescale factors alpha of a step, for the correction group:
    // [tile][step parity][row] floats.
    static constexpr uint32_t ALPHA_OFF = SLOT_OFF + STAGES * SLOT_BYTES;
    static constexpr uint32_t BAR_OFF = ALPHA_OFF + Q_TILES * 2 * kBM * 4;
    static constexpr int BAR_QFULL = 0;
    static constexpr int BAR_KVFULL = 1;
    static constexpr int BAR_KVEMPTY = BAR_KVFULL + STAGES;
    static constexpr int BAR_SFULL = BAR_KVEMPTY + STAGES;   // [tile][S buffer]
    // P barriers are per S buffer too: the softmax may finish steps j and j+1
    // before the issuer consumes P(j), and one barrier per tile would then
    // have two completed phases that a parity wait cannot tell apart.
    static constexpr int BAR_PFULL = BAR_SFULL + 2 * Q_TILES;  // [tile][S buffer]
    static constexpr int BAR_PVDONE = BAR_PFULL + 2 * Q_TILES; // [tile]
    static constexpr int BAR_OFULL = BAR_PVDONE + Q_TILES;     // [tile]
    static constexpr int BAR_OSTAGED = BAR_OFULL + Q_TILES;    // [tile] bf16 O_t staged (one arrival per warp)
    // [tile][step parity]: the step's alpha published (one arrival per softmax
    // warp); O rescaled for the step, or found to need none (one arrival per
    // correction warp).
    static constexpr int BAR_ALPHA = BAR_OSTAGED + Q_TILES;
    static constexpr int BAR_OREADY = BAR_ALPHA + 2 * Q_TILES;
    static constexpr int BAR_DRAIN = BAR_OREADY + 2 * Q_TILES;
    static constexpr int NUM_BARS = BAR_DRAIN + 1;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;  // [0] tmem base, [1] abort
    static constexpr uint32_t BYTES = MISC_OFF + 16;
    static constexpr size_t ALLOC_BYTES = BYTES + 1024;  // slack for 1024 alignment

    // tensor memory columns (32-bit each; 512 allocated): two S buffers of BN
    // columns per tile in [0, 256) (P_t(j) is packed over the first BN/2
    // columns of the buffer S_t(j) came from), O_t in [256, 512).
    static constexpr uint32_t TMEM_COLS = 512;
    __host__ __device__ static constexpr uint32_t S_COL(int t, int b) { return (2 * t + b) * BN; }
    __host__ __device__ static constexpr uint32_t O_COL(int t) { return 256 + t * D; }

    static_assert(2 * Q_TILES * BN <= 256, "S buffers overflow their half of TMEM");
    static_assert(256 + Q_TILES * D <= 512, "O region overflows TMEM");
    static_assert(ALLOC_BYTES <= 232448, "shared memory over the 227 KB per-CTA limit");
    static_assert(ALLOC_BYTES > 232448 / 2, "two CTAs per SM would contend for TMEM");
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 128 && D % 64 == 0, "tile shape");

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

template <int D, bool F8>
__device__ __forceinline__ void tp_forward(const FwdParams& p) {
    using L = LayoutTP<D, F8>;
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
    // Launched with programmatic stream serialization: nothing here reads or
    // writes global memory before the grid before it in the stream has
    // completed (griddep_wait), and a grid launched the same way after this one
    // (the next forward, or fa_combine's merge of these partial states) may be
    // scheduled once every CTA here has started; it waits in turn.
    griddep_wait();
    if (threadIdx.x == 0) griddep_launch_dependents();

    Work<QT> w;
    compute_work<QT, BN>(p, blockIdx.x, w);

    if (threadIdx.x == 0) {
        mbar_init(bar(L::BAR_QFULL), 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar(L::BAR_KVFULL + s), 1);
            mbar_init(bar(L::BAR_KVEMPTY + s), 1);
        }
        for (int t = 0; t < QT; ++t) {
            mbar_init(bar(L::BAR_SFULL + 2 * t + 0), 1);
            mbar_init(bar(L::BAR_SFULL + 2 * t + 1), 1);
            mbar_init(bar(L::BAR_PFULL + 2 * t + 0), kBM);
            mbar_init(bar(L::BAR_PFULL + 2 * t + 1), kBM);
            mbar_init(bar(L::BAR_PVDONE + t), 1);
            mbar_init(bar(L::BAR_OFULL + t), 1);
            mbar_init(bar(L::BAR_OSTAGED + t), 4);
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar(L::BAR_ALPHA + 2 * t + b), 4);
                mbar_init(bar(L::BAR_OREADY + 2 * t + b), 4);
            }
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
        // The whole warp runs the loop (uniform values); one elected lane issues.
        if (w.nmax > 0) {
            const bool leader = elect_one();
            int nvalid = 0;
#pragma unroll
            for (int t = 0; t < QT; ++t) nvalid += (w.n[t] > 0) ? 1 : 0;
            // (The failure-detection test hook withholds the Q tiles so that the
            // issuer's bounded wait runs out; nothing else changes.)
            if (leader && !p.test_withhold_q) mbar_arrive_expect_tx(bar(L::BAR_QFULL), nvalid * L::Q_TILE_BYTES);
#pragma unroll
            for (int t = 0; t < QT; ++t) {
                if (leader && w.n[t] > 0 && !p.test_withhold_q) {
#pragma unroll
                    for (int c = 0; c < L::CHUNKS; ++c)
                        tma_load_3d(sbase + L::Q_OFF + t * L::Q_TILE_BYTES + c * (kBM * 128),
                                    &p.tm_q, bar(L::BAR_QFULL), L::CHUNK_ELEMS * c, w.qbase + w.q0 + t * kBM,
                                    w.zq);
                }
            }
            // Entry e of the sequence: K_0; then for step j: K_{j+1} (if any), V_j.
            const int total = 2 * w.nmax;
            RingPos<ST> pos;
            int issued = 0;
            bool ok = true;
            for (int e = 0; e < total; ++e) {
                bool is_v;
                int tile;
                if (e == 0) {
                    is_v = false;
                    tile = 0;
                } else if (e == total - 1) {
                    is_v = true;
                    tile = w.nmax - 1;
                } else {
                    is_v = ((e - 1) & 1) != 0;  // odd offsets within a step: V_j
                    tile = is_v ? (e - 1) >> 1 : ((e - 1) >> 1) + 1;
                }
                if (e >= ST) {
                    ok = wait_phase(bar(L::BAR_KVEMPTY + pos.slot), pos.phase ^ 1u, p, abort_flag,
                                    kStatusWaitKvEmpty);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
                if (leader) {
                    mbar_arrive_expect_tx(bar(L::BAR_KVFULL + pos.slot), L::SLOT_BYTES);
                    const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
                    const int row = w.kbase + (w.kv_tile0 + tile) * BN;
#pragma unroll
                    for (int c = 0; c < L::CHUNKS; ++c)
                        tma_load_3d(sbase + L::SLOT_OFF + pos.slot * L::SLOT_BYTES + c * (BN * 128), map,
                                    bar(L::BAR_KVFULL + pos.slot), L::CHUNK_ELEMS * c, row, w.zq);
                }
                issued = e + 1;
                pos.advance();
            }
            if (ok) {
                // Producer tail: wait until the issuer has released the last use
                // of every slot, so no tcgen05.commit arrival is still in flight
                // towards this CTA's shared memory when it exits.
                for (int e = max(0, total - ST); e < total && ok; ++e) {
                    ok = wait_phase(bar(L::BAR_KVEMPTY + e % ST), (e / ST) & 1, p, abort_flag,
                                    kStatusWaitKvEmpty);
                    ok = __all_sync(0xffffffffu, ok);
                }
            }
            if (!ok) {
                // Let every copy already issued land before the CTA goes away.
                wait_phase(bar(L::BAR_QFULL), 0, p, abort_flag, kStatusWaitDrain, false);
                for (int e = max(0, issued - ST); e < issued; ++e)
                    wait_phase(bar(L::BAR_KVFULL + e % ST), (e / ST) & 1, p, abort_flag,
                               kStatusWaitDrain, false);
            }
        }
      } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop, so descriptors and TMEM addresses stay in
        // warp-uniform registers; one elected lane issues each tcgen05 op.
        if (w.nmax > 0) {
            const bool leader = elect_one();
            auto wait_all = [&](uint32_t b, uint32_t parity, unsigned what) {
                return __all_sync(0xffffffffu, wait_phase(b, parity, p, abort_flag, what));
            };
            constexpr uint32_t IDESC_S =
                F8 ? make_idesc_e4m3(kBM, BN, false, false) : make_idesc_bf16(kBM, BN, false, false);
            constexpr uint32_t IDESC_O =
                F8 ? make_idesc_e4m3(kBM, D, false, true) : make_idesc_bf16(kBM, D, false, true);
            auto issue_s = [&](int t, int b, int slot) {
                const uint32_t qa = sbase + L::Q_OFF + t * L::Q_TILE_BYTES;
                const uint32_t kb = sbase + L::SLOT_OFF + slot * L::SLOT_BYTES;
#pragma unroll
                for (int kk = 0; kk < D / L::K_MMA; ++kk) {
                    const uint32_t in_row = (kk & 3) * 32;  // 16 bf16 = 32 bytes of a 128-byte row
                    const uint64_t a = make_sdesc_sw128(qa + (kk >> 2) * (kBM * 128) + in_row, 16, 1024);
                    const uint64_t bd = make_sdesc_sw128(kb + (kk >> 2) * (BN * 128) + in_row, 16, 1024);
                    if (leader) {
                        if constexpr (F8) umma_ss_f8(tmem + L::S_COL(t, b), a, bd, IDESC_S, kk > 0 ? 1u : 0u);
                        else umma_ss(tmem + L::S_COL(t, b), a, bd, IDESC_S, kk > 0 ? 1u : 0u);
                    }
                }
            };
            auto issue_pv = [&](int t, int b, int slot, bool accumulate) {
                const uint32_t vb = sbase + L::SLOT_OFF + slot * L::SLOT_BYTES;
#pragma unroll
                for (int kk = 0; kk < BN / L::K_MMA; ++kk) {
                    // V is MN-major: one MMA's K_MMA keys are K_MMA rows of 128
                    // bytes (2048 or 4096 bytes); 128-byte column chunks of d are
                    // BN*128 bytes apart. A = P, K_MMA keys = 8 TMEM columns.
                    const uint64_t bd = make_sdesc_sw128(vb + kk * (L::K_MMA * 128), BN * 128, 1024);
                    if (leader) {
                        if constexpr (F8)
                            umma_ts_f8(tmem + L::O_COL(t), tmem + L::S_COL(t, b) + kk * 8, bd, IDESC_O,
                                       (accumulate || kk > 0) ? 1u : 0u);
                        else
                            umma_ts(tmem + L::O_COL(t), tmem + L::S_COL(t, b) + kk * 8, bd, IDESC_O,
                                    (accumulate || kk > 0) ? 1u : 0u);
                    }
                }
            };

            RingPos<ST> pos;
            bool ok = wait_all(bar(L::BAR_QFULL), 0, kStatusWaitQ);
            if (ok) ok = wait_all(bar(L::BAR_KVFULL + pos.slot), pos.phase, kStatusWaitKvFull);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < QT; ++t) {
                    if (w.n[t] > 0) {
                        issue_s(t, 0, pos.slot);
                        if (leader) umma_commit(bar(L::BAR_SFULL + 2 * t + 0));
                    }
                }
                if (leader) umma_commit(bar(L::BAR_KVEMPTY + pos.slot));
                pos.advance();
            }
            for (int j = 0; j < w.nmax && ok; ++j) {
                // S_t(j+1) into the other S buffer. It overwrites P_t(j-1),
                // whose PV was issued in the previous step (MMAs run in order).
                if (j + 1 < w.nmax) {
                    ok = wait_all(bar(L::BAR_KVFULL + pos.slot), pos.phase, kStatusWaitKvFull);
                    if (!ok) break;
                    tc_fence_after();
                    const int b = (j + 1) & 1;
#pragma unroll
                    for (int t = 0; t < QT; ++t) {
                        if (j + 1 < w.n[t]) {
                            issue_s(t, b, pos.slot);
                            if (leader) umma_commit(bar(L::BAR_SFULL + 2 * t + b));
                        }
                    }
                    if (leader) umma_commit(bar(L::BAR_KVEMPTY + pos.slot));
                    pos.advance();
                }
                // O_t += P_t(j) V_j as each tile's P arrives.
                ok = wait_all(bar(L::BAR_KVFULL + pos.slot), pos.phase, kStatusWaitKvFull);
                if (!ok) break;
#pragma unroll
                for (int t = 0; t < QT; ++t) {
                    if (ok && j < w.n[t]) {
                        ok = wait_all(bar(L::BAR_PFULL + 2 * t + (j & 1)), (j >> 1) & 1, kStatusWaitP);
                        // ... and O_t rescaled for step j by the correction group.
                        if (ok) ok = wait_all(bar(L::BAR_OREADY + 2 * t + (j & 1)), (j >> 1) & 1, kStatusWaitO);
                        if (!ok) break;
                        tc_fence_after();
                        issue_pv(t, j & 1, pos.slot, j > 0);
                        if (leader) umma_commit(bar(L::BAR_PVDONE + t));
                        if (leader && j + 1 == w.n[t]) umma_commit(bar(L::BAR_OFULL + t));
                    }
                }
                if (!ok) break;
                if (leader) umma_commit(bar(L::BAR_KVEMPTY + pos.slot));
                pos.advance();
            }
            // Always wait for every MMA this thread issued before the CTA can
            // reach its teardown: on an abort no softmax waits for O_full, and
            // TMEM must not be released under an MMA in flight.
            if (leader) umma_commit(bar(L::BAR_DRAIN));
            wait_phase(bar(L::BAR_DRAIN), 0, p, abort_flag, kStatusWaitDrain, false);
        }
      }
    } else if (warp >= L::CORR_WARP0) {
        // ------------------------------------------------------------ correction
        // Warp CORR_WARP0 + 4 t + q rescales the O rows of lane quarter q of tile
        // t: per step j > 0 it reads the rows' alpha(j); if any differs from 1 it
        // waits for PV_t(j - 1) to finish and multiplies the rows' O by alpha(j)
        // in TMEM. Either way it then releases step j's PV (O_ready). Taking the
        // rescale out of the softmax's path lets the exponentials of step j run
        // while O is rescaled.
        const int t = (warp - L::CORR_WARP0) >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_field + L::O_COL(t);
        int n = w.n[0];
#pragma unroll
        for (int i = 1; i < QT; ++i)
            if (t == i) n = w.n[i];
        for (int j = 0; j < n; ++j) {
            const int b = j & 1;
            bool ok = wait_phase(bar(L::BAR_ALPHA + 2 * t + b), (j >> 1) & 1, p, abort_flag, kStatusWaitS);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            const float alpha = ld_shared_f32(sbase + L::ALPHA_OFF + ((t * 2 + b) * kBM + r) * 4);
            // O does not exist before the first PV (which overwrites it).
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                // PV_t(j-1) has finished writing O (its commit is PV_done phase j-1).
                ok = wait_phase(bar(L::BAR_PVDONE + t), (j - 1) & 1, p, abort_flag, kStatusWaitO);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc_fence_after();
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
                tmem_wait_st();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::BAR_OREADY + 2 * t + b));
        }
    } else {
        // ------------------------------------------------------------ softmax
        if constexpr (L::REG_SPLIT) setmaxnreg_inc<L::SOFTMAX_REGS>();
        const int t = (warp - L::SOFTMAX_WARP0) >> 2;
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        const int r = quarter * 32 + lane;
        const int q_row = w.q0 + t * kBM + r;
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tO = tmem + lane_field + L::O_COL(t);
        const float sl2 = p.scale_log2;
        int n = w.n[0];
#pragma unroll
        for (int i = 1; i < QT; ++i)
            if (t == i) n = w.n[i];

        float m = -INFINITY;       // exponent reference (base-2 units of scale*log2e*s)
        float m_true = -INFINITY;  // true running row max, same units
        float l = 0.f;             // running sum relative to m
        // The rounding error of each key tile's largest p when P is rounded to
        // bf16, relative to m like l. l + lc is the denominator of O (see RowOut).
        float lc = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int b = j & 1;
            const uint32_t tS = tmem + lane_field + L::S_COL(t, b);
            ok = wait_phase(bar(L::BAR_SFULL + 2 * t + b), (j >> 1) & 1, p, abort_flag,
                            kStatusWaitS);
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
            // this row + causal_off. Keys past the sequence end are zero fill
            // (or the next packed sequence's tokens), so they must become -inf.
            const int kv0 = (w.kv_tile0 + j) * BN;
            int valid = w.kv_end - kv0;
            if (p.causal) valid = min(valid, q_row + w.causal_off - kv0 + 1);
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
            const float s_max = max3f(a0, a1, fmaxf(a2, a3));
            const float m_tile = s_max * sl2;  // base-2 units
            m_true = fmaxf(m_true, m_tile);
            // The exponent reference m only moves when this tile's max exceeds it
            // by more than kRescaleSlack; otherwise every p = 2^(x - m) <= 2^slack
            // and the old reference is kept, so O and l need no rescale. The
            // result is the same: O/l and m + log2(l) do not depend on which
            // reference is used, only rounding does.
            // e4m3 P: a slack of kP8Slack and p = 2^(x - m + kP8Shift), so the
            // row's largest p lies in [2^6, 2^8], inside e4m3's range and mostly
            // in its normal range; l sums the same scaled p, and the LSE takes the
            // shift back out.
            const bool move = m_tile > m + (F8 ? kP8Slack : kRescaleSlack);
            const float m_new = move ? m_tile : m;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // all masked so far
            const float alpha = move ? ex2(m - m_use) : 1.f;
            const float neg = F8 ? kP8Shift - m_use : -m_use;

            // The accumulator's rescale for this step is the correction group's:
            // publish alpha (the step parity's slot is free: the correction group
            // read it two steps ago, before the PV this step's S waited behind).
            st_shared_f32(sbase + L::ALPHA_OFF + ((t * 2 + b) * kBM + r) * 4, alpha);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::BAR_ALPHA + 2 * t + b));

            // x = s*scale*log2e - m as packed fp32 pairs (one FFMA2 per two keys),
            // p = 2^x on the MUFU, row sums as four packed partial pairs.
            const uint64_t sl2x2 = f2pack(sl2, sl2);
            const uint64_t negx2 = f2pack(neg, neg);
            uint64_t part2[4] = {0ull, 0ull, 0ull, 0ull};
            if constexpr (F8) {
                // e4m3 P: four keys per TMEM column, key 4i + k in byte k of
                // column i; BN / 4 columns in stores of 8 (32 keys).
                static_assert(BN % 32 == 0, "e4m3 P in whole 8-column stores");
#pragma unroll
                for (int g = 0; g < BN / 32; ++g) {
                    uint32_t pk[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int c = g * 32 + 4 * i;
                        float x0, x1, x2, x3;
                        f2unpack(ffma2(f2pack(s[c], s[c + 1]), sl2x2, negx2), x0, x1);
                        f2unpack(ffma2(f2pack(s[c + 2], s[c + 3]), sl2x2, negx2), x2, x3);
                        const float e0 = ex2(x0);
                        const float e1 = ex2(x1);
                        const float e2 = ex2(x2);
                        const float e3 = ex2(x3);
                        part2[(2 * i) & 3] = fadd2(part2[(2 * i) & 3], f2pack(e0, e1));
                        part2[(2 * i + 1) & 3] = fadd2(part2[(2 * i + 1) & 3], f2pack(e2, e3));
                        pk[i] = pack_e4m3x4(e0, e1, e2, e3);
                    }
                    tmem_st8(tS + g * 8, pk);
                }
            } else {
#pragma unroll
            for (int cc = 0; cc < BN / 64; ++cc) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float x0, x1;
                    f2unpack(ffma2(f2pack(s[cc * 64 + 2 * i], s[cc * 64 + 2 * i + 1]), sl2x2, negx2),
                             x0, x1);
                    const float e0 = ex2(x0);
                    const float e1 = ex2(x1);
                    part2[i & 3] = fadd2(part2[i & 3], f2pack(e0, e1));
                    pk[i] = pack_bf16x2(e0, e1);
                }
                tmem_st32(tS + cc * 32, pk);  // P over the buffer's columns [32cc, 32cc+32)
            }
            if constexpr (BN % 64 == 32) {
                // The last 32 keys: 16 columns.
                constexpr int c0 = BN - 32;
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    f2unpack(ffma2(f2pack(s[c0 + 2 * i], s[c0 + 2 * i + 1]), sl2x2, negx2), x0, x1);
                    const float e0 = ex2(x0);
                    const float e1 = ex2(x1);
                    part2[i & 3] = fadd2(part2[i & 3], f2pack(e0, e1));
                    pk[i] = pack_bf16x2(e0, e1);
                }
                tmem_st16(tS + c0 / 2, pk);
            }
            }  // bf16 P
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(L::BAR_PFULL + 2 * t + b));
            float part[8];
            f2unpack(part2[0], part[0], part[1]);
            f2unpack(part2[1], part[2], part[3]);
            f2unpack(part2[2], part[4], part[5]);
            f2unpack(part2[3], part[6], part[7]);
            const float sum = ((part[0] + part[1]) + (part[2] + part[3])) +
                              ((part[4] + part[5]) + (part[6] + part[7]));
            l = l * alpha + sum;
            if constexpr (!F8) {
                // The tile's largest p exactly as computed above (same FMA and
                // ex2) and what rounding it to bf16 changed (exact: both lie
                // within a factor of two). 0 for a fully masked row.
                const float p_max = ex2(__fmaf_rn(s_max, sl2, neg));
                lc = lc * alpha + (round_bf16(p_max) - p_max);
            }
            m = m_new;
        }

        if (ok && n > 0) {
            ok = wait_phase(bar(L::BAR_OFULL + t), 0, p, abort_flag, kStatusWaitO);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) tc_fence_after();
        }
        // 8-bit inputs: the O scale is the V descale, and the reference carries
        // the P shift, which the LSE takes back out.
        const float o_scale = F8 ? p.o_scale : 1.f;
        const float m_out = F8 ? m - kP8Shift : m;
        const float l_o = F8 ? l : l + lc;
        if (ok && !p.split_mode && !p.varlen && n > 0) {
            // Plain mode: bf16 O_t staged in Q_t's shared memory (8-bit inputs: in
            // the K/V slots), written with TMA.
            const uint32_t staging = F8 ? sbase + L::SLOT_OFF : sbase + L::Q_OFF + t * L::Q_TILE_BYTES;
            store_tile_tma<D>(p, w.rm, w.zq, w.q0 + t * kBM, r, q_row, m_out, m_true, l, l_o, tO, staging,
                              bar(L::BAR_OSTAGED + t), abort_flag, o_scale);
        } else if (ok) {
            write_row<D>(p, w.rm, w.bh, w.split, q_row, n, m_out, m_true, l, l_o, tO, o_scale);
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::TMEM_COLS);
}

// bf16 Q, K, V.
template <int D>
__global__ void __launch_bounds__(LayoutTP<D>::THREADS, 1)
    fa_fwd_tp_kernel(const __grid_constant__ FwdParams p) {
    tp_forward<D, false>(p);
}

// e4m3 Q, K, V with per-tensor descales (FA-3 page, section 7.3: 8-bit inputs
// to both GEMMs, fp32 accumulation and fp32 softmax statistics).
template <int D>
__global__ void __launch_bounds__(LayoutTP<D, true>::THREADS, 1)
    fa_fwd_tp8_kernel(const __grid_constant__ FwdParams p) {
    tp_forward<D, true>(p);
}

}  // namespace fa
