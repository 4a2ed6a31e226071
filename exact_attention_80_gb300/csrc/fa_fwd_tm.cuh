// fa_fwd_tm.cuh — fused exact attention forward, two query tiles per CTA with
// P handed to the tensor core in TMEM.
//
// One CTA owns two query tiles of 128 rows of one (batch, head) and sweeps the
// keys those rows need in key tiles of BN = 128. Roles, by warp:
//   warp 0      TMA producer: Q tiles once, then K and V tiles into a ring of
//               STAGES shared-memory slots, in the order the issuer consumes
//               them: K_0, then per step j: V_j, K_{j+1}.
//   warp 1      tcgen05 issuer, owns the TMEM allocation. Step j, per tile t
//               as its P arrives: O_t += P_t(j) V_j (A = P_t from TMEM), then
//               at once S_t(j+1) = Q_t K_{j+1}^T into the same TMEM columns.
//   warps 2-3   idle.
//   warps 4..   one 128-thread softmax group per query tile: thread = row =
//               TMEM lane. Reads S_t(j), computes P_t(j) and writes it as
//               packed bf16 pairs over the first half of S_t's columns;
//               rescales its own row of O_t when the exponent reference moves;
//               deferred 1/l and LSE at the end.
// The two tiles alternate on the tensor core: while one tile's softmax runs,
// the MMAs of the other tile (its PV, then its next S) run, so the tensor and
// vector work of the two tiles overlap (the FlashAttention-T page, section
// "工程落地：参数、监控与未来演进", "Wavefront 调度"). Keeping P in TMEM
// spares the shared-memory store path and the async-proxy fence a P staged in
// shared memory needs; with O row-major each thread rescales its own row, so
// the softmax groups need no barrier of their own.
//
// tcgen05.mma operations of one thread run in issue order, so S_t(j+1),
// issued after O_t += P_t(j) V_j, overwrites P_t(j) only after that MMA has
// read it; the S_t(j+1) commit also covers the PV, so a softmax that sees
// S_t(j+1) may rescale O_t.
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
//
// Compile-time forms of the one body (tm_forward<D, F8, DUAL, PERSIST>):
//   F8       e4m3 Q, K, V: kind::f8f6f4 MMAs, P packed four e4m3 per TMEM
//            column, bf16 O staged in buffers of its own (fa_fwd_tm8_kernel).
//   DUAL     split-KV with one query tile: both tile slots on the same rows,
//            each with its own key split (tm_dual_control; fa_fwd_tmd_kernel,
//            fa_fwd_tm8d_kernel).
//   PERSIST  one CTA per SM walking several query units, the ring and the
//            barrier phases carried across them (tm_persist_control;
//            fa_fwd_tmp_kernel, fa_fwd_tmp8_kernel).
#pragma once

#include <type_traits>

#include "fa_fwd_common.cuh"

namespace fa {

// Per head dim: K/V ring depth and the setmaxnreg split (control warpgroup /
// softmax warpgroups), each the spill-free choice for that instantiation.
template <int D>
struct TmCfg;
template <>
struct TmCfg<64> {
    static constexpr int STAGES = 8, CTRL_REGS = 72, SOFTMAX_REGS = 216;
};
template <>
struct TmCfg<128> {
    static constexpr int STAGES = 5, CTRL_REGS = 88, SOFTMAX_REGS = 208;
};
// Persistent CTAs stage O in buffers of their own (the next unit's Q loads
// into the Q tiles meanwhile), which takes one K/V slot at d = 128.
template <int D>
struct TmPersistCfg {
    static constexpr int STAGES = D == 128 ? 4 : 8;
    // Spill-free at both head dims (104 / 200 spilled at d = 64 once the kernels
    // wait for the previous grid; 88 / 208 is also 2 % faster there).
    static constexpr int CTRL_REGS = 88, SOFTMAX_REGS = 208;
};
// 8-bit (e4m3) inputs: K/V slots are half the size, so the ring is deeper.
template <int D>
struct TmCfg8;
template <>
struct TmCfg8<64> {
    static constexpr int STAGES = 10, CTRL_REGS = 88, SOFTMAX_REGS = 208;
};
template <>
struct TmCfg8<128> {
    static constexpr int STAGES = 8, CTRL_REGS = 88, SOFTMAX_REGS = 208;
};

// F8: Q, K, V are e4m3 (one byte per element) and both MMAs are
// kind::f8f6f4; otherwise bf16 and kind::f16. PERSIST: persistent CTAs
// (plain mode), each walking several query units.
template <int D, bool F8 = false, bool PERSIST = false>
struct LayoutTM {
    using Cfg = std::conditional_t<F8, TmCfg8<D>, TmCfg<D>>;
    static constexpr int Q_TILES = 2;
    static constexpr int BN = 128;
    static constexpr bool PERSIST_BF16 = PERSIST && !F8;
    static constexpr int STAGES = PERSIST_BF16 ? TmPersistCfg<D>::STAGES : Cfg::STAGES;
    static constexpr int THREADS = (4 + 4 * Q_TILES) * 32;
    static constexpr int EB = F8 ? 1 : 2;              // input bytes per element
    // Swizzle row width: 128 bytes, or 64 when a whole row is 64 bytes (e4m3,
    // d = 64; 64-byte swizzle).
    static constexpr int ROW_BYTES = D * EB < 128 ? D * EB : 128;
    static constexpr int CHUNK_ELEMS = ROW_BYTES / EB; // elements per swizzle row
    static constexpr int CHUNKS = D / CHUNK_ELEMS;     // column chunks of a Q/K/V row
    static constexpr int K_MMA = 32 / EB;              // K elements per MMA instruction
    static constexpr int KSTEPS_ROW = ROW_BYTES / 32;  // MMA K steps per swizzle row

    // shared memory (offsets from a 1024-aligned base)
    static constexpr uint32_t Q_TILE_BYTES = kBM * D * EB;
    static constexpr uint32_t SLOT_BYTES = BN * D * EB;
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t SLOT_OFF = Q_OFF + Q_TILES * Q_TILE_BYTES;
    // bf16 O is staged for its TMA store in the tile's Q memory when that holds
    // a bf16 tile; 8-bit Q tiles are half that size, so F8 has buffers of its
    // own. Persistent bf16 CTAs stage each warp's 32 rows, 64 columns at a time,
    // in a 4 KB buffer per warp (the next unit's Q may be loading).
    static constexpr uint32_t OST_OFF = SLOT_OFF + STAGES * SLOT_BYTES;
    static constexpr uint32_t OST_WARP_BYTES = 32 * 128;
    static constexpr uint32_t OST_TILE_BYTES = F8 ? kBM * D * 2 : (PERSIST ? 4 * OST_WARP_BYTES : 0);
    static constexpr uint32_t BAR_OFF = OST_OFF + Q_TILES * OST_TILE_BYTES;
    static constexpr int BAR_QFULL = 0;                       // [tile] Q_t landed
    static constexpr int BAR_KVFULL = BAR_QFULL + Q_TILES;
    static constexpr int BAR_KVEMPTY = BAR_KVFULL + STAGES;
    static constexpr int BAR_SFULL = BAR_KVEMPTY + STAGES;  // [tile] S_t(j) (and PV_t(j-1)) done
    static constexpr int BAR_PFULL = BAR_SFULL + Q_TILES;   // [tile] P_t(j) in TMEM (one arrival per warp)
    static constexpr int BAR_OFULL = BAR_PFULL + Q_TILES;   // [tile] last PV_t finished
    // [tile] persistent CTAs: the unit's last S_t MMA finished, Q_t free (one
    // completion per unit in which the tile has keys)
    static constexpr int BAR_QEMPTY = BAR_OFULL + Q_TILES;
    static constexpr int BAR_DRAIN = BAR_QEMPTY + Q_TILES;
    static constexpr int NUM_BARS = BAR_DRAIN + 1;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;  // [0] tmem base, [1] abort
    static constexpr uint32_t BYTES = MISC_OFF + 16;
    static constexpr size_t ALLOC_BYTES = BYTES + 1024;  // slack for 1024 alignment

    // tensor memory columns (32-bit each; 512 allocated): S_t (P_t packed over
    // its first BN/2 columns), then O_t.
    static constexpr uint32_t TMEM_COLS = 512;
    __host__ __device__ static constexpr uint32_t S_COL(int t) { return t * BN; }
    __host__ __device__ static constexpr uint32_t O_COL(int t) { return 256 + t * D; }

    static_assert(Q_TILES * BN <= 256, "S region overflows its half of TMEM");
    static_assert(256 + Q_TILES * D <= 512, "O region overflows TMEM");
    static_assert(ALLOC_BYTES <= 232448, "shared memory over the 227 KB per-CTA limit");
    static_assert(ALLOC_BYTES > 232448 / 2, "two CTAs per SM would contend for TMEM");
    // A step holds V_j and K_{j+1} while it waits for V_{j+1} and K_{j+2}
    // (before it releases the first two), so the ring needs four slots.
    static_assert(D % 64 == 0 && STAGES >= 4, "tile shape and ring depth");
    static_assert(ROW_BYTES == 128 || ROW_BYTES == 64, "swizzle rows of 128 or 64 bytes");
    static_assert(!PERSIST || STAGES % 2 == 0, "persistent CTAs pair their K/V slots");

    // Register split: the sum is the launch allocation (THREADS x LAUNCH_REGS),
    // checked on the host.
    static constexpr bool REG_SPLIT = true;
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int CTRL_REGS = PERSIST_BF16 ? TmPersistCfg<D>::CTRL_REGS : Cfg::CTRL_REGS;
    static constexpr int SOFTMAX_REGS = PERSIST_BF16 ? TmPersistCfg<D>::SOFTMAX_REGS : Cfg::SOFTMAX_REGS;
    static_assert(128 * CTRL_REGS + 256 * SOFTMAX_REGS == THREADS * LAUNCH_REGS,
                  "register split must equal the launch allocation");
};

// Control warps of a dual-range CTA (split-KV with one query tile): the two
// query tiles hold the same rows, Q is loaded once (tile 0's buffer) and read by
// both tiles' S MMAs, and each tile streams the keys of its own split. K/V ring
// entries in consumption order: K^0_0, K^1_0, then per step j and tile t (if the
// tile has step j): V^t_j, then K^t_{j+1} if it has a next step. The issuer
// takes each tile's step as one unit: wait P_t, V^t_j, PV_t; wait K^t_{j+1},
// S_t(j+1); release both slots.
template <int D, bool F8>
__device__ __forceinline__ void tm_dual_control(const FwdParams& p, uint32_t sbase, uint32_t tmem,
                                                volatile uint32_t* abort_flag, int warp) {
    using L = LayoutTM<D, F8>;
    constexpr int BN = L::BN;
    constexpr int ST = L::STAGES;
    auto bar = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8u * i; };
    WorkDual w;
    compute_work_dual<BN>(p, blockIdx.x, w);
    if (w.nmax == 0) return;
    const bool leader = elect_one();
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (leader && !p.test_withhold_q) {
            mbar_arrive_expect_tx(bar(L::BAR_QFULL + 0), L::Q_TILE_BYTES);
#pragma unroll
            for (int c = 0; c < L::CHUNKS; ++c)
                tma_load_3d(sbase + L::Q_OFF + c * (kBM * L::ROW_BYTES), &p.tm_q, bar(L::BAR_QFULL + 0),
                            L::CHUNK_ELEMS * c, w.q0, w.zq);
        }
        RingPos<ST> pos;
        int issued = 0;
        bool ok = true;
        auto load_kv = [&](bool is_v, int t, int kv) -> bool {
            if (issued >= ST) {
                const bool okw = __all_sync(0xffffffffu, wait_phase(bar(L::BAR_KVEMPTY + pos.slot), pos.phase ^ 1u,
                                                                    p, abort_flag, kStatusWaitKvEmpty));
                if (!okw) return false;
            }
            if (leader) {
                mbar_arrive_expect_tx(bar(L::BAR_KVFULL + pos.slot), L::SLOT_BYTES);
                const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
                const int row = ((t ? w.kv_tile0[1] : w.kv_tile0[0]) + kv) * BN;
#pragma unroll
                for (int c = 0; c < L::CHUNKS; ++c)
                    tma_load_3d(sbase + L::SLOT_OFF + pos.slot * L::SLOT_BYTES + c * (BN * L::ROW_BYTES), map,
                                bar(L::BAR_KVFULL + pos.slot), L::CHUNK_ELEMS * c, row, w.zq);
            }
            ++issued;
            pos.advance();
            return true;
        };
        for (int t = 0; t < 2 && ok; ++t)
            if (w.n[t] > 0) ok = load_kv(false, t, 0);
        for (int j = 0; j < w.nmax && ok; ++j) {
            for (int t = 0; t < 2 && ok; ++t) {
                if (j < w.n[t]) {
                    ok = load_kv(true, t, j);
                    if (ok && j + 1 < w.n[t]) ok = load_kv(false, t, j + 1);
                }
            }
        }
        if (ok) {
            // Wait until the issuer has released every slot's last use, so no
            // tcgen05.commit arrival is in flight when the CTA exits.
            for (int e = max(0, issued - ST); e < issued && ok; ++e)
                ok = __all_sync(0xffffffffu, wait_phase(bar(L::BAR_KVEMPTY + e % ST), (e / ST) & 1, p,
                                                        abort_flag, kStatusWaitKvEmpty));
        } else {
            if (!p.test_withhold_q)
                wait_phase(bar(L::BAR_QFULL + 0), 0, p, abort_flag, kStatusWaitDrain, false);
            for (int e = max(0, issued - ST); e < issued; ++e)
                wait_phase(bar(L::BAR_KVFULL + e % ST), (e / ST) & 1, p, abort_flag, kStatusWaitDrain,
                           false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        auto wait_all = [&](uint32_t b, uint32_t parity, unsigned what) {
            return __all_sync(0xffffffffu, wait_phase(b, parity, p, abort_flag, what));
        };
        constexpr uint32_t IDESC_S =
            F8 ? make_idesc_e4m3(kBM, BN, false, false) : make_idesc_bf16(kBM, BN, false, false);
        constexpr uint32_t IDESC_O =
            F8 ? make_idesc_e4m3(kBM, D, false, true) : make_idesc_bf16(kBM, D, false, true);
        const uint64_t kmaj0 = make_sdesc_rows<L::ROW_BYTES>(sbase, 16, 8 * L::ROW_BYTES);
        const uint64_t vmn0 = make_sdesc_rows<L::ROW_BYTES>(sbase, BN * L::ROW_BYTES, 8 * L::ROW_BYTES);
        const uint32_t kmaj_lo = static_cast<uint32_t>(kmaj0);
        const uint32_t kmaj_hi = static_cast<uint32_t>(kmaj0 >> 32);
        const uint32_t vmn_lo = static_cast<uint32_t>(vmn0);
        const uint32_t vmn_hi = static_cast<uint32_t>(vmn0 >> 32);
        auto desc = [](uint32_t lo, uint32_t hi, uint32_t off) -> uint64_t {
            return (static_cast<uint64_t>(hi) << 32) | (lo + (off >> 4));
        };
        // S_t = Q K^T from the one Q tile; O_t += P_t V as in the two-tile kernel.
        auto issue_s = [&](int t, int slot) {
            const uint32_t kb = L::SLOT_OFF + slot * L::SLOT_BYTES;
#pragma unroll
            for (int kk = 0; kk < D / L::K_MMA; ++kk) {
                const uint32_t in_row = (kk % L::KSTEPS_ROW) * 32;
                const int ch = kk / L::KSTEPS_ROW;
                const uint64_t a = desc(kmaj_lo, kmaj_hi, L::Q_OFF + ch * (kBM * L::ROW_BYTES) + in_row);
                const uint64_t b = desc(kmaj_lo, kmaj_hi, kb + ch * (BN * L::ROW_BYTES) + in_row);
                if (leader) {
                    if constexpr (F8) umma_ss_f8(tmem + L::S_COL(t), a, b, IDESC_S, kk > 0 ? 1u : 0u);
                    else umma_ss(tmem + L::S_COL(t), a, b, IDESC_S, kk > 0 ? 1u : 0u);
                }
            }
        };
        auto issue_pv = [&](int t, int slot, bool accumulate) {
            const uint32_t vb = L::SLOT_OFF + slot * L::SLOT_BYTES;
#pragma unroll
            for (int kk = 0; kk < BN / L::K_MMA; ++kk) {
                const uint64_t b = desc(vmn_lo, vmn_hi, vb + kk * (L::K_MMA * L::ROW_BYTES));
                if (leader) {
                    if constexpr (F8)
                        umma_ts_f8(tmem + L::O_COL(t), tmem + L::S_COL(t) + kk * 8, b, IDESC_O,
                                   (accumulate || kk > 0) ? 1u : 0u);
                    else
                        umma_ts(tmem + L::O_COL(t), tmem + L::S_COL(t) + kk * 8, b, IDESC_O,
                                (accumulate || kk > 0) ? 1u : 0u);
                }
            }
        };
        RingPos<ST> pos;
        auto next_slot = [&](int& slot) -> bool {
            slot = pos.slot;
            if (!wait_all(bar(L::BAR_KVFULL + pos.slot), pos.phase, kStatusWaitKvFull)) return false;
            pos.advance();
            return true;
        };
        bool ok = wait_all(bar(L::BAR_QFULL + 0), 0, kStatusWaitQ);
        for (int t = 0; t < 2 && ok; ++t) {
            if (w.n[t] == 0) continue;
            int ks;
            ok = next_slot(ks);
            if (!ok) break;
            tc_fence_after();
            issue_s(t, ks);
            if (leader) umma_commit(bar(L::BAR_SFULL + t));
            if (leader) umma_commit(bar(L::BAR_KVEMPTY + ks));
        }
        for (int j = 0; j < w.nmax && ok; ++j) {
            for (int t = 0; t < 2 && ok; ++t) {
                if (j >= w.n[t]) continue;
                ok = wait_all(bar(L::BAR_PFULL + t), j & 1, kStatusWaitP);
                int vs = 0;
                if (ok) ok = next_slot(vs);
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, vs, j > 0);
                if (j + 1 < w.n[t]) {
                    int ks;
                    ok = next_slot(ks);
                    if (!ok) break;
                    issue_s(t, ks);
                    if (leader) umma_commit(bar(L::BAR_SFULL + t));
                    if (leader) umma_commit(bar(L::BAR_KVEMPTY + ks));
                } else {
                    if (leader) umma_commit(bar(L::BAR_OFULL + t));
                }
                if (leader) umma_commit(bar(L::BAR_KVEMPTY + vs));
            }
        }
        // Every MMA this thread issued must finish before TMEM can be freed.
        if (leader) umma_commit(bar(L::BAR_DRAIN));
        wait_phase(bar(L::BAR_DRAIN), 0, p, abort_flag, kStatusWaitDrain, false);
    }
}

// Unit of a persistent CTA's round k, or -1 when the round has none for it.
// A round walks gridDim.x consecutive units (one wave's worth, sharing heads in
// L2, the order compute_work gives them), forwards on even rounds and backwards
// on odd ones: under a causal mask a round's heaviest units come first, so a
// CTA that took one of them takes one of the lightest next.
__device__ __forceinline__ long long persist_unit(const FwdParams& p, int k) {
    const long long g = gridDim.x;
    const long long c = (k & 1) ? g - 1 - blockIdx.x : blockIdx.x;
    const long long lin = static_cast<long long>(k) * g + c;
    return lin < p.total_units ? lin : -1;
}

// Control warps of a persistent CTA (bf16, plain mode, dense): the producer and
// the issuer of tm_forward's one-unit CTA, run over the CTA's units with the
// K/V ring and every barrier's phase carried from unit to unit. Phases count
// per tile: SFULL_t and PFULL_t complete once per key step of the tile,
// QFULL_t, QEMPTY_t and OFULL_t once per unit in which the tile has keys.
//   The K/V ring holds pairs of slots: the entry of step j holds V_j and the K
//   tile the step's S MMAs read, K_{j+1}, or, at a unit's last step, K_0 of the
//   CTA's next unit (the CTA's first entry holds that unit's K_0 alone). The
//   issuer then waits for one entry and releases one per step, and the next
//   unit's first S MMAs read a K tile that is already resident.
//   Q_t of the next unit loads as soon as the unit's last S_t MMA has
//   completed: the issuer commits QEMPTY_t right after that MMA. Each waiter
//   of a barrier sees every one of its phases in turn (an mbarrier wait tells
//   phases apart by parity alone, so a waiter must never be two phases away
//   from the one it waits for): the producer has waited for the previous
//   QEMPTY_t phase before it issued the load that the next one releases. O_t of
//   the next unit is first written by its PV_t(0), which waits for P_t(0); the
//   softmax threads hand that P over only after their epilogue has read O_t out
//   of TMEM.
template <int D, bool F8>
__device__ __forceinline__ void tm_persist_control(const FwdParams& p, uint32_t sbase, uint32_t tmem,
                                                   volatile uint32_t* abort_flag, int warp) {
    using L = LayoutTM<D, F8, true>;
    constexpr uint32_t RB = L::ROW_BYTES;  // swizzle row bytes
    constexpr int QT = L::Q_TILES;
    constexpr int BN = L::BN;
    constexpr int NP = L::STAGES / 2;  // ring entries: slot pairs (V half, K half)
    static_assert(L::STAGES % 2 == 0 && NP >= 2, "the ring holds pairs of K/V slots");
    auto bar = [&](int i) -> uint32_t { return sbase + L::BAR_OFF + 8u * i; };
    auto v_half = [](int e) -> uint32_t { return L::SLOT_OFF + (2 * e) * L::SLOT_BYTES; };
    auto k_half = [](int e) -> uint32_t { return L::SLOT_OFF + (2 * e + 1) * L::SLOT_BYTES; };
    const int rounds = static_cast<int>((p.total_units + gridDim.x - 1) / gridDim.x);
    // The CTA's next unit with keys at round k or later: its work in w, its
    // round in k; false when there is none.
    auto next_unit = [&](int& k, Work<QT>& w) -> bool {
        for (; k < rounds; ++k) {
            const long long lin = persist_unit(p, k);
            if (lin < 0) continue;
            compute_work<QT, BN>(p, lin, w);
            if (w.nmax > 0) return true;
        }
        return false;
    };
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        const bool leader = elect_one();
        RingPos<NP> pos;
        int issued = 0;           // ring entries issued, all units
        int q_loads[QT] = {};     // Q_t loads issued
        bool ok = true;
        auto load_q = [&](const Work<QT>& u, int t) -> bool {
            if (u.n[t] == 0) return true;
            if (q_loads[t] > 0 &&
                !__all_sync(0xffffffffu, wait_phase(bar(L::BAR_QEMPTY + t), (q_loads[t] - 1) & 1, p,
                                                    abort_flag, kStatusWaitQ)))
                return false;
            if (leader && !p.test_withhold_q) {
                mbar_arrive_expect_tx(bar(L::BAR_QFULL + t), L::Q_TILE_BYTES);
#pragma unroll
                for (int c = 0; c < L::CHUNKS; ++c)
                    tma_load_3d(sbase + L::Q_OFF + t * L::Q_TILE_BYTES + c * (kBM * RB), &p.tm_q,
                                bar(L::BAR_QFULL + t), L::CHUNK_ELEMS * c, tile_row0(p, u.q0, t), u.zq);
            }
            ++q_loads[t];
            return true;
        };
        // One ring entry: V rows from vrow and K rows from krow of heads vz, kz
        // (a row < 0: that half stays empty).
        auto load_pair = [&](int vrow, int vz, int krow, int kz) -> bool {
            if (issued >= NP &&
                !__all_sync(0xffffffffu, wait_phase(bar(L::BAR_KVEMPTY + pos.slot), pos.phase ^ 1u, p,
                                                    abort_flag, kStatusWaitKvEmpty)))
                return false;
            if (leader) {
                const uint32_t full = bar(L::BAR_KVFULL + pos.slot);
                mbar_arrive_expect_tx(full, (vrow >= 0 ? L::SLOT_BYTES : 0u) + (krow >= 0 ? L::SLOT_BYTES : 0u));
                if (vrow >= 0) {
#pragma unroll
                    for (int c = 0; c < L::CHUNKS; ++c)
                        tma_load_3d(sbase + v_half(pos.slot) + c * (BN * RB), &p.tm_v, full, L::CHUNK_ELEMS * c,
                                    vrow, vz);
                }
                if (krow >= 0) {
#pragma unroll
                    for (int c = 0; c < L::CHUNKS; ++c)
                        tma_load_3d(sbase + k_half(pos.slot) + c * (BN * RB), &p.tm_k, full, L::CHUNK_ELEMS * c,
                                    krow, kz);
                }
            }
            ++issued;
            pos.advance();
            return true;
        };
        int k = 0;
        Work<QT> w;
        bool have = next_unit(k, w);
        if (have) {
            // Q_0, K_0 (the first entry), then Q_1, as in the one-unit CTA.
            ok = load_q(w, 0);
            if (ok) ok = load_pair(-1, 0, w.kv_tile0 * BN, w.zq);
            if (ok) ok = load_q(w, 1);
        }
        while (have && ok) {
            int kn = k + 1;
            Work<QT> wn;
            const bool have_next = next_unit(kn, wn);
            for (int j = 0; j < w.nmax && ok; ++j) {
                int krow = -1, kz = 0;
                if (j + 1 < w.nmax) {
                    krow = (w.kv_tile0 + j + 1) * BN;
                    kz = w.zq;
                } else if (have_next) {
                    krow = wn.kv_tile0 * BN;
                    kz = wn.zq;
                }
                ok = load_pair((w.kv_tile0 + j) * BN, w.zq, krow, kz);
            }
            if (ok && have_next) {
                ok = load_q(wn, 0);
                if (ok) ok = load_q(wn, 1);
            }
            w = wn;
            k = kn;
            have = have_next;
        }
        if (ok) {
            // Every entry's last use released: no commit arrival still in flight.
            for (int e = max(0, issued - NP); e < issued && ok; ++e)
                ok = __all_sync(0xffffffffu, wait_phase(bar(L::BAR_KVEMPTY + e % NP), (e / NP) & 1, p, abort_flag,
                                                        kStatusWaitKvEmpty));
        } else {
            // Let every copy already issued land before the CTA goes away.
#pragma unroll
            for (int t = 0; t < QT; ++t)
                if (q_loads[t] > 0 && !p.test_withhold_q)
                    wait_phase(bar(L::BAR_QFULL + t), (q_loads[t] - 1) & 1, p, abort_flag, kStatusWaitDrain, false);
            for (int e = max(0, issued - NP); e < issued; ++e)
                wait_phase(bar(L::BAR_KVFULL + e % NP), (e / NP) & 1, p, abort_flag, kStatusWaitDrain, false);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        const bool leader = elect_one();
        auto wait_all = [&](uint32_t b, uint32_t parity, unsigned what) {
            return __all_sync(0xffffffffu, wait_phase(b, parity, p, abort_flag, what));
        };
        constexpr uint32_t IDESC_S =
            F8 ? make_idesc_e4m3(kBM, BN, false, false) : make_idesc_bf16(kBM, BN, false, false);
        constexpr uint32_t IDESC_O =
            F8 ? make_idesc_e4m3(kBM, D, false, true) : make_idesc_bf16(kBM, D, false, true);
        const uint64_t kmaj0 = make_sdesc_rows<L::ROW_BYTES>(sbase, 16, 8 * RB);
        const uint64_t vmn0 = make_sdesc_rows<L::ROW_BYTES>(sbase, BN * RB, 8 * RB);
        const uint32_t kmaj_lo = static_cast<uint32_t>(kmaj0);
        const uint32_t kmaj_hi = static_cast<uint32_t>(kmaj0 >> 32);
        const uint32_t vmn_lo = static_cast<uint32_t>(vmn0);
        const uint32_t vmn_hi = static_cast<uint32_t>(vmn0 >> 32);
        auto desc = [](uint32_t lo, uint32_t hi, uint32_t off) -> uint64_t {
            return (static_cast<uint64_t>(hi) << 32) | (lo + (off >> 4));
        };
        // S_t = Q_t K^T from the K tile at shared offset kb; O_t += P_t V from vb.
        // One MMA takes 32 bytes of K (16 bf16 or 32 e4m3) of a swizzle row; P is
        // packed two bf16 or four e4m3 per TMEM column, so one MMA's keys are 8
        // columns.
        auto issue_s = [&](int t, uint32_t kb) {
            const uint32_t qa = L::Q_OFF + t * L::Q_TILE_BYTES;
#pragma unroll
            for (int kk = 0; kk < D / L::K_MMA; ++kk) {
                const uint32_t in_row = (kk % L::KSTEPS_ROW) * 32;
                const int ch = kk / L::KSTEPS_ROW;
                const uint64_t a = desc(kmaj_lo, kmaj_hi, qa + ch * (kBM * RB) + in_row);
                const uint64_t b = desc(kmaj_lo, kmaj_hi, kb + ch * (BN * RB) + in_row);
                if (leader) {
                    if constexpr (F8) umma_ss_f8(tmem + L::S_COL(t), a, b, IDESC_S, kk > 0 ? 1u : 0u);
                    else umma_ss(tmem + L::S_COL(t), a, b, IDESC_S, kk > 0 ? 1u : 0u);
                }
            }
        };
        auto issue_pv = [&](int t, uint32_t vb, bool accumulate) {
#pragma unroll
            for (int kk = 0; kk < BN / L::K_MMA; ++kk) {
                const uint64_t b = desc(vmn_lo, vmn_hi, vb + kk * (L::K_MMA * RB));
                if (leader) {
                    if constexpr (F8)
                        umma_ts_f8(tmem + L::O_COL(t), tmem + L::S_COL(t) + kk * 8, b, IDESC_O,
                                   (accumulate || kk > 0) ? 1u : 0u);
                    else
                        umma_ts(tmem + L::O_COL(t), tmem + L::S_COL(t) + kk * 8, b, IDESC_O,
                                (accumulate || kk > 0) ? 1u : 0u);
                }
            }
        };
        // Phase parities carried across units: bit t of sbits = parity of the
        // tile's earlier key steps (PFULL_t), of qbits = parity of its earlier
        // Q_t loads (QFULL_t).
        uint32_t sbits = 0, qbits = 0;
        RingPos<NP> pos;  // the entry in use
        bool ok = true;
        bool first = true;
        constexpr bool kKvWaitMid1 = (D >= 128);
        int k = 0;
        Work<QT> w;
        while (ok && next_unit(k, w)) {
            // pos: the entry whose K half holds this unit's K_0 (the previous
            // unit's last entry, already waited for; or the CTA's first).
            if (first) {
                ok = wait_all(bar(L::BAR_KVFULL + pos.slot), pos.phase, kStatusWaitKvFull);
                first = false;
            }
            if (ok) {
#pragma unroll
                for (int t = 0; t < QT; ++t) {
                    if (ok && w.n[t] > 0) {
                        ok = wait_all(bar(L::BAR_QFULL + t), (qbits >> t) & 1u, kStatusWaitQ);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(t, k_half(pos.slot));
                        if (leader) umma_commit(bar(L::BAR_SFULL + t));
                        if (w.n[t] == 1 && leader) umma_commit(bar(L::BAR_QEMPTY + t));
                    }
                }
            }
            if (ok) {
                // That entry's V half was read by the previous unit's last PVs,
                // issued before these S MMAs.
                if (leader) umma_commit(bar(L::BAR_KVEMPTY + pos.slot));
                pos.advance();
                ok = wait_all(bar(L::BAR_KVFULL + pos.slot), pos.phase, kStatusWaitKvFull);
            }
            for (int j = 0; j < w.nmax && ok; ++j) {
                const uint32_t vb = v_half(pos.slot), kb = k_half(pos.slot);
                const bool k_next = (j + 1 < w.nmax);
                RingPos<NP> nxt = pos;
                nxt.advance();
                if (j < w.n[0]) {
                    ok = wait_all(bar(L::BAR_PFULL + 0), (sbits ^ static_cast<uint32_t>(j)) & 1u, kStatusWaitP);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(0, vb, j > 0);
                    if (j + 1 < w.n[0]) {
                        issue_s(0, kb);
                        if (leader) umma_commit(bar(L::BAR_SFULL + 0));
                        if (j + 2 == w.n[0] && leader) umma_commit(bar(L::BAR_QEMPTY + 0));
                    } else {
                        if (leader) umma_commit(bar(L::BAR_OFULL + 0));
                    }
                }
                if (!kKvWaitMid1 && k_next) {
                    ok = wait_all(bar(L::BAR_KVFULL + nxt.slot), nxt.phase, kStatusWaitKvFull);
                    if (!ok) break;
                }
                const bool act1 = j < w.n[1];
                if (act1) {
                    ok = wait_all(bar(L::BAR_PFULL + 1), ((sbits >> 1) ^ static_cast<uint32_t>(j)) & 1u, kStatusWaitP);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(1, vb, j > 0);
                }
                if (kKvWaitMid1 && k_next) {
                    ok = wait_all(bar(L::BAR_KVFULL + nxt.slot), nxt.phase, kStatusWaitKvFull);
                    if (!ok) break;
                }
                if (act1) {
                    if (j + 1 < w.n[1]) {
                        issue_s(1, kb);
                        if (leader) umma_commit(bar(L::BAR_SFULL + 1));
                        if (j + 2 == w.n[1] && leader) umma_commit(bar(L::BAR_QEMPTY + 1));
                    } else {
                        if (leader) umma_commit(bar(L::BAR_OFULL + 1));
                    }
                }
                // A unit's last entry stays: its K half is the next unit's K_0.
                if (k_next) {
                    if (leader) umma_commit(bar(L::BAR_KVEMPTY + pos.slot));
                    pos = nxt;
                }
            }
#pragma unroll
            for (int t = 0; t < QT; ++t) {
                sbits ^= static_cast<uint32_t>(w.n[t] & 1) << t;
                qbits ^= static_cast<uint32_t>(w.n[t] > 0 ? 1 : 0) << t;
            }
            ++k;
        }
        // The last unit's last entry.
        if (!first && leader) umma_commit(bar(L::BAR_KVEMPTY + pos.slot));
        // Every MMA this thread issued must finish before TMEM can be freed.
        if (leader) umma_commit(bar(L::BAR_DRAIN));
        wait_phase(bar(L::BAR_DRAIN), 0, p, abort_flag, kStatusWaitDrain, false);
    }
}

// DUAL: split-KV with one query tile, both tiles on the same rows (see
// tm_dual_control); the softmax groups then take their tile's own split.
// M64: one 64-row query tile per CTA (fa_fwd_rows with 64 rows): M = 64 MMAs,
// whose accumulator rows 16 q + i sit in TMEM lanes 32 q + i (i < 16) of lane
// quarter q; lanes 16-31 of each quarter hold no row.
template <int D, bool F8, bool DUAL = false, bool PERSIST = false, bool M64 = false>
__device__ __forceinline__ void tm_forward(const FwdParams& p) {
    using L = LayoutTM<D, F8, PERSIST>;
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


    if (threadIdx.x == 0) {
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar(L::BAR_KVFULL + s), 1);
            mbar_init(bar(L::BAR_KVEMPTY + s), 1);
        }
        for (int t = 0; t < QT; ++t) {
            mbar_init(bar(L::BAR_QFULL + t), 1);
            mbar_init(bar(L::BAR_SFULL + t), 1);
            mbar_init(bar(L::BAR_PFULL + t), 4);  // one arrival per warp of the group
            mbar_init(bar(L::BAR_OFULL + t), 1);
            mbar_init(bar(L::BAR_QEMPTY + t), 1);
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
      // The work record is derived inside each role, after its register limit
      // is set, so that no role carries fields it does not use.
      if constexpr (PERSIST) {
        tm_persist_control<D, F8>(p, sbase, tmem, abort_flag, warp);
      } else if constexpr (DUAL) {
        tm_dual_control<D, F8>(p, sbase, tmem, abort_flag, warp);
      } else {
      Work<QT> w;
      compute_work<QT, BN>(p, blockIdx.x, w);
      if (warp == 0) {
        // ------------------------------------------------------------ producer
        // The whole warp runs the loop (uniform values); one elected lane issues.
        if (w.nmax > 0) {
            const bool leader = elect_one();
            // Q_t of each tile with work, on its own barrier. (The failure-
            // detection test hook withholds the Q tiles so that the issuer's
            // bounded wait runs out; nothing else changes.)
            auto load_q = [&](int t) {
                if (leader && w.n[t] > 0 && !p.test_withhold_q) {
                    mbar_arrive_expect_tx(bar(L::BAR_QFULL + t), L::Q_TILE_BYTES);
#pragma unroll
                    for (int c = 0; c < L::CHUNKS; ++c)
                        tma_load_3d(sbase + L::Q_OFF + t * L::Q_TILE_BYTES + c * (kBM * L::ROW_BYTES),
                                    &p.tm_q, bar(L::BAR_QFULL + t), L::CHUNK_ELEMS * c, w.qbase + tile_row0(p, w.q0, t),
                                    w.zq);
                }
            };
            // Q_0, K_0, then Q_1: the first S can start after two tiles' bytes.
            load_q(0);
            // Entry e of the sequence: K_0; then for step j: V_j, K_{j+1} (if any).
            const int total = 2 * w.nmax;
            RingPos<ST> pos;
            int issued = 0;
            bool ok = true;
            for (int e = 0; e < total; ++e) {
                const bool is_v = (e & 1) != 0;  // K_j at e = 2j, V_j at e = 2j + 1
                const int kv = e >> 1;
                if (e >= ST) {
                    ok = wait_phase(bar(L::BAR_KVEMPTY + pos.slot), pos.phase ^ 1u, p, abort_flag,
                                    kStatusWaitKvEmpty);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
                if (leader) {
                    mbar_arrive_expect_tx(bar(L::BAR_KVFULL + pos.slot), L::SLOT_BYTES);
                    const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
                    const int row = w.kbase + (w.kv_tile0 + kv) * BN;
#pragma unroll
                    for (int c = 0; c < L::CHUNKS; ++c)
                        tma_load_3d(sbase + L::SLOT_OFF + pos.slot * L::SLOT_BYTES + c * (BN * L::ROW_BYTES), map,
                                    bar(L::BAR_KVFULL + pos.slot), L::CHUNK_ELEMS * c, row, w.zq);
                }
                issued = e + 1;
                pos.advance();
                if (e == 0) load_q(1);
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
#pragma unroll
                for (int t = 0; t < QT; ++t)
                    if (w.n[t] > 0 && !p.test_withhold_q && issued > 0)
                        wait_phase(bar(L::BAR_QFULL + t), 0, p, abort_flag, kStatusWaitDrain, false);
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
            constexpr int MMA_M = M64 ? 64 : kBM;
            constexpr uint32_t IDESC_S =
                F8 ? make_idesc_e4m3(MMA_M, BN, false, false) : make_idesc_bf16(MMA_M, BN, false, false);
            constexpr uint32_t IDESC_O =
                F8 ? make_idesc_e4m3(MMA_M, D, false, true) : make_idesc_bf16(MMA_M, D, false, true);
            // Descriptors are built once; an operand at byte offset `off` from a
            // base adds off >> 4 to the low word (the 14-bit start field never
            // carries: shared addresses stay below 2^18).
            // Q, K: K-major; V: MN-major (8-row groups 8 swizzle rows apart).
            const uint64_t kmaj0 = make_sdesc_rows<L::ROW_BYTES>(sbase, 16, 8 * L::ROW_BYTES);
            const uint64_t vmn0 = make_sdesc_rows<L::ROW_BYTES>(sbase, BN * L::ROW_BYTES, 8 * L::ROW_BYTES);
            const uint32_t kmaj_lo = static_cast<uint32_t>(kmaj0);
            const uint32_t kmaj_hi = static_cast<uint32_t>(kmaj0 >> 32);
            const uint32_t vmn_lo = static_cast<uint32_t>(vmn0);
            const uint32_t vmn_hi = static_cast<uint32_t>(vmn0 >> 32);
            auto desc = [](uint32_t lo, uint32_t hi, uint32_t off) -> uint64_t {
                return (static_cast<uint64_t>(hi) << 32) | (lo + (off >> 4));
            };
            auto issue_s = [&](int t, int slot) {
                const uint32_t qa = L::Q_OFF + t * L::Q_TILE_BYTES;
                const uint32_t kb = L::SLOT_OFF + slot * L::SLOT_BYTES;
                // One MMA takes 32 bytes of K (16 bf16 or 32 e4m3) of a swizzle row.
                if constexpr (F8) {
#pragma unroll
                    for (int kk = 0; kk < D / L::K_MMA; ++kk) {
                        const uint32_t in_row = (kk % L::KSTEPS_ROW) * 32;
                        const int ch = kk / L::KSTEPS_ROW;
                        if (leader)
                            umma_ss_f8(tmem + L::S_COL(t),
                                       desc(kmaj_lo, kmaj_hi, qa + ch * (kBM * L::ROW_BYTES) + in_row),
                                       desc(kmaj_lo, kmaj_hi, kb + ch * (BN * L::ROW_BYTES) + in_row), IDESC_S,
                                       kk > 0 ? 1u : 0u);
                    }
                } else {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t in_row = (kk & 3) * 32;  // 16 bf16 = 32 bytes of a 128-byte row
                        if (leader)
                            umma_ss(tmem + L::S_COL(t), desc(kmaj_lo, kmaj_hi, qa + (kk >> 2) * (kBM * 128) + in_row),
                                    desc(kmaj_lo, kmaj_hi, kb + (kk >> 2) * (BN * 128) + in_row), IDESC_S,
                                    kk > 0 ? 1u : 0u);
                    }
                }
            };
            // O_t += P_t V: A = P_t packed two bf16 (four e4m3) per TMEM column,
            // so one MMA's K keys (16 bf16 or 32 e4m3) are 8 columns; B = V
            // MN-major (K key rows of one swizzle row each, K/8 swizzle atoms;
            // column chunks of d BN swizzle rows apart).
            auto issue_pv = [&](int t, int slot, bool accumulate) {
                const uint32_t vb = L::SLOT_OFF + slot * L::SLOT_BYTES;
                if constexpr (F8) {
#pragma unroll
                    for (int kk = 0; kk < BN / L::K_MMA; ++kk)
                        if (leader)
                            umma_ts_f8(tmem + L::O_COL(t), tmem + L::S_COL(t) + kk * 8,
                                       desc(vmn_lo, vmn_hi, vb + kk * (L::K_MMA * L::ROW_BYTES)), IDESC_O,
                                       (accumulate || kk > 0) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk)
                        if (leader)
                            umma_ts(tmem + L::O_COL(t), tmem + L::S_COL(t) + kk * 8,
                                    desc(vmn_lo, vmn_hi, vb + kk * 2048), IDESC_O,
                                    (accumulate || kk > 0) ? 1u : 0u);
                }
            };

            // K/V entries in consumption order: K_0, then per step j: V_j, K_{j+1}.
            RingPos<ST> pos;
            int slot_v = 0, slot_k = 0;  // slots of V_j and K_{j+1} for the current step
            auto wait_kv = [&](int j) -> bool {  // V_j, then K_{j+1} if any step needs it
                slot_v = pos.slot;
                if (!wait_all(bar(L::BAR_KVFULL + pos.slot), pos.phase, kStatusWaitKvFull)) return false;
                pos.advance();
                if (j + 1 < w.nmax) {
                    slot_k = pos.slot;
                    if (!wait_all(bar(L::BAR_KVFULL + pos.slot), pos.phase, kStatusWaitKvFull)) return false;
                    pos.advance();
                }
                return true;
            };
            bool ok = wait_all(bar(L::BAR_KVFULL + pos.slot), pos.phase, kStatusWaitKvFull);
            if (ok) {
#pragma unroll
                for (int t = 0; t < QT; ++t) {
                    if (ok && w.n[t] > 0) {
                        ok = wait_all(bar(L::BAR_QFULL + t), 0, kStatusWaitQ);
                        if (!ok) break;
                        tc_fence_after();
                        issue_s(t, pos.slot);
                        if (leader) umma_commit(bar(L::BAR_SFULL + t));
                    }
                }
            }
            if (ok) {
                if (leader) umma_commit(bar(L::BAR_KVEMPTY + pos.slot));
                pos.advance();
                ok = wait_kv(0);
            }
            // Per step: tile 0's PV and next S; tile 1's PV; tile 1's next S. The
            // next step's K/V waits go where the MMA queue holds the most work:
            // between tile 1's PV and S for d = 128 (PV of N = 128), after tile
            // 0's batch for d = 64 (a shorter PV). Each group of waits and
            // commits then sits behind queued MMAs, so the tensor core does not
            // idle while the issuing thread synchronises.
            constexpr bool kKvWaitMid1 = (D >= 128);
            for (int j = 0; j < w.nmax && ok; ++j) {
                const int sv = slot_v, sk = slot_k;
                const bool k_next = (j + 1 < w.nmax);
                if (j < w.n[0]) {
                    ok = wait_all(bar(L::BAR_PFULL + 0), j & 1, kStatusWaitP);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(0, sv, j > 0);
                    if (j + 1 < w.n[0]) {
                        issue_s(0, sk);
                        if (leader) umma_commit(bar(L::BAR_SFULL + 0));
                    } else {
                        if (leader) umma_commit(bar(L::BAR_OFULL + 0));
                    }
                }
                if (!kKvWaitMid1 && k_next) {
                    ok = wait_kv(j + 1);
                    if (!ok) break;
                }
                const bool act1 = j < w.n[1];
                if (act1) {
                    ok = wait_all(bar(L::BAR_PFULL + 1), j & 1, kStatusWaitP);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(1, sv, j > 0);
                }
                if (kKvWaitMid1 && k_next) {
                    ok = wait_kv(j + 1);
                    if (!ok) break;
                }
                if (act1) {
                    if (j + 1 < w.n[1]) {
                        issue_s(1, sk);
                        if (leader) umma_commit(bar(L::BAR_SFULL + 1));
                    } else {
                        if (leader) umma_commit(bar(L::BAR_OFULL + 1));
                    }
                }
                // V_j and K_{j+1} are released together after the step's last MMA,
                // so no commit sits between tile 1's PV and the next K/V waits.
                if (leader) umma_commit(bar(L::BAR_KVEMPTY + sv));
                if (k_next && leader) umma_commit(bar(L::BAR_KVEMPTY + sk));
            }
            // Always wait for every MMA this thread issued before the CTA can
            // reach its teardown: on an abort no softmax waits for O_full, and
            // TMEM must not be released under an MMA in flight.
            if (leader) umma_commit(bar(L::BAR_DRAIN));
            wait_phase(bar(L::BAR_DRAIN), 0, p, abort_flag, kStatusWaitDrain, false);
        }
      }
      }  // !DUAL
    } else {
        // ------------------------------------------------------------ softmax
        if constexpr (L::REG_SPLIT) setmaxnreg_inc<L::SOFTMAX_REGS>();
        const int t = (warp - 4) >> 2;
        const int quarter = warp & 3;  // TMEM lane quarter this warp may access
        // The query row of this thread's TMEM lane; with 64-row tiles only
        // lanes 0-15 of each quarter hold one (the others run along for the
        // warp-collective TMEM accesses and write nothing).
        const int r = M64 ? quarter * 16 + (lane & 15) : quarter * 32 + lane;
        // Persistent CTAs walk their units (persist_unit); the phases of S_t
        // and O_t carry over: s_phase counts the tile's earlier key steps,
        // o_phase its earlier units with keys. A one-unit CTA runs the body once.
        const int rounds = PERSIST ? static_cast<int>((p.total_units + gridDim.x - 1) / gridDim.x) : 1;
        int s_phase = 0, o_phase = 0;
        bool ok = true;
        for (int k = 0; k < rounds && ok; ++k) {
        long long lin = blockIdx.x;
        if constexpr (PERSIST) {
            lin = persist_unit(p, k);
            if (lin < 0) continue;
        }
        std::conditional_t<DUAL, WorkDual, Work<QT>> w;
        if constexpr (DUAL) compute_work_dual<BN>(p, lin, w);
        else compute_work<QT, BN>(p, lin, w);
        const int q_row = (M64 && lane >= 16) ? (1 << 30) : (DUAL ? w.q0 : tile_row0(p, w.q0, t)) + r;
        // This tile's key split: the CTA's, or its own in a dual-range CTA.
        int kv_tile0_t, kv_end_t, split_t;
        if constexpr (DUAL) {
            kv_tile0_t = t ? w.kv_tile0[1] : w.kv_tile0[0];
            kv_end_t = t ? w.kv_end[1] : w.kv_end[0];
            split_t = t ? w.split[1] : w.split[0];
        } else {
            kv_tile0_t = w.kv_tile0;
            kv_end_t = w.kv_end;
            split_t = w.split;
        }
        const uint32_t lane_field = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t tS = tmem + lane_field + L::S_COL(t);
        const uint32_t tO = tmem + lane_field + L::O_COL(t);
        const float sl2 = p.scale_log2;
        // e4m3 P: with the reference at most kP8Slack below the true row max,
        // p = 2^(x - m + kP8Shift) <= 2^8 stays inside e4m3's range (448) and
        // the row's largest p is at least 2^6, so most of P is in e4m3's normal
        // range. l sums the same scaled p, so O / l is unchanged; the LSE takes
        // the shift back out.
        constexpr float kSlack = F8 ? kP8Slack : kRescaleSlack;
        int n = w.n[0];
#pragma unroll
        for (int i = 1; i < QT; ++i)
            if (t == i) n = w.n[i];

        float m = -INFINITY;       // exponent reference (base-2 units of scale*log2e*s)
        float m_true = -INFINITY;  // true running row max, same units
        float l = 0.f;             // running sum relative to m
        // bf16 P: the rounding error of each key tile's largest p, relative to m
        // like l. l + lc is the denominator of O (see RowOut).
        float lc = 0.f;
        for (int j = 0; j < n; ++j) {
            // tcgen05.ld/st are warp-collective: the whole warp leaves together.
            ok = wait_phase_warp(bar(L::BAR_SFULL + t), (s_phase + j) & 1, p, abort_flag, kStatusWaitS);
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
            const int kv0 = (kv_tile0_t + j) * BN;
            int valid = kv_end_t - kv0;
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
            const bool move = m_tile > m + kSlack;
            const float m_new = move ? m_tile : m;
            const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // all masked so far
            const float alpha = move ? ex2(m - m_use) : 1.f;
            const float neg = F8 ? kP8Shift - m_use : -m_use;

            // x = s*scale*log2e - m as packed fp32 pairs (one FFMA2 per two keys),
            // p = 2^x on the MUFU, row sums as four packed partial pairs; P goes
            // over S_t's first BN/2 columns as packed bf16 pairs, 32 columns
            // (64 keys) at a time.
            const uint64_t sl2x2 = f2pack(sl2, sl2);
            const uint64_t negx2 = f2pack(neg, neg);
            uint64_t part2[4] = {0ull, 0ull, 0ull, 0ull};
            if constexpr (F8) {
                // e4m3 P: four keys per column, 32 columns (128 keys) at a time.
#pragma unroll
                for (int h = 0; h < BN / 128; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int c = h * 128 + 4 * i;
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
                    tmem_st32(tS + h * 32, pk);
                }
            } else {
#pragma unroll
                for (int h = 0; h < BN / 64; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int c = h * 64 + 2 * i;
                        float x0, x1;
                        f2unpack(ffma2(f2pack(s[c], s[c + 1]), sl2x2, negx2), x0, x1);
                        const float e0 = ex2(x0);
                        const float e1 = ex2(x1);
                        part2[i & 3] = fadd2(part2[i & 3], f2pack(e0, e1));
                        pk[i] = pack_bf16x2(e0, e1);
                    }
                    tmem_st32(tS + h * 32, pk);
                }
            }

            // O_t(j-1) is complete (the S_t(j) commit covers PV_t(j-1)); rescale
            // the rows whose reference moved. tcgen05.ld/st are warp-collective,
            // so the warp takes this branch together (alpha = 1 rows multiply by 1).
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
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::BAR_PFULL + t));

            float part[8];
            f2unpack(part2[0], part[0], part[1]);
            f2unpack(part2[1], part[2], part[3]);
            f2unpack(part2[2], part[4], part[5]);
            f2unpack(part2[3], part[6], part[7]);
            const float sum = ((part[0] + part[1]) + (part[2] + part[3])) +
                              ((part[4] + part[5]) + (part[6] + part[7]));
            l = l * alpha + sum;
            if constexpr (!F8) {
                // The tile's largest p exactly as the loop above computed it (the
                // same FMA and ex2), and what rounding it to bf16 changed (exact:
                // both lie within a factor of two). 0 for a fully masked row.
                const float p_max = ex2(__fmaf_rn(s_max, sl2, neg));
                lc = lc * alpha + (round_bf16(p_max) - p_max);
            }
            m = m_new;
        }

        if (ok && n > 0) {
            ok = wait_phase_warp(bar(L::BAR_OFULL + t), o_phase & 1, p, abort_flag, kStatusWaitO);
            if (ok) tc_fence_after();
        }
        // A tile slot the CTA does not own (one tile per CTA, fa_fwd_rows) writes
        // nothing: its rows belong to another CTA.
        if (!DUAL && !PERSIST && t >= p.tiles_per_cta) ok = false;
        if constexpr (PERSIST && !F8) {
            // Plain mode, dense: bf16 O staged per warp in its own buffer.
            if (ok && n > 0)
                store_rows_tma_buf<D>(p, w.rm, w.zq, q_row - r, r, q_row, m, m_true, l, l + lc, tO,
                                      sbase + L::OST_OFF + t * L::OST_TILE_BYTES + quarter * L::OST_WARP_BYTES);
            else if (ok)
                write_row<D>(p, w.rm, w.bh, 0, q_row, n, m, m_true, l, l + lc, tO);
        } else if constexpr (F8) {
            // Dense layouts only (the host rejects varlen). Plain mode: bf16
            // o_scale * O_t / l staged in the tile's own buffer and written with
            // TMA. Split mode: the partial state, O scaled by o_scale, per row.
            if (ok && !p.split_mode && n > 0)
                store_rows_tma<D>(p, w.rm, w.zq, q_row - r, r, q_row, m - kP8Shift, m_true, l, l, tO,
                                  sbase + L::OST_OFF + t * L::OST_TILE_BYTES, p.o_scale);
            else if (ok && (!DUAL || split_t < p.num_splits))
                write_row<D>(p, w.rm, w.bh, split_t, q_row, n, m - kP8Shift, m_true, l, l, tO, p.o_scale);
        } else {
            if (ok && !M64 && !p.split_mode && !p.varlen && n > 0) {
                // Plain mode: bf16 O_t staged in Q_t's shared memory, written with TMA
                // stores per warp (128-row tiles; 64-row tiles write per row).
                store_rows_tma<D>(p, w.rm, w.zq, q_row - r, r, q_row, m, m_true, l, l + lc, tO,
                                  sbase + L::Q_OFF + t * L::Q_TILE_BYTES);
            } else if (ok && (!DUAL || split_t < p.num_splits)) {
                write_row<D>(p, w.rm, w.bh, split_t, q_row, n, m, m_true, l, l + lc, tO);
            }
        }
        s_phase += n;
        o_phase += n > 0 ? 1 : 0;
        }  // units
        // Persistent CTAs leave their last TMA stores' shared-memory reads for
        // here (store_rows_tma_buf waits for a warp's earlier ones before it
        // overwrites its buffer).
        if constexpr (PERSIST) {
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
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
__global__ void __launch_bounds__(LayoutTM<D>::THREADS, 1)
    fa_fwd_tm_kernel(const __grid_constant__ FwdParams p) {
    tm_forward<D, false>(p);
}

// bf16, one 64-row query tile per CTA (fa_fwd_rows with 64 rows).
template <int D>
__global__ void __launch_bounds__(LayoutTM<D>::THREADS, 1)
    fa_fwd_tm64_kernel(const __grid_constant__ FwdParams p) {
    tm_forward<D, false, false, false, true>(p);
}

// e4m3 Q, K, V with per-tensor descales (FA-3 page, section 7.3: 8-bit inputs
// to both GEMMs, fp32 accumulation and fp32 softmax statistics).
template <int D>
__global__ void __launch_bounds__(LayoutTM<D, true>::THREADS, 1)
    fa_fwd_tm8_kernel(const __grid_constant__ FwdParams p) {
    tm_forward<D, true>(p);
}

// Persistent CTAs (plain mode, dense): grid min(units, SMs), each CTA walking
// its units with persist_unit; bf16 and e4m3 inputs.
template <int D>
__global__ void __launch_bounds__(LayoutTM<D, false, true>::THREADS, 1)
    fa_fwd_tmp_kernel(const __grid_constant__ FwdParams p) {
    tm_forward<D, false, false, true>(p);
}
template <int D>
__global__ void __launch_bounds__(LayoutTM<D, true, true>::THREADS, 1)
    fa_fwd_tmp8_kernel(const __grid_constant__ FwdParams p) {
    tm_forward<D, true, false, true>(p);
}

// Dual-range split-KV CTAs (one query tile), bf16 and e4m3 inputs.
template <int D>
__global__ void __launch_bounds__(LayoutTM<D>::THREADS, 1)
    fa_fwd_tmd_kernel(const __grid_constant__ FwdParams p) {
    tm_forward<D, false, true>(p);
}
template <int D>
__global__ void __launch_bounds__(LayoutTM<D, true>::THREADS, 1)
    fa_fwd_tm8d_kernel(const __grid_constant__ FwdParams p) {
    tm_forward<D, true, true>(p);
}

}  // namespace fa
