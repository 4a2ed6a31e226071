// fa_fwd_sp.cuh — fused exact attention forward, P staged in shared memory.
//
// Used for head dims 64 and 128. One CTA owns two query tiles of 128 rows of
// one (batch, head) and sweeps the keys those rows need in key tiles of
// BN = 128. Roles, by warp:
//   warp 0      TMA producer: Q tiles once, then K and V tiles into a ring of
//               STAGES shared-memory slots, in the order the issuer consumes
//               them: K_0, then per step j: K_{j+1}, V_j.
//   warp 1      tcgen05 issuer (one thread), owns the TMEM allocation. Step j:
//               S_t(j+1) = Q_t K_{j+1}^T for each tile as soon as that tile's
//               softmax has read S_t(j) out of TMEM, then the PV product of
//               step j once the tiles' P has arrived (operands in shared memory).
//   warps 2-3   idle.
//   warps 4..   one 128-thread softmax group per query tile: thread = row =
//               TMEM lane. Reads S_t(j) into registers and frees it at once,
//               so the next S is computed during the softmax; writes P_t(j)
//               (bf16) into a swizzled shared-memory tile for the PV MMA;
//               rescales O_t in TMEM when the exponent reference moves;
//               deferred 1/l and LSE at the end.
// Wide MMAs keep the tensor core at its full per-instruction rate, and the
// softmax of one step overlaps the S and PV MMAs of its neighbours (the
// tensor/vector overlap the FlashAttention-T page asks for, section
// "工程落地：参数、监控与未来演进", "Wavefront 调度").
//
// PV for d = 128 is computed transposed, O^T += V^T P^T: the head dim (128)
// is the MMA's M (= TMEM lanes) and the query rows of both tiles are its
// N = 256 columns, so one batch of 8 MMAs covers the whole step (instead of
// two batches of N = 128): fewer, wider instructions from the single issuing
// thread. The softmax group of tile t then holds O_t^T in TMEM columns
// [256 + 128t, 384 + 128t), one head-dim index per lane; a rescale multiplies
// column q by row q's factor, which the row's thread publishes in shared
// memory. For d = 64 (M = 64 would use a different TMEM lane layout) PV stays
// row-major, O_t += P_t V_j, one batch of N = 64 per tile.
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
struct SpCfg;
template <>
struct SpCfg<64> {
    static constexpr int Q_TILES = 2, BN = 128, STAGES = 8;
};
template <>
struct SpCfg<128> {
    static constexpr int Q_TILES = 2, BN = 128, STAGES = 3;
};

template <int D>
struct LayoutSP {
    static constexpr int Q_TILES = SpCfg<D>::Q_TILES;
    static constexpr int BN = SpCfg<D>::BN;
    static constexpr int STAGES = SpCfg<D>::STAGES;
    static constexpr int THREADS = (4 + 4 * Q_TILES) * 32;
    static constexpr int CHUNKS = D / 64;  // 64-element (128-byte) column chunks

    // PV transposed (O^T in TMEM, one head-dim index per lane); see above.
    static constexpr bool O_T = (D == 128);

    // shared memory (offsets from a 1024-aligned base)
    static constexpr uint32_t Q_TILE_BYTES = kBM * D * 2;
    static constexpr uint32_t P_TILE_BYTES = kBM * BN * 2;
    static constexpr uint32_t SLOT_BYTES = BN * D * 2;
    static constexpr uint32_t Q_OFF = 0;
    // P of all tiles as one K-major operand of Q_TILES*128 rows: 64-key chunk
    // c of row (128 t + r) is the 128-byte line P_OFF + c*P_CHUNK + (128 t + r)*128.
    static constexpr uint32_t P_OFF = Q_OFF + Q_TILES * Q_TILE_BYTES;
    static constexpr uint32_t P_CHUNK = Q_TILES * kBM * 128;
    static constexpr uint32_t P_TILE = kBM * 128;  // offset of tile t's rows in a chunk
    static constexpr uint32_t SLOT_OFF = P_OFF + Q_TILES * P_TILE_BYTES;
    static constexpr uint32_t BAR_OFF = SLOT_OFF + STAGES * SLOT_BYTES;
    static constexpr int BAR_QFULL = 0;
    static constexpr int BAR_KVFULL = 1;
    static constexpr int BAR_KVEMPTY = BAR_KVFULL + STAGES;
    // S_full and PV_done are shared by the tiles (one commit after the step's
    // S MMAs / PV MMAs of all tiles): each costs the issuing thread as much as
    // an MMA. A tile only waits for phases below its own step count, and no
    // phase can run two ahead of an active tile, so shared parity waits hold.
    static constexpr int BAR_SFULL = BAR_KVEMPTY + STAGES;   // S(j) of every tile in TMEM
    static constexpr int BAR_SFREE = BAR_SFULL + 1;          // [tile] S_t read by softmax
    static constexpr int BAR_PFULL = BAR_SFREE + Q_TILES;    // [tile] P_t in smem
    static constexpr int BAR_PVDONE = BAR_PFULL + Q_TILES;   // PV(j) of every tile finished
    static constexpr int BAR_OFULL = BAR_PVDONE + 1;         // [tile] last PV_t finished
    static constexpr int BAR_DRAIN = BAR_OFULL + Q_TILES;
    static constexpr int NUM_BARS = BAR_DRAIN + 1;
    static constexpr uint32_t MISC_OFF = BAR_OFF + NUM_BARS * 8;  // [0] tmem base, [1] abort
    // Per-row factors a tile's softmax group exchanges (O^T rescale and
    // epilogue): [tile][row] fp32.
    static constexpr uint32_t ROWF_OFF = MISC_OFF + 16;
    static constexpr uint32_t BYTES = ROWF_OFF + Q_TILES * kBM * 4;
    static constexpr size_t ALLOC_BYTES = BYTES + 1024;  // slack for 1024 alignment

    // tensor memory columns (32-bit each; 512 allocated)
    static constexpr uint32_t TMEM_COLS = 512;
    __host__ __device__ static constexpr uint32_t S_COL(int t) { return t * BN; }
    __host__ __device__ static constexpr uint32_t O_COL(int t) { return 256 + t * D; }

    static_assert(Q_TILES * BN <= 256, "S region overflows its half of TMEM");
    static_assert(256 + Q_TILES * D <= 512, "O region overflows TMEM");
    static_assert(ALLOC_BYTES <= 232448, "shared memory over the 227 KB per-CTA limit");
    static_assert(ALLOC_BYTES > 232448 / 2, "two CTAs per SM would contend for TMEM");
    static_assert(BN == 128 && D % 64 == 0 && STAGES >= 3, "tile shape");
    static_assert(!O_T || (D == kBM && Q_TILES == 2), "transposed PV: M = d = 128, N = 256");

    // Register split: see LayoutTP.
    static constexpr bool REG_SPLIT = (Q_TILES == 2);
    static constexpr int LAUNCH_REGS = 168;
    static constexpr int CTRL_REGS = 72;
    static constexpr int SOFTMAX_REGS = 216;
    static_assert(!REG_SPLIT || 128 * CTRL_REGS + 256 * SOFTMAX_REGS == THREADS * LAUNCH_REGS,
                  "register split must equal the launch allocation");
};

// Writes a query tile's result from O_t^T (TMEM lane = head-dim index,
// column = row of the tile; not read when n == 0). Run by all 128 threads of
// the tile's softmax group: thread r publishes row r's factor (1/l in plain
// mode, the move from the lazy reference to the split's true max in split
// mode) and row r's scalars, and after the group's barrier writes head-dim
// index r of every row; a warp writes 32 consecutive head-dim entries of a row.
template <int D, int QT>
__device__ __forceinline__ void write_tile_t(const FwdParams& p, const Work<QT>& w, int t, int r, int n,
                                             float m, float m_true, float l, uint32_t tO, float* rowf,
                                             int nbar, bool ok) {
    const int lane = r & 31;
    const int row0 = w.q0 + t * kBM;     // first query row of the tile
    const int rows_valid = p.Nq - row0;  // rows q < rows_valid exist
    float fac;
    if (!p.split_mode) fac = (l > 0.f) ? 1.f / l : 0.f;
    else fac = (l > 0.f && m != m_true) ? ex2(m - m_true) : 1.f;
    rowf[r] = fac;
    if (named_bar_or(nbar, kBM, !ok)) return;  // some warp of the group failed

    constexpr float kLn2 = 0.69314718055994530942f;
    const size_t part0 = (static_cast<size_t>(w.split) * p.BH + w.bh) * p.Nq + row0;
    if (r < rows_valid) {
        if (!p.split_mode) {
            p.lse[static_cast<size_t>(w.bh) * p.Nq + row0 + r] = (l > 0.f) ? (m + lg2(l)) * kLn2 : -INFINITY;
        } else {
            p.ws_m[part0 + r] = (l > 0.f) ? m_true * kLn2 : -INFINITY;
            p.ws_l[part0 + r] = l * fac;
        }
    }
    const bool odd = (lane & 1) != 0;
#pragma unroll 1
    for (int cc = 0; cc < kBM / 32; ++cc) {
        uint32_t o[32];
        if (n > 0) tmem_ld32(tO + cc * 32, o);
        const float4* f4 = reinterpret_cast<const float4*>(rowf + cc * 32);
        float f[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float4 v4 = f4[i];
            f[4 * i] = v4.x;
            f[4 * i + 1] = v4.y;
            f[4 * i + 2] = v4.z;
            f[4 * i + 3] = v4.w;
        }
        if (n > 0) {
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
        }
        float v[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(o[i]) * f[i];
        if (!p.split_mode) {
            // Lane pairs swap values so that each lane stores two adjacent
            // head-dim entries (one 32-bit word) of one row: the even lane of
            // row 2i, the odd lane of row 2i+1.
            __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(p.o) +
                                (static_cast<size_t>(w.bh) * p.Nq + row0) * D + (r & ~1);
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float recv = __shfl_xor_sync(0xffffffffu, odd ? v[2 * i] : v[2 * i + 1], 1);
                const uint32_t word = odd ? pack_bf16x2(recv, v[2 * i + 1]) : pack_bf16x2(v[2 * i], recv);
                const int q = cc * 32 + 2 * i + (odd ? 1 : 0);
                if (q < rows_valid) *reinterpret_cast<uint32_t*>(ob + static_cast<size_t>(q) * D) = word;
            }
        } else {
            float* wb = p.ws_o + part0 * D + r;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int q = cc * 32 + i;
                if (q < rows_valid) wb[static_cast<size_t>(q) * D] = v[i];
            }
        }
    }
}

template <int D>
__global__ void __launch_bounds__(LayoutSP<D>::THREADS, 1)
    fa_fwd_sp_kernel(const __grid_constant__ FwdParams p) {
    using L = LayoutSP<D>;
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
    compute_work<QT, BN>(p, w);

    if (threadIdx.x == 0) {
        mbar_init(bar(L::BAR_QFULL), 1);
        for (int s = 0; s < ST; ++s) {
            mbar_init(bar(L::BAR_KVFULL + s), 1);
            mbar_init(bar(L::BAR_KVEMPTY + s), 1);
        }
        mbar_init(bar(L::BAR_SFULL), 1);
        mbar_init(bar(L::BAR_PVDONE), 1);
        for (int t = 0; t < QT; ++t) {
            mbar_init(bar(L::BAR_SFREE + t), kBM);
            mbar_init(bar(L::BAR_PFULL + t), kBM);
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
            // (The failure-detection test hook withholds the Q tiles so that the
            // issuer's bounded wait runs out; nothing else changes.)
            if (!p.test_withhold_q) mbar_arrive_expect_tx(bar(L::BAR_QFULL), nvalid * L::Q_TILE_BYTES);
#pragma unroll
            for (int t = 0; t < QT; ++t) {
                if (w.n[t] > 0 && !p.test_withhold_q) {
#pragma unroll
                    for (int c = 0; c < L::CHUNKS; ++c)
                        tma_load_3d(sbase + L::Q_OFF + t * L::Q_TILE_BYTES + c * (kBM * 128),
                                    &p.tm_q, bar(L::BAR_QFULL), 64 * c, w.q0 + t * kBM, w.bh);
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
                    if (!ok) break;
                }
                mbar_arrive_expect_tx(bar(L::BAR_KVFULL + pos.slot), L::SLOT_BYTES);
                const CUtensorMap* map = is_v ? &p.tm_v : &p.tm_k;
                const int row = (w.kv_tile0 + tile) * BN;
#pragma unroll
                for (int c = 0; c < L::CHUNKS; ++c)
                    tma_load_3d(sbase + L::SLOT_OFF + pos.slot * L::SLOT_BYTES + c * (BN * 128), map,
                                bar(L::BAR_KVFULL + pos.slot), 64 * c, row, w.bh);
                issued = e + 1;
                pos.advance();
            }
            if (ok) {
                // Producer tail: wait until the issuer has released the last use
                // of every slot, so no tcgen05.commit arrival is still in flight
                // towards this CTA's shared memory when it exits.
                for (int e = max(0, total - ST); e < total && ok; ++e)
                    ok = wait_phase(bar(L::BAR_KVEMPTY + e % ST), (e / ST) & 1, p, abort_flag,
                                    kStatusWaitKvEmpty);
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
        if (lane == 0 && w.nmax > 0) {
            constexpr uint32_t IDESC_S = make_idesc_bf16(kBM, BN, false, false);
            constexpr uint32_t IDESC_O = make_idesc_bf16(kBM, D, false, true);
            // Descriptors are built once; an operand at byte offset `off` from a
            // base adds off >> 4 to the low word (the 14-bit start field never
            // carries: shared addresses stay below 2^18).
            const uint64_t kmaj0 = make_sdesc_sw128(sbase, 16, 1024);          // K-major tiles
            const uint64_t vmn0 = make_sdesc_sw128(sbase, BN * 128, 1024);     // V, MN-major
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
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t in_row = (kk & 3) * 32;  // 16 bf16 = 32 bytes of a 128-byte row
                    umma_ss(tmem + L::S_COL(t), desc(kmaj_lo, kmaj_hi, qa + (kk >> 2) * (kBM * 128) + in_row),
                            desc(kmaj_lo, kmaj_hi, kb + (kk >> 2) * (BN * 128) + in_row), IDESC_S,
                            kk > 0 ? 1u : 0u);
                }
            };
            // O_t += P_t V_j (row-major O). P is K-major like Q; V is MN-major:
            // 16 keys = two 8-row swizzle atoms (2048 bytes), 64-column chunks
            // of d BN*128 bytes apart.
            auto issue_pv = [&](int t, int slot, bool accumulate) {
                const uint32_t pa = L::P_OFF + t * L::P_TILE;
                const uint32_t vb = L::SLOT_OFF + slot * L::SLOT_BYTES;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    umma_ss(tmem + L::O_COL(t), desc(kmaj_lo, kmaj_hi, pa + (kk >> 2) * L::P_CHUNK + (kk & 3) * 32),
                            desc(vmn_lo, vmn_hi, vb + kk * 2048), IDESC_O,
                            (accumulate || kk > 0) ? 1u : 0u);
            };
            // O^T += V_j^T P^T over `rows` query rows starting at tile t0: A is
            // the V slot read MN-major (M = d), B the P rows read K-major
            // (N = query rows, 128 bytes apart).
            constexpr uint32_t IDESC_OT2 = make_idesc_bf16(D, 2 * kBM, true, false);
            constexpr uint32_t IDESC_OT1 = make_idesc_bf16(D, kBM, true, false);
            auto issue_pv_t = [&](int t0, bool both, int slot, bool accumulate) {
                const uint32_t pb = L::P_OFF + t0 * L::P_TILE;
                const uint32_t vb = L::SLOT_OFF + slot * L::SLOT_BYTES;
                const uint32_t idesc = both ? IDESC_OT2 : IDESC_OT1;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)
                    umma_ss(tmem + L::O_COL(t0), desc(vmn_lo, vmn_hi, vb + kk * 2048),
                            desc(kmaj_lo, kmaj_hi, pb + (kk >> 2) * L::P_CHUNK + (kk & 3) * 32), idesc,
                            (accumulate || kk > 0) ? 1u : 0u);
            };

            RingPos<ST> pos;
            bool ok = wait_phase(bar(L::BAR_QFULL), 0, p, abort_flag, kStatusWaitQ);
            if (ok) ok = wait_phase(bar(L::BAR_KVFULL + pos.slot), pos.phase, p, abort_flag,
                                    kStatusWaitKvFull);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int t = 0; t < QT; ++t)
                    if (w.n[t] > 0) issue_s(t, pos.slot);
                umma_commit(bar(L::BAR_SFULL));
                umma_commit(bar(L::BAR_KVEMPTY + pos.slot));
                pos.advance();
            }
            for (int j = 0; j < w.nmax && ok; ++j) {
                // S_t(j+1) as soon as the softmax has read S_t(j) out of TMEM.
                if (j + 1 < w.nmax) {
                    ok = wait_phase(bar(L::BAR_KVFULL + pos.slot), pos.phase, p, abort_flag,
                                    kStatusWaitKvFull);
                    if (!ok) break;
                    // Every tile still active at step j must have read S(j) before
                    // S(j+1) exists, even one that needs no S(j+1): otherwise
                    // two phases of the shared S_full barrier could complete
                    // before that tile's last parity wait.
#pragma unroll
                    for (int t = 0; t < QT; ++t) {
                        if (ok && j < w.n[t]) {
                            ok = wait_phase(bar(L::BAR_SFREE + t), j & 1, p, abort_flag, kStatusWaitS);
                            if (!ok) break;
                            if (j + 1 < w.n[t]) {
                                tc_fence_after();
                                issue_s(t, pos.slot);
                            }
                        }
                    }
                    if (!ok) break;
                    umma_commit(bar(L::BAR_SFULL));
                    umma_commit(bar(L::BAR_KVEMPTY + pos.slot));
                    pos.advance();
                }
                ok = wait_phase(bar(L::BAR_KVFULL + pos.slot), pos.phase, p, abort_flag,
                                kStatusWaitKvFull);
                if (!ok) break;
                if constexpr (L::O_T) {
                    // One transposed PV batch over the tiles active at step j
                    // (N = 256 for both; N = 128 when one tile has finished).
#pragma unroll
                    for (int t = 0; t < QT; ++t) {
                        if (ok && j < w.n[t])
                            ok = wait_phase(bar(L::BAR_PFULL + t), j & 1, p, abort_flag, kStatusWaitP);
                    }
                    if (!ok) break;
                    tc_fence_after();
                    const bool a0 = j < w.n[0], a1 = j < w.n[1];
                    issue_pv_t(a0 ? 0 : 1, a0 && a1, pos.slot, j > 0);
                } else {
                    // O_t += P_t(j) V_j as each tile's P arrives.
#pragma unroll
                    for (int t = 0; t < QT; ++t) {
                        if (ok && j < w.n[t]) {
                            ok = wait_phase(bar(L::BAR_PFULL + t), j & 1, p, abort_flag, kStatusWaitP);
                            if (!ok) break;
                            tc_fence_after();
                            issue_pv(t, pos.slot, j > 0);
                        }
                    }
                    if (!ok) break;
                }
                // PV_done before O_full: the last PV_done arrival then lands
                // before the softmax (waiting on O_full) lets the CTA exit.
                umma_commit(bar(L::BAR_PVDONE));
#pragma unroll
                for (int t = 0; t < QT; ++t)
                    if (j + 1 == w.n[t]) umma_commit(bar(L::BAR_OFULL + t));
                umma_commit(bar(L::BAR_KVEMPTY + pos.slot));
                pos.advance();
            }
            // Always wait for every MMA this thread issued before the CTA can
            // reach its teardown: on an abort no softmax waits for O_full, and
            // TMEM must not be released under an MMA in flight.
            umma_commit(bar(L::BAR_DRAIN));
            wait_phase(bar(L::BAR_DRAIN), 0, p, abort_flag, kStatusWaitDrain, false);
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
        // Row-major O: this row's accumulator. O^T: head-dim index r of every row.
        const uint32_t tO = tmem + lane_field + L::O_COL(t);
        // This row's 128-byte lines of the swizzled P operand (one per 64-key chunk).
        const uint32_t p_row = sbase + L::P_OFF + t * L::P_TILE + r * 128;
        const uint32_t swz = static_cast<uint32_t>(r & 7);
        // O^T path: the tile's per-row factors and its group's named barrier.
        float* rowf = reinterpret_cast<float*>(smem + L::ROWF_OFF) + t * kBM;
        const int nbar = 1 + t;
        const float sl2 = p.scale_log2;
        int n = w.n[0];
#pragma unroll
        for (int i = 1; i < QT; ++i)
            if (t == i) n = w.n[i];

        float m = -INFINITY;       // exponent reference (base-2 units of scale*log2e*s)
        float m_true = -INFINITY;  // true running row max, same units
        float l = 0.f;             // running sum relative to m
        // `ok` is uniform within a warp. On the O^T path a warp whose wait
        // failed does no more work but still meets its group at the next named
        // barrier, whose reduction then lets the whole group leave together.
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            if (ok) {
                ok = wait_phase(bar(L::BAR_SFULL), j & 1, p, abort_flag, kStatusWaitS);
                // tcgen05.ld/st are warp-collective: the whole warp leaves together.
                ok = __all_sync(0xffffffffu, ok);
            }
            if constexpr (!L::O_T) {
                if (!ok) break;
            }
            float alpha = 1.f, m_new = m;
            uint32_t pk[BN / 2];  // P as packed bf16 pairs
            float part[8];
            if (ok) {
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
                // S_t(j) is in registers: the issuer may overwrite it with S_t(j+1).
                tc_fence_before();
                mbar_arrive(bar(L::BAR_SFREE + t));

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
                // The exponent reference m only moves when this tile's max exceeds
                // it by more than kRescaleSlack; otherwise every p = 2^(x - m) <=
                // 2^slack and the old reference is kept, so O and l need no
                // rescale. The result is the same: O/l and m + log2(l) do not
                // depend on which reference is used, only rounding does.
                const bool move = m_tile > m + kRescaleSlack;
                m_new = move ? m_tile : m;
                const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // all masked so far
                alpha = move ? ex2(m - m_use) : 1.f;
                const float neg = -m_use;

                // x = s*scale*log2e - m as packed fp32 pairs (one FFMA2 per two
                // keys), p = 2^x on the MUFU, row sums as four packed partial pairs.
                const uint64_t sl2x2 = f2pack(sl2, sl2);
                const uint64_t negx2 = f2pack(neg, neg);
                uint64_t part2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int i = 0; i < BN / 2; ++i) {
                    float x0, x1;
                    f2unpack(ffma2(f2pack(s[2 * i], s[2 * i + 1]), sl2x2, negx2), x0, x1);
                    const float e0 = ex2(x0);
                    const float e1 = ex2(x1);
                    part2[i & 3] = fadd2(part2[i & 3], f2pack(e0, e1));
                    pk[i] = pack_bf16x2(e0, e1);
                }
                f2unpack(part2[0], part[0], part[1]);
                f2unpack(part2[1], part[2], part[3]);
                f2unpack(part2[2], part[4], part[5]);
                f2unpack(part2[3], part[6], part[7]);
            }

            if (j > 0) {
                // PV(j-1) must be done before P_t is overwritten and before O_t
                // is rescaled.
                if (ok) {
                    ok = wait_phase(bar(L::BAR_PVDONE), (j - 1) & 1, p, abort_flag, kStatusWaitO);
                    ok = __all_sync(0xffffffffu, ok);
                    if (ok) tc_fence_after();
                }
                if constexpr (L::O_T) {
                    // Column q of O_t^T belongs to row q: publish this row's
                    // factor; the group rescales together when any row moved.
                    rowf[r] = alpha;
                    if (named_bar_or(nbar, kBM, !ok || alpha != 1.f)) {
                        if (named_bar_or(nbar, kBM, !ok)) {
                            ok = false;
                            break;
                        }
#pragma unroll 1
                        for (int cc = 0; cc < kBM / 32; ++cc) {
                            uint32_t o[32];
                            tmem_ld32(tO + cc * 32, o);
                            const float4* f4 = reinterpret_cast<const float4*>(rowf + cc * 32);
                            float f[32];
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                const float4 v4 = f4[i];
                                f[4 * i] = v4.x;
                                f[4 * i + 1] = v4.y;
                                f[4 * i + 2] = v4.z;
                                f[4 * i + 3] = v4.w;
                            }
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                float x0, x1;
                                f2unpack(fmul2(f2pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])),
                                               f2pack(f[2 * i], f[2 * i + 1])),
                                         x0, x1);
                                o[2 * i] = __float_as_uint(x0);
                                o[2 * i + 1] = __float_as_uint(x1);
                            }
                            tmem_st32(tO + cc * 32, o);
                        }
                        tmem_wait_st();
                        // Every factor read before any row publishes the next one.
                        named_bar_sync(nbar, kBM);
                    }
                } else {
                    if (!ok) break;
                    if (__any_sync(0xffffffffu, alpha != 1.f)) {
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
                }
            }
            // (O^T path, step 0 only: a failed warp goes on to the next barrier.)
            if (!ok) continue;

            // P_t(j) into the 128-byte-swizzled K-major operand: 16-byte unit u
            // of a row's 128-byte line lands at position u ^ (row % 8).
#pragma unroll
            for (int c = 0; c < BN / 64; ++c) {
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_shared_v4(p_row + c * L::P_CHUNK + ((u ^ swz) << 4), pk[c * 32 + u * 4 + 0],
                                 pk[c * 32 + u * 4 + 1], pk[c * 32 + u * 4 + 2], pk[c * 32 + u * 4 + 3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(L::BAR_PFULL + t));
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
        if constexpr (L::O_T) {
            write_tile_t<D, QT>(p, w, t, r, n, m, m_true, l, tO, rowf, nbar, ok);
        } else {
            if (ok) write_row<D>(p, w.bh, w.split, q_row, n, m, m_true, l, tO);
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, L::TMEM_COLS);
}

}  // namespace fa
