// fa_fwd_common.cuh — pieces shared by the forward kernels: work partition,
// bounded mbarrier waits, K/V ring positions and the per-row epilogue.
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
// e4m3 P: a smaller slack and a fixed shift, p = 2^(x - m + kP8Shift) with
// x - m <= kP8Slack, so p <= 2^8 (e4m3 saturates at 448) and the row's largest
// p is at least 2^6 (e4m3 is normal from 2^-6 up).
constexpr float kP8Slack = 2.0f;
constexpr float kP8Shift = 6.0f;

// Ring position (slot, phase parity) of a sequence of K/V entries.
template <int ST>
struct RingPos {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void advance() {
        if (++slot == ST) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// Where a query row's output goes: O row (in units of d elements) =
// o_base + q * o_stride, LSE index = lse_base + q, for row q of the sequence;
// split partials at (split * BH + bh) * Nq + q. Rows q >= len_q are not written.
struct RowMap {
    long long o_base;
    long long lse_base;
    int o_stride;
    int len_q;
};

// Work owned by one CTA.
template <int Q_TILES>
struct Work {
    int bh;        // batch * H + head (work row)
    int zq;        // head coordinate of the Q/K/V/O tensor maps (bh, or h for varlen)
    int qbase;     // token of the sequence's first query row (0 unless varlen)
    int kbase;     // token of the sequence's first key (0 unless varlen)
    int q0;        // first query row of the unit, within the sequence
    int split;     // key split index (0 in plain mode)
    int kv_tile0;  // first key tile of the split, within the sequence
    int kv_end;    // exclusive key bound of the split (for masking), within the sequence
    int causal_off;  // causal: key j visible to query row i iff j <= i + causal_off
    RowMap rm;
    int n[Q_TILES];  // key tiles each query tile visits
    int nmax;
};

// First query row of tile slot t (0 or 1) of a unit that starts at row q0.
// Under a causal mask, with two slots, the slots are reversed: slot 0 takes
// the unit's later rows, whose tile sees one more key tile. The MMA issuer
// serves slot 0 first in every key step, so the tile that ends last, and sets
// when the unit's epilogue and the next unit can run, is served first.
__device__ __forceinline__ int tile_row0(const FwdParams& p, int q0, int t) {
    const int bm = p.bm64 ? 64 : kBM;
    return q0 + ((p.causal && p.tiles_per_cta == 2) ? 1 - t : t) * bm;
}

// Unit `lin` (blockIdx.x for a one-unit CTA; a persistent CTA walks lin =
// blockIdx.x + k * gridDim.x).
template <int QT, int BN>
__device__ __forceinline__ void compute_work(const FwdParams& p, long long lin, Work<QT>& w) {
    // CTA order: key splits fastest; then heads in groups of p.head_group
    // (sized so one group is about one wave of CTAs), and within a group the
    // query units heaviest first (last rows first under a causal mask) across
    // the group's heads. CTAs running together share a few heads' K/V in L2,
    // and long causal units start before short ones.
    w.split = static_cast<int>(lin % p.num_splits);
    lin /= p.num_splits;
    const long long per_group = static_cast<long long>(p.head_group) * p.n_units;
    const int group = static_cast<int>(lin / per_group);
    const int r = static_cast<int>(lin % per_group);
    const int heads_here = min(p.head_group, p.BH - group * p.head_group);
    const int unit = p.n_units - 1 - r / heads_here;
    w.bh = group * p.head_group + r % heads_here;
    // Query rows per tile: 128, or 64 for the 64-row tiles of fa_fwd_rows.
    const int bm = p.bm64 ? 64 : kBM;
    w.q0 = unit * p.tiles_per_cta * bm;
    // The sequence's rows and keys: the whole head (dense), or the packed
    // sequence b of a variable-length batch.
    int len_q = p.Nq, len_k = p.Nk;
    w.zq = w.bh;
    w.qbase = 0;
    w.kbase = 0;
    w.rm.o_base = static_cast<long long>(w.bh) * p.Nq;
    w.rm.lse_base = w.rm.o_base;
    w.rm.o_stride = 1;
    if (p.varlen) {
        const int b = w.bh / p.H;
        const int h = w.bh - b * p.H;
        const int cq0 = p.cu_q[b], cq1 = p.cu_q[b + 1], ck0 = p.cu_k[b], ck1 = p.cu_k[b + 1];
        const bool valid = 0 <= cq0 && cq0 <= cq1 && cq1 <= p.total_q && cq1 - cq0 <= p.Nq &&
                           0 <= ck0 && ck0 <= ck1 && ck1 <= p.Nk;
        if (!valid) {
            // Nothing is read or written for a sequence whose offsets are broken.
            if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSeqlens);
            len_q = 0;
            len_k = 0;
        } else {
            len_q = cq1 - cq0;
            len_k = ck1 - ck0;
        }
        w.zq = h;
        w.qbase = valid ? cq0 : 0;
        w.kbase = valid ? ck0 : 0;
        w.rm.o_base = static_cast<long long>(w.qbase) * p.H + h;
        w.rm.lse_base = static_cast<long long>(h) * p.total_q + w.qbase;
        w.rm.o_stride = p.H;
    }
    w.rm.len_q = len_q;
    w.causal_off = p.causal_br ? len_k - len_q : 0;
    const int total_tiles = (len_k + BN - 1) / BN;
    const int t0 = min(w.split * p.kv_tiles_per_split, total_tiles);
    const int t1 = min(t0 + p.kv_tiles_per_split, total_tiles);
    w.kv_tile0 = t0;
    w.kv_end = min(len_k, t1 * BN);
    w.nmax = 0;
#pragma unroll
    for (int t = 0; t < QT; ++t) {
        const int row0 = tile_row0(p, w.q0, t);
        int n = 0;
        if (t < p.tiles_per_cta && row0 < len_q) {
            int end = t1;
            if (p.causal) {
                // Keys up to the tile's last row + causal_off; none if that is < 0.
                const int last_key = min(row0 + bm - 1, len_q - 1) + w.causal_off;
                end = min(end, last_key < 0 ? 0 : last_key / BN + 1);
            }
            n = max(0, end - t0);
        }
        w.n[t] = n;
        w.nmax = max(w.nmax, n);
    }
}

// Work of a dual-range CTA: split-KV with one query tile (Nq <= 128, dense).
// Both query tiles of the CTA hold the same 128 rows; tile t takes key split
// 2 * pair + t, so the two tiles still alternate on the tensor core. A tile
// whose split index is past the last split has no work and writes nothing.
struct WorkDual {
    int bh;
    int zq;
    int q0;           // 0: the one query tile
    int causal_off;
    RowMap rm;
    int split[2];     // key split of each tile (may be >= num_splits: no such split)
    int kv_tile0[2];  // first key tile of each tile's split
    int kv_end[2];    // exclusive key bound of each tile's split
    int n[2];
    int nmax;
};

// Pair `lin` of the dual-range grid: heads slowest, split pairs fastest.
template <int BN>
__device__ __forceinline__ void compute_work_dual(const FwdParams& p, long long lin, WorkDual& w) {
    const int pairs = (p.num_splits + 1) / 2;
    const int pair = static_cast<int>(lin % pairs);
    w.bh = static_cast<int>(lin / pairs);
    w.zq = w.bh;
    w.q0 = 0;
    w.rm.o_base = static_cast<long long>(w.bh) * p.Nq;
    w.rm.lse_base = w.rm.o_base;
    w.rm.o_stride = 1;
    w.rm.len_q = p.Nq;
    w.causal_off = p.causal_br ? p.Nk - p.Nq : 0;
    const int total_tiles = (p.Nk + BN - 1) / BN;
    w.nmax = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int s = 2 * pair + t;
        w.split[t] = s;
        const int t0 = min(s * p.kv_tiles_per_split, total_tiles);
        const int t1 = min(t0 + p.kv_tiles_per_split, total_tiles);
        w.kv_tile0[t] = t0;
        w.kv_end[t] = min(p.Nk, t1 * BN);
        int end = t1;
        if (p.causal) {
            const int last_key = min(kBM, p.Nq) - 1 + w.causal_off;
            end = min(end, last_key < 0 ? 0 : last_key / BN + 1);
        }
        w.n[t] = (s < p.num_splits) ? max(0, end - t0) : 0;
        w.nmax = max(w.nmax, w.n[t]);
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

// wait_phase for a whole warp that waits together: every lane polls, and the
// loop's exits are warp votes, so the warp runs it as one (no divergent exits
// to reconverge from). True once every lane has seen the phase complete; false
// as wait_phase returns false (abort raised elsewhere, or this warp's wait ran
// past the limit, which raises it).
__device__ __forceinline__ bool wait_phase_warp(uint32_t bar, uint32_t parity, const FwdParams& p,
                                                volatile uint32_t* abort_flag, unsigned what,
                                                bool honor_abort = true) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
    const long long start = clock64();
    while (true) {
        if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
        if (honor_abort && __any_sync(0xffffffffu, *abort_flag != 0u)) return false;
        if (__any_sync(0xffffffffu, clock64() - start > p.wait_limit)) {
            if ((threadIdx.x & 31) == 0) {
                *abort_flag = 1u;
                atomicOr(p.status, what);
            }
            __syncwarp();
            return false;
        }
    }
}

// One query row's output, written 32 fp32 columns at a time from the final
// accumulator row: normalised O (bf16) and LSE in plain mode, or the
// unnormalised partial state (O, m, l) in split mode. Deferred normalisation:
// one division per row, at the write.
//
// Two row sums arrive: `l`, the sum of the exponentials as computed (fp32, for
// the LSE and the partial l), and `l_o`, the denominator of O: the sum of the
// weights the PV MMA actually multiplied V by (P rounded to bf16), as far as
// the softmax tracked them (l plus the rounding error of each key tile's
// largest p). O / l_o keeps the dominant keys' weights consistent with the
// rounded P, so a row dominated by one key gives that key's V up to the output
// rounding. Paths that do not track the rounding pass l_o = l.
template <int D>
struct RowOut {
    bool row_ok;
    bool split;
    float f;   // plain: o_scale/l_o; split: move from the lazy reference m to m_true
    float fo;  // split: the factor on the partial O, f * o_scale * l / l_o (l takes f alone)
    size_t row_idx, lse_idx, part_idx;
    float m, m_true, l;

    // `o_scale` multiplies O, normalised (plain mode) or partial (split mode):
    // the V descale of 8-bit inputs, 1 otherwise. In split mode O is scaled by
    // l / l_o, so that the partial (u, l) satisfies u / l = O / l_o.
    __device__ __forceinline__ RowOut(const FwdParams& p, const RowMap& rm, int bh, int split_idx,
                                      int q_row, float m_, float m_true_, float l_, float l_o,
                                      float o_scale = 1.f)
        : row_ok(q_row < rm.len_q), split(p.split_mode != 0), m(m_), m_true(m_true_), l(l_) {
        row_idx = static_cast<size_t>(rm.o_base + static_cast<long long>(q_row) * rm.o_stride);
        lse_idx = static_cast<size_t>(rm.lse_base + q_row);
        part_idx = (static_cast<size_t>(split_idx) * p.BH + bh) * p.Nq + q_row;
        if (!split) {
            f = (l_o > 0.f) ? o_scale / l_o : 0.f;
            fo = f;
        } else {
            f = (l > 0.f && m != m_true) ? ex2(m - m_true) : 1.f;
            fo = f * o_scale * ((l_o > 0.f && l_o != l) ? l / l_o : 1.f);
        }
    }
    // Columns [32 cc, 32 cc + 32) of the row, fp32 bits (zero when the row saw
    // no key); `o` is scaled in place.
    __device__ __forceinline__ void chunk(const FwdParams& p, int cc, uint32_t (&o)[32]) const {
        if (!split) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * f, __uint_as_float(o[2 * i + 1]) * f);
            if (row_ok) {
                uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + row_idx * D + cc * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
        } else {
            if (fo != 1.f) {
                const uint64_t f2 = f2pack(fo, fo);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float x0, x1;
                    f2unpack(fmul2(f2pack(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), f2),
                             x0, x1);
                    o[2 * i] = __float_as_uint(x0);
                    o[2 * i + 1] = __float_as_uint(x1);
                }
            }
            if (row_ok) {
                uint4* dst = reinterpret_cast<uint4*>(p.ws_o + part_idx * D + cc * 32);
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
        }
    }
    // The row's scalars: LSE (plain) or the partial m, l (split).
    __device__ __forceinline__ void finish(const FwdParams& p) const {
        if (!row_ok) return;
        constexpr float kLn2 = 0.69314718055994530942f;
        if (!split) {
            p.lse[lse_idx] = (l > 0.f) ? (m + lg2(l)) * kLn2 : -INFINITY;
        } else {
            p.ws_m[part_idx] = (l > 0.f) ? m_true * kLn2 : -INFINITY;
            p.ws_l[part_idx] = l * f;
        }
    }
};

// Writes one query row's result from its TMEM accumulator row (lane address
// tO, D fp32 columns; not read when n == 0), a chunk at a time.
template <int D>
__device__ __forceinline__ void write_row(const FwdParams& p, const RowMap& rm, int bh, int split,
                                          int q_row, int n, float m, float m_true, float l, float l_o,
                                          uint32_t tO, float o_scale = 1.f) {
    const RowOut<D> out(p, rm, bh, split, q_row, m, m_true, l, l_o, o_scale);
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
        out.chunk(p, cc, o);
    }
    out.finish(p);
}

// Plain-mode epilogue of one 128-row query tile, run by the tile's 128
// softmax threads (thread r = row r = TMEM lane r): o_scale * O_t / l as bf16
// is staged at `q_tile` (128 x D bf16: the tile's own bf16 Q shared memory,
// free once the tile's last PV has finished, as every S MMA reading Q came
// before it; or a staging buffer of that size) in the 128-byte-swizzled
// layout a Q load through the same kind of tensor map produces, and the
// group's first warp writes the tile with TMA tensor stores (rows past Nq are
// clipped). `bh` is the head coordinate of the O tensor map. `staged` is an
// mbarrier expecting one arrival per warp. Returns false if the bounded wait
// for the staging ran out. Dense layouts only: a packed variable-length
// sequence's tile would spill into the next sequence's rows.
template <int D>
__device__ __forceinline__ bool store_tile_tma(const FwdParams& p, const RowMap& rm, int bh, int q_row0,
                                               int r, int q_row, float m, float m_true, float l,
                                               float l_o, uint32_t tO, uint32_t q_tile, uint32_t staged,
                                               volatile uint32_t* abort_flag, float o_scale = 1.f) {
    const int lane = r & 31;
    const RowOut<D> out(p, rm, bh, 0, q_row, m, m_true, l, l_o, o_scale);
    const uint32_t swz = static_cast<uint32_t>(r & 7);
#pragma unroll 1
    for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(tO + cc * 32, o);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * out.f, __uint_as_float(o[2 * i + 1]) * out.f);
        // 32 columns = four 16-byte units of the row's line in 64-column chunk cc/2.
        const uint32_t line = q_tile + (cc >> 1) * (kBM * 128) + r * 128;
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
            const uint32_t u = static_cast<uint32_t>((cc & 1) * 4 + uu);
            st_shared_v4(line + ((u ^ swz) << 4), pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2], pk[4 * uu + 3]);
        }
    }
    out.finish(p);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(staged);
    bool ok = true;
    if (r < 32) {
        ok = __all_sync(0xffffffffu, wait_phase(staged, 0, p, abort_flag, kStatusWaitO));
        if (ok && lane == 0) {
#pragma unroll
            for (int c = 0; c < D / 64; ++c) tma_store_3d(&p.tm_o, q_tile + c * (kBM * 128), 64 * c, q_row0, bh);
            bulk_commit_group();
            bulk_wait_group_read0();  // shared memory read before the CTA exits
        }
    }
    return ok;
}

// Plain-mode epilogue of one 128-row query tile, per warp: o_scale * O_t / l as
// bf16, one 64-column chunk at a time. Each warp stages its own 32 rows of the
// chunk at `q_tile` (a 128 x D bf16 area: the tile's own bf16 Q shared memory,
// free once the tile's last PV has finished, or a buffer of that size) in the
// 128-byte-swizzled layout of the O tensor map, and writes them at once with a
// TMA tensor store of a 32-row x 64-column box (rows past the sequence are
// clipped; a warp whose rows all lie past it stores nothing). No warp waits for
// another; each waits for its own stores to have read shared memory before it
// leaves. `bh` is the head coordinate of the O tensor map (box rows 32).
template <int D>
__device__ __forceinline__ void store_rows_tma(const FwdParams& p, const RowMap& rm, int bh, int q_row0,
                                               int r, int q_row, float m, float m_true, float l,
                                               float l_o, uint32_t tO, uint32_t q_tile, float o_scale = 1.f) {
    const int lane = r & 31;
    const int quarter = r >> 5;
    const RowOut<D> out(p, rm, bh, 0, q_row, m, m_true, l, l_o, o_scale);
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    const int wrow0 = q_row0 + quarter * 32;
    const bool any_row = wrow0 < rm.len_q;
#pragma unroll 1
    for (int c = 0; c < D / 64; ++c) {
        uint32_t a[32], b[32];
        tmem_ld32(tO + c * 64, a);
        tmem_ld32(tO + c * 64 + 32, b);
        tmem_wait_ld();
        const uint32_t line = q_tile + c * (kBM * 128) + r * 128;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t x0 = hh ? b[2 * i] : a[2 * i];
                const uint32_t x1 = hh ? b[2 * i + 1] : a[2 * i + 1];
                pk[i] = pack_bf16x2(__uint_as_float(x0) * out.f, __uint_as_float(x1) * out.f);
            }
#pragma unroll
            for (int uu = 0; uu < 4; ++uu) {
                const uint32_t u = static_cast<uint32_t>(hh * 4 + uu);
                st_shared_v4(line + ((u ^ swz) << 4), pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2], pk[4 * uu + 3]);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && any_row) {
            tma_store_3d(&p.tm_o, q_tile + c * (kBM * 128) + quarter * (32 * 128), 64 * c, wrow0, bh);
            bulk_commit_group();
        }
    }
    out.finish(p);
    if (lane == 0) bulk_wait_group_read0();
    __syncwarp();
}

// store_rows_tma for persistent CTAs: the warp stages its 32 rows one
// 64-column chunk at a time in its own 4 KB buffer `buf` (32 rows x 128 bytes,
// the layout of one 32-row box of the O tensor map). Before each chunk it waits
// until its earlier TMA stores (this unit's previous chunk, or the previous
// unit's last) have read the buffer; the wait for the last chunk is left to
// the next call, or to the end of the kernel.
template <int D>
__device__ __forceinline__ void store_rows_tma_buf(const FwdParams& p, const RowMap& rm, int bh, int q_row0,
                                                   int r, int q_row, float m, float m_true, float l,
                                                   float l_o, uint32_t tO, uint32_t buf) {
    const int lane = r & 31;
    const int quarter = r >> 5;
    const RowOut<D> out(p, rm, bh, 0, q_row, m, m_true, l, l_o);
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    const int wrow0 = q_row0 + quarter * 32;
    const bool any_row = wrow0 < rm.len_q;
    const uint32_t line = buf + lane * 128;
#pragma unroll 1
    for (int c = 0; c < D / 64; ++c) {
        uint32_t a[32], b[32];
        tmem_ld32(tO + c * 64, a);
        tmem_ld32(tO + c * 64 + 32, b);
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
        tmem_wait_ld();
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t x0 = hh ? b[2 * i] : a[2 * i];
                const uint32_t x1 = hh ? b[2 * i + 1] : a[2 * i + 1];
                pk[i] = pack_bf16x2(__uint_as_float(x0) * out.f, __uint_as_float(x1) * out.f);
            }
#pragma unroll
            for (int uu = 0; uu < 4; ++uu) {
                const uint32_t u = static_cast<uint32_t>(hh * 4 + uu);
                st_shared_v4(line + ((u ^ swz) << 4), pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2], pk[4 * uu + 3]);
            }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && any_row) {
            tma_store_3d(&p.tm_o, buf, 64 * c, wrow0, bh);
            bulk_commit_group();
        }
    }
    out.finish(p);
}

}  // namespace fa
