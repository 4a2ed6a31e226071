/*
 * fa.h — exact scaled-dot-product attention forward on GB300 (sm_103a).
 *
 * What is computed (per batch b and head h, rows i of Q, keys j of K/V):
 *     S = scale * Q K^T            (optionally causal: key j visible to query i iff j <= i + c)
 *     O = softmax_row(S) V          (exact softmax, no approximation of the definition)
 *     LSE_i = ln sum_j exp(S_ij)    (natural log, in units of the scaled score)
 * The result is the plain definition of attention; the kernels reach it tile by
 * tile with the two-level online softmax ("Inside FlashAttention-3：面向 Hopper
 * 架构的 IO-Aware 精确注意力机制深度解析", section 二 "核心算法：Two-Level 在线
 * Softmax 的再回顾": running max m, running sum l, accumulator rescaled by
 * exp(m_old - m_new); and "AI 大模型之 FlashAttention_02", section "warp之间怎样
 * 减少通信": the division by l is deferred to the final write).
 *
 * Conventions shared by every entry point
 *  - Layout: Q, K, V, O are row-major contiguous bf16 tensors [B][H][N][d]
 *    (N = Nq for Q and O, Nk for K and V); LSE is fp32 [B][H][Nq].
 *  - Every pointer is a DEVICE pointer owned by the caller. The library
 *    allocates nothing, frees nothing and never synchronises (except
 *    fa_device_status, which says so).
 *  - Calls are asynchronous on `stream`; the return value covers argument
 *    validation and the launch only. Device-side failures surface at the
 *    caller's next synchronisation, or as FA_ERR_TIMEOUT from fa_device_status.
 *  - d must be 64, 128 or 256. Any other head dim is an error, never a silent
 *    fallback (the FlashAttention_02 page, sections 4.4 and 8, warns that
 *    frameworks silently switch backends for unsupported head dims).
 *  - `causal` selects the mask: FA_CAUSAL_NONE (0); FA_CAUSAL_TOP_LEFT (1),
 *    key j visible to query i iff j <= i; FA_CAUSAL_BOTTOM_RIGHT (2), iff
 *    j <= i + (Nk - Nq), so the last query row sees every key (the usual
 *    alignment when Nq new queries attend to a cache of Nk keys). Any other
 *    value is FA_ERR_CAUSAL. The two alignments coincide when Nq = Nk. The
 *    FlashAttention_02 page, section "正确性与部署边界", leaves square/non-square
 *    alignment to the implementation's documentation: this is it.
 *  - A query row that sees no key (bottom-right with Nq > Nk: its first Nq - Nk
 *    rows) gets O = 0 and LSE = -inf; in split mode its partial state is
 *    m = -inf, l = 0, O = 0, like an empty split.
 *  - `scale` must be finite and > 0; it is used exactly as given (float32).
 *  - q, k, v, o and the workspace must be 16-byte aligned; lse 4-byte aligned.
 *  - The output buffers must not overlap the inputs.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_NULL = 1,       /* a required pointer is NULL */
    FA_ERR_ALIGN = 2,      /* a pointer is not aligned as stated above */
    FA_ERR_SHAPE = 3,      /* B, H, Nq or Nk < 1, or a size overflows 32/64-bit indexing */
    FA_ERR_HEADDIM = 4,    /* d is not 64, 128 or 256 */
    FA_ERR_SPLITS = 5,     /* num_splits < 1 or > FA_MAX_SPLITS */
    FA_ERR_WORKSPACE = 6,  /* workspace pointer NULL or misaligned */
    FA_ERR_CUDA = 7,       /* a CUDA runtime or driver call failed (no device, launch, tensor-map encode) */
    FA_ERR_TIMEOUT = 8,    /* a kernel gave up on a bounded wait (reported by fa_device_status) */
    FA_ERR_SCALE = 9,      /* scale is not finite or not > 0 */
    FA_ERR_SCRATCH = 10,   /* fa_fwd_splitkv_static: partial states exceed FA_STATIC_SCRATCH_BYTES */
    FA_ERR_CAUSAL = 11,    /* causal is not FA_CAUSAL_NONE, _TOP_LEFT or _BOTTOM_RIGHT */
    FA_ERR_SEQLENS = 12,   /* fa_fwd_varlen: cu_seqlens not a valid partition (from fa_device_status) */
    FA_ERR_TILE = 13       /* fa_fwd_rows: rows_per_cta not offered for this head dim */
} fa_status;

#define FA_CAUSAL_NONE 0
#define FA_CAUSAL_TOP_LEFT 1
#define FA_CAUSAL_BOTTOM_RIGHT 2

#define FA_MAX_SPLITS 256

/*
 * fa_fwd — fused attention forward, one launch.
 *   q    [B][H][Nq][d] bf16 (read)        k, v [B][H][Nk][d] bf16 (read)
 *   o    [B][H][Nq][d] bf16 (written)     lse  [B][H][Nq] fp32 (written)
 * Work partition: each work unit is the query tiles of one (b, h) that one CTA
 * owns, swept over all keys they need ("AI 大模型之 FlashAttention_02", section
 * "从头级并行转向序列级并行": query tiles of one head go to different CTAs, no
 * cross-CTA reduction). Causal tiles that lie wholly above the diagonal are
 * skipped. One CTA per unit, except at d = 64 and 128 when the units fill at
 * least four waves of CTAs (four per SM) and are short (Nk within 16 key tiles
 * of 128, or 32 for non-causal d = 128): then one persistent CTA per SM walks
 * its share of the units in order, so that a unit's Q load and start-up
 * overlap the previous unit's last key steps. The result is the same bit for
 * bit either way.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int Nq, int Nk, int d, float scale, int causal,
                 cudaStream_t stream);

/*
 * fa_splitkv_workspace_bytes — size in bytes of the workspace fa_fwd_splitkv
 * writes and fa_combine reads, for the given shape and split count (0 when an
 * argument is out of range). Workspace layout, fp32, in this order:
 *   O_part [S][B][H][Nq][d]   unnormalised partial outputs  (u of each split)
 *   m      [S][B][H][Nq]      partial row max, natural-log units of the scaled score
 *   l      [S][B][H][Nq]      partial row sum, relative to that split's m
 * ("AI 大模型之 FlashAttention_02", section "工程实操 沿键切分的归约与沿查询切分的
 * 区别", subsection "接口与实现约束": a split scheme must state its split axis,
 * each group's output responsibility, the partial-statistics layout and the
 * merge operator; this comment and fa_combine's are that statement.)
 */
size_t fa_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits);

/*
 * fa_fwd_splitkv — split-KV forward: writes partial states, no final output.
 * Split axis: keys. With T = ceil(Nk / BN) key tiles (BN = 128 keys for
 * d <= 128, 96 for d = 256) and P = ceil(T / num_splits), split s owns key tiles
 * [s*P, min((s+1)*P, T)). Trailing splits may be empty; an empty split (or a
 * row whose keys in that split are all masked) writes m = -inf, l = 0, O = 0
 * (same section, subsection "扩展验证组合": the empty-tail rule; the true key
 * count Nk masks the last tile). Same q/k/v/shape rules as fa_fwd; `workspace`
 * must hold fa_splitkv_workspace_bytes(B, H, Nq, d, num_splits) bytes.
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* workspace,
                         int B, int H, int Nq, int Nk, int d, float scale, int causal,
                         int num_splits, cudaStream_t stream);

/*
 * fa_combine — merge operator for the split partial states ("AI 大模型之
 * FlashAttention_02", section "工程实操 沿键切分的归约与沿查询切分的区别",
 * subsection "逐步计算与预期结果", steps 2-3): per row
 *     M = max_s m_s,  w_s = exp(m_s - M),  L = sum_s w_s l_s,
 *     O = (sum_s w_s O_s) / L  -> bf16,   LSE = M + ln L.
 * (Normalising each split first and averaging is the wrong merge the page
 * warns against; it is not what this computes.) Reads the workspace written
 * by fa_fwd_splitkv with the same B, H, Nq, d, num_splits; writes o and lse
 * exactly as fa_fwd does.
 */
fa_status fa_combine(const void* workspace, void* o, float* lse,
                     int B, int H, int Nq, int d, int num_splits, cudaStream_t stream);

/*
 * fa_fwd_varlen — fused forward over a batch of variable-length sequences held
 * as one ragged, token-major packed tensor (the FA-3 page, "Inside
 * FlashAttention-3：面向 Hopper 架构的 IO-Aware 精确注意力机制深度解析", section
 * 7.2 "cuDNN 集成": variable-length sequences through ragged tensors).
 *
 *   q, o:  bf16 [total_q][H][d]      k, v: bf16 [total_k][H][d]
 *   lse:   fp32 [H][total_q]
 *   cu_seqlens_q, cu_seqlens_k: DEVICE int32 [B + 1]; sequence b owns query
 *   tokens cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key tokens
 *   cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1. Required: cu[0] >= 0,
 *   nondecreasing, cu_seqlens_q[B] <= total_q, cu_seqlens_k[B] <= total_k, and
 *   every query length <= max_seqlen_q.
 *
 * Each sequence is its own attention problem: its queries see only its keys,
 * and the causal mask (top-left or bottom-right) is placed by its own lengths.
 * Sequences may be empty; queries with no key get O = 0, LSE = -inf. Tokens
 * past cu_seqlens_q[B] are not written. Offsets that break the requirements
 * are found on the device: that sequence is neither read nor written and
 * fa_device_status later reports FA_ERR_SEQLENS. Host checks: pointers
 * (cu arrays 4-byte aligned), 1 <= max_seqlen_q <= total_q, causal, d, scale.
 * Launches ceil(max_seqlen_q / 256) (d <= 128; 128 for d = 256) query units per
 * (sequence, head); units past a sequence's end exit at once.
 */
fa_status fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                        const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H,
                        int total_q, int total_k, int max_seqlen_q, int d, float scale,
                        int causal, cudaStream_t stream);

/*
 * fa_fwd_fp8 — fused forward on 8-bit inputs (the FA-3 page, section 7.3
 * "BF16 / FP8 支持": e4m3 operands for both GEMMs, fp32 accumulation, and the
 * softmax max and sum kept in fp32).
 *
 *   q [B][H][Nq][d], k, v [B][H][Nk][d]: e4m3 codes, one byte each (OCP 8-bit
 *   floating point, E4M3: bias 7, no infinities, max 448), 16-byte aligned.
 *   The value of a code c of Q is decode(c) * q_descale (K, V likewise).
 *   o [B][H][Nq][d] bf16 (written), lse [B][H][Nq] fp32 (written).
 *
 * Computes the same function as fa_fwd on those values: O = softmax(scale *
 * Q K^T [+ mask]) V, LSE = ln of the softmax denominator. S is exact up to fp32
 * accumulation. P is rounded to e4m3 per element for the PV GEMM: P is scaled
 * so that each row's largest element lies in [2^6, 2^8], and the row sum l
 * is taken before the rounding. So O carries a rounding error of relative
 * size about 2^-4 / sqrt(3) per term, which averages over the keys. The LSE
 * does not carry it.
 * d = 64, 128 or 256 (else FA_ERR_HEADDIM). No varlen; the split-KV form is
 * fa_fwd_fp8_splitkv. causal as fa_fwd. FA_ERR_SCALE if a descale is not finite and > 0,
 * or if scale * q_descale * k_descale is not.
 */
fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, float q_descale,
                     float k_descale, float v_descale, void* o, float* lse, int B, int H,
                     int Nq, int Nk, int d, float scale, int causal, cudaStream_t stream);

/*
 * fa_fwd_fp8_splitkv — fa_fwd_splitkv on e4m3 inputs: the key axis split as
 * fa_fwd_splitkv splits it, partial states written to a workspace of
 * fa_splitkv_workspace_bytes(B, H, Nq, d, num_splits) bytes in the same fp32
 * layout, merged by fa_combine. The partial O includes the V descale; m and l
 * are those of the encoded values' scores. Arguments and status codes as
 * fa_fwd_fp8, plus num_splits (FA_ERR_SPLITS) and the workspace
 * (FA_ERR_WORKSPACE).
 */
fa_status fa_fwd_fp8_splitkv(const void* q, const void* k, const void* v, float q_descale,
                             float k_descale, float v_descale, void* workspace, int B, int H,
                             int Nq, int Nk, int d, float scale, int causal, int num_splits,
                             cudaStream_t stream);

/*
 * fa_bwd_workspace_bytes — bytes of the fp32 workspace fa_bwd needs, with the
 * query rows of each head padded to Nq_pad = 128 * ceil(Nq / 128): a dQ
 * accumulator [B][H][Nq_pad][d], then -LSE log2(e) and -D, each
 * [B][H][Nq_pad]. 0 when an argument is out of range (d must be 64, 128 or 256).
 */
size_t fa_bwd_workspace_bytes(int B, int H, int Nq, int d);

/*
 * fa_bwd — attention backward: dQ, dK, dV of O = softmax(scale Q K^T [+ mask]) V
 * for the upstream gradient dO ("AI 大模型之 FlashAttention_02", sections
 * "warp之间怎样减少通信" and "训练与部署 切分与归约的反向一致性": dK and dV are
 * accumulated across query rows, a reduction direction the forward does not
 * have).
 *   q, o, dout [B][H][Nq][d] bf16, k, v [B][H][Nk][d] bf16 (read);
 *   lse [B][H][Nq] fp32: the LSE fa_fwd wrote for the same q, k, v, causal, scale;
 *   dq [B][H][Nq][d], dk, dv [B][H][Nk][d] bf16 (written);
 *   workspace: fa_bwd_workspace_bytes(B, H, Nq, d) bytes, 16-byte aligned.
 * With P = exp(scale Q K^T - LSE): dV = P^T dO, dS = P * (dO V^T - D) with
 * D_i = sum_c dO_ic O_ic, dQ = scale dS K, dK = scale dS^T Q. Responsibilities:
 * a preprocess launch forms D and LSE log2(e) per padded row and zeroes the
 * fp32 dQ accumulator; the main launch runs one CTA per (head, 128-key tile),
 * which accumulates its keys' dK and dV over all query tiles in fp32 and adds
 * its dS K to the dQ accumulator (fp32 atomic adds, across key tiles); a last
 * launch writes dQ = scale times the accumulator in bf16. d = 64, 128 or 256
 * (else FA_ERR_HEADDIM; at 256 each key tile takes two CTAs, one per half of
 * the head dim); causal as fa_fwd.
 * Three launches on `stream`, no synchronisation.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                 const float* lse, void* dq, void* dk, void* dv, void* workspace, int B, int H,
                 int Nq, int Nk, int d, float scale, int causal, cudaStream_t stream);

/*
 * fa_fwd_rows — fa_fwd with the query rows a CTA owns chosen by the caller:
 * the query-tile sweep of the long-sequence workload (B = 1, H = 8,
 * N = 8192: query tiles split across CTAs, with several tile sizes; "AI 大模型之
 * FlashAttention_02", section "从头级并行转向序列级并行", and the tile sizes
 * of section "本册配套实验验证记录"). rows_per_cta = 256 is fa_fwd's own
 * choice at d <= 128: two 128-row tiles that alternate on the tensor core.
 * rows_per_cta = 128 gives each CTA one 128-row tile (the other tile slot
 * idles), so twice as many CTAs share the GPU and each computes alone.
 * rows_per_cta = 64 (d <= 128) gives each CTA one 64-row tile computed with
 * M = 64 MMAs, whose accumulator rows take 16 of each 32-lane TMEM quarter.
 * At d = 256 only 128 is offered (fa_fwd's choice there). Other values:
 * FA_ERR_TILE. Arguments, layouts and the other status codes are those of
 * fa_fwd; the result equals fa_fwd's bit for bit.
 */
fa_status fa_fwd_rows(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int Nq, int Nk, int d, float scale, int causal, int rows_per_cta,
                      cudaStream_t stream);

/*
 * fa_fwd_grid_ctas — number of work units (CTAs of one unit each) fa_fwd
 * (num_splits = 1) or fa_fwd_splitkv would run for this shape (fa_fwd launches
 * one persistent CTA per SM instead when the units fill four waves and are
 * short, see fa_fwd): B * H * ceil(Nq / BM) * num_splits,
 * BM = 256 query rows per CTA for d <= 128 (two 128-row tiles) and 128 for
 * d = 256 ("AI 大模型之 FlashAttention_02", section "从头级并行转向序列级并行" and
 * the printed CTA counts of section "本册配套实验验证记录"). Split-KV launches
 * with num_splits >= 2, Nq <= 128 and d <= 128 run two splits per CTA (the two
 * query-tile slots of a CTA hold the same rows, each with its own split), so
 * they launch B * H * ceil(num_splits / 2) CTAs. fa_fwd_fp8 and
 * fa_fwd_fp8_splitkv launch the same grids as fa_fwd and fa_fwd_splitkv.
 * Returns -1 when an argument is out of range. Host-only; launches nothing.
 */
long long fa_fwd_grid_ctas(int B, int H, int Nq, int d, int num_splits);

/*
 * fa_device_status — SYNCHRONISES `stream`, then reads the library's device
 * error word: FA_OK; FA_ERR_TIMEOUT if any kernel since the last clear gave up
 * on a bounded wait (it then exits cleanly and leaves its outputs undefined);
 * else FA_ERR_SEQLENS if fa_fwd_varlen met offsets that are not a valid
 * partition. `clear` != 0 resets the word. FA_ERR_CUDA if the read fails.
 */
fa_status fa_device_status(cudaStream_t stream, int clear);

/*
 * fa_fwd_splitkv_static — split-KV forward plus merge that allocates nothing
 * and takes no workspace argument. The pages have no counterpart to this
 * entry point; it exists for callers that cannot call cudaMalloc: a host
 * program or framework that owns every byte of device memory through its own
 * allocator and budget (so a library allocation would go unaccounted or fail),
 * or a serving loop where an allocation could block on device-wide
 * synchronisation at the wrong moment.
 *
 * It computes exactly what fa_fwd_splitkv followed by fa_combine computes
 * (same kernels, same split rule, same o/lse output contract as fa_fwd), but
 * keeps the partial states in one statically sized device buffer of
 * FA_STATIC_SCRATCH_BYTES that the library defines. Every GPU that loads the
 * library holds that buffer until the process exits.
 *   - The partial states, fa_splitkv_workspace_bytes(B, H, Nq, d, num_splits)
 *     bytes, must fit in FA_STATIC_SCRATCH_BYTES; larger problems return
 *     FA_ERR_SCRATCH before any CUDA call (use fewer splits, or fa_fwd_splitkv
 *     with your own workspace).
 *   - The first call on a device looks up that device's address of the buffer
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture. The address is cached per device and CUDA
 *     context: after cudaDeviceReset, or once the primary context has been
 *     released and re-created, the next call looks it up again (so that call,
 *     too, belongs before any capture) and no stale address is ever used.
 *   - Pointers, alignment, shapes, scale, mask and split count are checked
 *     before the size test and before any CUDA call: a refused call queues no
 *     work and leaves the buffer untouched.
 *   - All calls on a device share the one buffer and it keeps the last call's
 *     contents. Nothing in it needs to start at zero: the split kernel writes
 *     every entry the merge reads. Calls whose work overlaps on the GPU (other
 *     streams, other host threads) race on the buffer and give wrong results;
 *     order them on one stream or with events.
 * Arguments and the other status codes are those of fa_fwd plus num_splits.
 */
#define FA_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)
fa_status fa_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                                int B, int H, int Nq, int Nk, int d, float scale, int causal,
                                int num_splits, cudaStream_t stream);

/*
 * fa_test_fwd_withheld_q — failure-detection test hook (not for production
 * use). Launches the fa_fwd kernel (scale 1, non-causal) with its Q tile loads
 * withheld and every mbarrier wait bounded by `wait_limit_cycles` SM cycles
 * (2^16 .. 2^31). The MMA issuer's wait for Q then runs out before any MMA is
 * issued; the kernel raises its abort flag, the other roles leave at their
 * next wait, in-flight K/V copies are waited for, TMEM is freed and the kernel
 * exits without touching o or lse. A following fa_device_status returns
 * FA_ERR_TIMEOUT, and the CUDA context stays usable. No fault, trap or hang is
 * involved: only a wait that nothing will satisfy, with a bound.
 */
fa_status fa_test_fwd_withheld_q(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int H, int Nq, int Nk, int d, long long wait_limit_cycles,
                                 cudaStream_t stream);

/* fa_status_string — static, human-readable name of a status code. */
const char* fa_status_string(fa_status status);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
