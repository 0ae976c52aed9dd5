// Paged GQA decode over bfloat16 or 8-bit (e4m3) K/V pages: TMA page staging,
// mbarrier pipeline, tensor-core tile products, online softmax, fused split
// merge.  sm_103a.  Included by the decode_tma_*.cu files, each of which
// instantiates one (head dimension, page type, merge variant).
//
// Decode attention reads every cached K/V byte once and does G multiply-adds
// per element, far below the tensor cores' ridge point, so the kernel is built
// around keeping HBM busy (the pages: moving KV tensors from global memory to
// the compute cores takes far longer than the matrix products, "Advanced
// Optimizations: MQA, GQA, and PagedAttention", section "The Memory Bandwidth
// Bottleneck").
//
// Unit of work.  A pool block [block_size, Hkv, D] is contiguous, all KV heads
// of a token side by side.  A CTA therefore works on a group of HG KV heads at
// once (HG = 8 for Llama-style GQA) and one TMA box fetches a page slice for
// the whole group: [rows, HG heads, 128 bytes x D/64] — at Hkv = 8, D = 128,
// block_size = 16 that is the entire 32 KB block, one contiguous read.  The
// tensor map lists the pool's dimensions as (d_lo 64, slot, head-half, block)
// so the box lands in shared memory head-major, [head-half][slot][64], which
// keeps the 128-byte swizzle conflict-free for ldmatrix over tokens.
//
// Structure of a CTA (one per span of the tile sequence, see partition.cuh;
// the grid is one CTA per SM):
//   * warp NC (producer): walks the span's tiles (T = 128 / HG tokens of one
//     (sequence, head group); 256 / HG for 8-bit pages, so that a stage holds
//     64 KB either way), keeps a 32-entry window of block ids in
//     registers (plus the next window in flight), and issues one
//     cp.async.bulk.tensor per page for K and one for V into a ring of stages
//     guarded by "full" (transaction bytes) and "empty" mbarriers.  Reading the
//     pages inside the attention kernel is the block-read + attention fusion
//     of "Modern LLM Inference ...", section 8.3.
//   * warps 0..NC-1 (consumers): warp (hgi, mt, tg) owns KV head hgi of the
//     group, query rows [16 mt, 16 mt + 16) of that head's G-row group and
//     tokens [tg TW, (tg+1) TW) of every tile.  S = q K^T and O += P V run on
//     mma.sync m16n8k16 (bf16 in, fp32 accumulate) fed by ldmatrix from the
//     swizzled stage; the running max / sum softmax runs on the fp32
//     accumulators in base-2 units.  When TG > 1 the token groups of a head
//     combine through shared memory at the end of a piece; the tg == 0 warps
//     then write the output rows (whole run) or a normalised partial and its
//     log2-sum-exp (split run).  After the tile loop a split run is merged by
//     the warp whose arrival completed it, with register loads of the pieces
//     (merge variant 0); in the shared-merge variant (1: cooperative launch,
//     long runs) all its pieces' warps merge it, each taking a share of the
//     rows; in variant 2 (runs over 2 to 5 spans) pieces only write their
//     partials and a second kernel merges every split run over all SMs.
//   * 8-bit pages: K and V fragments come straight from the stage by
//     ldmatrix and are widened to f16 in registers (cvt.rn.f16x2.e4m3x2);
//     both products run on f16 mma.sync, the per-head scales fold into the
//     logit multiplier and the epilogue.
//
// Every wait is bounded (kWaitNs); a wait that gives up latches
// PGD_ERR_TIMEOUT, marks the CTA aborted and lets every warp leave.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <limits.h>
#include <math.h>

#include <atomic>
#include <mutex>

#include "partition.cuh"

namespace pgd {
namespace tma {

constexpr uint64_t kWaitNs = 2000000000ull;  // 2 s
// With automatic splits, use fewer spans than CTAs when the call has fewer than
// this many tiles per CTA: tiny calls then split runs into fewer pieces.
constexpr int kMinTilesPerCta = 2;
constexpr int kSmemBudget = 227 * 1024;

// ----------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of `bar` with the given parity; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// The same wait taken by a whole warp: every lane waits (so every lane sees
// the phase complete), then the warp takes one decision.  Without the vote,
// lanes near the limit could decide differently and the ones that went on
// would meet the warp's next shuffle or mma without the others.
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Relaxed (morally strong, unordered) read: a later fence makes it an acquire.
__device__ __forceinline__ int ld_relaxed(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// A split run's counter word: pieces arrived in the low bits, and a flag bit
// that the last arriver flips as it sets the count back to zero.
constexpr int kRunFlagShift = 30;
constexpr int kRunCountMask = (1 << kRunFlagShift) - 1;

// Bounded wait until the flag bit of the run word at p differs from `old`
// (acquire, GPU scope).  Only used under a cooperative launch, where the CTA
// that flips it is resident; false after kWaitNs.
__device__ __forceinline__ bool wait_flip(const int* p, int old) {
    if (((ld_acquire(p) >> kRunFlagShift) & 1) != old) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        __nanosleep(32);
        if (((ld_acquire(p) >> kRunFlagShift) & 1) != old) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
}

// L2 policy for data read exactly once per call (the K/V pages).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "l"(policy)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D; bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// D = A(16x16, row) * B(16x8, col) + D; f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Two e4m3 values (low byte -> low half) to two f16: exact, every e4m3 value
// is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}

// The low (bytes 0, 1) and high (bytes 2, 3) pair of a word of 8-bit codes
// as f16x2.  e4m3: the exact values.  int8: the word must hold the codes with
// their sign bits flipped (w ^ 0x80808080); each byte is then placed as the
// low byte under an 0x64 high byte, and that f16 is 1024 + (code + 128) =
// code + kI8Bias (exponent 10, the byte as the low mantissa bits), exact.  The
// kernel takes the bias out of the sums it enters (see kI8Bias).
template <bool INT8>
__device__ __forceinline__ uint32_t widen_lo(uint32_t w) {
    if constexpr (INT8) return __byte_perm(w, 0x64646464u, 0x5140);
    else return e4m3x2_to_f16x2((uint16_t)(w & 0xffffu));
}
template <bool INT8>
__device__ __forceinline__ uint32_t widen_hi(uint32_t w) {
    if constexpr (INT8) return __byte_perm(w, 0x64646464u, 0x5342);
    else return e4m3x2_to_f16x2((uint16_t)(w >> 16));
}
// int8 pages: every widened code carries +1152.  In q . k that adds
// 1152 * sum_d q[d] to every score of a query row (subtracted with the logit
// multiplier); in P V it adds 1152 * sum_t P[t] to every output column of a
// row (the f16 P values fed to the products are summed beside them and the
// term subtracted at the piece's end).
constexpr float kI8Bias = 1152.f;

__device__ __forceinline__ float2 f16x2_to_float2(uint32_t w) {
    return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

// Two bf16 (one 32-bit word) to two f16.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&w);
    const float2 f = __bfloat1622float2(b);
    return pack_f16(f.x, f.y);
}

// ----------------------------------------------------------------- configuration
template <int D_, int HG_, int MT_, int TG_, bool ROWS16_, bool FP8_ = false, int MV_ = 0,
          bool INT8_ = false, bool PB_ = false>
struct Cfg {
    static constexpr int D = D_;
    static constexpr int HG = HG_;            // KV heads per unit of work
    static constexpr int MT = MT_;            // m16 row tiles of one head's query group
    static constexpr int TG = TG_;            // token groups per tile
    static constexpr bool ROWS16 = ROWS16_;   // rows 8..15 of an m-tile in use
    static constexpr bool FP8 = FP8_;         // 8-bit K/V pages, f16 products
    static constexpr bool INT8 = INT8_;       // 8-bit pages hold int8 codes (else e4m3)
    static constexpr bool PB = PB_;           // 8-bit pages with a scale per block and KV head
    // merge variant of split runs: 0 the last arriver merges with register
    // loads; 1 (SHARE, cooperative launch) all pieces' warps merge a share of
    // the rows; 2 (SEP) no merge here: pieces write partials, and a second
    // kernel (merge_runs_kernel) merges them
    static constexpr int MV = MV_;
    static constexpr bool SHARE = MV_ == 1;
    static constexpr bool SEP = MV_ == 2;
    // 128-byte rows of a head in a page box: D/64 for bf16, 1 for 8-bit D = 128
    static constexpr int HALVES = FP8 ? D / 128 : D / 64;
    static constexpr int HH = HG * HALVES;    // 128-byte head rows per token in a tile
    // tokens per tile: 128 token-heads per stage tensor (16 KB of 8-bit rows
    // would leave the consumers' per-tile work too thin: 256 there)
    static constexpr int T = (FP8 ? 256 : 128) / HG;
    static constexpr int NC = HG * MT * TG;   // consumer warps
    static constexpr int THREADS = (NC + 1) * 32;
    static constexpr int TW = T / TG;         // tokens per consumer warp per tile
    // a warp's slice is processed in chunks of CH tokens (8-bit pages: at
    // most 32, which bounds the score registers)
    static constexpr int CH = (FP8 && TW > 32) ? 32 : TW;
    static constexpr int TENSOR_BYTES = HH * T * 128;   // K (or V) bytes of a stage
    static constexpr int STAGE_BYTES = 2 * TENSOR_BYTES;
    static constexpr int ROWS = ROWS16 ? 16 : 8;
    // per-block scales of 8-bit pages: pages of a tile (block_size >= 8)
    static constexpr int MAXP = FP8 ? (T / 8 < 32 ? T / 8 : 32) : 1;
    static constexpr int COMB_FLOATS = (TG - 1) * HG * MT * ROWS * (D + 2);
    static constexpr int COMB_BYTES = COMB_FLOATS * 4;
    static constexpr int STATIC_RESERVE = 4096;  // static smem + alignment slack
    static constexpr int STAGES_FIT = (kSmemBudget - STATIC_RESERVE - COMB_BYTES) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    // dynamic smem: [1024 align slack][stages][comb]
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + COMB_BYTES;
    static_assert(!FP8 || D == 128, "8-bit pages: head_dim 128");
    static_assert(!INT8 || FP8, "int8 codes are 8-bit pages");
    static_assert(!PB || FP8, "per-block scales are for 8-bit pages");
    static_assert(STAGES >= 2, "pipeline needs at least two stages");
    static_assert(TW % 16 == 0, "a warp's token slice must be whole k16 steps");
    static_assert(TW % CH == 0 && CH % 16 == 0, "chunks must split the slice in k16 steps");
    static_assert(NC <= 8, "at most 8 consumer warps");
};

// A run whose pieces this warp brought to completion: merged after the tile loop.
struct MergeJob {
    int64_t t0;     // first tile of the run
    int64_t c0;     // CTA of its first piece
    int npieces;
    int first_is_tail;
    int b, kvh;     // b < 0: no job
    int k;          // shared merge: this warp's piece of the run; -1: merge all rows
    int flag;       // shared merge: the run's flag before this piece arrived
};

// What the producer tells the consumers about the tile in a stage.
struct StageDesc {
    int64_t run_start;  // flat index of tile 0 of the (b, unit) run
    int b, unit, n_valid, flags;
    int n_b;            // tiles of the run
    int tok0;           // sequence position of the tile's first token
    int L;              // sequence length
    int pad;
};

// Offset (in elements) of query row r of KV head kvh of sequence b in q / out
// [B, q_len, Hq, D]: row r is query token r / G, head kvh * G + r % G.
__device__ __forceinline__ int64_t qrow_offset(const DecodeArgs& a, int b, int kvh, int r) {
    const int G = a.group;
    return (((int64_t)b * a.q_len + r / G) * a.hq + (int64_t)kvh * G + r % G) * a.d;
}

// Merge the pieces of a split run for query rows [r_lo, r_hi) of head `hgi` of
// the group (KV head `kvh` of sequence `b`) and write them to `out`.  Log-sum-exp combination in base 2: with lse_k = m_k +
// log2 l_k and o_k the normalised partial of piece k,
//     out = sum_k 2^(lse_k - M) o_k / sum_k 2^(lse_k - M),  M = max_k lse_k,
// accumulated online.  The lanes cover a row's columns with float4 reads, and
// each lane keeps kMergeRows slots: a slot is a row pass, or (PHASED, when the
// warp's rows fit one pass) every slot takes the same rows and piece phase x
// (pieces x, x + RU, ...), the slots folded together at the end.  kPieceBatch
// pieces per slot are read before any is used, so a lane has 16 loads in
// flight.  Runs after the tile loop, when the loop's accumulators are dead.
constexpr int kPieceBatch = 4;
constexpr int kMergeRows = 4;
static_assert(kShareMinLoads == 6 * kMergeRows * kPieceBatch, "six batches of merge loads");

__device__ __forceinline__ void lse_fold(float& M, float& W, float4& acc, float e, float w,
                                         float4 v) {
    // (M, W, acc) holds acc = sum_k 2^(lse_k - M) o_k and W = sum_k 2^(lse_k - M);
    // add a term that is (e, w, v) in the same form: a piece is (lse, 1, o),
    // another slot is (M', W', acc')
    // explicit roundings: every merge of this kernel rounds the same way,
    // whatever the compiler would contract
    const float nm = fmaxf(M, e);
    const float base = nm == -INFINITY ? 0.f : nm;
    const float sa = fast_exp2(M - base), sb = fast_exp2(e - base);
    M = nm;
    W = __fmaf_rn(W, sa, __fmul_rn(w, sb));
    acc.x = __fmaf_rn(acc.x, sa, __fmul_rn(v.x, sb));
    acc.y = __fmaf_rn(acc.y, sa, __fmul_rn(v.y, sb));
    acc.z = __fmaf_rn(acc.z, sa, __fmul_rn(v.z, sb));
    acc.w = __fmaf_rn(acc.w, sa, __fmul_rn(v.w, sb));
}

template <class C, bool PHASED>
__device__ __forceinline__ void merge_pieces(const DecodeArgs& a, int64_t t0, int64_t N, int64_t P,
                                          int64_t c0, int npieces, bool first_is_tail, int hgi,
                                          int r_lo, int r_hi, int b, int kvh) {
    constexpr int D = C::D;
    constexpr int CPR = D / 4;             // float4 chunks per row
    constexpr int RPP = 32 / CPR;          // rows per pass
    constexpr int RU = kMergeRows;
    constexpr int PB = kPieceBatch;
    const int lane = threadIdx.x % 32;
    const int rows = a.q_len * a.group;    // query rows per KV head
    const int piece_rows = C::HG * rows;
    const int col = (lane % CPR) * 4;
    constexpr int npe = PHASED ? 1 : RU;  // row passes per round
    constexpr int rep = RU / npe;          // piece phases per row pass
    for (int rb = r_lo; rb < r_hi; rb += RPP * npe) {
        int r[RU], ph[RU];
        bool rok[RU];
        int64_t pr[RU];
        float4 acc[RU];
        float M[RU], W[RU];
#pragma unroll
        for (int x = 0; x < RU; ++x) {
            ph[x] = x / npe;
            r[x] = rb + (x % npe) * RPP + lane / CPR;
            rok[x] = ph[x] < rep && r[x] < r_hi;
            pr[x] = (int64_t)(hgi * rows + r[x]);
            acc[x] = make_float4(0.f, 0.f, 0.f, 0.f);
            M[x] = -INFINITY;
            W[x] = 0.f;
        }
        for (int k0 = 0; k0 < npieces; k0 += PB * rep) {
            float4 v[RU][PB];
            float e[RU][PB];
#pragma unroll
            for (int u = 0; u < PB; ++u) {
#pragma unroll
                for (int x = 0; x < RU; ++x) {
                    const int k = k0 + ph[x] + rep * u;
                    const bool ok = rok[x] && k < npieces;
                    // with P > N every non-empty span holds one tile: piece k is
                    // the owner of tile t0 + k; otherwise the pieces are CTAs
                    // c0, c0 + 1, ...
                    const int64_t c = P > N ? (ok ? span_owner(t0 + k, N, P) : 0) : c0 + k;
                    const int64_t sl = c * 2 + ((first_is_tail && k == 0) ? 1 : 0);
                    v[x][u] = ok ? __ldcg(reinterpret_cast<const float4*>(
                                       a.part_o + (sl * piece_rows + pr[x]) * D + col))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                    e[x][u] = ok ? __ldcg(a.part_lse + sl * piece_rows + pr[x]) : -INFINITY;
                }
            }
#pragma unroll
            for (int x = 0; x < RU; ++x) {
#pragma unroll
                for (int u = 0; u < PB; ++u) lse_fold(M[x], W[x], acc[x], e[x][u], 1.f, v[x][u]);
            }
        }
        // fold the other piece phases of a row pass into its first slot
#pragma unroll
        for (int x = npe; x < RU; ++x) {
            if (rok[x]) lse_fold(M[x % npe], W[x % npe], acc[x % npe], M[x], W[x], acc[x]);
        }
#pragma unroll
        for (int x = 0; x < RU; ++x) {
            if (x >= npe || !rok[x]) continue;
            const float w = W[x] > 0.f ? 1.f / W[x] : 0.f;  // no token in any piece: zeros
            uint2 pk;
            pk.x = pack_bf16(acc[x].x * w, acc[x].y * w);
            pk.y = pack_bf16(acc[x].z * w, acc[x].w * w);
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) +
                                      qrow_offset(a, b, kvh, r[x]) + col) = pk;
        }
    }
}

// ----------------------------------------------------------------- the kernel
template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    decode_tma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, DecodeArgs a) {
    constexpr int S = C::STAGES;
    constexpr int D = C::D;
    constexpr int T = C::T;
    extern __shared__ uint8_t dyn_smem[];
    __shared__ int64_t scratch[C::THREADS > 98 ? C::THREADS : 98];
    __shared__ SpanStart ss;
    __shared__ __align__(8) uint64_t full_bar[S];
    __shared__ __align__(8) uint64_t empty_bar[S];
    __shared__ __align__(8) uint64_t comb_bar;
    __shared__ StageDesc desc[S];
    __shared__ MergeJob jobs[C::NC][2];  // per consumer warp and partial slot
    // 8-bit pages with per-block scales: K (0) and V (1) scale of every head
    // of the unit for each page of the tile in a stage
    __shared__ float qsc[C::PB ? S : 1][2][C::HG][C::PB ? C::MAXP : 1];
    __shared__ volatile int aborted;

    uint8_t* stage_base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(dyn_smem) + 1023) & ~uintptr_t(1023));
    float* comb = reinterpret_cast<float*>(stage_base + S * C::STAGE_BYTES);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int bs = a.block_size;
    // page geometry of a tile: R rows per box, T / R boxes (pages) per tile
    const int R = bs < T ? bs : T;
    const int log_r = __ffs(R) - 1;

    // 8-bit pages with per-block scales: the producer publishes each stage's
    // scales after issuing its copies, with a second arrival on the stage
    constexpr bool pbs = C::PB;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(smem_u32(&full_bar[s]), pbs ? 2 : 1);
            mbar_init(smem_u32(&empty_bar[s]), C::NC * 32);
        }
        mbar_init(smem_u32(&comb_bar), C::NC * 32);
        for (int w = 0; w < C::NC; ++w) jobs[w][0].b = jobs[w][1].b = -1;
        aborted = 0;
        fence_barrier_init();
    }
    find_span_start(a.seq_lens, a.B, a.units, T, a.q_len, a.window, a.max_blocks, bs,
                    a.num_parts, a.auto_parts ? kMinTilesPerCta : 1, scratch, &ss,
                    a.tile_base, a.run_cost);  // ends with __syncthreads

    // Sequences that own no tiles: length 0 gives zeros, an out-of-range length
    // gives NaN and latches PGD_ERR_SEQ_LEN.  CTA b % P writes sequence b.
    for (int b = blockIdx.x; b < a.B; b += gridDim.x) {
        const int L = a.seq_lens[b];
        if (L != 0 && seq_len_ok(L, a.max_blocks, bs)) continue;
        if (L != 0 && threadIdx.x == 0) latch_error(a.err, PGD_ERR_SEQ_LEN);
        const __nv_bfloat16 fill = __float2bfloat16_rn(L == 0 ? 0.f : NAN);
        __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(a.out) + (int64_t)b * a.q_len * a.hq * D;
        for (int i = threadIdx.x; i < a.q_len * a.hq * D; i += blockDim.x) ob[i] = fill;
    }
    const int64_t r0 = ss.r0, r1 = ss.r1;
    const int W = ss.run_cost;
    const int n_tiles = ss.n_tiles;  // real tiles (a span may hold cost slots only)
    if (n_tiles == 0) return;

    if (warp == C::NC) {
        // ============================================================ producer
        TileCursor cur = cursor_at(ss, a.seq_lens, a.units, T, a.q_len, a.window, a.max_blocks,
                                   bs, W);
        const uint64_t policy = policy_evict_first();
        const uint32_t box_bytes = (uint32_t)(C::HH * R * 128);
        // Block-id window: lane l holds block_table[win_b][win_lb + l]; the next
        // 32 entries are loaded ahead into nxt_id so that walking a run meets
        // the table's latency once per window, not once per tile.
        int win_b = -1, win_lb = 0, win_id = -1, nxt_id = -1;
        auto table_row = [&](int b, int lb) -> int {
            const int idx = lb + lane;
            return idx < a.max_blocks ? a.block_table[(int64_t)b * a.max_blocks + idx] : -1;
        };
        int issued = 0;  // stages armed with expect_tx
        int L = a.seq_lens[cur.b];
        int L_b = cur.b;
        for (int it = 0; it < n_tiles; ++it) {
            const int s = it % S;
            const uint32_t ph = (uint32_t)(it / S) & 1u;
            const int64_t x = cur.run_start + cur.i;  // virtual index of the tile
            if (cur.b != L_b) {
                L = a.seq_lens[cur.b];
                L_b = cur.b;
            }
            const int tok0 = (cur.first + cur.i) * T;
            const int n_valid = min(T, L - tok0);
            const int npg = bs < T ? (n_valid + bs - 1) / bs : 1;
            // pages wholly before the earliest token any query reads are not
            // fetched (a windowed cache may have released them)
            const int lo_min = a.window > 0 ? max(0, L - a.q_len - a.window + 1) : 0;
            const int skip = (bs < T && lo_min > tok0) ? (lo_min - tok0) / bs : 0;
            const int lb0 = tok0 / bs;
            const int slot0 = bs < T ? 0 : tok0 % bs;
            if (cur.b != win_b || lb0 < win_lb || lb0 + npg > win_lb + 32) {
                if (cur.b == win_b && lb0 == win_lb + 32) {
                    win_id = nxt_id;
                    win_lb += 32;
                } else {
                    win_b = cur.b;
                    win_lb = lb0;
                    win_id = table_row(win_b, win_lb);
                }
                nxt_id = table_row(win_b, win_lb + 32);
            }
            const int64_t phys = __shfl_sync(0xffffffffu, win_id, (lb0 - win_lb + lane) & 31);
            const bool want = lane >= skip && lane < npg;
            const bool ok = want && phys >= 0 && phys < a.num_blocks;
            const bool bad = __any_sync(0xffffffffu, want && !ok);
            const int nok = __popc(__ballot_sync(0xffffffffu, ok));
            // per-block scales of page `lane` for the unit's heads, loaded
            // before the wait and published after the copies are issued;
            // pages not fetched get 0 (their tokens are masked, their V rows
            // zeroed, so the factor only has to be finite)
            float ksv[C::HG], vsv[C::HG];
            if constexpr (pbs) {
                const int64_t sb = ok ? (int64_t)phys * a.hkv + (int64_t)cur.unit * C::HG : -1;
#pragma unroll
                for (int h = 0; h < C::HG; ++h) {
                    ksv[h] = sb >= 0 ? __ldg(a.k_scale + sb + h) : 0.f;
                    vsv[h] = sb >= 0 ? __ldg(a.v_scale + sb + h) : 0.f;
                }
            }
            const int flags =
                segment_flags(x, cur.run_start, cur.n_b, r0, r1) | (bad ? kTileBad : 0);

            if (!mbar_wait_warp(smem_u32(&empty_bar[s]), ph ^ 1u)) {
                if (lane == 0) {
                    latch_error(a.err, PGD_ERR_TIMEOUT);
                    aborted = 1;
                }
                break;
            }
            if (__any_sync(0xffffffffu, aborted)) break;
            const uint32_t fb = smem_u32(&full_bar[s]);
            if (lane == 0) {
                desc[s] = StageDesc{cur.run_start, cur.b, cur.unit, n_valid, flags, cur.n_b,
                                    tok0, L, 0};
                mbar_arrive_expect_tx(fb, (uint32_t)nok * box_bytes * 2u);
                if (bad) latch_error(a.err, PGD_ERR_BLOCK_ID);
            }
            ++issued;
            __syncwarp();
            if (ok) {
                // page `lane` of the tile: K box then V box, all HG heads
                const uint32_t dst = smem_u32(stage_base + s * C::STAGE_BYTES) + lane * box_bytes;
                const int hh0 = cur.unit * C::HH;
                tma_load_4d(dst, &tmap_k, fb, 0, slot0, hh0, (int)phys, policy);
                tma_load_4d(dst + C::TENSOR_BYTES, &tmap_v, fb, 0, slot0, hh0, (int)phys, policy);
            }
            if constexpr (pbs) {
                if (lane < C::MAXP) {
#pragma unroll
                    for (int h = 0; h < C::HG; ++h) {
                        qsc[s][0][h][lane] = ksv[h];
                        qsc[s][1][h][lane] = vsv[h];
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(fb);  // second arrival: the scales are in place
            }
            cursor_next(cur, a.seq_lens, a.B, a.units, T, a.q_len, a.window, a.max_blocks, bs,
                        W);
        }
        // Do not leave while copies this CTA issued may still land.
        if (lane == 0) {
            const int first = issued > S ? issued - S : 0;
            for (int it = first; it < issued; ++it) {
                if (!mbar_wait(smem_u32(&full_bar[it % S]), (uint32_t)(it / S) & 1u)) break;
            }
        }
        return;
    }

    const int rows = a.q_len * a.group;  // query rows per KV head
    constexpr int RPP = 32 / (D / 4);    // rows per merge pass

    // ================================================================ consumers
    const int tg = warp % C::TG;
    const int mt = (warp / C::TG) % C::MT;
    const int hgi = warp / (C::TG * C::MT);
    const int gid = lane >> 2, tig = lane & 3;
    const int tw0 = tg * C::TW;
    const int G = a.group;               // query row r is (token r / G, head r % G)
    const int row0 = mt * 16 + gid;      // row of accumulator rows c0,c1
    const int row1 = row0 + 8;           // row of c2,c3
    const bool row0_ok = row0 < rows;
    const bool row1_ok = C::ROWS16 && row1 < rows;
    const int piece_rows = C::HG * rows; // rows of a partial result
    const int hh_mine = hgi * C::HALVES; // my head's first head-half in a page box
    // Query token of each of my rows: attends to positions [lo, hi) with
    // hi = L - q_len + i + 1 and lo = hi - window (clamped at 0) when windowed.
    const int qi0 = row0 / G, qi1 = row1 / G;

    uint32_t qa[D / 16][4];
    float o[D / 8][4];
    // logit multiplier (base-2 units; times the K scale of 8-bit pages) and the
    // V scale of 8-bit pages, set per piece
    float s_mul = a.scale_log2, v_mul = 1.f;
    // int8 pages: the K bias term of each row's scores (1152 * sum_d q) and
    // the running sums of the f16 P values (for the V bias term); 0 otherwise
    float qc0 = 0.f, qc1 = 0.f, cp0 = 0.f, cp1 = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    bool seg_bad = false;
    uint32_t comb_phase = 0;

    // Lane-dependent parts of the ldmatrix addresses.
    const int lm_mi = lane >> 3, lm_i = lane & 7;
    // byte offset of (token t, head-half h of my head) row in a tensor of a stage
    auto row_off = [&](int t, int h) -> uint32_t {
        const int p = t >> log_r, r = t & (R - 1);
        return (uint32_t)(((p * C::HH + hh_mine + h) * R + r) * 128);
    };

    // Load the query rows this warp owns for (sequence q_seq, KV head q_kvh) as
    // mma A fragments (and, for 8-bit pages, that head's scales).
    auto load_q = [&](int q_seq, int q_kvh) {
        const __nv_bfloat16* qb = static_cast<const __nv_bfloat16*>(a.q);
        const uint32_t* q0 = reinterpret_cast<const uint32_t*>(
            qb + (row0_ok ? qrow_offset(a, q_seq, q_kvh, row0) : 0));
        const uint32_t* q1 = reinterpret_cast<const uint32_t*>(
            qb + (row1_ok ? qrow_offset(a, q_seq, q_kvh, row1) : 0));
        if constexpr (C::FP8) {
            // f16 fragments with the head dimension permuted inside each
            // 16-wide step: mma k-slots (2 tig, 2 tig + 1) and (2 tig + 8,
            // 2 tig + 9) hold d = 16 ks + 4 tig + (0, 1) and + (2, 3), so
            // that one 32-bit read of an 8-bit K row feeds both B registers.
            // The dot product does not depend on the order of d.
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int c = ks * 8 + 2 * tig;  // word of columns 16ks + 4 tig
                qa[ks][0] = row0_ok ? bf16x2_to_f16x2(__ldg(q0 + c)) : 0u;
                qa[ks][1] = row1_ok ? bf16x2_to_f16x2(__ldg(q1 + c)) : 0u;
                qa[ks][2] = row0_ok ? bf16x2_to_f16x2(__ldg(q0 + c + 1)) : 0u;
                qa[ks][3] = row1_ok ? bf16x2_to_f16x2(__ldg(q1 + c + 1)) : 0u;
            }
            if constexpr (C::INT8) {
                // the sum of this lane's f16 q values of each row, over the
                // lanes of the row's quad: the whole row
                float q0s = 0.f, q1s = 0.f;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const float2 x0 = f16x2_to_float2(qa[ks][0]), x2 = f16x2_to_float2(qa[ks][2]);
                    const float2 x1 = f16x2_to_float2(qa[ks][1]), x3 = f16x2_to_float2(qa[ks][3]);
                    q0s += (x0.x + x0.y) + (x2.x + x2.y);
                    q1s += (x1.x + x1.y) + (x3.x + x3.y);
                }
                q0s += __shfl_xor_sync(0xffffffffu, q0s, 1);
                q0s += __shfl_xor_sync(0xffffffffu, q0s, 2);
                q1s += __shfl_xor_sync(0xffffffffu, q1s, 1);
                q1s += __shfl_xor_sync(0xffffffffu, q1s, 2);
                qc0 = kI8Bias * q0s;
                qc1 = kI8Bias * q1s;
            }
            if constexpr (pbs) {  // scales per page, applied per n-tile
                s_mul = a.scale_log2;
                v_mul = 1.f;
            } else {
                s_mul = a.scale_log2 * __ldg(a.k_scale + q_kvh);
                v_mul = __ldg(a.v_scale + q_kvh);
            }
        } else {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const int c = ks * 8 + tig;  // 32-bit word index of columns 16ks + 2 tig
                qa[ks][0] = row0_ok ? __ldg(q0 + c) : 0u;
                qa[ks][1] = row1_ok ? __ldg(q1 + c) : 0u;
                qa[ks][2] = row0_ok ? __ldg(q0 + c + 4) : 0u;
                qa[ks][3] = row1_ok ? __ldg(q1 + c + 4) : 0u;
            }
        }
    };
    // Prefetch the first piece's query rows while its pages are in flight.
    int pre_seq = -1, pre_kvh = -1;
    {
        const TileCursor c0 = cursor_at(ss, a.seq_lens, a.units, T, a.q_len, a.window,
                                        a.max_blocks, bs, W);
        pre_seq = c0.b;
        pre_kvh = c0.unit * C::HG + hgi;
        load_q(pre_seq, pre_kvh);
    }

    for (int it = 0; it < n_tiles; ++it) {
        const int s = it % S;
        const uint32_t ph = (uint32_t)(it / S) & 1u;
        if (!mbar_wait_warp(smem_u32(&full_bar[s]), ph)) {
            if (lane == 0) {
                latch_error(a.err, PGD_ERR_TIMEOUT);
                aborted = 1;
            }
            break;
        }
        if (__any_sync(0xffffffffu, aborted)) break;
        const StageDesc dsc = desc[s];
        uint8_t* st = stage_base + s * C::STAGE_BYTES;
        // the CTA's final piece of a split run reads its run's counter now
        // (relaxed; the merge after the loop fences first), so that if every
        // other piece is in already it skips its fence and arrival
        int pre_cnt = 0;
        if (!C::SHARE && !C::SEP && it == n_tiles - 1 && tg == 0 && (dsc.flags & kSegEnd) &&
            (dsc.flags & kSegPartial))
            pre_cnt = ld_relaxed(a.counters +
                                 ((int64_t)dsc.b * a.hkv + dsc.unit * C::HG + hgi) * C::MT + mt);
        const uint32_t k_u = smem_u32(st);
        const uint32_t v_u = k_u + C::TENSOR_BYTES;
        const int kvh = dsc.unit * C::HG + hgi;

        if (dsc.flags & kSegStart) {
            // New piece: its query rows (unless prefetched at the start).
            if (dsc.b != pre_seq || kvh != pre_kvh) load_q(dsc.b, kvh);
            pre_seq = -1;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
            m0 = m1 = -INFINITY;
            l0 = l1 = 0.f;
            cp0 = cp1 = 0.f;
            seg_bad = false;
        }
        seg_bad |= (dsc.flags & kTileBad) != 0;

        const int n_valid = dsc.n_valid;
        // tile-local tokens before `v_lo` (pages not fetched: before every
        // query's window) or from n_valid on (past the end) hold tail slots or
        // stale data: zero their V rows so 0 * (NaN or Inf) never reaches O
        const int lo_min = a.window > 0 ? max(0, dsc.L - a.q_len - a.window + 1) : 0;
        const int v_lo = max(0, lo_min - dsc.tok0);
        const bool active = tw0 < n_valid && tw0 + C::TW > v_lo;
        // (both ends clamped to my slice: with several token groups or chunks
        // a slice can end before n_valid while the window starts inside it)
        const int z_hi = min(tw0 + C::TW, max(tw0, v_lo));        // zero [tw0, z_hi) ...
        const int z_lo2 = min(tw0 + C::TW, max(tw0, n_valid));    // ... and [z_lo2, tw0 + TW)
        const bool zeroed = active && (z_hi > tw0 || z_lo2 < tw0 + C::TW);
        if (zeroed) {
            const int n1 = z_hi - tw0;
            const int nz = n1 + (tw0 + C::TW - z_lo2);
            for (int idx = lane; idx < nz * 8 * C::HALVES; idx += 32) {
                const int j = idx / (8 * C::HALVES);
                const int t = j < n1 ? tw0 + j : z_lo2 + (j - n1);
                const int rem = idx % (8 * C::HALVES);
                *reinterpret_cast<uint4*>(st + C::TENSOR_BYTES + row_off(t, rem / 8) +
                                          (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
            }
            __syncwarp();
        }

        if (active) {
#pragma unroll 1
            for (int c0 = tw0; c0 < tw0 + C::TW; c0 += C::CH) {  // CH-token chunks of my slice
                if (c0 >= n_valid || c0 + C::CH <= v_lo) continue;
                // ---- S = q K^T over the chunk's CH tokens
                float sc[C::CH / 8][4];
#pragma unroll
                for (int j = 0; j < C::CH / 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
                if constexpr (C::FP8) {
                    // lane (gid, tig) needs bytes 16 ks + 4 tig .. +3 of token row
                    // c0 + 8 j + gid, widened to the two f16 B registers: one
                    // ldmatrix.x4 brings them for n-tiles (jp, jp + 1) x k-steps
                    // (ks, ks + 1)
#pragma unroll
                    for (int ks = 0; ks < D / 16; ks += 2) {
#pragma unroll
                        for (int jp = 0; jp < C::CH / 8; jp += 2) {
                            const int tok = c0 + (jp + (lm_mi & 1)) * 8 + lm_i;
                            const int kc = ks + (lm_mi >> 1);
                            uint32_t w[4];
                            ldsm_x4(k_u + row_off(tok, 0) + ((kc ^ lm_i) << 4), w[0], w[1], w[2],
                                    w[3]);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                if constexpr (C::INT8) w[q] ^= 0x80808080u;
                                mma_f16(sc[jp + (q & 1)], qa[ks + (q >> 1)],
                                        widen_lo<C::INT8>(w[q]), widen_hi<C::INT8>(w[q]));
                            }
                        }
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const int h = ks / 4;
                        const int kc = (ks % 4) * 2 + (lm_mi & 1);
#pragma unroll
                        for (int np = 0; np < C::CH / 16; ++np) {
                            const int tok = c0 + np * 16 + (lm_mi >> 1) * 8 + lm_i;
                            uint32_t b0, b1, b2, b3;
                            ldsm_x4(k_u + row_off(tok, h) + ((kc ^ lm_i) << 4), b0, b1, b2, b3);
                            mma_bf16(sc[2 * np], qa[ks], b0, b1);
                            mma_bf16(sc[2 * np + 1], qa[ks], b2, b3);
                        }
                    }
                }
                // ---- mask (causal / window, per row), scale to base-2 units, running max
                const int hi0 = dsc.L - a.q_len + qi0 + 1 - dsc.tok0;   // tile-local bounds
                const int hi1 = dsc.L - a.q_len + qi1 + 1 - dsc.tok0;
                const int lo0 = a.window > 0 ? hi0 - a.window : INT_MIN;
                const int lo1 = a.window > 0 ? hi1 - a.window : INT_MIN;
                float mx0 = -INFINITY, mx1 = -INFINITY;
                // logit multiplier of each n-tile (8 tokens, one page): with
                // per-block scales, times the K scale of the tile's page
                float smj[C::CH / 8];
#pragma unroll
                for (int j = 0; j < C::CH / 8; ++j) smj[j] = s_mul;
                if constexpr (pbs) {
#pragma unroll
                    for (int j = 0; j < C::CH / 8; ++j)
                        smj[j] = s_mul * qsc[s][0][hgi][(c0 + 8 * j) >> log_r];
                }
                // every row sees all of this warp's tokens (the usual case): no mask
                const bool full = c0 + C::CH <= dsc.L - a.q_len + 1 - dsc.tok0 &&
                                  (a.window == 0 || c0 >= dsc.L - a.window - dsc.tok0);
                if (full) {
#pragma unroll
                    for (int j = 0; j < C::CH / 8; ++j) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            if constexpr (C::INT8) {
                                sc[j][e] = fmaf(sc[j][e], smj[j], -qc0 * smj[j]);
                                sc[j][2 + e] = fmaf(sc[j][2 + e], smj[j], -qc1 * smj[j]);
                            } else {
                                sc[j][e] *= smj[j];
                                sc[j][2 + e] *= smj[j];
                            }
                            mx0 = fmaxf(mx0, sc[j][e]);
                            mx1 = fmaxf(mx1, sc[j][2 + e]);
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < C::CH / 8; ++j) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int tok = c0 + j * 8 + tig * 2 + e;
                            const bool v0 = tok < hi0 && tok >= lo0;
                            const bool v1 = tok < hi1 && tok >= lo1;
                            sc[j][e] = v0 ? fmaf(sc[j][e], smj[j], -qc0 * smj[j]) : -INFINITY;
                            sc[j][2 + e] = v1 ? fmaf(sc[j][2 + e], smj[j], -qc1 * smj[j])
                                              : -INFINITY;
                            mx0 = fmaxf(mx0, sc[j][e]);
                            mx1 = fmaxf(mx1, sc[j][2 + e]);
                        }
                    }
                }
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                if (C::ROWS16) {
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                }
                const float mn0 = fmaxf(m0, mx0);
                const float mn1 = C::ROWS16 ? fmaxf(m1, mx1) : 0.f;
                const float base0 = mn0 == -INFINITY ? 0.f : mn0;
                const float base1 = mn1 == -INFINITY ? 0.f : mn1;
                const float alpha0 = fast_exp2(m0 - base0);
                const float alpha1 = C::ROWS16 ? fast_exp2(m1 - base1) : 1.f;
                m0 = mn0;
                if (C::ROWS16) m1 = mn1;
                float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
                for (int j = 0; j < C::CH / 8; ++j) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        sc[j][e] = fast_exp2(sc[j][e] - base0);
                        ps0 += sc[j][e];
                        if (C::ROWS16) {
                            sc[j][2 + e] = fast_exp2(sc[j][2 + e] - base1);
                            ps1 += sc[j][2 + e];
                        } else {
                            sc[j][2 + e] = 0.f;
                        }
                    }
                }
                l0 = l0 * alpha0 + ps0;
                if (C::ROWS16) l1 = l1 * alpha1 + ps1;
                if constexpr (C::INT8) {
                    cp0 *= alpha0;
                    if (C::ROWS16) cp1 *= alpha1;
                }
                if (__any_sync(0xffffffffu, alpha0 != 1.f || alpha1 != 1.f)) {
#pragma unroll
                    for (int n = 0; n < D / 8; ++n) {
                        o[n][0] *= alpha0;
                        o[n][1] *= alpha0;
                        o[n][2] *= alpha1;
                        o[n][3] *= alpha1;
                    }
                }
                // ---- O += P V
#pragma unroll
                for (int kk = 0; kk < C::CH / 16; ++kk) {
                    if constexpr (C::FP8) {
                        // 8-bit V straight from the stage: a transposed 16-bit ldmatrix
                        // gives lane (gid, tig) tokens (2 tig, 2 tig + 1) x bytes
                        // d = (2 gid, 2 gid + 1) of a 16-byte chunk; one byte permute
                        // puts the two tokens of d = 2 gid in the low half and those of
                        // 2 gid + 1 in the high half, each an e4m3x2 B operand.  n-tile
                        // 2 c + par then holds d = 16 c + 2 j + par for B column j, so
                        // the output columns come out permuted (undone where O is stored).
                        uint32_t pa[4];
                        if constexpr (pbs) {
                            // per-block V scales folded into P (the row sums
                            // above use P itself)
                            const float v0 = qsc[s][1][hgi][(c0 + 16 * kk) >> log_r];
                            const float v1 = qsc[s][1][hgi][(c0 + 16 * kk + 8) >> log_r];
                            pa[0] = pack_f16(sc[2 * kk][0] * v0, sc[2 * kk][1] * v0);
                            pa[1] = pack_f16(sc[2 * kk][2] * v0, sc[2 * kk][3] * v0);
                            pa[2] = pack_f16(sc[2 * kk + 1][0] * v1, sc[2 * kk + 1][1] * v1);
                            pa[3] = pack_f16(sc[2 * kk + 1][2] * v1, sc[2 * kk + 1][3] * v1);
                        } else {
                            pa[0] = pack_f16(sc[2 * kk][0], sc[2 * kk][1]);
                            pa[1] = pack_f16(sc[2 * kk][2], sc[2 * kk][3]);
                            pa[2] = pack_f16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
                            pa[3] = pack_f16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
                        }
                        if constexpr (C::INT8) {  // the f16 P values the products take
                            const float2 a0 = f16x2_to_float2(pa[0]), a2 = f16x2_to_float2(pa[2]);
                            cp0 += (a0.x + a0.y) + (a2.x + a2.y);
                            if (C::ROWS16) {
                                const float2 a1 = f16x2_to_float2(pa[1]);
                                const float2 a3 = f16x2_to_float2(pa[3]);
                                cp1 += (a1.x + a1.y) + (a3.x + a3.y);
                            }
                        }
                        const int tok = c0 + kk * 16 + (lm_mi & 1) * 8 + lm_i;
#pragma unroll
                        for (int c2 = 0; c2 < D / 32; ++c2) {
                            const int vc = c2 * 2 + (lm_mi >> 1);
                            uint32_t r[4];
                            ldsm_x4_t(v_u + row_off(tok, 0) + ((vc ^ lm_i) << 4), r[0], r[1], r[2],
                                      r[3]);
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                r[q] = __byte_perm(r[q], 0u, 0x3120);
                                if constexpr (C::INT8) r[q] ^= 0x80808080u;
                            }
#pragma unroll
                            for (int h = 0; h < 2; ++h) {  // chunk 2 c2 + h: r[2h] tokens 0-7, r[2h+1] 8-15
                                const int n = 4 * c2 + 2 * h;
                                mma_f16(o[n], pa, widen_lo<C::INT8>(r[2 * h]),
                                        widen_lo<C::INT8>(r[2 * h + 1]));
                                mma_f16(o[n + 1], pa, widen_hi<C::INT8>(r[2 * h]),
                                        widen_hi<C::INT8>(r[2 * h + 1]));
                            }
                        }
                        continue;
                    }
                    uint32_t pa[4];
                    pa[0] = pack_bf16(sc[2 * kk][0], sc[2 * kk][1]);
                    pa[1] = pack_bf16(sc[2 * kk][2], sc[2 * kk][3]);
                    pa[2] = pack_bf16(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
                    pa[3] = pack_bf16(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
                    const int tok = c0 + kk * 16 + (lm_mi & 1) * 8 + lm_i;
#pragma unroll
                    for (int dp = 0; dp < D / 16; ++dp) {
                        const int h = dp / 4;
                        const int vc = (dp % 4) * 2 + (lm_mi >> 1);
                        uint32_t b0, b1, b2, b3;
                        ldsm_x4_t(v_u + row_off(tok, h) + ((vc ^ lm_i) << 4), b0, b1, b2, b3);
                        mma_bf16(o[2 * dp], pa, b0, b1);
                        mma_bf16(o[2 * dp + 1], pa, b2, b3);
                    }
                }
            }
        }

        // ---- release the stage
        if (zeroed) fence_proxy_async();
        __syncwarp();
        mbar_arrive(smem_u32(&empty_bar[s]));

        if (!(dsc.flags & kSegEnd)) continue;

        // ================================================ end of a piece: combine
        if constexpr (C::INT8) {
            // every output column of a row got 1152 * (the row's f16 P sum)
            float ct0 = cp0 + __shfl_xor_sync(0xffffffffu, cp0, 1);
            ct0 += __shfl_xor_sync(0xffffffffu, ct0, 2);
            float ct1 = cp1 + __shfl_xor_sync(0xffffffffu, cp1, 1);
            ct1 += __shfl_xor_sync(0xffffffffu, ct1, 2);
            ct0 *= kI8Bias;
            ct1 *= kI8Bias;
#pragma unroll
            for (int n = 0; n < D / 8; ++n) {
                o[n][0] -= ct0;
                o[n][1] -= ct0;
                o[n][2] -= ct1;
                o[n][3] -= ct1;
            }
        }
        float lt0 = l0 + __shfl_xor_sync(0xffffffffu, l0, 1);
        lt0 += __shfl_xor_sync(0xffffffffu, lt0, 2);
        float lt1 = l1 + __shfl_xor_sync(0xffffffffu, l1, 1);
        lt1 += __shfl_xor_sync(0xffffffffu, lt1, 2);
        if (C::TG > 1) {
            constexpr int RS = D + 2;  // row stride: D outputs, then m and l
            const int grp = hgi * C::MT + mt;
            if (tg > 0) {
                float* cb = comb + ((tg - 1) * C::HG * C::MT + grp) * C::ROWS * RS;
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    *reinterpret_cast<float2*>(cb + gid * RS + n * 8 + tig * 2) =
                        make_float2(o[n][0], o[n][1]);
                    if (C::ROWS16)
                        *reinterpret_cast<float2*>(cb + (gid + 8) * RS + n * 8 + tig * 2) =
                            make_float2(o[n][2], o[n][3]);
                }
                if (tig == 0) {
                    cb[gid * RS + D] = m0;
                    cb[gid * RS + D + 1] = lt0;
                    if (C::ROWS16) {
                        cb[(gid + 8) * RS + D] = m1;
                        cb[(gid + 8) * RS + D + 1] = lt1;
                    }
                }
            }
            mbar_arrive(smem_u32(&comb_bar));
            if (!mbar_wait_warp(smem_u32(&comb_bar), comb_phase)) {
                if (lane == 0) {
                    latch_error(a.err, PGD_ERR_TIMEOUT);
                    aborted = 1;
                }
                break;
            }
            comb_phase ^= 1u;
            if (tg == 0) {
#pragma unroll 1
                for (int t2 = 1; t2 < C::TG; ++t2) {
                    const float* cb = comb + ((t2 - 1) * C::HG * C::MT + grp) * C::ROWS * RS;
                    const float om0 = cb[gid * RS + D], ol0 = cb[gid * RS + D + 1];
                    const float nm0 = fmaxf(m0, om0);
                    const float nb0 = nm0 == -INFINITY ? 0.f : nm0;
                    const float sa0 = fast_exp2(m0 - nb0), sb0 = fast_exp2(om0 - nb0);
                    m0 = nm0;
                    lt0 = lt0 * sa0 + ol0 * sb0;
                    float sa1 = 1.f, sb1 = 0.f;
                    if (C::ROWS16) {
                        const float om1 = cb[(gid + 8) * RS + D], ol1 = cb[(gid + 8) * RS + D + 1];
                        const float nm1 = fmaxf(m1, om1);
                        const float nb1 = nm1 == -INFINITY ? 0.f : nm1;
                        sa1 = fast_exp2(m1 - nb1);
                        sb1 = fast_exp2(om1 - nb1);
                        m1 = nm1;
                        lt1 = lt1 * sa1 + ol1 * sb1;
                    }
#pragma unroll
                    for (int n = 0; n < D / 8; ++n) {
                        const float2 u = *reinterpret_cast<const float2*>(cb + gid * RS + n * 8 +
                                                                          tig * 2);
                        o[n][0] = o[n][0] * sa0 + u.x * sb0;
                        o[n][1] = o[n][1] * sa0 + u.y * sb0;
                        if (C::ROWS16) {
                            const float2 w = *reinterpret_cast<const float2*>(
                                cb + (gid + 8) * RS + n * 8 + tig * 2);
                            o[n][2] = o[n][2] * sa1 + w.x * sb1;
                            o[n][3] = o[n][3] * sa1 + w.y * sb1;
                        }
                    }
                }
            }
            mbar_arrive(smem_u32(&comb_bar));
            if (!mbar_wait_warp(smem_u32(&comb_bar), comb_phase)) {
                if (lane == 0) {
                    latch_error(a.err, PGD_ERR_TIMEOUT);
                    aborted = 1;
                }
                break;
            }
            comb_phase ^= 1u;
        }
        if (tg != 0) continue;

        // ---- write: whole run -> out (bf16); split run -> partial (fp32) + lse
        // a row that saw no token (window / causal range outside this piece, or
        // a query before the sequence start) has l = 0: zeros, lse = -inf
        const float inv0 = seg_bad ? NAN : (lt0 > 0.f ? v_mul / lt0 : 0.f);
        const float inv1 = seg_bad ? NAN : (lt1 > 0.f ? v_mul / lt1 : 0.f);
        if (!(dsc.flags & kSegPartial)) {
            __nv_bfloat16* o0 = static_cast<__nv_bfloat16*>(a.out) +
                                (row0_ok ? qrow_offset(a, dsc.b, kvh, row0) : 0);
            __nv_bfloat16* o1 = static_cast<__nv_bfloat16*>(a.out) +
                                (row1_ok ? qrow_offset(a, dsc.b, kvh, row1) : 0);
            if constexpr (C::FP8) {
                // n-tiles 2c, 2c+1 hold d = 16 c + 4 tig + (0, 2) and (1, 3)
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    if (row0_ok)
                        *reinterpret_cast<uint2*>(o0 + 16 * c + 4 * tig) =
                            make_uint2(pack_bf16(o[2 * c][0] * inv0, o[2 * c + 1][0] * inv0),
                                       pack_bf16(o[2 * c][1] * inv0, o[2 * c + 1][1] * inv0));
                    if (row1_ok)
                        *reinterpret_cast<uint2*>(o1 + 16 * c + 4 * tig) =
                            make_uint2(pack_bf16(o[2 * c][2] * inv1, o[2 * c + 1][2] * inv1),
                                       pack_bf16(o[2 * c][3] * inv1, o[2 * c + 1][3] * inv1));
                }
            } else {
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    if (row0_ok)
                        *reinterpret_cast<uint32_t*>(o0 + n * 8 + tig * 2) =
                            pack_bf16(o[n][0] * inv0, o[n][1] * inv0);
                    if (row1_ok)
                        *reinterpret_cast<uint32_t*>(o1 + n * 8 + tig * 2) =
                            pack_bf16(o[n][2] * inv1, o[n][3] * inv1);
                }
            }
            continue;
        }
        // The pieces of run [t0, t0 + n_b): with P <= N every span holds at
        // least one tile, so they are CTAs c0..c1; with P > N every span holds
        // at most one tile, so piece k is the owner of tile t0 + k.
        const int64_t t0 = dsc.run_start;
        const int64_t N = ss.n_total, P = ss.parts;
        const int64_t c0 = span_owner(t0, N, P);
        const int npieces = P > N ? dsc.n_b : (int)(span_owner(t0 + dsc.n_b - 1, N, P) - c0 + 1);
        const bool first_is_tail = P <= N && span_begin(c0, N, P) < t0;
        const int prow0 = hgi * rows + row0, prow1 = hgi * rows + row1;  // rows of the piece
        const int64_t slot = (int64_t)blockIdx.x * 2 + ((dsc.flags & kSegSlot1) ? 1 : 0);
        {
            float* po = a.part_o + slot * piece_rows * D;
            if constexpr (C::FP8) {
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
                    if (row0_ok)
                        *reinterpret_cast<float4*>(po + (int64_t)prow0 * D + 16 * c + 4 * tig) =
                            make_float4(o[2 * c][0] * inv0, o[2 * c + 1][0] * inv0,
                                        o[2 * c][1] * inv0, o[2 * c + 1][1] * inv0);
                    if (row1_ok)
                        *reinterpret_cast<float4*>(po + (int64_t)prow1 * D + 16 * c + 4 * tig) =
                            make_float4(o[2 * c][2] * inv1, o[2 * c + 1][2] * inv1,
                                        o[2 * c][3] * inv1, o[2 * c + 1][3] * inv1);
                }
            } else {
#pragma unroll
                for (int n = 0; n < D / 8; ++n) {
                    if (row0_ok)
                        *reinterpret_cast<float2*>(po + (int64_t)prow0 * D + n * 8 + tig * 2) =
                            make_float2(o[n][0] * inv0, o[n][1] * inv0);
                    if (row1_ok)
                        *reinterpret_cast<float2*>(po + (int64_t)prow1 * D + n * 8 + tig * 2) =
                            make_float2(o[n][2] * inv1, o[n][3] * inv1);
                }
            }
            if (tig == 0) {
                float* pl = a.part_lse + slot * piece_rows;
                if (row0_ok)
                    pl[prow0] = seg_bad ? 0.f : (lt0 > 0.f ? m0 + fast_log2(lt0) : -INFINITY);
                if (row1_ok)
                    pl[prow1] = seg_bad ? 0.f : (lt1 > 0.f ? m1 + fast_log2(lt1) : -INFINITY);
            }
        }
        if constexpr (C::SEP) continue;  // merged by the run-merge kernel after this one
        // Publish the partial and count it; the warp that brings the count to
        // the number of pieces sets it back to zero and flips the run's flag
        // bit.  Shared merge (cooperative launch, a merge of more than six
        // batches of loads whose rows split): every piece's warp, after its tile
        // loop, waits for the flip and merges a share of the rows.  Otherwise
        // the last warp merges all rows.  No second kernel, no atomics at the
        // end.
        const int pre = __shfl_sync(0xffffffffu, pre_cnt, 0);
        // final piece, every other piece counted: no fence, no arrival (this
        // warp merges after its loop, reading its own rows after __syncwarp)
        const bool known_last = !C::SHARE && it == n_tiles - 1 &&
                                (pre & kRunCountMask) == npieces - 1;
        if (!known_last) __threadfence();
        __syncwarp();
        if (lane == 0) {
            int* word = a.counters + ((int64_t)dsc.b * a.hkv + kvh) * C::MT + mt;
            const int js = (dsc.flags & kSegSlot1) ? 1 : 0;  // one piece per partial slot and CTA
            const int old = known_last ? pre : atomicAdd(word, 1);
            const int flag = (old >> kRunFlagShift) & 1;  // cannot flip before I arrive
            const bool last = (old & kRunCountMask) == npieces - 1;

            if constexpr (C::SHARE) {
                const int nr = min(rows - mt * 16, C::ROWS);
                constexpr int RPP = 32 / (D / 4);          // rows per merge pass
                const bool shared = min(npieces, nr) >= 2 &&
                                    (nr + RPP - 1) / RPP * npieces > kShareMinLoads;
                if (last) {
                    if (shared) {
                        __threadfence();  // every piece's partial is visible before the flip
                        st_release(word, (flag ^ 1) << kRunFlagShift);
                    } else {
                        *word = (flag ^ 1) << kRunFlagShift;  // nobody waits on this flip
                    }
                }
                if (shared) {
                    const int k = P > N ? (int)(ss.r0 - t0) : (int)(blockIdx.x - c0);
                    jobs[warp][js] =
                        MergeJob{t0, c0, npieces, first_is_tail ? 1 : 0, dsc.b, kvh, k, flag};
                } else if (last) {
                    jobs[warp][js] =
                        MergeJob{t0, c0, npieces, first_is_tail ? 1 : 0, dsc.b, kvh, -1, 0};
                }
            } else if (last) {
                *word = (flag ^ 1) << kRunFlagShift;
                jobs[warp][js] =
                    MergeJob{t0, c0, npieces, first_is_tail ? 1 : 0, dsc.b, kvh, -1, 0};
            }
        }
    }
    // ---- merge the split runs recorded above
    if constexpr (C::SEP) return;  // (none: the run-merge kernel merges them)
    if (__any_sync(0xffffffffu, aborted)) return;
    const int r_mine = mt * 16, r_end = min(rows, r_mine + C::ROWS);
#pragma unroll 1
    for (int j = 0; j < 2; ++j) {
        const MergeJob jb = jobs[warp][j];
        if (jb.b < 0) continue;
        int m_lo = r_mine, m_hi = r_end;
        if (C::SHARE && jb.k >= 0) {
            // the first min(pieces, rows) pieces' warps each merge a share of
            // the rows, once every piece is in
            const int nr = r_end - r_mine;
            const int nm = min(jb.npieces, nr);
            if (jb.k >= nm) continue;
            m_lo = r_mine + jb.k * nr / nm;
            m_hi = r_mine + (jb.k + 1) * nr / nm;
            int ok = 1;
            if (lane == 0)
                ok = wait_flip(a.counters + ((int64_t)jb.b * a.hkv + jb.kvh) * C::MT + mt,
                               jb.flag) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) latch_error(a.err, PGD_ERR_TIMEOUT);
                return;
            }
        }
        __threadfence();
        if (m_hi - m_lo <= RPP)
            merge_pieces<C, true>(a, jb.t0, ss.n_total, ss.parts, jb.c0, jb.npieces,
                                  jb.first_is_tail != 0, hgi, m_lo, m_hi, jb.b, jb.kvh);
        else
            merge_pieces<C, false>(a, jb.t0, ss.n_total, ss.parts, jb.c0, jb.npieces,
                                   jb.first_is_tail != 0, hgi, m_lo, m_hi, jb.b, jb.kvh);
    }
}

// Co-resident CTAs per SM of one instantiation on `dev` (the current device),
// after setting its dynamic shared memory limit there.  The attribute applies
// to the current device only, so both are kept per device; the first launch
// on a device does the set-up under a lock (two host threads may make their
// first launch together), later ones read one atomic.  0 on failure.
template <class C>
int resident_per_sm(int dev, cudaError_t* err) {
    static std::atomic<int> per_sm[kMaxDevices] = {};
    static std::mutex mu;
    *err = cudaSuccess;
    if (dev < 0 || dev >= kMaxDevices) {
        *err = cudaErrorInvalidDevice;
        return 0;
    }
    int n = per_sm[dev].load(std::memory_order_acquire);
    if (n > 0) return n;
    std::lock_guard<std::mutex> lock(mu);
    n = per_sm[dev].load(std::memory_order_relaxed);
    if (n > 0) return n;
    cudaError_t e = cudaFuncSetAttribute(decode_tma_kernel<C>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_tma_kernel<C>, C::THREADS,
                                                          C::SMEM_BYTES);
    if (e == cudaSuccess && n < 1) e = cudaErrorLaunchOutOfResources;
    if (e != cudaSuccess) {
        *err = e;
        return 0;
    }
    per_sm[dev].store(n, std::memory_order_release);
    return n;
}

template <class C>
cudaError_t launch_cfg(const DecodeArgs& a, const CUtensorMap& mk, const CUtensorMap& mv,
                       int num_sms, int dev, cudaStream_t s) {
    cudaError_t e0;
    const int per_sm = resident_per_sm<C>(dev, &e0);
    if (per_sm < 1) return e0;
    if constexpr (C::SHARE) {
        // the shared merge waits on other CTAs: only a grid resident at once,
        // launched cooperatively
        if (a.num_parts > per_sm * num_sms) return cudaErrorCooperativeLaunchTooLarge;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(a.num_parts);
        cfg.blockDim = dim3(C::THREADS);
        cfg.dynamicSmemBytes = C::SMEM_BYTES;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_tma_kernel<C>, mk, mv, a);
        if (e != cudaSuccess) return e;
    } else {
        decode_tma_kernel<C><<<a.num_parts, C::THREADS, C::SMEM_BYTES, s>>>(mk, mv, a);
    }
    return cudaGetLastError();
}

// Token groups per tile of t tokens for (HG, MT): up to 8 consumer warps, >= 16
// tokens each.
constexpr int token_groups(int t, int hg, int mt) {
    const int by_tokens = t / 16;
    const int by_warps = 8 / (hg * mt) > 0 ? 8 / (hg * mt) : 1;
    return by_tokens < by_warps ? by_tokens : by_warps;
}

template <int D, int HG, int MT, bool R16, bool FP8, int MV, bool INT8, bool PB>
cudaError_t launch_hg(const DecodeArgs& a, const Pool& p, cudaStream_t s) {
    constexpr int TG = token_groups((FP8 ? 256 : 128) / HG, HG, MT);
    const int idx = HG == 1 ? 0 : HG == 2 ? 1 : HG == 4 ? 2 : 3;
    return launch_cfg<Cfg<D, HG, MT, TG, R16, FP8, MV, INT8, PB>>(
        a, p.tmap_k[idx], p.tmap_v[idx], p.num_sms, p.device, s);
}

template <int D, int MT, bool R16, bool FP8, int MV, bool INT8, bool PB>
cudaError_t launch_mt(const DecodeArgs& a, const Pool& p, cudaStream_t s) {
    switch (a.hg) {
        case 1: return launch_hg<D, 1, MT, R16, FP8, MV, INT8, PB>(a, p, s);
        case 2: return launch_hg<D, 2, MT, R16, FP8, MV, INT8, PB>(a, p, s);
        case 4:
            if constexpr (MT <= 2) return launch_hg<D, 4, MT, R16, FP8, MV, INT8, PB>(a, p, s);
            break;
        case 8:
            if constexpr (MT == 1) return launch_hg<D, 8, MT, R16, FP8, MV, INT8, PB>(a, p, s);
            break;
    }
    return cudaErrorInvalidValue;
}

// FP8: 8-bit K/V pages (head_dim 128 only), INT8: of int8 codes (else e4m3),
// PB: with a scale per block and KV head (else per KV head).
// MV: merge variant (see Cfg).  The shared variant (1) returns
// cudaErrorCooperativeLaunchTooLarge when the grid cannot be resident at once.
template <int D, bool FP8, int MV, bool INT8 = false, bool PB = false>
cudaError_t launch_tma_d(const DecodeArgs& a, const Pool& p, cudaStream_t s) {
    const int rows = a.q_len * a.group;  // query rows per KV head
    if (rows <= 8) return launch_mt<D, 1, false, FP8, MV, INT8, PB>(a, p, s);
    if (rows <= 16) return launch_mt<D, 1, true, FP8, MV, INT8, PB>(a, p, s);
    if (rows <= 32) return launch_mt<D, 2, true, FP8, MV, INT8, PB>(a, p, s);
    if (rows <= 48) return launch_mt<D, 3, true, FP8, MV, INT8, PB>(a, p, s);
    return launch_mt<D, 4, true, FP8, MV, INT8, PB>(a, p, s);
}

}  // namespace tma
}  // namespace pgd
