// Log-sum-exp merge of split-KV partial results, and the rows no decode CTA
// writes (empty and invalid sequences).
//
// A piece of a (sequence, KV head) run computed by one CTA leaves, per query
// row, its normalised output o_c and its base-2 log-sum-exp
// lse_c = m_c + log2(l_c).  The full softmax over the union of the pieces is
//
//     lse* = log2 sum_c 2^lse_c,    out = sum_c 2^(lse_c - lse*) o_c,
//
// evaluated with the largest lse_c subtracted first.  This is the combine step
// of split-KV decoding (FlashDecoding, listed among the vLLM optimisations in
// "Modern LLM Inference ...", section 8.3); it keeps the softmax exact, as the
// same notes say of FlashAttention's online softmax.
//
// merge_kernel: one CTA per sequence; used after the CUDA-core kernel, whose
// units are single KV heads (a run is one (sequence, KV head) pair).  Runs that were not split
// are left alone (the decode kernel wrote them), sequences of length 0 get
// zeros, and sequences whose length is out of range get NaN and latch
// PGD_ERR_SEQ_LEN.
#include <cuda_bf16.h>
#include <math.h>

#include "partition.cuh"

namespace pgd {
namespace {

constexpr int kMergeThreads = 128;

template <typename T>
__device__ __forceinline__ T cvt(float x);
template <>
__device__ __forceinline__ float cvt<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 cvt<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <typename T>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(DecodeArgs a) {
    const int b = blockIdx.x;
    const int D = a.d;
    const int G = a.group;
    T* __restrict__ out_b = static_cast<T*>(a.out) + (int64_t)b * a.hq * D;
    const int L = a.seq_lens[b];

    if (!seq_len_ok(L, a.max_blocks, a.block_size) || L == 0) {
        const float fill = (L == 0) ? 0.f : NAN;
        if (L != 0 && threadIdx.x == 0) latch_error(a.err, PGD_ERR_SEQ_LEN);
        for (int i = threadIdx.x; i < a.hq * D; i += blockDim.x) out_b[i] = cvt<T>(fill);
        return;
    }

    const int64_t N = a.tile_base[a.B];
    const int64_t P = a.num_parts;
    const int n_b = tiles_of(L, a.max_blocks, a.block_size, a.tile_tokens, 1, 0);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int nwarps = blockDim.x / 32;

    for (int r = warp; r < a.hq; r += nwarps) {
        const int kvh = r / G, j = r % G;
        const int64_t t0 = a.tile_base[b] + (int64_t)kvh * n_b;
        const int64_t c0 = span_owner(t0, N, P);
        const int64_t c1 = span_owner(t0 + n_b - 1, N, P);
        if (c0 == c1) continue;  // written whole by the decode kernel

        // CTAs whose span is empty (more CTAs than tiles) wrote nothing: skip them.
        float lse_max = -INFINITY;
        for (int64_t c = c0; c <= c1; ++c) {
            const int64_t sb = span_begin(c, N, P);
            if (sb == span_begin(c + 1, N, P)) continue;
            const int64_t slot = c * 2 + (sb < t0 ? 1 : 0);
            lse_max = fmaxf(lse_max, a.part_lse[slot * G + j]);
        }
        float wsum = 0.f;
        for (int d = lane; d < D; d += 32) {
            float acc = 0.f;
            wsum = 0.f;
            for (int64_t c = c0; c <= c1; ++c) {
                const int64_t sb = span_begin(c, N, P);
                if (sb == span_begin(c + 1, N, P)) continue;
                const int64_t slot = c * 2 + (sb < t0 ? 1 : 0);
                const float w = fast_exp2(a.part_lse[slot * G + j] - lse_max);
                wsum += w;
                acc += w * a.part_o[(slot * G + j) * D + d];
            }
            out_b[(int64_t)r * D + d] = cvt<T>(acc / wsum);
        }
    }
}

constexpr int kRunMergeMaxThreads = 256;
constexpr int kRunMergeItems = 2;   // (row, 4 columns) items a thread takes at once
constexpr int kRunMergePieces = 4;  // pieces whose loads are issued before any fold (the
                                    // decode kernel's merge batch, kPieceBatch)

// (M, W, acc) holds acc = sum_k 2^(lse_k - M) o_k and W = sum_k 2^(lse_k - M);
// add piece (e, v), keeping the larger exponent as the reference.  The same
// explicit roundings as the decode kernel's own merge (a fused multiply-add of
// the rescaled sum and the rounded product), so that a run merged here or
// inside the decode kernel gives the same bits.
__device__ __forceinline__ void fold_piece(float& M, float& W, float4& acc, float e, float4 v) {
    const float nm = fmaxf(M, e);
    const float base = nm == -INFINITY ? 0.f : nm;
    const float sa = fast_exp2(M - base), sb = fast_exp2(e - base);
    M = nm;
    W = __fmaf_rn(W, sa, __fmul_rn(1.f, sb));
    acc.x = __fmaf_rn(acc.x, sa, __fmul_rn(v.x, sb));
    acc.y = __fmaf_rn(acc.y, sa, __fmul_rn(v.y, sb));
    acc.z = __fmaf_rn(acc.z, sa, __fmul_rn(v.z, sb));
    acc.w = __fmaf_rn(acc.w, sa, __fmul_rn(v.w, sb));
}

// Span arithmetic of partition.cuh with a 32-bit unsigned division whenever
// the numerator and divisor fit (every shape this merge is planned for): the
// 64-bit division routine is most of the time between the tile table's
// arrival and the partial loads.
__device__ __forceinline__ int64_t floor_div(int64_t num, int64_t den) {
    if (num >= 0 && num <= 0x7fffffff && den <= 0x7fffffff)
        return (int64_t)((uint32_t)num / (uint32_t)den);
    return num / den;
}
__device__ __forceinline__ int64_t owner_of(int64_t x, int64_t N, int64_t P) {
    return floor_div((x + 1) * P - 1, N);  // span_owner
}
__device__ __forceinline__ int64_t begin_of(int64_t c, int64_t N, int64_t P) {
    return floor_div(c * N, P);  // span_begin
}

// Merge of the split runs the TMA decode kernel's separate-merge variant leaves
// (its pieces only write partials: when runs cover a few spans, the merges a
// decode would fuse all wait at the end of the step for partials written just
// before).  One CTA per (run, head of the unit); a thread takes two (row, 4
// columns) items and, for four pieces at a time, first issues every load and
// then folds the pieces in order, so one batch costs one round trip.  The
// CTAs (at most 256 threads) fit the GPU in one wave at the shapes this merge
// is planned for.  The pieces and their partial slots follow from the spans
// exactly as in the decode kernel: with P <= N spans every span holds a tile,
// so the pieces are CTAs c0 .. c1; with P > N each holds at most one, so piece
// k is the owner of tile t0 + k.  Runs held whole by one span, and sequences
// without tiles, were written by the decode kernel and are left alone.
__global__ void __launch_bounds__(kRunMergeMaxThreads) merge_runs_kernel(DecodeArgs a) {
    constexpr int D = 128;
    constexpr int CPR = D / 4;  // float4 items per row
    constexpr int I = kRunMergeItems, K = kRunMergePieces;
    const int b = blockIdx.x / a.units, u = blockIdx.x % a.units, hgi = blockIdx.y;
    // all from the decode's tile table in device memory (the lengths may sit in
    // host memory): a sequence spans units * (tiles + W) virtual slots, or none
    const int64_t N = a.tile_base[a.B], P = a.tile_base[a.B + 1];
    const int W = (int)a.tile_base[a.B + 2];
    const int64_t slots = a.tile_base[b + 1] - a.tile_base[b];
    if (slots == 0) return;
    const int n_b = (int)(slots / a.units) - W;
    const int64_t t0 = a.tile_base[b] + (int64_t)u * (n_b + W) + W;  // run's first real tile
    const int64_t c0 = owner_of(t0, N, P);
    const int64_t c1 = owner_of(t0 + n_b - 1, N, P);
    if (c0 == c1) return;
    const bool dense = P <= N;
    const int npieces = dense ? (int)(c1 - c0 + 1) : n_b;
    const bool first_is_tail = dense && begin_of(c0, N, P) < t0;
    const int G = a.group, rows = a.q_len * G;
    const int piece_rows = a.hg * rows;
    const int kvh = u * a.hg + hgi;
    const int n_items = rows * CPR;
    for (int base = threadIdx.x; base < n_items; base += blockDim.x * I) {
        int64_t pr[I];
        int col[I];
        bool ok[I];
        float M[I], Wt[I];
        float4 acc[I];
#pragma unroll
        for (int i = 0; i < I; ++i) {
            const int item = base + i * blockDim.x;
            ok[i] = item < n_items;
            const int r = ok[i] ? item / CPR : 0;
            col[i] = ok[i] ? (item % CPR) * 4 : 0;
            pr[i] = (int64_t)hgi * rows + r;
            M[i] = -INFINITY;
            Wt[i] = 0.f;
            acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int k0 = 0; k0 < npieces; k0 += K) {
            int64_t sl[K];  // partial slots of this batch's pieces
#pragma unroll
            for (int j = 0; j < K; ++j) {
                const int k = k0 + j < npieces ? k0 + j : npieces - 1;
                const int64_t c = dense ? c0 + k : owner_of(t0 + k, N, P);
                sl[j] = c * 2 + ((first_is_tail && k == 0) ? 1 : 0);
            }
            float e[I][K];
            float4 v[I][K];
#pragma unroll
            for (int i = 0; i < I; ++i) {
#pragma unroll
                for (int j = 0; j < K; ++j) {
                    const bool ld = ok[i] && k0 + j < npieces;
                    e[i][j] = ld ? __ldg(a.part_lse + sl[j] * piece_rows + pr[i]) : -INFINITY;
                    v[i][j] = ld ? __ldg(reinterpret_cast<const float4*>(
                                       a.part_o + (sl[j] * piece_rows + pr[i]) * D + col[i]))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
            // every entry of the batch is folded, those past the last piece as
            // (-inf, 0): the decode kernel's merge folds its batches of four the
            // same way (kPieceBatch)
#pragma unroll
            for (int i = 0; i < I; ++i) {
#pragma unroll
                for (int j = 0; j < K; ++j) fold_piece(M[i], Wt[i], acc[i], e[i][j], v[i][j]);
            }
        }
#pragma unroll
        for (int i = 0; i < I; ++i) {
            if (!ok[i]) continue;
            const int r = (base + i * blockDim.x) / CPR;
            const float w = Wt[i] > 0.f ? 1.f / Wt[i] : 0.f;  // no token in any piece: zeros
            __nv_bfloat162 lo = __floats2bfloat162_rn(acc[i].x * w, acc[i].y * w);
            __nv_bfloat162 hi = __floats2bfloat162_rn(acc[i].z * w, acc[i].w * w);
            uint2 pk;
            pk.x = *reinterpret_cast<uint32_t*>(&lo);
            pk.y = *reinterpret_cast<uint32_t*>(&hi);
            const int64_t orow = ((int64_t)b * a.q_len + r / G) * a.hq + (int64_t)kvh * G + r % G;
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + orow * D + col[i]) = pk;
        }
    }
}

}  // namespace

cudaError_t launch_merge_runs(const DecodeArgs& a, cudaStream_t s) {
    if (a.B == 0 || a.d != 128) return a.B == 0 ? cudaSuccess : cudaErrorInvalidValue;
    // threads for two items each, a multiple of 32 (items = rows * 32)
    const int items = a.q_len * a.group * (128 / 4);
    int threads = (items / kRunMergeItems + 31) / 32 * 32;
    threads = threads < kRunMergeMaxThreads ? threads : kRunMergeMaxThreads;
    merge_runs_kernel<<<dim3((unsigned)(a.B * a.units), (unsigned)a.hg), threads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_merge(const DecodeArgs& a, int dtype, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    if (dtype == PGD_F32) merge_kernel<float><<<a.B, kMergeThreads, 0, s>>>(a);
    else merge_kernel<__nv_bfloat16><<<a.B, kMergeThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pgd
