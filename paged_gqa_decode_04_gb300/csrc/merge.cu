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
// One CTA per sequence; used after the CUDA-core kernel, whose units are single
// KV heads (a run is one (sequence, KV head) pair).  Runs that were not split
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

}  // namespace

cudaError_t launch_merge(const DecodeArgs& a, int dtype, cudaStream_t s) {
    if (a.B == 0) return cudaSuccess;
    if (dtype == PGD_F32) merge_kernel<float><<<a.B, kMergeThreads, 0, s>>>(a);
    else merge_kernel<__nv_bfloat16><<<a.B, kMergeThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pgd
