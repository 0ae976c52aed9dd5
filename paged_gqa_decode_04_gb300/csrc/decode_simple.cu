// Plain CUDA-core decode kernel: float32 and bfloat16 pools, any block size.
//
// One CTA per span of the tile sequence (see partition.cuh).  For each piece of
// a (sequence, KV head) run inside the span, the four warps take the group's
// query rows in turn; a warp walks the piece token by token, lanes splitting
// the head dimension, with a running max / running sum (online) softmax:
//
//     m' = max(m, s_t);  l' = l 2^(m - m') + 2^(s_t - m');
//     o' = o 2^(m - m') + 2^(s_t - m') v_t                   (base-2 logits)
//
// which is the exact softmax of the Attention(Q,K,V) equation evaluated in one
// pass ("Modern LLM Inference ...", "Linear Attention vs. FlashAttention
// (Online Softmax)": FlashAttention keeps the softmax exact).  This kernel is
// the float32 path; bfloat16 and 8-bit pages take the TMA pipeline of
// decode_tma.cuh.
#include <cuda_bf16.h>
#include <math.h>

#include "partition.cuh"

namespace pgd {
namespace {

constexpr int kSimpleThreads = 128;
constexpr int kSimpleWarps = kSimpleThreads / 32;

template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
    return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

template <int D, typename T>
__global__ void __launch_bounds__(kSimpleThreads) decode_simple_kernel(DecodeArgs a) {
    constexpr int DPL = D / 32;  // head-dim elements per lane
    __shared__ int64_t scratch[kSimpleThreads];
    __shared__ SpanStart ss;
    find_span_start(a.seq_lens, a.B, a.units, a.tile_tokens, 1, 0, a.max_blocks, a.block_size,
                    a.num_parts, 1, scratch, &ss, a.tile_base);
    if (ss.r0 >= ss.r1) return;

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const T* __restrict__ q = static_cast<const T*>(a.q);
    const T* __restrict__ kp = static_cast<const T*>(a.k_pool);
    const T* __restrict__ vp = static_cast<const T*>(a.v_pool);
    T* __restrict__ out = static_cast<T*>(a.out);
    const int G = a.group;

    TileCursor cur = cursor_at(ss, a.seq_lens, a.units, a.tile_tokens, 1, 0, a.max_blocks,
                               a.block_size);
    int64_t x = ss.r0;
    while (x < ss.r1) {
        const int64_t run_end = cur.run_start + cur.n_b;
        const int64_t piece_end = run_end < ss.r1 ? run_end : ss.r1;
        const int flags = segment_flags(x, cur.run_start, cur.n_b, ss.r0, ss.r1);
        const int L = a.seq_lens[cur.b];
        const int i_end = (int)(piece_end - cur.run_start);
        const int t_begin = cur.i * a.tile_tokens;
        const int t_end = min(L, i_end * a.tile_tokens);
        const int b = cur.b, kvh = cur.unit;  // one KV head per unit here

        for (int j = warp; j < G; j += kSimpleWarps) {
            const int h = kvh * G + j;
            float qf[DPL], o[DPL];
            const T* qrow = q + ((int64_t)b * a.hq + h) * D + lane * DPL;
#pragma unroll
            for (int e = 0; e < DPL; ++e) {
                qf[e] = ld_f(qrow + e);
                o[e] = 0.f;
            }
            float m = -INFINITY, l = 0.f;
            bool bad = false;
            for (int t = t_begin; t < t_end; ++t) {
                const int64_t phys = a.block_table[(int64_t)b * a.max_blocks + t / a.block_size];
                if (phys < 0 || phys >= a.num_blocks) {
                    bad = true;
                    continue;
                }
                const int64_t row =
                    ((phys * a.block_size + t % a.block_size) * a.hkv + kvh) * (int64_t)D +
                    lane * DPL;
                float dot = 0.f;
#pragma unroll
                for (int e = 0; e < DPL; ++e) dot += qf[e] * ld_f(kp + row + e);
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
                const float s = dot * a.scale_log2;
                const float m_new = fmaxf(m, s);
                const float alpha = fast_exp2(m - m_new);
                const float p = fast_exp2(s - m_new);
                l = l * alpha + p;
#pragma unroll
                for (int e = 0; e < DPL; ++e) o[e] = o[e] * alpha + p * ld_f(vp + row + e);
                m = m_new;
            }
            if (bad && lane == 0) latch_error(a.err, PGD_ERR_BLOCK_ID);
            const float inv = bad ? NAN : 1.f / l;
            if (!(flags & kSegPartial)) {
                T* orow = out + ((int64_t)b * a.hq + h) * D + lane * DPL;
#pragma unroll
                for (int e = 0; e < DPL; ++e) orow[e] = from_f<T>(o[e] * inv);
            } else {
                const int64_t slot = (int64_t)blockIdx.x * 2 + ((flags & kSegSlot1) ? 1 : 0);
                float* prow = a.part_o + (slot * G + j) * D + lane * DPL;
#pragma unroll
                for (int e = 0; e < DPL; ++e) prow[e] = o[e] * inv;
                if (lane == 0) a.part_lse[slot * G + j] = bad ? 0.f : m + fast_log2(l);
            }
        }
        // advance past this piece
        x = piece_end;
        cur.i = i_end - 1;
        cursor_next(cur, a.seq_lens, a.B, a.units, a.tile_tokens, 1, 0, a.max_blocks,
                    a.block_size);
    }
}

}  // namespace

cudaError_t launch_decode_simple(const DecodeArgs& a, int dtype, cudaStream_t s) {
    dim3 grid(a.num_parts), block(kSimpleThreads);
    if (dtype == PGD_F32) {
        if (a.d == 64) decode_simple_kernel<64, float><<<grid, block, 0, s>>>(a);
        else decode_simple_kernel<128, float><<<grid, block, 0, s>>>(a);
    } else {
        if (a.d == 64) decode_simple_kernel<64, __nv_bfloat16><<<grid, block, 0, s>>>(a);
        else decode_simple_kernel<128, __nv_bfloat16><<<grid, block, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace pgd
