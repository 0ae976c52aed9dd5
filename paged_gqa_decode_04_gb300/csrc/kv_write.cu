// Device side of the KV write path (include/paged_kv_manager.h): store the
// new tokens' K/V rows into their pool slots, and copy whole blocks for
// copy-on-write.  Both are plain coalesced copies in 16-byte vectors: a token
// row (Hkv * D elements) and a block (block_size rows) are contiguous in the
// pool [num_blocks, block_size, Hkv, D].
#include <stdint.h>

#include "paged_kv_manager.h"
#include "pgd_internal.h"

namespace pgd {
namespace {

constexpr int kWriteThreads = 256;

// One warp per new token: copy its K row and V row (row_vec 16-byte vectors
// each) to slot slot_mapping[i].
__global__ void __launch_bounds__(kWriteThreads)
    append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                  const int32_t* __restrict__ slots, int n, int64_t n_slots, int row_vec,
                  uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, int* err) {
    const int warp = (blockIdx.x * kWriteThreads + threadIdx.x) / 32;
    const int lane = threadIdx.x % 32;
    if (warp >= n) return;
    const int64_t slot = slots[warp];
    if (slot < 0 || slot >= n_slots) {
        if (lane == 0) atomicCAS(err, 0, PGD_ERR_BLOCK_ID);
        return;
    }
    const uint4* ks = k_new + (int64_t)warp * row_vec;
    const uint4* vs = v_new + (int64_t)warp * row_vec;
    uint4* kd = k_pool + slot * row_vec;
    uint4* vd = v_pool + slot * row_vec;
    for (int i = lane; i < row_vec; i += 32) {
        kd[i] = ks[i];
        vd[i] = vs[i];
    }
}

// Block y of the grid copies chunk blockIdx.x of block pair y (K and V), and,
// for 8-bit pages with a scale per block and KV head (k_scale / v_scale
// non-null, [num_blocks][hkv]), chunk 0 also copies the pair's scale rows: a
// copied block keeps the range its codes were written with.
__global__ void __launch_bounds__(kWriteThreads)
    copy_blocks_kernel(const int32_t* __restrict__ src, const int32_t* __restrict__ dst,
                       int64_t num_blocks, int64_t block_vec, uint4* __restrict__ k_pool,
                       uint4* __restrict__ v_pool, float* __restrict__ k_scale,
                       float* __restrict__ v_scale, int hkv, int* err) {
    const int pair = blockIdx.y;
    const int64_t s = src[pair], d = dst[pair];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicCAS(err, 0, PGD_ERR_BLOCK_ID);
        return;
    }
    if (k_scale && blockIdx.x == 0) {
        for (int h = threadIdx.x; h < hkv; h += kWriteThreads) {
            k_scale[d * hkv + h] = k_scale[s * hkv + h];
            v_scale[d * hkv + h] = v_scale[s * hkv + h];
        }
    }
    const int64_t per = (block_vec + gridDim.x - 1) / gridDim.x;
    const int64_t lo = blockIdx.x * per;
    const int64_t hi = lo + per < block_vec ? lo + per : block_vec;
    for (int64_t i = lo + threadIdx.x; i < hi; i += kWriteThreads) {
        k_pool[d * block_vec + i] = k_pool[s * block_vec + i];
        v_pool[d * block_vec + i] = v_pool[s * block_vec + i];
    }
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace pgd

using namespace pgd;

extern "C" int paged_kv_append(pgd_pool_t pool, const void* k_new, const void* v_new,
                               const int32_t* slot_mapping, int n, void* stream) {
    if (!pool || n < 0) return PGD_ERR_ARG;
    if (n == 0) return PGD_OK;
    if (!k_new || !v_new || !slot_mapping) return PGD_ERR_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 3))
        return PGD_ERR_ALIGN;
    const Pool& p = pool_desc(pool);
    const int elt = p.dtype == PGD_F32 ? 4 : p.dtype == PGD_BF16 ? 2 : 1;
    const int row_vec = p.hkv * p.d * elt / 16;  // D is 64 or 128: whole vectors
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return PGD_ERR_CUDA;
    if (prev != p.device && cudaSetDevice(p.device) != cudaSuccess) return PGD_ERR_CUDA;
    const int warps_per_cta = kWriteThreads / 32;
    append_kernel<<<(n + warps_per_cta - 1) / warps_per_cta, kWriteThreads, 0,
                    static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), slot_mapping, n,
        p.num_blocks * p.block_size, row_vec, static_cast<uint4*>(const_cast<void*>(p.k)),
        static_cast<uint4*>(const_cast<void*>(p.v)), p.err);
    const cudaError_t e = cudaGetLastError();
    if (prev != p.device) cudaSetDevice(prev);
    return e == cudaSuccess ? PGD_OK : PGD_ERR_CUDA;
}

extern "C" int paged_kv_copy_blocks(pgd_pool_t pool, const int32_t* src, const int32_t* dst, int n,
                                    void* stream) {
    if (!pool || n < 0) return PGD_ERR_ARG;
    if (n == 0) return PGD_OK;
    if (!src || !dst) return PGD_ERR_ARG;
    if (n > 65535) return PGD_ERR_SHAPE;  // grid y limit
    const Pool& p = pool_desc(pool);
    const int elt = p.dtype == PGD_F32 ? 4 : p.dtype == PGD_BF16 ? 2 : 1;
    const int64_t block_vec = (int64_t)p.block_size * p.hkv * p.d * elt / 16;
    const int chunks = (int)((block_vec + 4095) / 4096);  // <= 64 KB of each tensor per CTA
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return PGD_ERR_CUDA;
    if (prev != p.device && cudaSetDevice(p.device) != cudaSuccess) return PGD_ERR_CUDA;
    copy_blocks_kernel<<<dim3(chunks, n), kWriteThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        src, dst, p.num_blocks, block_vec, static_cast<uint4*>(const_cast<void*>(p.k)),
        static_cast<uint4*>(const_cast<void*>(p.v)),
        p.scale_per_block ? const_cast<float*>(p.k_scale) : nullptr,
        p.scale_per_block ? const_cast<float*>(p.v_scale) : nullptr, p.hkv, p.err);
    const cudaError_t e = cudaGetLastError();
    if (prev != p.device) cudaSetDevice(prev);
    return e == cudaSuccess ? PGD_OK : PGD_ERR_CUDA;
}
