// paged_gqa_decode_noalloc: the decode step for callers that cannot allocate
// device memory.
//
// Who needs it.  A library embedded in a host runtime that owns every byte of
// device memory (an inference server's plugin interface, a framework with its
// own caching allocator and a fixed memory budget) may be handed no allocator
// at all, and calling cudaMalloc behind the runtime's back would break its
// accounting.  Latency-critical callers avoid cudaMalloc / cudaFree because
// they can synchronise the whole device.  Both still need the split-KV scratch
// (partial results, tile prefix table, per-run counters) that
// paged_gqa_decode normally takes as a caller-provided workspace.
//
// How.  The scratch lives in one file-scope __device__ array of a fixed size,
// which the CUDA module reserves on every device that loads this library and
// keeps until the process exits.  The host never dereferences the symbol: on
// a device's first call, with that device current, cudaGetSymbolAddress turns
// it into the device address that the kernel is given.  Each call then clears
// the per-run counters (the only part that must start at zero) with an
// asynchronous memset on the caller's stream and runs the same decode as
// paged_gqa_decode with that address as its workspace.  Nothing here calls
// cudaMalloc, cudaFree or any allocating routine.
#include <mutex>

#include "pgd_internal.h"

namespace pgd {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on `dev` (looked up once per device,
// with `dev` current); nullptr if the lookup failed.
void* scratch_on(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        int prev = -1;
        if (cudaGetDevice(&prev) != cudaSuccess) return nullptr;
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return nullptr;
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (prev != dev) cudaSetDevice(prev);
        if (e != cudaSuccess || !p) return nullptr;
        g_scratch_ptr[dev] = p;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace pgd

extern "C" size_t paged_gqa_noalloc_scratch_bytes(void) { return pgd::kNoAllocScratchBytes; }

extern "C" int paged_gqa_decode_noalloc(pgd_pool_t pool, const void* q, int B, int Hq,
                                        const int32_t* block_table, int max_blocks,
                                        const int32_t* seq_lens, float scale, void* out,
                                        int num_splits, void* stream) {
    if (!pool) return PGD_ERR_ARG;
    size_t need = 0;
    int rc = paged_gqa_workspace_size(pool, B, Hq, num_splits, &need);
    if (rc != PGD_OK) return rc;
    if (need > pgd::kNoAllocScratchBytes) return PGD_ERR_TOO_LARGE;
    if (B == 0) return paged_gqa_decode(pool, q, B, Hq, block_table, max_blocks, seq_lens, scale,
                                        out, nullptr, 0, num_splits, stream);
    const pgd::Pool& p = pgd::pool_desc(pool);
    const int dev = p.device;
    unsigned char* scratch = static_cast<unsigned char*>(pgd::scratch_on(dev));
    if (!scratch) return PGD_ERR_CUDA;
    // Every argument check before anything is enqueued: a refused call must
    // not touch the shared array, which another call may be using.
    pgd::Plan plan;
    pgd::WorkspaceLayout wl;
    rc = pgd::check_decode(p, q, B, 1, Hq, block_table, max_blocks, seq_lens, 0, scale, out,
                           scratch, pgd::kNoAllocScratchBytes, num_splits, &plan, &wl);
    if (rc != PGD_OK) return rc;

    // The array keeps whatever the previous call left; only the counters must
    // start at zero.
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return PGD_ERR_CUDA;
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) return PGD_ERR_CUDA;
    const cudaError_t e = cudaMemsetAsync(scratch + wl.counters_off, 0,
                                          wl.tile_base_off - wl.counters_off,
                                          static_cast<cudaStream_t>(stream));
    if (prev != dev) cudaSetDevice(prev);
    if (e != cudaSuccess) return PGD_ERR_CUDA;
    return paged_gqa_decode(pool, q, B, Hq, block_table, max_blocks, seq_lens, scale, out,
                            scratch, pgd::kNoAllocScratchBytes, num_splits, stream);
}
