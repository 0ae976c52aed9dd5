// Diagnostic: exercise the bounded-wait path of the pipeline kernels without
// faulting anything.  One thread initialises an mbarrier that nothing will
// ever arrive on and waits on it with the same helper the decode kernel uses,
// but with a caller-chosen limit; when the limit passes it latches
// PGD_ERR_TIMEOUT in the pool's error word and returns, so the context stays
// usable and the host reads the status with paged_gqa_get_error.
#include "decode_tma.cuh"

namespace pgd {
namespace {

__global__ void wait_timeout_kernel(uint64_t limit_ns, int* err) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = tma::smem_u32(&bar);
    tma::mbar_init(b, 1);
    tma::fence_barrier_init();
    if (!tma::mbar_wait(b, 0, limit_ns)) latch_error(err, PGD_ERR_TIMEOUT);
}

}  // namespace
}  // namespace pgd

extern "C" int paged_gqa_selftest_wait_timeout(pgd_pool_t pool, int64_t limit_us, void* stream) {
    if (!pool || limit_us < 1 || limit_us > 1000000) return PGD_ERR_ARG;
    const pgd::Pool& p = pgd::pool_desc(pool);
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return PGD_ERR_CUDA;
    if (prev != p.device && cudaSetDevice(p.device) != cudaSuccess) return PGD_ERR_CUDA;
    pgd::wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(
        (uint64_t)limit_us * 1000ull, p.err);
    const cudaError_t e = cudaGetLastError();
    if (prev != p.device) cudaSetDevice(prev);
    return e == cudaSuccess ? PGD_OK : PGD_ERR_CUDA;
}
