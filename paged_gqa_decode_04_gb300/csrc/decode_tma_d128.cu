// The TMA decode kernel instantiated for head_dim 128, and the dispatch on
// head_dim (head_dim 64 lives in decode_tma_d64.cu).
#include "decode_tma.cuh"

namespace pgd {
namespace tma {
template cudaError_t launch_tma_d<128>(const DecodeArgs&, const Pool&, cudaStream_t);
extern template cudaError_t launch_tma_d<64>(const DecodeArgs&, const Pool&, cudaStream_t);
extern template cudaError_t launch_tma_d<128, true>(const DecodeArgs&, const Pool&, cudaStream_t);
}  // namespace tma

cudaError_t launch_decode_tma(const DecodeArgs& a, const Pool& p, cudaStream_t s) {
    const int idx = a.hg == 1 ? 0 : a.hg == 2 ? 1 : a.hg == 4 ? 2 : 3;
    if (!p.tmap_ok[idx]) return cudaErrorInvalidValue;
    if (p.dtype == PGD_FP8_E4M3) return tma::launch_tma_d<128, true>(a, p, s);
    if (a.d == 64) return tma::launch_tma_d<64>(a, p, s);
    return tma::launch_tma_d<128>(a, p, s);
}

}  // namespace pgd
