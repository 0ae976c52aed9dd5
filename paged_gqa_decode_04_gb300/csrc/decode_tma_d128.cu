// The TMA decode kernel instantiated for head_dim 128 (bf16 pages, last-arriver
// merge), and the dispatch on head_dim, page type and merge variant.  The other
// instantiations live in their own translation units so that they compile in
// parallel.
#include "decode_tma.cuh"

namespace pgd {
namespace tma {
template cudaError_t launch_tma_d<128, false, 0>(const DecodeArgs&, const Pool&, cudaStream_t);
extern template cudaError_t launch_tma_d<128, false, 1>(const DecodeArgs&, const Pool&,
                                                        cudaStream_t);
extern template cudaError_t launch_tma_d<128, false, 2>(const DecodeArgs&, const Pool&,
                                                        cudaStream_t);
extern template cudaError_t launch_tma_d<64, false, 0>(const DecodeArgs&, const Pool&,
                                                       cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 0>(const DecodeArgs&, const Pool&,
                                                       cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 1>(const DecodeArgs&, const Pool&,
                                                       cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 2>(const DecodeArgs&, const Pool&,
                                                       cudaStream_t);
}  // namespace tma

cudaError_t launch_decode_tma(const DecodeArgs& a, const Pool& p, cudaStream_t s) {
    const int idx = a.hg == 1 ? 0 : a.hg == 2 ? 1 : a.hg == 4 ? 2 : 3;
    if (!p.tmap_ok[idx]) return cudaErrorInvalidValue;
    const bool fp8 = p.dtype == PGD_FP8_E4M3;
    if (a.d == 128 && a.merge_variant == 1) {
        const cudaError_t e = fp8 ? tma::launch_tma_d<128, true, 1>(a, p, s)
                                  : tma::launch_tma_d<128, false, 1>(a, p, s);
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        cudaGetLastError();  // not resident at once: the last-arriver variant instead
    }
    if (a.d == 128 && a.merge_variant == 2)
        return fp8 ? tma::launch_tma_d<128, true, 2>(a, p, s)
                   : tma::launch_tma_d<128, false, 2>(a, p, s);
    if (fp8) return tma::launch_tma_d<128, true, 0>(a, p, s);
    if (a.d == 64) return tma::launch_tma_d<64, false, 0>(a, p, s);
    return tma::launch_tma_d<128, false, 0>(a, p, s);
}

}  // namespace pgd
