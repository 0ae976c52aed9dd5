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
extern template cudaError_t launch_tma_d<128, true, 0, true>(const DecodeArgs&, const Pool&,
                                                             cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 1, true>(const DecodeArgs&, const Pool&,
                                                             cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 2, true>(const DecodeArgs&, const Pool&,
                                                             cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 0, false, true>(const DecodeArgs&,
                                                                    const Pool&, cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 1, false, true>(const DecodeArgs&,
                                                                    const Pool&, cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 2, false, true>(const DecodeArgs&,
                                                                    const Pool&, cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 0, true, true>(const DecodeArgs&,
                                                                   const Pool&, cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 1, true, true>(const DecodeArgs&,
                                                                   const Pool&, cudaStream_t);
extern template cudaError_t launch_tma_d<128, true, 2, true, true>(const DecodeArgs&,
                                                                   const Pool&, cudaStream_t);
}  // namespace tma

namespace {
// The 8-bit instantiation for merge variant MV of the pool's code and scale
// granularity.
template <int MV>
cudaError_t launch_q8(const DecodeArgs& a, const Pool& p, cudaStream_t s) {
    const bool i8 = p.dtype == PGD_INT8;
    if (a.scale_per_block)
        return i8 ? tma::launch_tma_d<128, true, MV, true, true>(a, p, s)
                  : tma::launch_tma_d<128, true, MV, false, true>(a, p, s);
    return i8 ? tma::launch_tma_d<128, true, MV, true>(a, p, s)
              : tma::launch_tma_d<128, true, MV>(a, p, s);
}
}  // namespace

cudaError_t launch_decode_tma(const DecodeArgs& a, const Pool& p, cudaStream_t s) {
    const int idx = a.hg == 1 ? 0 : a.hg == 2 ? 1 : a.hg == 4 ? 2 : 3;
    if (!p.tmap_ok[idx]) return cudaErrorInvalidValue;
    const bool q8 = p.dtype == PGD_FP8_E4M3 || p.dtype == PGD_INT8;
    if (a.d == 128 && a.merge_variant == 1) {
        const cudaError_t e = q8 ? launch_q8<1>(a, p, s) : tma::launch_tma_d<128, false, 1>(a, p, s);
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        cudaGetLastError();  // not resident at once: the last-arriver variant instead
    }
    if (a.d == 128 && a.merge_variant == 2)
        return q8 ? launch_q8<2>(a, p, s) : tma::launch_tma_d<128, false, 2>(a, p, s);
    if (q8) return launch_q8<0>(a, p, s);
    if (a.d == 64) return tma::launch_tma_d<64, false, 0>(a, p, s);
    return tma::launch_tma_d<128, false, 0>(a, p, s);
}

}  // namespace pgd
