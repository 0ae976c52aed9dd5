// The TMA decode kernel for 8-bit K/V pages of e4m3 codes with a scale per
// block and KV head, head_dim 128, separate-merge variant
// (pieces write partials; the run-merge kernel merges them).
#include "decode_tma.cuh"

namespace pgd {
namespace tma {
template cudaError_t launch_tma_d<128, true, 2, false, true>(const DecodeArgs&, const Pool&,
                                                           cudaStream_t);
}  // namespace tma
}  // namespace pgd
