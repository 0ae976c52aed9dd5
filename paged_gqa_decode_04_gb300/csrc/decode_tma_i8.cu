// The TMA decode kernel for 8-bit K/V pages of int8 codes, head_dim 128,
// last-arriver merge.
#include "decode_tma.cuh"

namespace pgd {
namespace tma {
template cudaError_t launch_tma_d<128, true, 0, true>(const DecodeArgs&, const Pool&, cudaStream_t);
}  // namespace tma
}  // namespace pgd
