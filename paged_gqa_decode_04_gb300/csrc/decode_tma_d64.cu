// The TMA decode kernel instantiated for head_dim 64.
#include "decode_tma.cuh"

namespace pgd {
namespace tma {
template cudaError_t launch_tma_d<64, false, 0>(const DecodeArgs&, const Pool&, cudaStream_t);
}  // namespace tma
}  // namespace pgd
