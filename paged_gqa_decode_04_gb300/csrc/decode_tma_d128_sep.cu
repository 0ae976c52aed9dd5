// The TMA decode kernel for head_dim 128 (bf16 pages), separate-merge variant
// (pieces write partials; the run-merge kernel merges them).
#include "decode_tma.cuh"

namespace pgd {
namespace tma {
template cudaError_t launch_tma_d<128, false, 2>(const DecodeArgs&, const Pool&, cudaStream_t);
}  // namespace tma
}  // namespace pgd
