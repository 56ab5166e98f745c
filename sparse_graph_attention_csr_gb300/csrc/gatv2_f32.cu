// GATv2 kernels instantiated for float storage.
#include "gatv2.cuh"

namespace sga {
template cudaError_t gatv2_fwd_t<float>(const Gatv2Args &, cudaStream_t);
template cudaError_t gatv2_bwd_t<float>(const Gatv2Args &, cudaStream_t);
}  // namespace sga
