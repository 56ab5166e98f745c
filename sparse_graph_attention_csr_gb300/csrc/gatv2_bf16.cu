// GATv2 kernels instantiated for __nv_bfloat16 storage.
#include "gatv2.cuh"

namespace sga {
template cudaError_t gatv2_fwd_t<__nv_bfloat16>(const Gatv2Args &, cudaStream_t);
template cudaError_t gatv2_bwd_t<__nv_bfloat16>(const Gatv2Args &, cudaStream_t);
}  // namespace sga
