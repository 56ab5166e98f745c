// GAT edge-attention kernels instantiated for both storage dtypes.
#include "gat.cuh"

namespace sga {
template cudaError_t gat_fwd_t<float>(const GatArgs &, cudaStream_t);
template cudaError_t gat_bwd_t<float>(const GatArgs &, cudaStream_t);
template cudaError_t gat_fwd_t<__nv_bfloat16>(const GatArgs &, cudaStream_t);
template cudaError_t gat_bwd_t<__nv_bfloat16>(const GatArgs &, cudaStream_t);
}  // namespace sga
