// Graph Transformer kernels instantiated for __nv_bfloat16 storage.
#include "gt.cuh"

namespace sga {
template cudaError_t gt_fwd_t<__nv_bfloat16>(const GtArgs &, cudaStream_t);
template cudaError_t gt_bwd_t<__nv_bfloat16>(const GtArgs &, cudaStream_t);
}  // namespace sga
