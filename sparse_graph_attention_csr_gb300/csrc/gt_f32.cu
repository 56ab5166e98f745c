// Graph Transformer kernels instantiated for float storage.
#include "gt.cuh"

namespace sga {
template cudaError_t gt_fwd_t<float>(const GtArgs &, cudaStream_t);
template cudaError_t gt_bwd_t<float>(const GtArgs &, cudaStream_t);
}  // namespace sga
