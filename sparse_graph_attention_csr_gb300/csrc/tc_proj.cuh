// GATv2 projections FL = X W_l and FR = X W_r on the tcgen05 tensor cores.
//
// One persistent CTA per SM (4 warps).  W_l and W_r are staged once per CTA
// as one K-major operand B of 2*H*D rows (FL columns, then FR columns).  For
// each 128-row tile of X the CTA stages the tile (cp.async, double-buffered:
// the next tile loads while the current one finishes), one thread issues the
// K/16 MMAs of shape 128 x 2HD x 16 into a TMEM accumulator, and the four
// warps read their 32 rows each back with tcgen05.ld.
//
// Outputs are rounded correctly to bf16 (they decide LeakyReLU branches
// downstream): an fp32 result whose bf16 rounding is not settled by the bound
// 2 * 2^-24 |x||w| + ulp (see gemm.cuh) is recomputed exactly from the shared
// memory tiles with an error-free TwoSum cascade, one warp per element.
#pragma once

#include "common.cuh"

namespace sga {

struct TcProj {
    const __nv_bfloat16 *X, *Wl, *Wr;
    __nv_bfloat16 *FL, *FR;
    int64_t M;      // rows of X
    int K;          // input width F: multiple of 16, <= 192
    int HD;         // output width per projection: multiple of 32, <= 128
    int32_t *err;
};

inline bool tc_proj_supported(int K, int HD) {
    return K % 16 == 0 && K >= 16 && K <= 192 && HD % 32 == 0 && HD <= 128;   // 2 HD % 64 == 0
}

// Launch on stream s (tc_proj.cu).
cudaError_t tc_proj(const TcProj &p, cudaStream_t s);

}  // namespace sga
