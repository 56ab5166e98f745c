// GATv2 projections FL = X W_l and FR = X W_r on the tcgen05 tensor cores.
//
// Persistent CTAs over 128-row tiles of X: TMA streams the tiles, one lane
// issues the 128 x 2HD x 16 MMAs into two TMEM accumulators (W_l and W_r
// staged once per CTA as one K-major operand, FL columns then FR columns),
// and eight epilogue warps drain them (see tc_proj.cu).
//
// Outputs are rounded correctly to bf16 (they decide LeakyReLU branches
// downstream): an fp32 result whose bf16 rounding is not settled by the bound
// 2 * 2^-24 |x||w| + ulp (see gemm.cuh) is recomputed exactly from the shared
// memory tiles with an error-free TwoSum cascade.
#pragma once

#include "common.cuh"

namespace sga {

struct TcProj {
    const __nv_bfloat16 *X, *Wl, *Wr;
    __nv_bfloat16 *FL, *FR;
    int64_t M;      // rows of X
    int K;          // input width F: multiple of 64, <= 192
    int HD;         // output width per projection: multiple of 32, <= 128
    int32_t *err;
};

inline bool tc_proj_supported(int K, int HD) {
    // K in 64-column TMA boxes (128-byte rows); 2 HD columns of one MMA, 32-column epilogue chunks
    return K % 64 == 0 && K >= 64 && K <= 192 && HD % 32 == 0 && HD >= 32 && HD <= 128;
}

// Launch on stream s (tc_proj.cu).
cudaError_t tc_proj(const TcProj &p, cudaStream_t s);

}  // namespace sga
