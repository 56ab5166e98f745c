// GATv2 input gradient dX = dFL W_l^T + dFR W_r^T on the tcgen05 tensor cores,
// operands streamed by the Tensor Memory Accelerator.
//
// dFL and dFR are the workspace's bf16 (hi, lo) rows [M][2 HD] (hi then lo,
// about 16 significant bits of the fp32 gradients); W_l, W_r are [F][HD] bf16.
// With K running over [dFL hi | dFL lo | dFR hi | dFR lo] (4 HD) and the
// weights repeated [W_l | W_l | W_r | W_r], dX is one K-major product
// (M x F x 4 HD) per 128-row tile, accumulated in fp32 in TMEM and rounded to
// bf16 once.
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace sga {

struct TcDx {
    const __nv_bfloat16 *dfl, *dfr;   // [M][2 HD]: hi row then lo row
    const __nv_bfloat16 *Wl, *Wr;     // [F][HD]
    __nv_bfloat16 *dX;                // [M][F]
    int64_t M;
    int F, HD;
    int32_t *err;                     // device error word (timed-out waits)
};

// HD in {64, 128}; F a multiple of 32 in [32, 256] (one MMA's N; the epilogue
// moves 32 accumulator columns at a time); M < 2^31.
inline bool tc_dx_supported(int F, int HD, int64_t M) {
    return (HD == 64 || HD == 128) && F % 32 == 0 && F >= 32 && F <= 256 && M < (int64_t(1) << 31);
}

// Launch on stream s (tc_dx.cu).
cudaError_t tc_dx(const TcDx &p, cudaStream_t s);

// Weight gradients dW_l = X^T dFL, dW_r = X^T dFR over node slabs: each CTA
// takes slab_rows consecutive nodes (a multiple of 64) and writes fp32
// partials part[w][slab][F][HD] (w = 0: dW_l, 1: dW_r), reduced afterwards in
// slab order.  Both operands are node-major in memory; they are loaded by TMA
// as 64 x 64 boxes and consumed as MN-major tcgen05 operands.
struct TcDw {
    const __nv_bfloat16 *X;            // [M][F]
    const __nv_bfloat16 *dfl, *dfr;    // [M][2 HD]: hi row then lo row
    float *part;                       // [2][slabs][F][HD]
    int64_t M;
    int F, HD;
    int slab_rows, slabs;
    int32_t *err;
};

// F == 128 (one MMA's M), HD in {64, 128}.
inline bool tc_dw_supported(int F, int HD, int64_t M) {
    return F == 128 && (HD == 64 || HD == 128) && M < (int64_t(1) << 31);
}

// Nodes per weight-gradient slab: a multiple of 64, at least 256, at most two
// slabs per SM; slabs = ceil(M / rows).
inline int dw_slab_rows(int64_t M, int num_sms) {
    const int64_t per = (M + 2 * (int64_t)num_sms - 1) / (2 * (int64_t)num_sms);
    const int64_t r = per < 256 ? 256 : per;
    return (int)((r + 63) / 64 * 64);
}

cudaError_t tc_dw(const TcDw &p, cudaStream_t s);

// TMA descriptor of a row-major [rows][cols] bf16 matrix with rows of
// row_elems elements, boxes of box_cols x box_rows, 128-byte swizzle (the
// K-major tile layout of tc.cuh), out-of-range elements read as zero.
cudaError_t bf16_tensor_map(CUtensorMap *m, const __nv_bfloat16 *base, int64_t rows, int64_t cols,
                            int64_t row_elems, uint32_t box_cols, uint32_t box_rows);

}  // namespace sga
