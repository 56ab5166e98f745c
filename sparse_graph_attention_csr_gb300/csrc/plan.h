// Host-side plan object and the launch interfaces the kernels expose to api.cu.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <vector>

#include "../../include/sga.h"

namespace sga {

// Degree partition of one CSR (rows or transposed rows).  Rows with degree >
// split_threshold are split rows; each is cut into chunks of chunk_len edges.
struct Partition {
    int32_t n_split = 0, n_chunks = 0;
    int32_t *split_rows = nullptr;  // [n_split] ascending row ids
    int32_t *chunk_ptr = nullptr;   // [n_split + 1] chunk range of each split row
    int32_t *chunk_row = nullptr;   // [n_chunks]
    int32_t *chunk_beg = nullptr;   // [n_chunks] first edge (absolute CSR offset)
    int32_t *chunk_end = nullptr;   // [n_chunks] one past the last edge
};

// Byte offsets of the regions of the caller's workspace.
struct WorkspaceLayout {
    size_t delta = 0;      // [N, H] f32          Delta_i = dOut_i . out_i
    size_t fwd_ml = 0;     // [n_chunks, H, 2] f32 chunk softmax stats (max, sum), log2 units
    size_t fwd_acc = 0;    // [n_chunks, H*D] f32  chunk unnormalised accumulators
    size_t bwd_row = 0;    // [n_chunks, 4, H*D] f32 chunk partial sums (dQ: A, B; dFL: A, B, da A, B)
    size_t bwd_rowc = 0;   // [n_chunks, H] f32   chunk part of Delta
    size_t da_split = 0;   // [n_split, H*D] f32  GATv2 da contribution of each split row
    size_t bwd_col = 0;    // [t_n_chunks, 2*H*D] f32 chunk partial dK,dV / dFR
    size_t dfl = 0;        // [N, H*D] f32 GATv2 dFL
    size_t dfr = 0;        // [N, H*D] f32 GATv2 dFR
    size_t da_part = 0;    // [da_blocks, H*D] f32 GATv2 partial da
    size_t dw_part = 0;    // [dw_slabs, 2, F, H*D] f32 GATv2 partial dW_l, dW_r
    size_t fix = 0;        // int32 count, then [fix_cap] int2 projection elements to round exactly
    int32_t fix_cap = 0;
    size_t total = 0;
    int32_t da_blocks = 0;
    int32_t dw_slabs = 0;
};

}  // namespace sga

struct sga_plan {
    int64_t N = 0, E = 0;
    int H = 0, D = 0, F = 0;
    sga_dtype dt = SGA_F32;
    int split_threshold = 256, chunk_len = 128;
    const int32_t *indptr = nullptr;   // graph the plan was built from
    const int32_t *indices = nullptr;
    int32_t *t_indptr = nullptr;       // [N + 1]
    int32_t *t_dst = nullptr;          // [E]
    sga::Partition rows, cols;         // partitions of the CSR and the transposed CSR
    int32_t *d_err = nullptr;          // device error word
    void *ws = nullptr;
    size_t ws_bytes = 0;
    sga::WorkspaceLayout layout;
    int64_t device_bytes = 0;
    int num_sms = 0;
    std::vector<void *> owned;         // device allocations freed by plan_free
};

namespace sga {

// ---- plan builders (plan.cu) ----
sga_status plan_build(sga_plan *p, cudaStream_t s);
void plan_free(sga_plan *p);
void set_cuda_error(cudaError_t e);
int get_cuda_error();

// ---- Graph Transformer (gt.cu) ----
struct GtArgs {
    const int32_t *indptr, *indices;
    const int32_t *t_indptr, *t_dst;
    const void *Q, *K, *V, *out, *dOut;
    const float *lse;
    void *out_w, *dQ, *dK, *dV;
    float *lse_w;
    int64_t N;
    int H, D;
    int split_threshold;
    Partition rows, cols;
    float *ws_ml, *ws_acc, *ws_delta, *ws_row, *ws_rowc, *ws_col;
    int32_t *d_err;
};
template <typename T> cudaError_t gt_fwd_t(const GtArgs &a, cudaStream_t s);
template <typename T> cudaError_t gt_bwd_t(const GtArgs &a, cudaStream_t s);

// ---- GATv2 (gatv2.cu) ----
struct Gatv2Args {
    const int32_t *indptr, *indices;
    const int32_t *t_indptr, *t_dst;
    const void *X, *Wl, *Wr, *a, *FL, *FR, *out, *dOut;
    const float *lse;
    void *FL_w, *FR_w, *out_w, *dX, *dWl, *dWr, *da;
    float *lse_w;
    int64_t N;
    int F, H, D;
    float slope;
    int split_threshold;
    Partition rows, cols;
    float *ws_ml, *ws_acc, *ws_delta, *ws_row, *ws_rowc, *ws_col, *ws_da, *ws_da_split, *ws_dw;
    float *ws_dfl, *ws_dfr;        // [N, H*D] fp32
    int32_t *ws_fix_count;
    int2 *ws_fix_list;
    int fix_cap;
    int da_blocks, dw_slabs;
    int32_t *d_err;
};
template <typename T> cudaError_t gatv2_fwd_t(const Gatv2Args &a, cudaStream_t s);
template <typename T> cudaError_t gatv2_bwd_t(const Gatv2Args &a, cudaStream_t s);

}  // namespace sga
