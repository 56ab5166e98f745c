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
    int32_t *chunk_split = nullptr; // [n_chunks] index of the chunk's split row
    int32_t *next = nullptr;        // [1] next item of a launch that takes its items dynamically
    // Items a warp claims with one atomic on `next` in passes that take them
    // in batches: the largest power of two whose chunks (the longest items,
    // at the head of the list) stay within three quarters of a resident
    // warp's average share of the edges, so no warp starts with more than
    // its share.
    int32_t batch = 1;
    // [n_split] chunks of each split row finished in the current launch of an
    // edge kernel that merges split rows itself (the last chunk to finish
    // merges the row and sets the count back to 0); zero between launches
    int32_t *arrive = nullptr;
    // The work items of an edge kernel in walking order: every chunk of a split
    // row (in chunk order), then every row of degree <= the threshold, by
    // descending degree (ties by id) or by ascending id.  n_items entries;
    // item x < n_chunks is chunk x.  nullptr: no list (chunks, then all rows
    // by id, split rows skipped at run time).
    int64_t n_items = 0;
    int4 *items = nullptr;          // [n_items] (row, first edge, end edge, 0)
    int32_t *order = nullptr;       // [N] all rows by descending degree (inspection; descending walks)
};

// Byte offsets of the regions of the caller's workspace.
struct WorkspaceLayout {
    size_t delta = 0;      // [N, H] f32          Delta_i = dOut_i . out_i (normalised weights)
    size_t lse_n = 0;      // [N, H] f32          lse_i + ln Z_i (backward row normalisation)
    size_t zt = 0;         // [N, H] f32          block-sparse plans: tile part of Z_i
    size_t bsr_lse_t = 0;  // [H, N_pad] f32      block-sparse plans: lse + ln Z, head-major
    size_t bsr_delta_t = 0;// [H, N_pad] f32      and Delta (N_pad: N rounded up to 128)
    size_t bias_t = 0;     // [E, H] f32          edge-bias plans: the bias in transposed order
    size_t gat_colc = 0;   // [t_n_chunks, H] f32 GAT plans: source-pass chunk parts of der
    size_t fwd_ml = 0;     // [n_chunks, H, 2] f32 chunk softmax stats (max, sum), log2 units
    size_t fwd_acc = 0;    // [n_chunks, H*D] f32  chunk unnormalised accumulators
    size_t bwd_row = 0;    // [n_chunks, 4, H*D] f32 chunk partial sums (dQ: A, B; dFL: A, B, da A, B)
    size_t bwd_rowc = 0;   // [n_chunks, H, 2] f32 chunk parts of C = sum p dP and Z = sum p
    size_t da_split = 0;   // [n_split, H*D] f32  GATv2 da contribution of each split row
    size_t bwd_col = 0;    // [t_n_chunks, 2*H*D] f32 chunk partial dK,dV / dFR
    size_t dfl = 0;        // [N, H*D] f32 GATv2 dFL
    size_t dfr = 0;        // [N, H*D] f32 GATv2 dFR
    size_t da_part = 0;    // [da_blocks, H*D] f32 GATv2 partial da
    size_t dw_part = 0;    // [dw_slabs, 2, F, H*D] f32 GATv2 partial dW_l, dW_r
    size_t fix = 0;        // int32 count, then [fix_cap] int2 projection elements to round exactly
    size_t agg_val = 0;    // [n_chunks, H*D] f32  min/max aggregation: chunk extremes
    size_t agg_pos = 0;    // [n_chunks, H*D] i32  their edge positions
    size_t agg_col = 0;    // [t_n_chunks, H*D] f32 backward: chunk sums of split sources
    int32_t fix_cap = 0;
    size_t total = 0;
    int32_t da_blocks = 0;
    int32_t dw_slabs = 0;
};

// Block-sparse split of the CSR (tensor-core forward): 128-row panels x
// 16-source column tiles with at least min_nnz edges are kept, each with one
// 16-bit source mask per panel row; all other edges form a residual CSR.
struct TileSet {
    int32_t min_nnz = 0;            // 0: no block-sparse representation
    int32_t n_panels = 0, n_tiles = 0;
    int64_t E_res = 0;
    int32_t *tile_ptr = nullptr;    // [n_panels + 1]
    int32_t *tile_col = nullptr;    // [n_tiles] column tile (sources 16c .. 16c+15)
    uint16_t *tile_bits = nullptr;  // [n_tiles + 1][128] source masks per panel row (the last: all zero)
    uint64_t *tile_bits_t = nullptr;// [n_tiles + 1][2][16] transposed: bit i of (t, half, c) = row 64 half + i has source c
    int32_t *r_indptr = nullptr;    // [N + 1] residual CSR
    int32_t *r_indices = nullptr;   // [E_res]
    // column view for the dK/dV pass: column panels of 128 sources (8 tile
    // columns); one entry per (row panel, column panel) pair holding a kept
    // tile, entries of a column panel in ascending row-panel order
    int32_t n_cpanels = 0, n_entries = 0;
    int32_t *ct_ptr = nullptr;      // [n_cpanels + 1]
    int32_t *ct_panel = nullptr;    // [n_entries] row panel
    int32_t *ct_tile = nullptr;     // [n_entries][8] tile index per tile column, -1: none
    // order in which the persistent kernels take panels: by descending kept
    // tiles (row panels) or entries (column panels), panels without any left out
    int32_t n_active = 0, n_cactive = 0;
    int4 *panel_info = nullptr;       // [n_active] (row panel, first tile, end tile, 0)
    int4 *cpanel_info = nullptr;      // [n_cactive] (column panel, first entry, end entry, 0)
};

}  // namespace sga

struct sga_plan {
    int64_t N = 0, E = 0;
    int H = 0, D = 0, F = 0;
    int layer = SGA_LAYER_ATTENTION;   // what the plan's workspace serves
    int schedule = SGA_SCHED_STREAM;   // thread mapping of the GT CSR forward
    sga_dtype dt = SGA_F32;
    int split_threshold = 256, chunk_len = 128;
    const int32_t *indptr = nullptr;   // graph the plan was built from
    const int32_t *indices = nullptr;
    int32_t *t_indptr = nullptr;       // [N + 1]
    int32_t *t_dst = nullptr;          // [E]
    int32_t *t_eid = nullptr;          // [E] CSR edge of each transposed entry (edge-bias plans)
    int edge_bias = 0;                 // plan serves gt_attn_bias_fwd/bwd
    int keep_eid = 0;                  // plan keeps t_eid (edge-bias and aggregation plans)
    int row_order = 1;                 // 1: rows walked by descending degree, 2: by ascending id
    sga::Partition rows, cols;         // partitions of the CSR and the transposed CSR
    sga::TileSet tiles;                // block-sparse split (tiles.min_nnz > 0)
    sga_plan *residual = nullptr;      // plan over the residual CSR (block-sparse plans)
    size_t residual_ws = 0;            // offset of the residual plan's workspace
    int32_t *d_err = nullptr;          // device error word
    void *ws = nullptr;
    size_t ws_bytes = 0;
    sga::WorkspaceLayout layout;
    int64_t device_bytes = 0;
    int num_sms = 0;
    std::vector<void *> owned;         // device allocations freed by plan_free
};

namespace sga {

// ---- plan builders (plan.cu, bsr.cu) ----
sga_status plan_build(sga_plan *p, cudaStream_t s);
sga_status bsr_build(sga_plan *p, cudaStream_t s);   // fills p->tiles (plan-owned memory)
void plan_free(sga_plan *p);
void set_cuda_error(cudaError_t e);
int get_cuda_error();

// Device exclusive prefix sum of n int32 (out may alias in); tmp holds
// scan_tmp_elems(n) int32.
int64_t scan_tmp_elems(int64_t n);
cudaError_t exclusive_scan(const int32_t *in, int32_t *out, int64_t n, int32_t *tmp, cudaStream_t s);

// Stable LSD radix sort of (key, value) int32 pairs by the low `bits` bits of
// the non-negative keys (plan.cu); the sorted pairs end in (*ka, *va).
int64_t radix_hist_elems(int64_t n);
cudaError_t radix_sort_pairs(int32_t **ka, int32_t **va, int32_t **kb, int32_t **vb, int64_t n,
                             int bits, int32_t *hist, int32_t *scan_tmp, cudaStream_t s);

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
    float *ws_lse;                 // [N, H] lse + ln Z written by the dQ pass
    // optional [N, H] terms added to each row's C = sum p dP and Z = sum p:
    // the share of edges that another pass (the block-sparse tiles)
    // handles; nullptr: none
    const float *delta_in, *z_in;
    // optional score bias [E, H] fp32 (CSR order; nullptr: none), its copy in
    // transposed order (workspace), the transposed position -> CSR edge map,
    // and the bias gradient dL/db [E, H] fp32
    const float *bias;
    float *bias_t, *dbias;
    const int32_t *t_eid;
    int64_t E;
    int32_t *d_err;
};
template <typename T> cudaError_t gt_fwd_t(const GtArgs &a, cudaStream_t s);
template <typename T> cudaError_t gt_bwd_t(const GtArgs &a, cudaStream_t s);
// GT forward with an alternative thread mapping (gt_sched.cu)
template <typename T> cudaError_t gt_fwd_sched_t(const GtArgs &a, int schedule, cudaStream_t s);

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
    float *ws_lse;                 // [N, H] lse + ln Z written by the destination pass
    float *ws_dfl, *ws_dfr;        // [N, H*D] fp32
    int32_t *ws_fix_count;
    int2 *ws_fix_list;
    int fix_cap;
    int da_blocks, dw_slabs;
    int32_t *d_err;
};
template <typename T> cudaError_t gatv2_fwd_t(const Gatv2Args &a, cudaStream_t s);

// ---- block-sparse tensor-core forward (bsr_fwd.cu) ----
struct BsrArgs {
    const void *Q, *K, *V;      // [N, H, D] bf16
    void *out;                  // in: residual forward, out: merged
    float *lse;                 // likewise
    const int32_t *tile_ptr, *tile_col;
    const uint16_t *tile_bits;      // [n_tiles + 1][128]: the last tile is all zero
    const int4 *panel_info;         // [n_active] (row panel, first tile, end tile, 0), most tiles first
    int64_t N;
    int H, D;
    int n_panels, n_tiles, n_active;
    int num_sms;
    int32_t *d_err;
};
bool bsr_fwd_supported(sga_dtype dt, int D);
cudaError_t launch_bsr_fwd(const BsrArgs &a, cudaStream_t s);

struct BsrBwdArgs {
    const void *Q, *K, *V, *dOut;   // [N, H, D] bf16
    const float *lse;               // [N, H] the forward's lse (Delta pass)
    float *delta_t;                 // [N, H] tile part of C = sum p dP (written by the Delta pass)
    float *z_t;                     // [N, H] tile part of Z = sum p (written by the Delta pass)
    const float *delta;             // [N, H] full Delta (read by the dQ and dK/dV passes)
    const float *lse_n;             // [N, H] lse + ln Z (read by the dQ and dK/dV passes)
    void *dQ, *dK, *dV;             // in: residual gradients, out: with the tile part added
    const int32_t *tile_ptr, *tile_col;
    const uint16_t *tile_bits;      // [n_tiles + 1][128]: the last tile is all zero
    const uint64_t *tile_bits_t;    // [n_tiles + 1][2][16] the same masks by (half, source)
    const int32_t *ct_ptr, *ct_panel, *ct_tile;
    const int4 *panel_info;         // [n_active] (row panel, first tile, end tile, 0), most tiles first
    const int4 *cpanel_info;        // [n_cactive] (column panel, first entry, end entry, 0), most first
    float *lse_t, *delta_t_hm;      // [H][N_pad] head-major copies of lse_n and delta (dK/dV pass)
    int64_t N, N_pad;               // N_pad: N rounded up to 128
    int H, D;
    int n_panels, n_cpanels, n_tiles, n_active, n_cactive;
    int num_sms;
    int32_t *d_err;
};
// Delta pass (delta_t), dQ pass, dK/dV pass (bsr_bwd.cu).
cudaError_t launch_bsr_bwd_delta(const BsrBwdArgs &a, cudaStream_t s);
cudaError_t launch_bsr_bwd_dq(const BsrBwdArgs &a, cudaStream_t s);
cudaError_t launch_bsr_bwd_dkdv(const BsrBwdArgs &a, cudaStream_t s);
template <typename T> cudaError_t gatv2_bwd_t(const Gatv2Args &a, cudaStream_t s);

// ---- GAT edge attention (gat.cu) ----
struct GatArgs {
    const int32_t *indptr, *indices;
    const int32_t *t_indptr, *t_dst;
    const void *Fv, *dOut;          // [N, H, D] projected features, upstream gradient
    const float *el, *er, *lse;     // [N, H] score halves, forward lse
    void *out_w, *dFv;              // [N, H, D]
    float *lse_w, *del, *der;       // [N, H]
    int64_t N;
    int H, D;
    float slope;
    int split_threshold;
    Partition rows, cols;
    float *ws_ml, *ws_acc;          // forward chunk partials (as the GT forward)
    float *ws_rowc;                 // [n_chunks, H, 4] destination-pass chunk sums C, Z, A, B
    float *ws_delta, *ws_lse;       // [N, H] Delta and lse + ln Z
    float *ws_col, *ws_colc;        // [t_n_chunks, H*D], [t_n_chunks, H] source-pass chunk sums
    int32_t *d_err;
};
template <typename T> cudaError_t gat_fwd_t(const GatArgs &a, cudaStream_t s);
template <typename T> cudaError_t gat_bwd_t(const GatArgs &a, cudaStream_t s);

// ---- min / max aggregation (agg.cu) ----
struct AggArgs {
    const int32_t *indptr, *indices;
    const void *X, *dOut;   // [N, HD] in the layer dtype
    void *out, *dX;         // likewise
    int32_t *arg;           // [N, HD] winning source node (-1: empty row); nullptr: not written
    uint8_t *mask;          // [E, R] win-mask bytes (R = 16-byte chunks of a row); nullptr: not written
    const int32_t *t_dst, *t_eid;   // transposed CSR and its CSR edge map
    int64_t N, E;
    int HD;
    int split_threshold;
    int num_sms;
    Partition rows, cols;
    float *ws_val;          // forward: chunk extremes [n_chunks, HD]; backward: chunk sums [t_n_chunks, HD]
    int32_t *ws_pos;
    int32_t *d_err;
};
template <typename T> cudaError_t agg_fwd_t(const AggArgs &a, bool is_max, cudaStream_t s);
template <typename T> cudaError_t agg_bwd_t(const AggArgs &a, cudaStream_t s);

}  // namespace sga
