/*
 * sga.h -- C ABI of the fused CSR edge-attention library (sm_103a).
 *
 * What it computes (the method of "On Efficient Scaling of GNNs via IO-Aware
 * Layers Implementations", Yandex Research blog post, "Attention-based layers"
 * paragraph, and the arXiv abstract of the same paper): attention layers of the
 * Graph Transformer and GATv2 kind over a graph stored as CSR sorted by
 * destination.  For every destination row the kernels gather the neighbour
 * rows, score them per head, run an online softmax and accumulate the weighted
 * values; the E x H edge scores are never written to device memory.  The
 * backward pass recomputes the weights from the per-row log-sum-exp saved by
 * the forward pass (the FlashAttention-2 idea the blog post names).  Rows of
 * very high degree ("super nodes", DF-GNN abstract; "degree-aware tiling" in
 * the blog post's aggregation paragraph) are cut into chunks whose partial
 * softmax statistics are merged in a fixed order.
 *
 * Conventions shared by every call
 *  - Graph: indptr[N+1] and indices[E], int32, DEVICE memory.  Row i is the
 *    destination; indices[indptr[i] .. indptr[i+1]) are its sources j.
 *    Duplicate entries count as separate edges.  N < 2^31, E < 2^31.
 *  - Node tensors are [N, H, D] row-major in the call's dtype (one node's heads
 *    contiguous).  lse is [N, H] float32, natural log; an empty row gives
 *    out = 0 and lse = -inf.  All tensor pointers are DEVICE pointers aligned
 *    to 16 bytes; the caller owns every buffer it passes.
 *  - Supported shapes: D in {32, 64, 128}; H >= 1; H*D <= 1024; GATv2 input
 *    width F a multiple of 8 with 8 <= F <= 1024.  Anything else returns
 *    SGA_EUNSUPPORTED.
 *  - dtype: SGA_F32 or SGA_BF16 for every tensor of a call except lse (always
 *    float32).  Arithmetic accumulates in float32.
 *  - Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  Every
 *    compute call is asynchronous on that stream.  sga_plan_create and
 *    sga_read_device_error synchronise it.
 *  - Errors: no call throws or aborts; each returns an sga_status.  Argument
 *    errors are detected on the host before any launch.  SGA_ECUDA means a CUDA
 *    runtime call failed; sga_last_cuda_error() returns its code.
 */
#ifndef SGA_H
#define SGA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SGA_OK = 0,
    SGA_EINVAL = 1,         /* bad argument: null pointer, misalignment, plan mismatch, invalid CSR */
    SGA_EUNSUPPORTED = 2,   /* shape or dtype outside the supported set */
    SGA_ECUDA = 3,          /* a CUDA runtime call failed */
    SGA_EWORKSPACE = 4,     /* workspace missing or smaller than sga_plan_workspace_bytes() */
    SGA_EDEVICE_CHECK = 5,  /* a device-side range check fired (see sga_read_device_error) */
    SGA_ELIMIT = 6          /* input needs more than gt_attn_fwd_noalloc's fixed scratch */
} sga_status;

typedef enum { SGA_F32 = 0, SGA_BF16 = 1 } sga_dtype;

/* Opaque, host-owned plan for one graph and one layer shape. */
typedef struct sga_plan sga_plan;

/* Layer a plan serves (its workspace layout). */
typedef enum {
    SGA_LAYER_ATTENTION = 0,  /* Graph Transformer (in_features = 0) or GATv2 (in_features > 0) */
    SGA_LAYER_MINMAX = 1,     /* min / max neighbourhood aggregation (agg_minmax_fwd/bwd) */
    SGA_LAYER_GAT = 2         /* GAT edge attention (gat_attn_fwd/bwd) */
} sga_layer;

/* Plan options.  Zero (or a NULL pointer) selects the default of each field. */
typedef struct {
    int32_t split_threshold;  /* rows of degree > this are split (default: 256, doubled while
                                 8x it stays within E / (16 x the SMs), the edges one resident
                                 warp takes on average, up to 4096) */
    int32_t chunk_len;        /* edges per chunk of a split row (default: half the threshold) */
    int32_t in_features;      /* GATv2 input width F; 0 for a Graph Transformer plan */
    int32_t tile_min_nnz;     /* > 0: block-sparse tensor-core forward, see below; 0: off */
    int32_t layer;            /* sga_layer (default SGA_LAYER_ATTENTION) */
    int32_t schedule;         /* sga_schedule of the Graph Transformer CSR forward (default 0) */
    int32_t edge_bias;        /* 1: the plan also serves gt_attn_bias_fwd/bwd (keeps the CSR edge
                                 of every transposed entry: 4 more bytes per edge) */
    int32_t row_order;        /* order in which the edge kernels walk rows (and transposed rows):
                                 1 (default): by descending degree, ties by id (long rows first
                                 balances the persistent warps); 2: by ascending id.  Results are
                                 bit-identical either way */
} sga_plan_opts;

/* Thread mapping of the Graph Transformer forward over the CSR (the backward
 * and the GATv2 passes always use the edge stream).  The pages contrast
 * neighbour-parallel with feature-parallel kernels (IO-aware layers arXiv
 * abstract) and schedule the score and aggregation stages with different
 * mappings (DF-GNN abstract, "bi-level thread scheduling").  Results agree
 * with the default up to fp32 rounding order. */
typedef enum {
    SGA_SCHED_STREAM = 0,   /* warps over rows, groups of lanes over a row's features, several
                               neighbours per step staged through a shared-memory ring */
    SGA_SCHED_FEATURE = 1,  /* warp per row, lanes over features, one neighbour at a time, direct loads */
    SGA_SCHED_BILEVEL = 2   /* scores edge-parallel (a lane per edge), aggregation feature-parallel */
} sga_schedule;

/* Build a plan: validates the CSR on the device (indptr[0] = 0, monotone,
 * indptr[N] = E, 0 <= indices < N), builds the transposed CSR (sources ->
 * ascending destinations) and the degree partitions of both.
 * Block-sparse plans (opts->tile_min_nnz > 0; bf16, D in {64, 128}):
 * the "block-sparse graph representation that enables the use of tensor
 * cores" of the IO-aware layers blog post ("Attention-based layers"
 * paragraph).  Destinations are grouped in panels of 128 rows and sources in
 * column tiles of 16; every (panel, tile) pair with at least tile_min_nnz edges
 * is kept with one 16-bit source mask per panel row, all other edges form a
 * residual CSR.  gt_attn_fwd then computes the kept tiles on the tcgen05
 * tensor cores and the residual edges with the CSR kernels, merged by
 * log-sum-exp.  gt_attn_bwd computes the tile part of the row term Delta on
 * the tensor cores, runs the residual CSR backward with it, then adds the
 * tiles' dQ (row panels) and dK/dV (column panels of 128 sources) from
 * tensor-core products (FlashAttention-2 style).  A
 * mask holds a (destination, source) pair once: the first edge of a pair in a
 * kept tile sets its bit and any repeat of it (its own softmax term) joins the
 * residual CSR.  Other shapes and dtypes return SGA_EUNSUPPORTED.
 * indptr/indices: device pointers, read only during this call.
 * The plan owns device memory for the transposed CSR and partitions (freed by
 * sga_plan_destroy).  Synchronises `stream`.  Returns SGA_EINVAL for an
 * invalid CSR, leaving *out NULL. */
sga_status sga_plan_create(const int32_t *indptr, const int32_t *indices, int64_t N, int64_t E,
                           int H, int D, sga_dtype dt, const sga_plan_opts *opts,
                           void *stream, sga_plan **out);

/* Bytes of device workspace every compute call of this plan needs (may be 0). */
size_t sga_plan_workspace_bytes(const sga_plan *plan);

/* Attach caller-owned device workspace (256-byte aligned, at least
 * sga_plan_workspace_bytes()).  Calls that use the same plan must not overlap
 * on the device: they share this workspace and the plan's own per-launch
 * state (the counter from which the edge kernels take their work items,
 * zeroed on the stream before each launch, and the arrival counts of split
 * rows merged inside the kernels, back at zero when a launch ends).
 * Different plans may run concurrently. */
sga_status sga_plan_set_workspace(sga_plan *plan, void *d_workspace, size_t bytes);

void sga_plan_destroy(sga_plan *plan);

/* Graph Transformer forward: s_ij = q_i . k_j / sqrt(D) per head, softmax over
 * the row, out_i = sum_j p_ij v_j, lse_i = log sum_j exp(s_ij).
 * Q, K, V, out: [N, H, D] in dt; lse: [N, H] float32.  The graph arguments must
 * be the ones the plan was built from. */
sga_status gt_attn_fwd(const sga_plan *plan, const int32_t *indptr, const int32_t *indices,
                       const void *Q, const void *K, const void *V, int64_t N, int64_t E, int H,
                       int D, sga_dtype dt, void *out, float *lse, void *stream);

/* Graph Transformer backward.  Recomputes p_ij = exp(s_ij - lse_i) and, with
 * Delta_i = dOut_i . out_i, dS_ij = p_ij (dOut_i . v_j - Delta_i):
 * dQ_i = sum_j dS_ij k_j / sqrt(D),  dK_j = sum_i dS_ij q_i / sqrt(D),
 * dV_j = sum_i p_ij dOut_i.  dK/dV walk the transposed CSR, so no atomics are
 * used and results are bitwise reproducible.  out/lse are the forward's. */
sga_status gt_attn_bwd(const sga_plan *plan, const int32_t *indptr, const int32_t *indices,
                       const void *Q, const void *K, const void *V, const void *out,
                       const float *lse, const void *dOut, int64_t N, int64_t E, int H, int D,
                       sga_dtype dt, void *dQ, void *dK, void *dV, void *stream);

/* Graph Transformer with an additive per-edge, per-head score bias (the
 * edge-feature term of "Masked Label Prediction: Unified Message Passing
 * Model", the Graph Transformer the IO-aware layers pages cite, in its
 * simplest form; DF-GNN's abstract names the AT-GNN family, GAT and Graph
 * Transformer): s_ij = q_i . k_j / sqrt(D) + bias[e, h] for the CSR entry e
 * of edge (i <- j).  bias: [E, H] float32 (both dtypes), device, 4-byte
 * aligned.  Needs a plan built with opts->edge_bias = 1 (CSR path, edge
 * stream schedule; block-sparse plans are refused).  The backward adds
 * dbias[E, H] float32 = dL/dbias = dS of every edge (written through the
 * plan's transposed-edge map by the dK/dV pass). */
sga_status gt_attn_bias_fwd(const sga_plan *plan, const int32_t *indptr, const int32_t *indices,
                            const void *Q, const void *K, const void *V, const float *bias,
                            int64_t N, int64_t E, int H, int D, sga_dtype dt, void *out, float *lse,
                            void *stream);
sga_status gt_attn_bias_bwd(const sga_plan *plan, const int32_t *indptr, const int32_t *indices,
                            const void *Q, const void *K, const void *V, const float *bias,
                            const void *out, const float *lse, const void *dOut, int64_t N,
                            int64_t E, int H, int D, sga_dtype dt, void *dQ, void *dK, void *dV,
                            float *dbias, void *stream);

/* GAT edge attention (the original graph attention score; GAT and the Graph
 * Transformer are the attention GNNs DF-GNN's abstract names): with the
 * projected features Fv [N, H, D] (in dt) and the two per-node halves of the
 * score el, er [N, H] (float32; el_i = a_l . Fv_i, er_j = a_r . Fv_j, dense
 * per-node dots the caller computes),
 *   e_ij = LeakyReLU_slope(el_i + er_j), p = softmax over the row,
 *   out_i = sum_j p_ij Fv_j, lse as above.
 * The backward returns the edge stage's gradients: dFv [N, H, D] (in dt; the
 * value path, sum over j's destinations of p dOut_i), del, der [N, H]
 * float32; the layer's dFL = dFv + a_l del + a_r der and the projection's
 * gradients are dense follow-ups.  Needs a plan built with
 * opts->layer = SGA_LAYER_GAT. */
sga_status gat_attn_fwd(const sga_plan *plan, const int32_t *indptr, const int32_t *indices,
                        const void *Fv, const float *el, const float *er, int64_t N, int64_t E,
                        int H, int D, float slope, sga_dtype dt, void *out, float *lse,
                        void *stream);
sga_status gat_attn_bwd(const sga_plan *plan, const int32_t *indptr, const int32_t *indices,
                        const void *Fv, const float *el, const float *er, const void *out,
                        const float *lse, const void *dOut, int64_t N, int64_t E, int H, int D,
                        float slope, sga_dtype dt, void *dFv, float *del, float *der,
                        void *stream);

/* GATv2 forward: FL = X W_l, FR = X W_r (X [N, F], W [F, H*D], FL/FR written as
 * [N, H, D] and kept for the backward pass); e_ij = sum_d a[h,d]
 * LeakyReLU_slope(FL[i,h,d] + FR[j,h,d]); out_i = sum_j softmax_j(e_ij) FR_j;
 * lse as above.  a: [H, D]. */
sga_status gatv2_fwd(const sga_plan *plan, const int32_t *indptr, const int32_t *indices,
                     const void *X, const void *W_l, const void *W_r, const void *a, int64_t N,
                     int64_t E, int F, int H, int D, float slope, sga_dtype dt, void *FL,
                     void *FR, void *out, float *lse, void *stream);

/* GATv2 backward by the chain rule through the softmax, LeakyReLU and both
 * projections: dX [N, F], dW_l, dW_r [F, H*D], da [H, D] (all in dt).
 * Reductions over nodes (dW, da) run in a fixed order: reproducible. */
sga_status gatv2_bwd(const sga_plan *plan, const int32_t *indptr, const int32_t *indices,
                     const void *X, const void *W_l, const void *W_r, const void *a,
                     const void *FL, const void *FR, const void *out, const float *lse,
                     const void *dOut, int64_t N, int64_t E, int F, int H, int D, float slope,
                     sga_dtype dt, void *dX, void *dW_l, void *dW_r, void *da, void *stream);

/* ---- min / max aggregation ------------------------------------------------
 *
 * The degree-aware reduction layer of "On Efficient Scaling of GNNs via
 * IO-Aware Layers Implementations" (arXiv abstract: degree-aware reduction
 * kernels; Yandex Research blog post, "Aggregation layers" paragraph):
 * out_i[f] = max (or min) over the sources j of row i of X_j[f], for every
 * element f of the node rows ([N, H, D] tensors read as [N, H*D]).  Needs a
 * plan built with opts->layer = SGA_LAYER_MINMAX (same N, E, H, D, dt).
 * The winner of an element is the first edge of the row in CSR order among
 * equal values; an empty row gives out = 0.  Values must not be NaN.  Rows
 * above the split threshold are cut into chunks whose partial extremes are
 * merged in chunk order; out is exact (bit-identical to the definition).
 * Optional outputs (NULL: not written):
 *   arg[N, H*D] int32 (16-byte aligned): the winning source node (-1 for an
 *     empty row);
 *   mask[E, R] bytes, R = H*D*sizeof(dt)/16 (sga_agg_mask_bytes): for CSR
 *     edge e and 16-byte chunk c of the row, bit x is set when e won
 *     element 8c + x (bf16) or 4c + x (fp32) of its row; the forward clears
 *     it first.  The backward takes it. */
typedef enum { SGA_AGG_MAX = 0, SGA_AGG_MIN = 1 } sga_agg_op;

sga_status agg_minmax_fwd(const sga_plan *plan, const int32_t *indptr, const int32_t *indices,
                          const void *X, int64_t N, int64_t E, int H, int D, sga_dtype dt,
                          sga_agg_op op, void *out, int32_t *arg, uint8_t *mask, void *stream);

/* Bytes of the forward's win mask for this plan (0 for other plans). */
size_t sga_agg_mask_bytes(const sga_plan *plan);

/* Backward of the min / max aggregation: dX_j[f] = sum of dOut_i[f] over the
 * rows i whose element f was won by an edge from j (mask from the forward).
 * One warp per source (or chunk of a high-degree source) walks its
 * destinations over the transposed CSR and reads a destination's dOut chunk
 * only where the mask has a bit; no atomics, sums in a fixed order
 * (reproducible). */
sga_status agg_minmax_bwd(const sga_plan *plan, const uint8_t *mask, const void *dOut, int64_t N,
                          int H, int D, sga_dtype dt, void *dX, void *stream);

/* ---- graph reordering ------------------------------------------------------
 *
 * "On Efficient Scaling of GNNs via IO-Aware Layers Implementations" (arXiv
 * abstract) studies graph reordering, which benefits neighbour-parallel
 * (gather-dominated) kernels: relabelled so that rows processed together
 * share neighbours, a graph's gathers hit the cache more often.  The pages
 * name no ordering; two are provided.  A user relabels once (graph and node
 * tensors) and runs the layers on the relabelled graph; the outputs are the
 * relabelled outputs (sga_permute_rows with inverse = 1 maps them back). */
typedef enum {
    SGA_ORDER_DEGREE = 0,  /* descending in-degree (times a node is gathered), ties by id */
    SGA_ORDER_RCM = 1      /* reverse Cuthill-McKee on the symmetrised graph: breadth-first
                              levels from each component's start node (least degree, least
                              id; components in that order), a level ordered by the position
                              of each node's earliest-placed neighbour in the level before,
                              then degree, then id; the whole order reversed.  Degree =
                              row degree + transposed degree (CSR entries) */
} sga_order;

/* perm[N] (device, int32) receives the new id of every node.  Exact and
 * deterministic (bit-identical to the sequential definition).  Allocates its
 * temporary device memory, frees it before returning, synchronises `stream`.
 * The CSR is checked on the device first (indptr[0] = 0, non-decreasing,
 * indptr[N] = E, sources in [0, N)): SGA_EINVAL if it is not valid. */
sga_status sga_reorder(const int32_t *indptr, const int32_t *indices, int64_t N, int64_t E,
                       sga_order method, int32_t *perm, void *stream);

/* The relabelled graph: new row perm[v] holds the sources of old row v as
 * perm[j], in their original order.  new_indptr[N+1], new_indices[E]: device,
 * caller-owned.  Synchronises `stream`.  The CSR (as for sga_reorder) and
 * perm (a permutation of 0..N-1: every entry in range, none repeated) are
 * checked on the device before anything is written: SGA_EINVAL otherwise. */
sga_status sga_relabel_csr(const int32_t *indptr, const int32_t *indices, int64_t N, int64_t E,
                           const int32_t *perm, int32_t *new_indptr, int32_t *new_indices,
                           void *stream);

/* Permute the rows of a node tensor (row_bytes a multiple of 16, buffers
 * 16-byte aligned and distinct): dst[perm[v]] = src[v], or with inverse = 1
 * dst[v] = src[perm[v]].  Asynchronous on `stream`.  perm should be a
 * permutation of 0..N-1 (sga_reorder's output is one); it is not checked
 * here, but a row whose perm entry lies outside [0, N) is skipped (nothing
 * is read or written for it), and a repeated entry leaves the rows it
 * targets to whichever copy lands last. */
sga_status sga_permute_rows(const void *src, int64_t N, int64_t row_bytes, const int32_t *perm,
                            int inverse, void *dst, void *stream);

const char *sga_status_string(sga_status s);

/* Last CUDA error code seen by a call that returned SGA_ECUDA (0 if none). */
int sga_last_cuda_error(void);

/* Device-side range checks: every gathered node id is checked against N before
 * it is dereferenced; a failing check skips the access and sets a bit in the
 * plan's device error word.  This call synchronises `stream`, reads the word
 * into *code, clears it, and returns SGA_EDEVICE_CHECK if it was non-zero. */
sga_status sga_read_device_error(const sga_plan *plan, void *stream, int32_t *code);

/* ---- forward without allocation ------------------------------------------
 *
 * No counterpart on the pages: this entry point exists for callers that must
 * not allocate device memory -- an engine that reserved all of its memory up
 * front, a plugin running inside another runtime that owns the device
 * memory, or a latency-critical loop that cannot afford cudaMalloc's implicit
 * device synchronisation.  It computes exactly what gt_attn_fwd computes
 * (same kernels) but needs no plan and no workspace: the split-row partition
 * and the chunk partials live in one file-scope static device array of
 * 32 MiB (sga_noalloc_scratch_bytes()), which every GPU that loads this
 * library holds until the process exits.
 *
 * Fixed choices and limits: rows of degree > 1024 are split into chunks of
 * 1024 edges; at most 4096 split rows and at most
 * 24 MiB / ((H*D + 2*H) * 4 bytes) chunks per call.  Larger inputs are
 * rejected with SGA_ELIMIT before any edge kernel runs.  The CSR is validated
 * on the device (SGA_EINVAL if invalid).
 *
 * Behaviour: the call synchronises `stream` once (it copies the split count
 * back to the host to size the launches), then launches the edge kernels
 * asynchronously on it.  The first call on a device looks up the array's
 * device address for that device (with that device current); make that
 * first call before any stream capture.  Every call shares the one array and
 * finds the previous call's data in it: calls that can overlap on the GPU
 * (other streams, other host threads) race and must be serialised by the
 * caller.  Allocates
 * nothing: no cudaMalloc, cudaFree or allocating library routine.
 *
 * Range checks: the CSR is validated before the edge kernels run, so their
 * own per-gather range check can fire only if indices change between the
 * validation and the gathers.  Such a failure skips the access and sets a bit
 * in a word of the static array, which sga_noalloc_read_device_error reads. */
sga_status gt_attn_fwd_noalloc(const int32_t *indptr, const int32_t *indices, const void *Q,
                               const void *K, const void *V, int64_t N, int64_t E, int H, int D,
                               sga_dtype dt, void *out, float *lse, void *stream);

/* Size in bytes of the static scratch array behind gt_attn_fwd_noalloc. */
size_t sga_noalloc_scratch_bytes(void);

/* Read and clear the device range-check word of gt_attn_fwd_noalloc on the
 * current device (0: no failed check since the last read).  Synchronises
 * `stream`; returns SGA_EDEVICE_CHECK if the word was non-zero.  It shares the
 * static array with gt_attn_fwd_noalloc, so it must not overlap such a call
 * on another stream. */
sga_status sga_noalloc_read_device_error(void *stream, int32_t *code);

/* ---- plan inspection (tests) -------------------------------------------- */

typedef struct {
    int64_t N, E;
    int32_t H, D, F, dtype;
    int32_t split_threshold, chunk_len;
    int32_t n_split, n_chunks;        /* CSR rows split, and their chunk count */
    int32_t t_n_split, t_n_chunks;    /* the same for the transposed CSR */
    int64_t plan_device_bytes;        /* device memory the plan owns */
    int32_t n_tiles;                  /* block-sparse plans: kept tiles */
    int32_t n_panels;                 /*   panels of 128 rows */
    int64_t E_residual;               /*   edges left in the residual CSR */
    int32_t n_entries;                /*   (row panel, 128-source column panel) pairs with a kept tile */
    int32_t reserved;
} sga_plan_info;

sga_status sga_plan_get_info(const sga_plan *plan, sga_plan_info *info);

typedef enum {
    SGA_ARR_T_INDPTR = 0,     /* [N+1] */
    SGA_ARR_T_DST = 1,        /* [E] */
    SGA_ARR_SPLIT_ROWS = 2,   /* [n_split] */
    SGA_ARR_CHUNK_PTR = 3,    /* [n_split+1] */
    SGA_ARR_CHUNK_ROW = 4,    /* [n_chunks] */
    SGA_ARR_CHUNK_BEG = 5,    /* [n_chunks] */
    SGA_ARR_CHUNK_END = 6,    /* [n_chunks] */
    SGA_ARR_T_SPLIT_ROWS = 7, /* transposed-CSR counterparts of 2..6 */
    SGA_ARR_T_CHUNK_PTR = 8,
    SGA_ARR_T_CHUNK_ROW = 9,
    SGA_ARR_T_CHUNK_BEG = 10,
    SGA_ARR_T_CHUNK_END = 11,
    SGA_ARR_TILE_PTR = 12,    /* [n_panels+1] block-sparse plans */
    SGA_ARR_TILE_COL = 13,    /* [n_tiles] */
    SGA_ARR_TILE_BITS = 14,   /* [n_tiles*64]: the [n_tiles][128] uint16 masks, as int32 words */
    SGA_ARR_R_INDPTR = 15,    /* [N+1] residual CSR */
    SGA_ARR_R_INDICES = 16,   /* [E_residual] */
    SGA_ARR_ROW_ORDER = 17,   /* [N] walking order of the rows (row_order plans) */
    SGA_ARR_T_ROW_ORDER = 18, /* [N] walking order of the transposed rows */
    SGA_ARR_T_EID = 19        /* [E] CSR edge of each transposed entry (edge-bias plans) */
} sga_plan_array;

/* Copy one plan array into caller HOST memory of `count` int32 (must equal the
 * array's length).  Synchronous. */
sga_status sga_plan_copy_array(const sga_plan *plan, sga_plan_array which, int32_t *host_out,
                               int64_t count);

/* ---- instrumentation ------------------------------------------------------ */

/* Kernels launched by this library since the process started (all threads). */
int64_t sga_launch_count(void);

typedef enum {
    SGA_KERN_NONE = 0,
    SGA_KERN_GT_FWD = 1, SGA_KERN_GT_FWD_MERGE = 2,
    SGA_KERN_GT_BWD_DQ = 3, SGA_KERN_GT_BWD_DKDV = 4, SGA_KERN_GT_BWD_MERGE = 5,
    SGA_KERN_GATV2_PROJ = 6, SGA_KERN_GATV2_FWD = 7, SGA_KERN_GATV2_FWD_MERGE = 8,
    SGA_KERN_GATV2_BWD_DST = 9, SGA_KERN_GATV2_BWD_SRC = 10, SGA_KERN_GATV2_BWD_MERGE = 11,
    SGA_KERN_GATV2_BWD_DX = 12, SGA_KERN_GATV2_BWD_DW = 13, SGA_KERN_GATV2_BWD_REDUCE = 14,
    SGA_KERN_BSR_FWD = 15, SGA_KERN_BSR_BWD_DELTA = 16, SGA_KERN_BSR_BWD_DQ = 17,
    SGA_KERN_BSR_BWD_DKDV = 18,
    SGA_KERN_AGG_FWD = 19, SGA_KERN_AGG_FWD_MERGE = 20, SGA_KERN_AGG_BWD = 21,
    SGA_KERN_AGG_BWD_MERGE = 22,
    SGA_KERN_GAT_FWD = 23, SGA_KERN_GAT_BWD_DST = 24, SGA_KERN_GAT_BWD_SRC = 25,
    SGA_KERN_COUNT = 26
} sga_kernel_id;
/* (Planned GATv2 passes merge their split rows inside the edge kernels --
 * the last chunk of a row to finish merges it -- so SGA_KERN_GATV2_FWD_MERGE
 * and SGA_KERN_GATV2_BWD_MERGE are no longer launched.  Graph Transformer
 * passes merge inside the edge kernels when a lane holds two or more 16-byte
 * chunks of a row (H*D above 256 bf16 or 128 fp32 elements) and the rows come
 * from the plan's item lists; otherwise (one chunk per lane, a forward with
 * rows walked in id order, the other edge schedules, gt_attn_fwd_noalloc)
 * split rows are merged by SGA_KERN_GT_FWD_MERGE and SGA_KERN_GT_BWD_MERGE
 * launches.) */

/* Time one kernel kind with CUDA events recorded on the launching stream
 * around each of its launches (at most 4096 launches per window).
 * sga_profile_stop synchronises those events and returns the summed device
 * time in milliseconds and the number of launches timed. */
sga_status sga_profile_start(sga_kernel_id which);
sga_status sga_profile_stop(double *total_ms, int64_t *launches);

#ifdef __cplusplus
}
#endif

#endif /* SGA_H */
