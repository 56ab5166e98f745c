// C ABI entry points: argument checks, plan lifetime, workspace layout,
// dtype dispatch and launch instrumentation.  See include/sga.h for the
// contract of every call.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"
#include "plan.h"

namespace sga {

namespace {

std::atomic<int64_t> g_launches{0};
thread_local int g_last_cuda = 0;

// One profiling window at a time, process wide.
struct Profiler {
    std::mutex mu;
    sga_kernel_id which = SGA_KERN_NONE;
    std::vector<cudaEvent_t> begin, end;
    int used = 0;
    bool open = false;
};
Profiler g_prof;
constexpr int kMaxProfiled = 4096;

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t round256(size_t b) { return (b + 255) & ~size_t(255); }

int da_blocks_for(int num_sms) { return std::max(1, num_sms * 2); }
// Split-K slabs of the weight-gradient GEMMs: at least 256 node rows each,
// at most two per SM.
int dw_slabs_for(int64_t N, int num_sms) {
    const int64_t s = (N + 255) / 256;
    return (int)std::min<int64_t>(std::max<int64_t>(s, 1), std::max(2 * num_sms, 1));
}

void compute_layout(sga_plan *p) {
    WorkspaceLayout &L = p->layout;
    const size_t HD = (size_t)p->H * p->D;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off += round256(bytes);
        return at;
    };
    if (p->layer == SGA_LAYER_MINMAX) {
        L.agg_val = take((size_t)std::max(p->rows.n_chunks, p->cols.n_chunks) * HD * 4);
        L.agg_pos = take((size_t)p->rows.n_chunks * HD * 4);
        L.total = off;
        return;
    }
    if (p->layer == SGA_LAYER_GAT) {
        L.delta = take((size_t)p->N * p->H * 4);
        L.lse_n = take((size_t)p->N * p->H * 4);
        L.fwd_ml = take((size_t)p->rows.n_chunks * p->H * 2 * 4);
        L.fwd_acc = take((size_t)p->rows.n_chunks * HD * 4);
        L.bwd_rowc = take((size_t)p->rows.n_chunks * p->H * 4 * 4);
        L.bwd_col = take((size_t)p->cols.n_chunks * HD * 4);
        L.gat_colc = take((size_t)p->cols.n_chunks * p->H * 4);
        L.total = off;
        return;
    }
    L.delta = take((size_t)p->N * p->H * 4);
    L.lse_n = take((size_t)p->N * p->H * 4);
    L.fwd_ml = take((size_t)p->rows.n_chunks * p->H * 2 * 4);
    L.fwd_acc = take((size_t)p->rows.n_chunks * HD * 4);
    L.bwd_row = take((size_t)p->rows.n_chunks * (p->F > 0 ? 4 : 2) * HD * 4);
    L.bwd_rowc = take((size_t)p->rows.n_chunks * p->H * 2 * 4);
    if (p->tiles.min_nnz > 0) {
        L.zt = take((size_t)p->N * p->H * 4);
        const size_t n_pad = (size_t)((p->N + 127) / 128) * 128;
        L.bsr_lse_t = take(n_pad * p->H * 4);
        L.bsr_delta_t = take(n_pad * p->H * 4);
    }
    if (p->edge_bias) L.bias_t = take((size_t)p->E * p->H * 4);
    L.bwd_col = take((size_t)p->cols.n_chunks * 2 * HD * 4);
    if (p->F > 0) {
        L.da_blocks = da_blocks_for(p->num_sms);
        L.dw_slabs = dw_slabs_for(p->N, p->num_sms);
        L.dfl = take((size_t)p->N * HD * 4);
        L.dfr = take((size_t)p->N * HD * 4);
        L.da_part = take((size_t)L.da_blocks * HD * 4);
        L.da_split = take((size_t)p->rows.n_split * HD * 4);
        L.dw_part = take((size_t)2 * L.dw_slabs * p->F * HD * 4);
        // about 0.6% of the projection outputs need exact rounding; room for 2%
        const int64_t cap = std::max<int64_t>(4096, (int64_t)p->N * HD * 2 / 50);
        L.fix_cap = (int32_t)std::min<int64_t>(cap, INT32_MAX / 16);
        L.fix = take(256 + (size_t)L.fix_cap * 8);
    }
    L.total = off;
}

template <typename P> P *ws_at(const sga_plan *p, size_t off) {
    return reinterpret_cast<P *>(static_cast<char *>(p->ws) + off);
}

sga_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return SGA_OK;
    g_last_cuda = (int)e;
    return SGA_ECUDA;
}

bool supported_shape(int H, int D) {
    return (D == 32 || D == 64 || D == 128) && H >= 1 && (int64_t)H * D <= 1024;
}

// Checks shared by every compute call.
sga_status check_call(const sga_plan *p, const int32_t *indptr, const int32_t *indices,
                      int64_t N, int64_t E, int H, int D, sga_dtype dt, int F) {
    if (!p) return SGA_EINVAL;
    if (dt != SGA_F32 && dt != SGA_BF16) return SGA_EUNSUPPORTED;
    if (!supported_shape(H, D)) return SGA_EUNSUPPORTED;
    if (indptr != p->indptr || indices != p->indices || N != p->N || E != p->E || H != p->H ||
        D != p->D || dt != p->dt || F != p->F)
        return SGA_EINVAL;
    if (p->layout.total > 0 && (!p->ws || p->ws_bytes < p->layout.total)) return SGA_EWORKSPACE;
    return SGA_OK;
}

// Every node tensor of a non-empty graph must be a 16-byte aligned pointer.
bool tensors_ok(int64_t N, std::initializer_list<const void *> ps) {
    if (N == 0) return true;
    for (const void *q : ps)
        if (!q || !aligned(q, 16)) return false;
    return true;
}

}  // namespace

void set_cuda_error(cudaError_t e) { g_last_cuda = (int)e; }
int get_cuda_error() { return g_last_cuda; }

void note_launch(sga_kernel_id which, cudaStream_t s, bool after) {
    if (after) g_launches.fetch_add(1, std::memory_order_relaxed);
    if (g_prof.which != which) return;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    if (g_prof.which != which) return;
    if (!after) {
        if (g_prof.used >= kMaxProfiled) return;
        if ((int)g_prof.begin.size() <= g_prof.used) {
            cudaEvent_t b, e;
            if (cudaEventCreate(&b) != cudaSuccess) return;
            if (cudaEventCreate(&e) != cudaSuccess) {
                cudaEventDestroy(b);
                return;
            }
            g_prof.begin.push_back(b);
            g_prof.end.push_back(e);
        }
        cudaEventRecord(g_prof.begin[g_prof.used], s);
        g_prof.open = true;
    } else if (g_prof.open) {
        cudaEventRecord(g_prof.end[g_prof.used], s);
        g_prof.used++;
        g_prof.open = false;
    }
}

}  // namespace sga

using namespace sga;

extern "C" {

const char *sga_status_string(sga_status s) {
    switch (s) {
        case SGA_OK: return "ok";
        case SGA_EINVAL: return "invalid argument";
        case SGA_EUNSUPPORTED: return "unsupported shape or dtype";
        case SGA_ECUDA: return "CUDA runtime error";
        case SGA_EWORKSPACE: return "workspace missing or too small";
        case SGA_EDEVICE_CHECK: return "device range check failed";
        case SGA_ELIMIT: return "input exceeds the fixed scratch of the no-allocation entry point";
    }
    return "unknown status";
}

int sga_last_cuda_error(void) { return get_cuda_error(); }

int64_t sga_launch_count(void) { return g_launches.load(); }

sga_status sga_plan_create(const int32_t *indptr, const int32_t *indices, int64_t N, int64_t E,
                           int H, int D, sga_dtype dt, const sga_plan_opts *opts, void *stream,
                           sga_plan **out) {
    if (!out) return SGA_EINVAL;
    *out = nullptr;
    if (!indptr || !aligned(indptr, 4)) return SGA_EINVAL;
    if (E > 0 && (!indices || !aligned(indices, 4))) return SGA_EINVAL;
    if (N < 0 || E < 0 || N >= INT32_MAX || E >= INT32_MAX) return SGA_EINVAL;
    if (dt != SGA_F32 && dt != SGA_BF16) return SGA_EUNSUPPORTED;
    if (!supported_shape(H, D)) return SGA_EUNSUPPORTED;
    sga_plan_opts o{};
    if (opts) o = *opts;
    if (o.split_threshold < 0 || o.chunk_len < 0 || o.in_features < 0 || o.tile_min_nnz < 0)
        return SGA_EINVAL;
    if (o.layer != SGA_LAYER_ATTENTION && o.layer != SGA_LAYER_MINMAX && o.layer != SGA_LAYER_GAT)
        return SGA_EINVAL;
    if (o.layer != SGA_LAYER_ATTENTION && (o.in_features != 0 || o.tile_min_nnz != 0)) return SGA_EINVAL;
    if (o.schedule < SGA_SCHED_STREAM || o.schedule > SGA_SCHED_BILEVEL) return SGA_EINVAL;
    if (o.edge_bias != 0 && o.edge_bias != 1) return SGA_EINVAL;
    if (o.row_order < 0 || o.row_order > 2) return SGA_EINVAL;
    if (o.edge_bias && (o.layer != SGA_LAYER_ATTENTION || o.in_features != 0 || o.tile_min_nnz != 0))
        return SGA_EUNSUPPORTED;
    if (o.tile_min_nnz > 0 && (!bsr_fwd_supported(dt, D) || o.tile_min_nnz > 128 * 16))
        return SGA_EUNSUPPORTED;
    if (o.in_features != 0 && (o.in_features % 8 != 0 || o.in_features > 1024))
        return SGA_EUNSUPPORTED;
    sga_plan *p = new (std::nothrow) sga_plan();
    if (!p) return SGA_EINVAL;
    p->N = N;
    p->E = E;
    p->H = H;
    p->D = D;
    p->F = o.in_features;
    p->layer = o.layer;
    p->schedule = o.schedule;
    p->edge_bias = o.edge_bias;
    p->keep_eid = o.edge_bias || o.layer == SGA_LAYER_MINMAX;   // (the aggregation backward's edge map)
    p->row_order = o.row_order == 2 ? 2 : 1;   // 0 (default) and 1: descending degree
    p->dt = dt;
    p->indptr = indptr;
    p->indices = indices;
    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&p->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (ce != cudaSuccess) {
        delete p;
        return cuda_status(ce);
    }
    // Split only rows that are long against a resident warp's average share
    // of the edges (16 warps per SM): the persistent warps walk items longest
    // first, so shorter rows already balance, and every split costs chunk
    // partials and a merge.
    int32_t t_default = 256;
    const int64_t per_warp = E / (16 * (int64_t)std::max(1, p->num_sms));
    while (t_default < 4096 && (int64_t)t_default * 8 <= per_warp) t_default *= 2;
    p->split_threshold = o.split_threshold > 0 ? o.split_threshold : t_default;
    p->chunk_len = o.chunk_len > 0 ? o.chunk_len : std::max(1, p->split_threshold / 2);
    sga_status st = plan_build(p, static_cast<cudaStream_t>(stream));
    if (st != SGA_OK) {
        delete p;
        return st;
    }
    p->tiles.min_nnz = o.tile_min_nnz;   // before the layout: block-sparse plans take more workspace
    compute_layout(p);
    if (o.tile_min_nnz > 0) {
        st = bsr_build(p, static_cast<cudaStream_t>(stream));
        sga_plan *rp = st == SGA_OK ? new (std::nothrow) sga_plan() : nullptr;
        if (st == SGA_OK && !rp) st = SGA_EINVAL;
        if (st == SGA_OK) {   // plan over the residual CSR
            rp->N = N;
            rp->E = p->tiles.E_res;
            rp->H = H;
            rp->D = D;
            rp->dt = dt;
            rp->split_threshold = p->split_threshold;
            rp->chunk_len = p->chunk_len;
            rp->row_order = p->row_order;
            rp->indptr = p->tiles.r_indptr;
            rp->indices = p->tiles.r_indices;
            rp->num_sms = p->num_sms;
            p->residual = rp;
            st = plan_build(rp, static_cast<cudaStream_t>(stream));
            if (st == SGA_OK) {
                compute_layout(rp);
                p->residual_ws = p->layout.total;
                p->layout.total += round256(rp->layout.total);
            }
        }
        if (st != SGA_OK) {
            sga_plan_destroy(p);
            return st;
        }
    }
    *out = p;
    return SGA_OK;
}

size_t sga_plan_workspace_bytes(const sga_plan *plan) { return plan ? plan->layout.total : 0; }

sga_status sga_plan_set_workspace(sga_plan *plan, void *d_workspace, size_t bytes) {
    if (!plan) return SGA_EINVAL;
    if (plan->layout.total > 0) {
        if (!d_workspace || !aligned(d_workspace, 256)) return SGA_EINVAL;
        if (bytes < plan->layout.total) return SGA_EWORKSPACE;
    }
    plan->ws = d_workspace;
    plan->ws_bytes = bytes;
    if (plan->residual) {
        plan->residual->ws = static_cast<char *>(d_workspace) + plan->residual_ws;
        plan->residual->ws_bytes = plan->residual->layout.total;
    }
    return SGA_OK;
}

void sga_plan_destroy(sga_plan *plan) {
    if (!plan) return;
    if (plan->residual) {
        plan_free(plan->residual);
        delete plan->residual;
        plan->residual = nullptr;
    }
    plan_free(plan);
    delete plan;
}

sga_status sga_plan_get_info(const sga_plan *p, sga_plan_info *info) {
    if (!p || !info) return SGA_EINVAL;
    info->N = p->N;
    info->E = p->E;
    info->H = p->H;
    info->D = p->D;
    info->F = p->F;
    info->dtype = (int32_t)p->dt;
    info->split_threshold = p->split_threshold;
    info->chunk_len = p->chunk_len;
    info->n_split = p->rows.n_split;
    info->n_chunks = p->rows.n_chunks;
    info->t_n_split = p->cols.n_split;
    info->t_n_chunks = p->cols.n_chunks;
    info->plan_device_bytes = p->device_bytes + (p->residual ? p->residual->device_bytes : 0);
    info->n_tiles = p->tiles.n_tiles;
    info->n_panels = p->tiles.n_panels;
    info->E_residual = p->tiles.E_res;
    info->n_entries = p->tiles.n_entries;
    return SGA_OK;
}

sga_status sga_plan_copy_array(const sga_plan *p, sga_plan_array which, int32_t *host_out,
                               int64_t count) {
    if (!p || (!host_out && count > 0)) return SGA_EINVAL;
    const int32_t *src = nullptr;
    int64_t n = 0;
    const Partition &R = p->rows, &C = p->cols;
    switch (which) {
        case SGA_ARR_T_INDPTR: src = p->t_indptr; n = p->N + 1; break;
        case SGA_ARR_T_DST: src = p->t_dst; n = p->E; break;
        case SGA_ARR_SPLIT_ROWS: src = R.split_rows; n = R.n_split; break;
        case SGA_ARR_CHUNK_PTR: src = R.chunk_ptr; n = R.n_split + 1; break;
        case SGA_ARR_CHUNK_ROW: src = R.chunk_row; n = R.n_chunks; break;
        case SGA_ARR_CHUNK_BEG: src = R.chunk_beg; n = R.n_chunks; break;
        case SGA_ARR_CHUNK_END: src = R.chunk_end; n = R.n_chunks; break;
        case SGA_ARR_T_SPLIT_ROWS: src = C.split_rows; n = C.n_split; break;
        case SGA_ARR_T_CHUNK_PTR: src = C.chunk_ptr; n = C.n_split + 1; break;
        case SGA_ARR_T_CHUNK_ROW: src = C.chunk_row; n = C.n_chunks; break;
        case SGA_ARR_T_CHUNK_BEG: src = C.chunk_beg; n = C.n_chunks; break;
        case SGA_ARR_T_CHUNK_END: src = C.chunk_end; n = C.n_chunks; break;
        case SGA_ARR_TILE_PTR: src = p->tiles.tile_ptr; n = p->tiles.min_nnz ? p->tiles.n_panels + 1 : 0; break;
        case SGA_ARR_TILE_COL: src = p->tiles.tile_col; n = p->tiles.n_tiles; break;
        case SGA_ARR_TILE_BITS:
            src = reinterpret_cast<const int32_t *>(p->tiles.tile_bits);
            n = (int64_t)p->tiles.n_tiles * 64;
            break;
        case SGA_ARR_R_INDPTR: src = p->tiles.r_indptr; n = p->tiles.min_nnz ? p->N + 1 : 0; break;
        case SGA_ARR_R_INDICES: src = p->tiles.r_indices; n = p->tiles.E_res; break;
        case SGA_ARR_ROW_ORDER: src = R.order; n = R.order ? p->N : 0; break;
        case SGA_ARR_T_ROW_ORDER: src = C.order; n = C.order ? p->N : 0; break;
        case SGA_ARR_T_EID: src = p->t_eid; n = p->t_eid ? p->E : 0; break;
        default: return SGA_EINVAL;
    }
    if (count != n) return SGA_EINVAL;
    if (n == 0) return SGA_OK;
    return cuda_status(cudaMemcpy(host_out, src, sizeof(int32_t) * (size_t)n, cudaMemcpyDeviceToHost));
}

sga_status sga_read_device_error(const sga_plan *p, void *stream, int32_t *code) {
    if (!p || !code) return SGA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, p->d_err, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e == cudaSuccess) e = cudaMemsetAsync(p->d_err, 0, sizeof(int32_t), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    *code = v;
    return v ? SGA_EDEVICE_CHECK : SGA_OK;
}

static GtArgs gt_args(const sga_plan *p) {
    GtArgs a{};
    a.indptr = p->indptr;
    a.indices = p->indices;
    a.t_indptr = p->t_indptr;
    a.t_dst = p->t_dst;
    a.N = p->N;
    a.H = p->H;
    a.D = p->D;
    a.split_threshold = p->split_threshold;
    a.rows = p->rows;
    a.cols = p->cols;
    a.d_err = p->d_err;
    if (p->ws) {
        a.ws_delta = ws_at<float>(p, p->layout.delta);
        a.ws_ml = ws_at<float>(p, p->layout.fwd_ml);
        a.ws_acc = ws_at<float>(p, p->layout.fwd_acc);
        a.ws_row = ws_at<float>(p, p->layout.bwd_row);
        a.ws_rowc = ws_at<float>(p, p->layout.bwd_rowc);
        a.ws_col = ws_at<float>(p, p->layout.bwd_col);
        a.ws_lse = ws_at<float>(p, p->layout.lse_n);
        if (p->edge_bias) a.bias_t = ws_at<float>(p, p->layout.bias_t);
    }
    a.E = p->E;
    a.t_eid = p->t_eid;
    return a;
}

sga_status gt_attn_fwd(const sga_plan *p, const int32_t *indptr, const int32_t *indices,
                       const void *Q, const void *K, const void *V, int64_t N, int64_t E, int H,
                       int D, sga_dtype dt, void *out, float *lse, void *stream) {
    if (p && p->layer != SGA_LAYER_ATTENTION) return SGA_EINVAL;
    sga_status st = check_call(p, indptr, indices, N, E, H, D, dt, p ? p->F : 0);
    if (st != SGA_OK) return st;
    if (!tensors_ok(N, {Q, K, V, out, lse})) return SGA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->residual) {   // block-sparse plan: residual edges on the CSR path, tiles on tcgen05
        GtArgs r = gt_args(p->residual);
        r.Q = Q;
        r.K = K;
        r.V = V;
        r.out_w = out;
        r.lse_w = lse;
        r.d_err = p->d_err;
        cudaError_t e = gt_fwd_t<__nv_bfloat16>(r, s);
        if (e != cudaSuccess) return cuda_status(e);
        BsrArgs b{};
        b.Q = Q;
        b.K = K;
        b.V = V;
        b.out = out;
        b.lse = lse;
        b.tile_ptr = p->tiles.tile_ptr;
        b.tile_col = p->tiles.tile_col;
        b.tile_bits = p->tiles.tile_bits;
        b.panel_info = p->tiles.panel_info;
        b.N = N;
        b.H = H;
        b.D = D;
        b.n_panels = p->tiles.n_panels;
        b.n_tiles = p->tiles.n_tiles;
        b.n_active = p->tiles.n_active;
        b.num_sms = p->num_sms;
        b.d_err = p->d_err;
        return cuda_status(launch_bsr_fwd(b, s));
    }
    GtArgs a = gt_args(p);
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.out_w = out;
    a.lse_w = lse;
    if (p->schedule != SGA_SCHED_STREAM)
        return cuda_status(dt == SGA_F32 ? gt_fwd_sched_t<float>(a, p->schedule, s)
                                         : gt_fwd_sched_t<__nv_bfloat16>(a, p->schedule, s));
    return cuda_status(dt == SGA_F32 ? gt_fwd_t<float>(a, s) : gt_fwd_t<__nv_bfloat16>(a, s));
}

sga_status gt_attn_bwd(const sga_plan *p, const int32_t *indptr, const int32_t *indices,
                       const void *Q, const void *K, const void *V, const void *out,
                       const float *lse, const void *dOut, int64_t N, int64_t E, int H, int D,
                       sga_dtype dt, void *dQ, void *dK, void *dV, void *stream) {
    if (p && p->layer != SGA_LAYER_ATTENTION) return SGA_EINVAL;
    sga_status st = check_call(p, indptr, indices, N, E, H, D, dt, p ? p->F : 0);
    if (st != SGA_OK) return st;
    if (!tensors_ok(N, {Q, K, V, out, lse, dOut, dQ, dK, dV})) return SGA_EINVAL;
    GtArgs a = gt_args(p->residual ? p->residual : p);
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.out = out;
    a.lse = lse;
    a.dOut = dOut;
    a.dQ = dQ;
    a.dK = dK;
    a.dV = dV;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (p->residual) {   // block-sparse plan: tiles on tcgen05 around the residual CSR passes
        BsrBwdArgs b{};
        b.Q = Q;
        b.K = K;
        b.V = V;
        b.dOut = dOut;
        b.lse = lse;
        b.delta_t = ws_at<float>(p, p->layout.delta);
        b.z_t = ws_at<float>(p, p->layout.zt);
        b.dQ = dQ;
        b.dK = dK;
        b.dV = dV;
        b.tile_ptr = p->tiles.tile_ptr;
        b.tile_col = p->tiles.tile_col;
        b.tile_bits = p->tiles.tile_bits;
        b.ct_ptr = p->tiles.ct_ptr;
        b.ct_panel = p->tiles.ct_panel;
        b.ct_tile = p->tiles.ct_tile;
        b.tile_bits_t = p->tiles.tile_bits_t;
        b.panel_info = p->tiles.panel_info;
        b.cpanel_info = p->tiles.cpanel_info;
        b.lse_t = ws_at<float>(p, p->layout.bsr_lse_t);
        b.delta_t_hm = ws_at<float>(p, p->layout.bsr_delta_t);
        b.N = N;
        b.N_pad = (N + 127) / 128 * 128;
        b.H = H;
        b.D = D;
        b.n_panels = p->tiles.n_panels;
        b.n_cpanels = p->tiles.n_cpanels;
        b.n_tiles = p->tiles.n_tiles;
        b.n_active = p->tiles.n_active;
        b.n_cactive = p->tiles.n_cactive;
        b.num_sms = p->num_sms;
        b.d_err = p->d_err;
        cudaError_t e = cudaMemsetAsync(b.delta_t, 0, sizeof(float) * (size_t)N * H, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(b.z_t, 0, sizeof(float) * (size_t)N * H, s);
        if (e == cudaSuccess) e = launch_bsr_bwd_delta(b, s);
        a.delta_in = b.delta_t;   // the residual rows' C and Z gain the tile parts
        a.z_in = b.z_t;
        a.d_err = p->d_err;
        if (e == cudaSuccess) e = gt_bwd_t<__nv_bfloat16>(a, s);
        b.delta = a.ws_delta;     // full (normalised) Delta of every row
        b.lse_n = a.ws_lse;       // and lse + ln Z
        if (e == cudaSuccess) e = launch_bsr_bwd_dq(b, s);
        if (e == cudaSuccess) e = launch_bsr_bwd_dkdv(b, s);
        return cuda_status(e);
    }
    return cuda_status(dt == SGA_F32 ? gt_bwd_t<float>(a, s) : gt_bwd_t<__nv_bfloat16>(a, s));
}

sga_status gt_attn_bias_fwd(const sga_plan *p, const int32_t *indptr, const int32_t *indices,
                            const void *Q, const void *K, const void *V, const float *bias,
                            int64_t N, int64_t E, int H, int D, sga_dtype dt, void *out, float *lse,
                            void *stream) {
    if (p && (p->layer != SGA_LAYER_ATTENTION || !p->edge_bias)) return SGA_EINVAL;
    sga_status st = check_call(p, indptr, indices, N, E, H, D, dt, 0);
    if (st != SGA_OK) return st;
    if (p->schedule != SGA_SCHED_STREAM || p->residual) return SGA_EUNSUPPORTED;
    if (!tensors_ok(N, {Q, K, V, out, lse})) return SGA_EINVAL;
    if (E > 0 && (!bias || !aligned(bias, 4))) return SGA_EINVAL;
    GtArgs a = gt_args(p);
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.out_w = out;
    a.lse_w = lse;
    a.bias = E > 0 ? bias : nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(dt == SGA_F32 ? gt_fwd_t<float>(a, s) : gt_fwd_t<__nv_bfloat16>(a, s));
}

sga_status gt_attn_bias_bwd(const sga_plan *p, const int32_t *indptr, const int32_t *indices,
                            const void *Q, const void *K, const void *V, const float *bias,
                            const void *out, const float *lse, const void *dOut, int64_t N,
                            int64_t E, int H, int D, sga_dtype dt, void *dQ, void *dK, void *dV,
                            float *dbias, void *stream) {
    if (p && (p->layer != SGA_LAYER_ATTENTION || !p->edge_bias)) return SGA_EINVAL;
    sga_status st = check_call(p, indptr, indices, N, E, H, D, dt, 0);
    if (st != SGA_OK) return st;
    if (p->residual) return SGA_EUNSUPPORTED;
    if (!tensors_ok(N, {Q, K, V, out, lse, dOut, dQ, dK, dV})) return SGA_EINVAL;
    if (E > 0 && (!bias || !dbias || !aligned(bias, 4) || !aligned(dbias, 4))) return SGA_EINVAL;
    GtArgs a = gt_args(p);
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.out = out;
    a.lse = lse;
    a.dOut = dOut;
    a.dQ = dQ;
    a.dK = dK;
    a.dV = dV;
    a.bias = E > 0 ? bias : nullptr;
    a.dbias = dbias;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(dt == SGA_F32 ? gt_bwd_t<float>(a, s) : gt_bwd_t<__nv_bfloat16>(a, s));
}

static Gatv2Args gatv2_args(const sga_plan *p, float slope) {
    Gatv2Args a{};
    a.indptr = p->indptr;
    a.indices = p->indices;
    a.t_indptr = p->t_indptr;
    a.t_dst = p->t_dst;
    a.N = p->N;
    a.F = p->F;
    a.H = p->H;
    a.D = p->D;
    a.slope = slope;
    a.split_threshold = p->split_threshold;
    a.rows = p->rows;
    a.cols = p->cols;
    a.d_err = p->d_err;
    a.da_blocks = p->layout.da_blocks;
    a.dw_slabs = p->layout.dw_slabs;
    if (p->ws) {
        a.ws_delta = ws_at<float>(p, p->layout.delta);
        a.ws_ml = ws_at<float>(p, p->layout.fwd_ml);
        a.ws_acc = ws_at<float>(p, p->layout.fwd_acc);
        a.ws_row = ws_at<float>(p, p->layout.bwd_row);
        a.ws_col = ws_at<float>(p, p->layout.bwd_col);
        a.ws_rowc = ws_at<float>(p, p->layout.bwd_rowc);
        a.ws_lse = ws_at<float>(p, p->layout.lse_n);
        a.ws_da = ws_at<float>(p, p->layout.da_part);
        a.ws_da_split = ws_at<float>(p, p->layout.da_split);
        a.ws_dw = ws_at<float>(p, p->layout.dw_part);
        a.ws_dfl = ws_at<float>(p, p->layout.dfl);
        a.ws_dfr = ws_at<float>(p, p->layout.dfr);
        a.ws_fix_count = ws_at<int32_t>(p, p->layout.fix);
        a.ws_fix_list = ws_at<int2>(p, p->layout.fix + 256);
        a.fix_cap = p->layout.fix_cap;
    }
    return a;
}

sga_status gatv2_fwd(const sga_plan *p, const int32_t *indptr, const int32_t *indices,
                     const void *X, const void *W_l, const void *W_r, const void *att, int64_t N,
                     int64_t E, int F, int H, int D, float slope, sga_dtype dt, void *FL, void *FR,
                     void *out, float *lse, void *stream) {
    if (p && p->F == 0) return SGA_EINVAL;
    sga_status st = check_call(p, indptr, indices, N, E, H, D, dt, F);
    if (st != SGA_OK) return st;
    if (!tensors_ok(N, {X, FL, FR, out, lse})) return SGA_EINVAL;
    if (!tensors_ok(1, {W_l, W_r, att})) return SGA_EINVAL;
    Gatv2Args a = gatv2_args(p, slope);
    a.X = X;
    a.Wl = W_l;
    a.Wr = W_r;
    a.a = att;
    a.FL_w = FL;
    a.FR_w = FR;
    a.out_w = out;
    a.lse_w = lse;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(dt == SGA_F32 ? gatv2_fwd_t<float>(a, s) : gatv2_fwd_t<__nv_bfloat16>(a, s));
}

sga_status gatv2_bwd(const sga_plan *p, const int32_t *indptr, const int32_t *indices,
                     const void *X, const void *W_l, const void *W_r, const void *att,
                     const void *FL, const void *FR, const void *out, const float *lse,
                     const void *dOut, int64_t N, int64_t E, int F, int H, int D, float slope,
                     sga_dtype dt, void *dX, void *dW_l, void *dW_r, void *da, void *stream) {
    if (p && p->F == 0) return SGA_EINVAL;
    sga_status st = check_call(p, indptr, indices, N, E, H, D, dt, F);
    if (st != SGA_OK) return st;
    if (!tensors_ok(N, {X, FL, FR, out, lse, dOut, dX})) return SGA_EINVAL;
    if (!tensors_ok(1, {W_l, W_r, att, dW_l, dW_r, da})) return SGA_EINVAL;
    Gatv2Args a = gatv2_args(p, slope);
    a.X = X;
    a.Wl = W_l;
    a.Wr = W_r;
    a.a = att;
    a.FL = FL;
    a.FR = FR;
    a.out = out;
    a.lse = lse;
    a.dOut = dOut;
    a.dX = dX;
    a.dWl = dW_l;
    a.dWr = dW_r;
    a.da = da;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(dt == SGA_F32 ? gatv2_bwd_t<float>(a, s) : gatv2_bwd_t<__nv_bfloat16>(a, s));
}

static AggArgs agg_args(const sga_plan *p) {
    AggArgs a{};
    a.indptr = p->indptr;
    a.indices = p->indices;
    a.t_dst = p->t_dst;
    a.t_eid = p->t_eid;
    a.N = p->N;
    a.E = p->E;
    a.HD = p->H * p->D;
    a.split_threshold = p->split_threshold;
    a.num_sms = p->num_sms;
    a.rows = p->rows;
    a.cols = p->cols;
    a.d_err = p->d_err;
    if (p->ws) {
        a.ws_val = ws_at<float>(p, p->layout.agg_val);
        a.ws_pos = ws_at<int32_t>(p, p->layout.agg_pos);
    }
    return a;
}

sga_status agg_minmax_fwd(const sga_plan *p, const int32_t *indptr, const int32_t *indices,
                          const void *X, int64_t N, int64_t E, int H, int D, sga_dtype dt,
                          sga_agg_op op, void *out, int32_t *arg, uint8_t *mask, void *stream) {
    if (p && p->layer != SGA_LAYER_MINMAX) return SGA_EINVAL;
    if (op != SGA_AGG_MAX && op != SGA_AGG_MIN) return SGA_EINVAL;
    sga_status st = check_call(p, indptr, indices, N, E, H, D, dt, 0);
    if (st != SGA_OK) return st;
    if (!tensors_ok(N, {X, out})) return SGA_EINVAL;
    if (arg && N > 0 && !aligned(arg, 16)) return SGA_EINVAL;
    AggArgs a = agg_args(p);
    a.X = X;
    a.out = out;
    a.arg = arg;
    a.mask = mask;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool mx = op == SGA_AGG_MAX;
    return cuda_status(dt == SGA_F32 ? agg_fwd_t<float>(a, mx, s) : agg_fwd_t<__nv_bfloat16>(a, mx, s));
}

size_t sga_agg_mask_bytes(const sga_plan *p) {
    if (!p || p->layer != SGA_LAYER_MINMAX) return 0;
    return (size_t)p->E * ((size_t)p->H * p->D * (p->dt == SGA_F32 ? 4 : 2) / 16);
}

sga_status agg_minmax_bwd(const sga_plan *p, const uint8_t *mask, const void *dOut, int64_t N,
                          int H, int D, sga_dtype dt, void *dX, void *stream) {
    if (!p || p->layer != SGA_LAYER_MINMAX) return SGA_EINVAL;
    if (N != p->N || H != p->H || D != p->D || dt != p->dt) return SGA_EINVAL;
    if (p->layout.total > 0 && (!p->ws || p->ws_bytes < p->layout.total)) return SGA_EWORKSPACE;
    if (!tensors_ok(N, {dOut, dX})) return SGA_EINVAL;
    if (p->E > 0 && !mask) return SGA_EINVAL;
    AggArgs a = agg_args(p);
    a.mask = const_cast<uint8_t *>(mask);
    a.dOut = dOut;
    a.dX = dX;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(dt == SGA_F32 ? agg_bwd_t<float>(a, s) : agg_bwd_t<__nv_bfloat16>(a, s));
}

static GatArgs gat_args(const sga_plan *p, float slope) {
    GatArgs a{};
    a.indptr = p->indptr;
    a.indices = p->indices;
    a.t_indptr = p->t_indptr;
    a.t_dst = p->t_dst;
    a.N = p->N;
    a.H = p->H;
    a.D = p->D;
    a.slope = slope;
    a.split_threshold = p->split_threshold;
    a.rows = p->rows;
    a.cols = p->cols;
    a.d_err = p->d_err;
    if (p->ws) {
        a.ws_delta = ws_at<float>(p, p->layout.delta);
        a.ws_lse = ws_at<float>(p, p->layout.lse_n);
        a.ws_ml = ws_at<float>(p, p->layout.fwd_ml);
        a.ws_acc = ws_at<float>(p, p->layout.fwd_acc);
        a.ws_rowc = ws_at<float>(p, p->layout.bwd_rowc);
        a.ws_col = ws_at<float>(p, p->layout.bwd_col);
        a.ws_colc = ws_at<float>(p, p->layout.gat_colc);
    }
    return a;
}

sga_status gat_attn_fwd(const sga_plan *p, const int32_t *indptr, const int32_t *indices,
                        const void *Fv, const float *el, const float *er, int64_t N, int64_t E,
                        int H, int D, float slope, sga_dtype dt, void *out, float *lse,
                        void *stream) {
    if (p && p->layer != SGA_LAYER_GAT) return SGA_EINVAL;
    sga_status st = check_call(p, indptr, indices, N, E, H, D, dt, 0);
    if (st != SGA_OK) return st;
    if (!tensors_ok(N, {Fv, out, lse, el, er})) return SGA_EINVAL;
    GatArgs a = gat_args(p, slope);
    a.Fv = Fv;
    a.el = el;
    a.er = er;
    a.out_w = out;
    a.lse_w = lse;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(dt == SGA_F32 ? gat_fwd_t<float>(a, s) : gat_fwd_t<__nv_bfloat16>(a, s));
}

sga_status gat_attn_bwd(const sga_plan *p, const int32_t *indptr, const int32_t *indices,
                        const void *Fv, const float *el, const float *er, const void *out,
                        const float *lse, const void *dOut, int64_t N, int64_t E, int H, int D,
                        float slope, sga_dtype dt, void *dFv, float *del, float *der,
                        void *stream) {
    if (p && p->layer != SGA_LAYER_GAT) return SGA_EINVAL;
    sga_status st = check_call(p, indptr, indices, N, E, H, D, dt, 0);
    if (st != SGA_OK) return st;
    if (!tensors_ok(N, {Fv, el, er, out, lse, dOut, dFv, del, der})) return SGA_EINVAL;
    GatArgs a = gat_args(p, slope);
    a.Fv = Fv;
    a.el = el;
    a.er = er;
    a.lse = lse;
    a.dOut = dOut;
    a.dFv = dFv;
    a.del = del;
    a.der = der;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return cuda_status(dt == SGA_F32 ? gat_bwd_t<float>(a, s) : gat_bwd_t<__nv_bfloat16>(a, s));
}

sga_status sga_profile_start(sga_kernel_id which) {
    if (which <= SGA_KERN_NONE || which >= SGA_KERN_COUNT) return SGA_EINVAL;
    std::lock_guard<std::mutex> lk(g_prof.mu);
    g_prof.which = which;
    g_prof.used = 0;
    g_prof.open = false;
    return SGA_OK;
}

sga_status sga_profile_stop(double *total_ms, int64_t *launches) {
    std::lock_guard<std::mutex> lk(g_prof.mu);
    double tot = 0.0;
    for (int i = 0; i < g_prof.used; ++i) {
        cudaError_t e = cudaEventSynchronize(g_prof.end[i]);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, g_prof.begin[i], g_prof.end[i]);
        if (e != cudaSuccess) {
            g_prof.which = SGA_KERN_NONE;
            return cuda_status(e);
        }
        tot += ms;
    }
    if (total_ms) *total_ms = tot;
    if (launches) *launches = g_prof.used;
    g_prof.which = SGA_KERN_NONE;
    g_prof.used = 0;
    g_prof.open = false;
    return SGA_OK;
}

}  // extern "C"
