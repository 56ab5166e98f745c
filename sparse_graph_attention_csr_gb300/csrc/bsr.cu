// Block-sparse split of a destination-sorted CSR for the tensor-core passes:
// the "block-sparse graph representation that enables the use of tensor
// cores" of the IO-aware layers blog post ("Attention-based layers"
// paragraph), which pays off on locally dense graphs.
//
// Rows form panels of 128 destinations, sources form column tiles of 16.  A
// (panel, tile) pair holding at least min_nnz edges is kept: its column index
// and one 16-bit source mask per panel row are stored.  A mask holds a
// (destination, source) pair once, so a repeated edge of a kept tile (the same
// pair again, later in CSR order) joins the residual: the softmax runs over
// edges, and the residual pass adds its term.  All other edges stay in a
// residual CSR, in their original order.
//
// The split is found by sorting the edges by (panel, tile, row within the
// panel, source within the tile), least significant key first, with stable
// radix passes: runs of equal (panel, tile) are the candidate tiles, and a
// repeated edge sits right after its first occurrence.  Nothing depends on
// the number of nodes beyond the int32 index range, and every array is
// determined by the graph and min_nnz (bit-exact).
#include <algorithm>
#include <numeric>
#include <vector>

#include "common.cuh"
#include "plan.h"

namespace sga {
namespace {

constexpr int kPanel = 128, kWidth = 16;

unsigned grid_of(int64_t n, int64_t cap = 65535) {
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>((n + 255) / 256, cap));
}

// destination row of every edge (a warp per row)
__global__ void edge_dst_kernel(const int32_t *__restrict__ indptr, int64_t N, int32_t *__restrict__ rows) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < N; i += nw)
        for (int32_t e = indptr[i] + lane; e < indptr[i + 1]; e += 32) rows[e] = (int32_t)i;
}

// least significant sort key: (row within the panel, source within the tile)
__global__ void key_low_kernel(const int32_t *__restrict__ rows, const int32_t *__restrict__ indices, int64_t E,
                               int32_t *__restrict__ key, int32_t *__restrict__ val) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += stride) {
        key[e] = ((rows[e] & (kPanel - 1)) << 4) | (indices[e] & (kWidth - 1));
        val[e] = (int32_t)e;
    }
}

// next key of the sorted edges: src[edge] >> shift (the tile, then the panel)
__global__ void key_gather_kernel(const int32_t *__restrict__ src, int shift, const int32_t *__restrict__ val,
                                  int64_t E, int32_t *__restrict__ key) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < E; k += stride) key[k] = src[val[k]] >> shift;
}

// run heads (a new (panel, tile) pair) and repeats (the same pair as the
// previous edge in sorted order) of the sorted edges
__global__ void run_flags_kernel(const int32_t *__restrict__ rows, const int32_t *__restrict__ indices,
                                 const int32_t *__restrict__ val, int64_t E, int32_t *__restrict__ head,
                                 uint8_t *__restrict__ rep) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < E; k += stride) {
        const int32_t e = val[k], r = rows[e], j = indices[e];
        int32_t h = 1;
        uint8_t rp = 0;
        if (k > 0) {
            const int32_t e1 = val[k - 1], r1 = rows[e1], j1 = indices[e1];
            h = (r >> 7) != (r1 >> 7) || (j >> 4) != (j1 >> 4);
            rp = r == r1 && j == j1;
        }
        head[k] = h;
        rep[k] = rp;
    }
}

__global__ void run_start_kernel(const int32_t *__restrict__ head, const int32_t *__restrict__ run_excl, int64_t E,
                                 int32_t *__restrict__ start) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < E; k += stride)
        if (head[k]) start[run_excl[k]] = (int32_t)k;
}

// keep[r] = run r holds at least min_nnz edges (keep[n_runs] = 0)
__global__ void run_keep_kernel(const int32_t *__restrict__ start, int64_t n_runs, int64_t E, int min_nnz,
                                int32_t *__restrict__ keep) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r <= n_runs; r += stride) {
        if (r == n_runs) {
            keep[r] = 0;
            continue;
        }
        const int64_t end = r + 1 < n_runs ? start[r + 1] : E;
        keep[r] = end - start[r] >= min_nnz;
    }
}

// column and panel of every kept tile
__global__ void tile_info_kernel(const int32_t *__restrict__ start, const int32_t *__restrict__ keep,
                                 const int32_t *__restrict__ tix, int64_t n_runs, const int32_t *__restrict__ val,
                                 const int32_t *__restrict__ rows, const int32_t *__restrict__ indices,
                                 int32_t *__restrict__ tile_col, int32_t *__restrict__ panel_count) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < n_runs; r += stride)
        if (keep[r]) {
            const int32_t e = val[start[r]];
            tile_col[tix[r]] = indices[e] >> 4;
            atomicAdd(&panel_count[rows[e] >> 7], 1);
        }
}

// mask bits of the kept, first-occurrence edges; residual flag of the others
__global__ void tile_bits_kernel(const int32_t *__restrict__ head, const int32_t *__restrict__ run_excl,
                                 const uint8_t *__restrict__ rep, const int32_t *__restrict__ keep,
                                 const int32_t *__restrict__ tix, const int32_t *__restrict__ val,
                                 const int32_t *__restrict__ rows, const int32_t *__restrict__ indices, int64_t E,
                                 uint32_t *__restrict__ bits32, uint8_t *__restrict__ res) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < E; k += stride) {
        const int32_t run = run_excl[k] + head[k] - 1, e = val[k];
        if (keep[run] && !rep[k]) {
            const int32_t r = rows[e], j = indices[e];
            const int64_t word = ((int64_t)tix[run] * kPanel + (r & (kPanel - 1))) >> 1;
            atomicOr(&bits32[word], (1u << (j & (kWidth - 1))) << ((r & 1) * 16));
            res[e] = 0;
        } else {
            res[e] = 1;
        }
    }
}

// residual edges per row (a warp per row)
__global__ void res_count_kernel(const int32_t *__restrict__ indptr, int64_t N, const uint8_t *__restrict__ res,
                                 int32_t *__restrict__ count) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < N; i += nw) {
        int n = 0;
        for (int32_t e = indptr[i] + lane; e < indptr[i + 1]; e += 32) n += res[e];
        for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(SGA_FULL_MASK, n, o);
        if (lane == 0) count[i] = n;
    }
}

// residual sources of every row, in CSR order (a warp per row)
__global__ void res_fill_kernel(const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices, int64_t N,
                                const uint8_t *__restrict__ res, const int32_t *__restrict__ r_indptr,
                                int32_t *__restrict__ r_indices) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < N; i += nw) {
        int32_t out = r_indptr[i];
        const int32_t b = indptr[i], end = indptr[i + 1];
        for (int32_t x0 = b; x0 < end; x0 += 32) {
            const int32_t x = x0 + lane;
            const bool take = x < end && res[x];
            const unsigned m = __ballot_sync(SGA_FULL_MASK, take);
            if (take) r_indices[out + __popc(m & ((1u << lane) - 1))] = indices[x];
            out += __popc(m);
        }
    }
}

// transposed masks for the column pass: word (t, half, c) holds in bit i
// whether row 64 half + i of tile t has source c
__global__ void tile_bits_t_kernel(const uint16_t *__restrict__ bits, int64_t n_tiles, uint64_t *__restrict__ bt) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n_tiles * 32; x += stride) {
        const int64_t t = x >> 5;
        const int hf = (int)(x >> 4) & 1, c = (int)x & 15;
        const uint16_t *b = bits + t * kPanel + hf * 64;
        uint64_t w = 0;
        for (int i = 0; i < 64; ++i) w |= (uint64_t)((b[i] >> c) & 1u) << i;
        bt[x] = w;
    }
}

int bits_for(int64_t max_value) {
    int b = 1;
    while (b < 31 && ((int64_t)1 << b) <= max_value) ++b;
    return b;
}

}  // namespace

sga_status bsr_build(sga_plan *p, cudaStream_t s) {
    TileSet &T = p->tiles;
    const int64_t N = p->N, E = p->E;
    T.n_panels = (int32_t)((N + kPanel - 1) / kPanel);
    std::vector<void *> tmp;
    auto fail = [&](cudaError_t e) {
        for (void *x : tmp) cudaFree(x);
        set_cuda_error(e);
        return SGA_ECUDA;
    };
    auto alloc = [&](void **ptr, size_t bytes, bool own) -> cudaError_t {
        cudaError_t e = cudaMalloc(ptr, std::max<size_t>(bytes, 16));
        if (e == cudaSuccess) {
            if (own) {
                p->owned.push_back(*ptr);
                p->device_bytes += (int64_t)bytes;
            } else {
                tmp.push_back(*ptr);
            }
        }
        return e;
    };
#define BSR_TRY(x)                                   \
    do {                                             \
        const cudaError_t e_ = (x);                  \
        if (e_ != cudaSuccess) return fail(e_);      \
    } while (0)
    const int64_t En = E + 1;   // run arrays hold up to E + 1 entries
    int32_t *rows, *ka, *va, *kb, *vb, *head, *run_excl, *hist, *scan_tmp, *panel_count;
    uint8_t *rep, *res;
    BSR_TRY(alloc((void **)&rows, 4 * (size_t)En, false));
    BSR_TRY(alloc((void **)&ka, 4 * (size_t)En, false));
    BSR_TRY(alloc((void **)&va, 4 * (size_t)En, false));
    BSR_TRY(alloc((void **)&kb, 4 * (size_t)En, false));
    BSR_TRY(alloc((void **)&vb, 4 * (size_t)En, false));
    BSR_TRY(alloc((void **)&head, 4 * (size_t)En, false));
    BSR_TRY(alloc((void **)&run_excl, 4 * (size_t)En, false));
    BSR_TRY(alloc((void **)&rep, (size_t)En, false));
    BSR_TRY(alloc((void **)&res, (size_t)En, false));
    BSR_TRY(alloc((void **)&panel_count, 4 * (size_t)(T.n_panels + 1), false));
    const int64_t hist_n = radix_hist_elems(En);
    BSR_TRY(alloc((void **)&hist, 4 * (size_t)hist_n, false));
    BSR_TRY(alloc((void **)&scan_tmp,
                  4 * (size_t)scan_tmp_elems(std::max<int64_t>({hist_n, En + 1, N + 1, (int64_t)T.n_panels + 1})),
                  false));
    BSR_TRY(alloc((void **)&T.tile_ptr, sizeof(int32_t) * (T.n_panels + 1), true));
    BSR_TRY(alloc((void **)&T.r_indptr, sizeof(int32_t) * (N + 1), true));
    BSR_TRY(cudaMemsetAsync(panel_count, 0, 4 * (size_t)(T.n_panels + 1), s));
    BSR_TRY(cudaMemsetAsync(T.r_indptr, 0, 4 * (size_t)(N + 1), s));

    // sort the edges by (panel, tile, row % 128, source % 16), ties in CSR order
    int64_t n_runs = 0;
    if (E > 0) {
        edge_dst_kernel<<<grid_of(N * 32), 256, 0, s>>>(p->indptr, N, rows);
        key_low_kernel<<<grid_of(E), 256, 0, s>>>(rows, p->indices, E, ka, va);
        BSR_TRY(cudaGetLastError());
        BSR_TRY(radix_sort_pairs(&ka, &va, &kb, &vb, E, 11, hist, scan_tmp, s));
        key_gather_kernel<<<grid_of(E), 256, 0, s>>>(p->indices, 4, va, E, ka);
        BSR_TRY(cudaGetLastError());
        BSR_TRY(radix_sort_pairs(&ka, &va, &kb, &vb, E, bits_for((N - 1) >> 4), hist, scan_tmp, s));
        key_gather_kernel<<<grid_of(E), 256, 0, s>>>(rows, 7, va, E, ka);
        BSR_TRY(cudaGetLastError());
        BSR_TRY(radix_sort_pairs(&ka, &va, &kb, &vb, E, bits_for((N - 1) >> 7), hist, scan_tmp, s));
        run_flags_kernel<<<grid_of(E), 256, 0, s>>>(rows, p->indices, va, E, head, rep);
        BSR_TRY(cudaGetLastError());
        BSR_TRY(exclusive_scan(head, run_excl, E, scan_tmp, s));
        int32_t last[2];
        BSR_TRY(cudaMemcpyAsync(&last[0], run_excl + E - 1, 4, cudaMemcpyDeviceToHost, s));
        BSR_TRY(cudaMemcpyAsync(&last[1], head + E - 1, 4, cudaMemcpyDeviceToHost, s));
        BSR_TRY(cudaStreamSynchronize(s));
        n_runs = (int64_t)last[0] + last[1];
    }
    // runs -> kept tiles (kb: run starts, vb: keep flags then tile index of each run;
    // both hold at most E + 1 entries)
    int32_t *start = kb, *keep = vb, *tix = ka;
    if (n_runs > 0) {
        run_start_kernel<<<grid_of(E), 256, 0, s>>>(head, run_excl, E, start);
        run_keep_kernel<<<grid_of(n_runs + 1), 256, 0, s>>>(start, n_runs, E, T.min_nnz, keep);
        BSR_TRY(cudaGetLastError());
        BSR_TRY(exclusive_scan(keep, tix, n_runs + 1, scan_tmp, s));
        int32_t nt = 0;
        BSR_TRY(cudaMemcpyAsync(&nt, tix + n_runs, 4, cudaMemcpyDeviceToHost, s));
        BSR_TRY(cudaStreamSynchronize(s));
        T.n_tiles = nt;
    }
    // one extra all-zero mask tile (index n_tiles) stands in for missing tiles
    BSR_TRY(alloc((void **)&T.tile_col, sizeof(int32_t) * (size_t)T.n_tiles, true));
    BSR_TRY(alloc((void **)&T.tile_bits, sizeof(uint16_t) * kPanel * (size_t)(T.n_tiles + 1), true));
    BSR_TRY(cudaMemsetAsync(T.tile_bits, 0, sizeof(uint16_t) * kPanel * (size_t)(T.n_tiles + 1), s));
    BSR_TRY(alloc((void **)&T.tile_bits_t, sizeof(uint64_t) * 32 * (size_t)(T.n_tiles + 1), true));
    BSR_TRY(cudaMemsetAsync(T.tile_bits_t, 0, sizeof(uint64_t) * 32 * (size_t)(T.n_tiles + 1), s));
    if (n_runs > 0) {
        tile_info_kernel<<<grid_of(n_runs), 256, 0, s>>>(start, keep, tix, n_runs, va, rows, p->indices,
                                                          T.tile_col, panel_count);
        tile_bits_kernel<<<grid_of(E), 256, 0, s>>>(head, run_excl, rep, keep, tix, va, rows, p->indices, E,
                                                    reinterpret_cast<uint32_t *>(T.tile_bits), res);
        BSR_TRY(cudaGetLastError());
    }
    if (T.n_tiles > 0) {
        tile_bits_t_kernel<<<grid_of((int64_t)T.n_tiles * 32), 256, 0, s>>>(T.tile_bits, T.n_tiles, T.tile_bits_t);
        BSR_TRY(cudaGetLastError());
    }
    BSR_TRY(exclusive_scan(panel_count, T.tile_ptr, T.n_panels + 1, scan_tmp, s));
    if (E > 0) {
        res_count_kernel<<<grid_of(N * 32), 256, 0, s>>>(p->indptr, N, res, T.r_indptr);
        BSR_TRY(cudaGetLastError());
    }
    BSR_TRY(exclusive_scan(T.r_indptr, T.r_indptr, N + 1, scan_tmp, s));
    int32_t e_res = 0;
    BSR_TRY(cudaMemcpyAsync(&e_res, T.r_indptr + N, 4, cudaMemcpyDeviceToHost, s));
    BSR_TRY(cudaStreamSynchronize(s));
    T.E_res = e_res;
    BSR_TRY(alloc((void **)&T.r_indices, sizeof(int32_t) * (size_t)T.E_res, true));
    if (T.E_res > 0) {
        res_fill_kernel<<<grid_of(N * 32), 256, 0, s>>>(p->indptr, p->indices, N, res, T.r_indptr, T.r_indices);
        BSR_TRY(cudaGetLastError());
    }
    BSR_TRY(cudaStreamSynchronize(s));
    for (void *x : tmp) cudaFree(x);
    tmp.clear();

    // column view (host, O(tiles)): entries (row panel, column panel of 8 tile
    // columns) in column-panel order, row panels ascending within each; and
    // the order in which the persistent kernels take panels: by descending
    // work (kept tiles, entries), ties by index, panels without work left out
    std::vector<int32_t> h_ptr(T.n_panels + 1), h_col(T.n_tiles);
    BSR_TRY(cudaMemcpy(h_ptr.data(), T.tile_ptr, sizeof(int32_t) * (T.n_panels + 1), cudaMemcpyDeviceToHost));
    if (T.n_tiles > 0)
        BSR_TRY(cudaMemcpy(h_col.data(), T.tile_col, sizeof(int32_t) * T.n_tiles, cudaMemcpyDeviceToHost));
    T.n_cpanels = T.n_panels;   // 128 sources per column panel, N sources
    std::vector<int32_t> c_ptr(T.n_cpanels + 1, 0);
    for (int32_t pn = 0; pn < T.n_panels; ++pn)
        for (int32_t t = h_ptr[pn]; t < h_ptr[pn + 1]; ++t)
            if (t == h_ptr[pn] || h_col[t] / 8 != h_col[t - 1] / 8) ++c_ptr[h_col[t] / 8 + 1];
    for (int32_t c = 0; c < T.n_cpanels; ++c) c_ptr[c + 1] += c_ptr[c];
    T.n_entries = c_ptr[T.n_cpanels];
    std::vector<int32_t> c_panel(T.n_entries), c_tile((size_t)T.n_entries * 8, -1), fillp(c_ptr);
    for (int32_t pn = 0; pn < T.n_panels; ++pn) {
        int32_t cur = -1;
        for (int32_t t = h_ptr[pn]; t < h_ptr[pn + 1]; ++t) {
            const int32_t cp = h_col[t] / 8;
            if (t == h_ptr[pn] || cp != h_col[t - 1] / 8) {
                cur = fillp[cp]++;
                c_panel[cur] = pn;
            }
            c_tile[(size_t)cur * 8 + h_col[t] % 8] = t;
        }
    }
    auto work_order = [](const std::vector<int32_t> &ptr) {
        std::vector<int32_t> o;
        for (int32_t i = 0; i + 1 < (int32_t)ptr.size(); ++i)
            if (ptr[i + 1] > ptr[i]) o.push_back(i);
        std::stable_sort(o.begin(), o.end(),
                         [&](int32_t a, int32_t b) { return ptr[a + 1] - ptr[a] > ptr[b + 1] - ptr[b]; });
        return o;
    };
    const std::vector<int32_t> p_order = work_order(h_ptr), c_order = work_order(c_ptr);
    T.n_active = (int32_t)p_order.size();
    T.n_cactive = (int32_t)c_order.size();
    std::vector<int4> p_info(T.n_active), c_info(T.n_cactive);
    for (int32_t k = 0; k < T.n_active; ++k) p_info[k] = make_int4(p_order[k], h_ptr[p_order[k]], h_ptr[p_order[k] + 1], 0);
    for (int32_t k = 0; k < T.n_cactive; ++k)
        c_info[k] = make_int4(c_order[k], c_ptr[c_order[k]], c_ptr[c_order[k] + 1], 0);
    BSR_TRY(alloc((void **)&T.ct_ptr, sizeof(int32_t) * (T.n_cpanels + 1), true));
    BSR_TRY(alloc((void **)&T.ct_panel, sizeof(int32_t) * T.n_entries, true));
    BSR_TRY(alloc((void **)&T.ct_tile, sizeof(int32_t) * 8 * (size_t)T.n_entries, true));
    BSR_TRY(alloc((void **)&T.panel_info, sizeof(int4) * T.n_active, true));
    BSR_TRY(alloc((void **)&T.cpanel_info, sizeof(int4) * T.n_cactive, true));
    BSR_TRY(cudaMemcpy(T.ct_ptr, c_ptr.data(), sizeof(int32_t) * (T.n_cpanels + 1), cudaMemcpyHostToDevice));
    if (T.n_entries > 0) {
        BSR_TRY(cudaMemcpy(T.ct_panel, c_panel.data(), sizeof(int32_t) * T.n_entries, cudaMemcpyHostToDevice));
        BSR_TRY(cudaMemcpy(T.ct_tile, c_tile.data(), sizeof(int32_t) * 8 * (size_t)T.n_entries,
                           cudaMemcpyHostToDevice));
    }
    if (T.n_active > 0)
        BSR_TRY(cudaMemcpy(T.panel_info, p_info.data(), sizeof(int4) * T.n_active, cudaMemcpyHostToDevice));
    if (T.n_cactive > 0)
        BSR_TRY(cudaMemcpy(T.cpanel_info, c_info.data(), sizeof(int4) * T.n_cactive, cudaMemcpyHostToDevice));
#undef BSR_TRY
    return SGA_OK;
}

}  // namespace sga
