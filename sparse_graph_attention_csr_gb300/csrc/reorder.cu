// Graph reordering on the device: relabel nodes so that rows processed
// together gather overlapping neighbour rows, which raises the cache hit rate
// of the gather kernels.  The IO-aware layers work ("On Efficient Scaling of
// GNNs via IO-Aware Layers Implementations", arXiv abstract) studies graph
// reordering and finds that it benefits neighbour-parallel (gather-dominated)
// kernels more consistently than feature-parallel ones; the pages name no
// particular ordering, so two classic ones are provided:
//
//  - SGA_ORDER_DEGREE: nodes by descending in-degree (the number of rows that
//    gather them), ties by ascending id.
//  - SGA_ORDER_RCM: reverse Cuthill-McKee on the symmetrised graph.  Written
//    as a level-synchronous breadth-first search that reproduces the
//    sequential algorithm exactly: within a component, a node of level L+1 is
//    placed by the earliest-placed neighbour of level L (its parent), then by
//    degree, then by id -- the order in which a queue-based Cuthill-McKee
//    appends it.  Components follow one another in the order of their start
//    nodes (the unvisited node of least degree, least id), and all components
//    advance one level per step.  Degree here is the row degree plus the
//    transposed degree (CSR entries, self-loops and duplicates included).
//
// The result is a permutation perm[v] = new id of node v.  sga_relabel_csr
// applies it to the graph (new row perm[v] = old row v with its sources
// mapped, in their original order) and sga_permute_rows to node tensors.
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "plan.h"

namespace sga {
namespace {

unsigned grid_n(int64_t n, int threads, int cap = 65535) {
    int64_t g = (n + threads - 1) / threads;
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>(g, cap));
}

__global__ void in_degree_kernel(const int32_t *__restrict__ indices, int64_t E, int32_t *__restrict__ indeg) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += stride)
        atomicAdd(&indeg[indices[e]], 1);
}

// key = max - indeg (descending in-degree as an ascending key), value = id
__global__ void degree_keys_kernel(const int32_t *__restrict__ indeg, int64_t N, int32_t maxdeg,
                                   int32_t *__restrict__ key, int32_t *__restrict__ val) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < N; v += stride) {
        key[v] = maxdeg - indeg[v];
        val[v] = (int32_t)v;
    }
}

// perm[order[p]] = p (or N - 1 - p for a reversed order)
__global__ void invert_kernel(const int32_t *__restrict__ order, int64_t N, int reverse, int32_t *__restrict__ perm) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < N; p += stride)
        perm[order[p]] = (int32_t)(reverse ? N - 1 - p : p);
}

// ---- connected components (minimum-id labels by hooking and pointer jumping)

__device__ __forceinline__ int32_t find_root(const int32_t *parent, int32_t x) {
    // parent values only decrease and parent[x] <= x, so this ends
    int32_t p = parent[x];
    while (p != x) {
        x = p;
        p = parent[x];
    }
    return x;
}

__global__ void cc_init_kernel(int32_t *parent, int64_t N) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < N; v += stride) parent[v] = (int32_t)v;
}

__global__ void cc_hook_kernel(const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices, int64_t N,
                               int32_t *parent, int32_t *changed) {
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t v = warp; v < N; v += nw) {
        const int32_t b = indptr[v], e = indptr[v + 1];
        for (int32_t x = b + lane; x < e; x += 32) {
            const int32_t u = indices[x];
            const int32_t ru = find_root(parent, u), rv = find_root(parent, (int32_t)v);
            if (ru != rv) {
                atomicMin(&parent[max(ru, rv)], min(ru, rv));
                *changed = 1;
            }
        }
    }
}

__global__ void cc_jump_kernel(int32_t *parent, int64_t N) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < N; v += stride)
        parent[v] = find_root(parent, (int32_t)v);
}

// component start key: min over members of (sym degree << 32 | id)
__global__ void comp_min_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ sdeg, int64_t N,
                                unsigned long long *minkey) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < N; v += stride)
        atomicMin(&minkey[parent[v]], ((unsigned long long)(uint32_t)sdeg[v] << 32) | (uint32_t)v);
}

__global__ void sym_degree_kernel(const int32_t *__restrict__ indptr, const int32_t *__restrict__ indeg, int64_t N,
                                  int32_t *__restrict__ sdeg) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < N; v += stride)
        sdeg[v] = indptr[v + 1] - indptr[v] + indeg[v];
}

// flag[v] = 1 for component roots (parent[v] == v)
__global__ void root_flag_kernel(const int32_t *__restrict__ parent, int64_t N, int32_t *__restrict__ flag) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v <= N; v += stride)
        flag[v] = v < N && parent[v] == (int32_t)v ? 1 : 0;
}

// the start node of every component, in root (ascending id of the root) order
__global__ void comp_starts_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ pos,
                                   const unsigned long long *__restrict__ minkey, int64_t N,
                                   int32_t *__restrict__ start_id, int32_t *__restrict__ start_deg) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < N; v += stride)
        if (parent[v] == (int32_t)v) {
            const unsigned long long k = minkey[v];
            start_id[pos[v]] = (int32_t)(k & 0xffffffffu);
            start_deg[pos[v]] = (int32_t)(k >> 32);
        }
}

// level 0: the sorted starts; rank within the level = component rank
__global__ void seed_level_kernel(const int32_t *__restrict__ front, int64_t n, int32_t *__restrict__ level,
                                  int32_t *__restrict__ lrank, const int32_t *__restrict__ parent,
                                  int32_t *__restrict__ comp_rank) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < n; r += stride) {
        const int32_t v = front[r];
        level[v] = 0;
        lrank[v] = (int32_t)r;
        comp_rank[parent[v]] = (int32_t)r;
    }
}

// every unvisited neighbour w of the frontier (both edge directions) takes
// the least rank among its frontier neighbours as its parent position
__global__ void expand_kernel(const int32_t *__restrict__ front, int64_t n, const int32_t *__restrict__ indptr,
                              const int32_t *__restrict__ indices, const int32_t *__restrict__ t_indptr,
                              const int32_t *__restrict__ t_dst, const int32_t *__restrict__ level,
                              int32_t *__restrict__ pp) {
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = warp; r < n; r += nw) {
        const int32_t u = front[r];
        for (int dir = 0; dir < 2; ++dir) {
            const int32_t *ptr = dir ? t_indptr : indptr;
            const int32_t *ids = dir ? t_dst : indices;
            const int32_t b = ptr[u], e = ptr[u + 1];
            for (int32_t x = b + lane; x < e; x += 32) {
                const int32_t w = ids[x];
                if (level[w] < 0) atomicMin(&pp[w], (int32_t)r);
            }
        }
    }
}

__global__ void cand_flag_kernel(const int32_t *__restrict__ level, const int32_t *__restrict__ pp, int64_t N,
                                 int32_t *__restrict__ flag) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v <= N; v += stride)
        flag[v] = v < N && level[v] < 0 && pp[v] != INT32_MAX ? 1 : 0;
}

// compact flagged nodes (ascending id) with a key per node
__global__ void compact_kernel(const int32_t *__restrict__ flag, const int32_t *__restrict__ pos, int64_t N,
                               const int32_t *__restrict__ keysrc, int32_t *__restrict__ key,
                               int32_t *__restrict__ val) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < N; v += stride)
        if (flag[v]) {
            key[pos[v]] = keysrc[v];
            val[pos[v]] = (int32_t)v;
        }
}

__global__ void gather_keys_kernel(const int32_t *__restrict__ val, int64_t n, const int32_t *__restrict__ keysrc,
                                   int32_t *__restrict__ key) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < n; r += stride) key[r] = keysrc[val[r]];
}

__global__ void set_level_kernel(const int32_t *__restrict__ front, int64_t n, int32_t L, int32_t *__restrict__ level,
                                 int32_t *__restrict__ lrank) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < n; r += stride) {
        level[front[r]] = L;
        lrank[front[r]] = (int32_t)r;
    }
}

// keys for the final order: component rank of each node's component
__global__ void node_comp_rank_kernel(const int32_t *__restrict__ parent, const int32_t *__restrict__ comp_rank,
                                      int64_t N, int32_t *__restrict__ out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < N; v += stride)
        out[v] = comp_rank[parent[v]];
}

__global__ void fill_kernel(int32_t *__restrict__ x, int64_t n, int32_t v) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) x[i] = v;
}

// destination (row) of every CSR entry
__global__ void edge_dst_kernel(const int32_t *__restrict__ indptr, int64_t N, int32_t *__restrict__ rows) {
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t v = warp; v < N; v += nw)
        for (int32_t x = indptr[v] + lane; x < indptr[v + 1]; x += 32) rows[x] = (int32_t)v;
}

__global__ void iota_kernel(int32_t *__restrict__ x, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n; v += stride) x[v] = (int32_t)v;
}

// ---- relabelling and row permutation

__global__ void relabel_degree_kernel(const int32_t *__restrict__ indptr, const int32_t *__restrict__ perm, int64_t N,
                                      int32_t *__restrict__ deg_new) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < N; v += stride)
        deg_new[perm[v]] = indptr[v + 1] - indptr[v];
}

__global__ void relabel_rows_kernel(const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                                    const int32_t *__restrict__ perm, int64_t N, const int32_t *__restrict__ new_ptr,
                                    int32_t *__restrict__ new_idx) {
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t v = warp; v < N; v += nw) {
        const int32_t b = indptr[v], e = indptr[v + 1], o = new_ptr[perm[v]];
        for (int32_t x = b + lane; x < e; x += 32) new_idx[o + (x - b)] = perm[indices[x]];
    }
}

// dst[perm[v]] = src[v] (forward) or dst[v] = src[perm[v]] (inverse), rows of
// `chunks` 16-byte chunks
__global__ void permute_rows_kernel(const uint4 *__restrict__ src, int64_t N, int64_t chunks,
                                    const int32_t *__restrict__ perm, int inverse, uint4 *__restrict__ dst) {
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t v = warp; v < N; v += nw) {
        const int64_t p = perm[v];
        if ((uint64_t)p >= (uint64_t)N) continue;   // not a node id: the row is skipped
        const int64_t from = inverse ? p : v, to = inverse ? v : p;
        for (int64_t c = lane; c < chunks; c += 32) dst[to * chunks + c] = src[from * chunks + c];
    }
}

// The device allocations of one reorder call (freed on every return path).
struct Scratch {
    std::vector<void *> ptrs;
    cudaError_t err = cudaSuccess;
    template <typename T> T *get(int64_t count) {
        if (err != cudaSuccess) return nullptr;
        void *p = nullptr;
        err = cudaMalloc(&p, (size_t)std::max<int64_t>(count, 1) * sizeof(T));
        if (err != cudaSuccess) return nullptr;
        ptrs.push_back(p);
        return static_cast<T *>(p);
    }
    ~Scratch() {
        for (void *p : ptrs) cudaFree(p);
    }
};

// Input checks of the entry points, run before any kernel indexes with the
// inputs.  Bits: 1 indptr[0] != 0, 2 indptr decreasing somewhere, 4
// indptr[N] != E, 8 a source id outside [0, N), 16 a perm entry outside
// [0, N), 32 a perm entry taken twice.
__global__ void check_csr_kernel(const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                                 int64_t N, int64_t E, int32_t *bad) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int bits = 0;
    if (t0 == 0) {
        if (indptr[0] != 0) bits |= 1;
        if ((int64_t)indptr[N] != E) bits |= 4;
    }
    for (int64_t i = t0; i < N; i += stride)
        if (indptr[i] > indptr[i + 1]) bits |= 2;
    for (int64_t e = t0; e < E; e += stride) {
        const int32_t j = indices[e];
        if (j < 0 || (int64_t)j >= N) bits |= 8;
    }
    if (bits) atomicOr(bad, bits);
}

__global__ void check_perm_kernel(const int32_t *__restrict__ perm, int64_t N, int32_t *seen, int32_t *bad) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int bits = 0;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < N; v += stride) {
        const int32_t p = perm[v];
        if (p < 0 || (int64_t)p >= N)
            bits |= 16;
        else if (atomicAdd(seen + p, 1) != 0)
            bits |= 32;
    }
    if (bits) atomicOr(bad, bits);
}

// Checks the CSR (indptr non-null) and the permutation (perm non-null) on
// `stream` and synchronises it; *bits receives the OR of the failed checks.
cudaError_t check_inputs(const int32_t *indptr, const int32_t *indices, int64_t N, int64_t E,
                         const int32_t *perm, cudaStream_t s, int32_t *bits) {
    Scratch m;
    int32_t *bad = m.get<int32_t>(1);
    int32_t *seen = perm ? m.get<int32_t>(N) : nullptr;
    if (m.err != cudaSuccess) return m.err;
    cudaError_t e = cudaMemsetAsync(bad, 0, sizeof(int32_t), s);
    if (e == cudaSuccess && indptr) {
        check_csr_kernel<<<grid_n(std::max(N, E), 256, 4096), 256, 0, s>>>(indptr, indices, N, E, bad);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess && perm && N > 0) {
        e = cudaMemsetAsync(seen, 0, sizeof(int32_t) * (size_t)N, s);
        if (e == cudaSuccess) {
            check_perm_kernel<<<grid_n(N, 256, 4096), 256, 0, s>>>(perm, N, seen, bad);
            e = cudaGetLastError();
        }
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(bits, bad, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);   // (the scratch is freed on return)
    return e;
}

int bits_for(int64_t maxval) {
    int b = 1;
    while (b < 31 && ((int64_t)1 << b) <= maxval) ++b;
    return b;
}

#define SGA_CK(x)                          \
    do {                                   \
        cudaError_t _e = (x);              \
        if (_e != cudaSuccess) return _e;  \
    } while (0)

cudaError_t reorder_impl(const int32_t *indptr, const int32_t *indices, int64_t N, int64_t E, int method,
                         int32_t *perm, cudaStream_t s) {
    Scratch m;
    const int64_t hist_n = radix_hist_elems(std::max<int64_t>(N, 1));
    int32_t *indeg = m.get<int32_t>(N + 1);
    int32_t *ka = m.get<int32_t>(N), *va = m.get<int32_t>(N), *kb = m.get<int32_t>(N), *vb = m.get<int32_t>(N);
    int32_t *hist = m.get<int32_t>(hist_n);
    int32_t *scan_tmp = m.get<int32_t>(scan_tmp_elems(std::max<int64_t>(hist_n, N + 1)));
    SGA_CK(m.err);
    SGA_CK(cudaMemsetAsync(indeg, 0, sizeof(int32_t) * (N + 1), s));
    if (E > 0) {
        in_degree_kernel<<<grid_n(E, 256, 8192), 256, 0, s>>>(indices, E, indeg);
        SGA_CK(cudaGetLastError());
    }
    if (method == SGA_ORDER_DEGREE) {
        const int32_t maxdeg = (int32_t)std::min<int64_t>(E, INT32_MAX - 1);
        degree_keys_kernel<<<grid_n(N, 256), 256, 0, s>>>(indeg, N, maxdeg, ka, va);
        SGA_CK(cudaGetLastError());
        SGA_CK(radix_sort_pairs(&ka, &va, &kb, &vb, N, bits_for(maxdeg), hist, scan_tmp, s));
        invert_kernel<<<grid_n(N, 256), 256, 0, s>>>(va, N, 0, perm);
        SGA_CK(cudaGetLastError());
        return cudaStreamSynchronize(s);
    }

    // ---- reverse Cuthill-McKee
    const int64_t hist_e = radix_hist_elems(std::max<int64_t>(E, 1));
    int32_t *t_indptr = m.get<int32_t>(N + 1);
    int32_t *eka = m.get<int32_t>(E), *eva = m.get<int32_t>(E), *ekb = m.get<int32_t>(E), *evb = m.get<int32_t>(E);
    int32_t *ehist = m.get<int32_t>(hist_e);
    int32_t *escan = m.get<int32_t>(scan_tmp_elems(std::max<int64_t>(hist_e, N + 1)));
    int32_t *sdeg = m.get<int32_t>(N), *parent = m.get<int32_t>(N), *flag = m.get<int32_t>(N + 1);
    int32_t *pos = m.get<int32_t>(N + 1), *level = m.get<int32_t>(N), *lrank = m.get<int32_t>(N);
    int32_t *pp = m.get<int32_t>(N), *comp_rank = m.get<int32_t>(N), *front = m.get<int32_t>(N);
    int32_t *dflag = m.get<int32_t>(1);
    unsigned long long *minkey = m.get<unsigned long long>(N);
    SGA_CK(m.err);
    auto host_i32 = [&](const int32_t *d, int32_t &h) -> cudaError_t {
        cudaError_t e = cudaMemcpyAsync(&h, d, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
        return e == cudaSuccess ? cudaStreamSynchronize(s) : e;
    };
    // transposed CSR: destinations of each source, ascending (stable sort by source)
    SGA_CK(cudaMemcpyAsync(t_indptr, indeg, sizeof(int32_t) * (N + 1), cudaMemcpyDeviceToDevice, s));
    SGA_CK(exclusive_scan(t_indptr, t_indptr, N + 1, escan, s));
    if (E > 0) {
        SGA_CK(cudaMemcpyAsync(eka, indices, sizeof(int32_t) * E, cudaMemcpyDeviceToDevice, s));
        edge_dst_kernel<<<grid_n(N * 32, 256, 1 << 20), 256, 0, s>>>(indptr, N, eva);
        SGA_CK(cudaGetLastError());
        SGA_CK(radix_sort_pairs(&eka, &eva, &ekb, &evb, E, bits_for(N - 1), ehist, escan, s));
    }
    const int32_t *t_dst = eva;
    sym_degree_kernel<<<grid_n(N, 256), 256, 0, s>>>(indptr, indeg, N, sdeg);
    SGA_CK(cudaGetLastError());

    // connected components of the symmetrised graph (label = least member id)
    cc_init_kernel<<<grid_n(N, 256), 256, 0, s>>>(parent, N);
    SGA_CK(cudaGetLastError());
    for (int it = 0;; ++it) {
        if (it > 4096) return cudaErrorUnknown;   // (converges in a few rounds)
        SGA_CK(cudaMemsetAsync(dflag, 0, sizeof(int32_t), s));
        cc_hook_kernel<<<grid_n(N * 32, 256, 1 << 20), 256, 0, s>>>(indptr, indices, N, parent, dflag);
        SGA_CK(cudaGetLastError());
        cc_jump_kernel<<<grid_n(N, 256), 256, 0, s>>>(parent, N);
        SGA_CK(cudaGetLastError());
        int32_t changed = 0;
        SGA_CK(host_i32(dflag, changed));
        if (!changed) break;
    }
    // component start nodes (least degree, then least id), components in start order
    SGA_CK(cudaMemsetAsync(minkey, 0xff, sizeof(unsigned long long) * N, s));
    comp_min_kernel<<<grid_n(N, 256), 256, 0, s>>>(parent, sdeg, N, minkey);
    root_flag_kernel<<<grid_n(N + 1, 256), 256, 0, s>>>(parent, N, flag);
    SGA_CK(cudaGetLastError());
    SGA_CK(exclusive_scan(flag, pos, N + 1, scan_tmp, s));
    int32_t n_comp = 0;
    SGA_CK(host_i32(pos + N, n_comp));
    comp_starts_kernel<<<grid_n(N, 256), 256, 0, s>>>(parent, pos, minkey, N, va, ka);
    SGA_CK(cudaGetLastError());
    // (ka = start degree, va = start id): ids first, then a stable sort by degree
    SGA_CK(cudaMemcpyAsync(kb, va, sizeof(int32_t) * n_comp, cudaMemcpyDeviceToDevice, s));
    std::swap(ka, kb);   // ka = ids as keys, kb = degrees (scratch now)
    SGA_CK(radix_sort_pairs(&ka, &va, &kb, &vb, n_comp, bits_for(N - 1), hist, scan_tmp, s));
    gather_keys_kernel<<<grid_n(n_comp, 256), 256, 0, s>>>(va, n_comp, sdeg, ka);
    SGA_CK(cudaGetLastError());
    SGA_CK(radix_sort_pairs(&ka, &va, &kb, &vb, n_comp, bits_for(2 * E + 1), hist, scan_tmp, s));
    SGA_CK(cudaMemcpyAsync(front, va, sizeof(int32_t) * n_comp, cudaMemcpyDeviceToDevice, s));
    SGA_CK(cudaMemsetAsync(level, 0xff, sizeof(int32_t) * N, s));
    seed_level_kernel<<<grid_n(n_comp, 256), 256, 0, s>>>(front, n_comp, level, lrank, parent, comp_rank);
    SGA_CK(cudaGetLastError());

    // breadth-first levels, all components at once
    int32_t n_front = n_comp, L = 0;
    while (n_front > 0) {
        fill_kernel<<<grid_n(N, 256), 256, 0, s>>>(pp, N, INT32_MAX);
        expand_kernel<<<grid_n((int64_t)n_front * 32, 256, 1 << 20), 256, 0, s>>>(front, n_front, indptr, indices,
                                                                                  t_indptr, t_dst, level, pp);
        cand_flag_kernel<<<grid_n(N + 1, 256), 256, 0, s>>>(level, pp, N, flag);
        SGA_CK(cudaGetLastError());
        SGA_CK(exclusive_scan(flag, pos, N + 1, scan_tmp, s));
        int32_t n_next = 0;
        SGA_CK(host_i32(pos + N, n_next));
        if (n_next == 0) break;
        // candidates in id order, then stable sorts by degree and by parent rank
        compact_kernel<<<grid_n(N, 256), 256, 0, s>>>(flag, pos, N, sdeg, ka, va);
        SGA_CK(cudaGetLastError());
        SGA_CK(radix_sort_pairs(&ka, &va, &kb, &vb, n_next, bits_for(2 * E + 1), hist, scan_tmp, s));
        gather_keys_kernel<<<grid_n(n_next, 256), 256, 0, s>>>(va, n_next, pp, ka);
        SGA_CK(cudaGetLastError());
        SGA_CK(radix_sort_pairs(&ka, &va, &kb, &vb, n_next, bits_for(n_front), hist, scan_tmp, s));
        SGA_CK(cudaMemcpyAsync(front, va, sizeof(int32_t) * n_next, cudaMemcpyDeviceToDevice, s));
        set_level_kernel<<<grid_n(n_next, 256), 256, 0, s>>>(front, n_next, ++L, level, lrank);
        SGA_CK(cudaGetLastError());
        n_front = n_next;
    }
    // Cuthill-McKee order = (component rank, level, rank within the level); reversed
    iota_kernel<<<grid_n(N, 256), 256, 0, s>>>(va, N);
    SGA_CK(cudaMemcpyAsync(ka, lrank, sizeof(int32_t) * N, cudaMemcpyDeviceToDevice, s));
    SGA_CK(radix_sort_pairs(&ka, &va, &kb, &vb, N, bits_for(N), hist, scan_tmp, s));
    gather_keys_kernel<<<grid_n(N, 256), 256, 0, s>>>(va, N, level, ka);
    SGA_CK(cudaGetLastError());
    SGA_CK(radix_sort_pairs(&ka, &va, &kb, &vb, N, bits_for(L), hist, scan_tmp, s));
    node_comp_rank_kernel<<<grid_n(N, 256), 256, 0, s>>>(parent, comp_rank, N, kb);
    gather_keys_kernel<<<grid_n(N, 256), 256, 0, s>>>(va, N, kb, ka);
    SGA_CK(cudaGetLastError());
    SGA_CK(radix_sort_pairs(&ka, &va, &kb, &vb, N, bits_for(n_comp), hist, scan_tmp, s));
    invert_kernel<<<grid_n(N, 256), 256, 0, s>>>(va, N, 1, perm);
    SGA_CK(cudaGetLastError());
    return cudaStreamSynchronize(s);
}

}  // namespace
}  // namespace sga

using namespace sga;

namespace {
bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
sga_status to_status(cudaError_t e) {
    if (e == cudaSuccess) return SGA_OK;
    set_cuda_error(e);
    return SGA_ECUDA;
}
}  // namespace

extern "C" sga_status sga_reorder(const int32_t *indptr, const int32_t *indices, int64_t N, int64_t E,
                                  sga_order method, int32_t *perm, void *stream) {
    if (!indptr || !perm || !aligned_to(indptr, 4) || !aligned_to(perm, 4)) return SGA_EINVAL;
    if (E > 0 && (!indices || !aligned_to(indices, 4))) return SGA_EINVAL;
    if (N < 0 || E < 0 || N >= INT32_MAX || E >= INT32_MAX / 2) return SGA_EINVAL;
    if (method != SGA_ORDER_DEGREE && method != SGA_ORDER_RCM) return SGA_EINVAL;
    if (N == 0) return SGA_OK;
    int32_t bits = 0;
    const cudaError_t e = check_inputs(indptr, indices, N, E, nullptr, static_cast<cudaStream_t>(stream), &bits);
    if (e != cudaSuccess) return to_status(e);
    if (bits) return SGA_EINVAL;
    return to_status(reorder_impl(indptr, indices, N, E, method, perm, static_cast<cudaStream_t>(stream)));
}

extern "C" sga_status sga_relabel_csr(const int32_t *indptr, const int32_t *indices, int64_t N, int64_t E,
                                      const int32_t *perm, int32_t *new_indptr, int32_t *new_indices,
                                      void *stream) {
    if (!indptr || !perm || !new_indptr) return SGA_EINVAL;
    if (E > 0 && (!indices || !new_indices)) return SGA_EINVAL;
    if (N < 0 || E < 0 || N >= INT32_MAX || E >= INT32_MAX) return SGA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t bits = 0;
    cudaError_t e = check_inputs(indptr, indices, N, E, perm, s, &bits);
    if (e != cudaSuccess) return to_status(e);
    if (bits) return SGA_EINVAL;
    Scratch m;
    int32_t *tmp = m.get<int32_t>(scan_tmp_elems(N + 1));
    if (m.err != cudaSuccess) return to_status(m.err);
    e = cudaMemsetAsync(new_indptr, 0, sizeof(int32_t) * (N + 1), s);
    if (e == cudaSuccess && N > 0) {
        relabel_degree_kernel<<<grid_n(N, 256), 256, 0, s>>>(indptr, perm, N, new_indptr);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = exclusive_scan(new_indptr, new_indptr, N + 1, tmp, s);
    if (e == cudaSuccess && E > 0) {
        relabel_rows_kernel<<<grid_n(N * 32, 256, 1 << 20), 256, 0, s>>>(indptr, indices, perm, N, new_indptr,
                                                                         new_indices);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);   // the scratch is freed on return
    return to_status(e);
}

extern "C" sga_status sga_permute_rows(const void *src, int64_t N, int64_t row_bytes, const int32_t *perm,
                                       int inverse, void *dst, void *stream) {
    if (N < 0 || row_bytes < 0 || row_bytes % 16 != 0) return SGA_EINVAL;
    if (N == 0 || row_bytes == 0) return SGA_OK;
    if (!src || !dst || !perm || src == dst || !aligned_to(src, 16) || !aligned_to(dst, 16)) return SGA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    permute_rows_kernel<<<grid_n(N * 32, 256, 1 << 20), 256, 0, s>>>(
        static_cast<const uint4 *>(src), N, row_bytes / 16, perm, inverse ? 1 : 0, static_cast<uint4 *>(dst));
    return to_status(cudaGetLastError());
}
