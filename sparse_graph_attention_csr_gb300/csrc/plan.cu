// Graph preprocessing on the device: CSR validation, the transposed CSR by a
// stable LSD radix sort of (source, destination) pairs, and the degree
// partition (split rows cut into fixed-length chunks) of both CSRs.
//
// The transposed CSR serves the backward pass, which needs each source's
// destinations to sum dK/dV (GT) or dFR (GATv2) without atomics.  The
// partition implements the super-node handling: DF-GNN's abstract names the
// bottleneck shift caused by super nodes, and the IO-aware layers blog post
// ("aggregation layers" paragraph) answers heavy-tailed degrees with
// degree-aware tiling and extra parallelism for high-degree nodes.
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "plan.h"

namespace sga {

namespace {

constexpr int kScanThreads = 512;
constexpr int kScanItems = 8;
constexpr int kScanTile = kScanThreads * kScanItems;  // 4096 elements per block

constexpr int kRadixBits = 8;
constexpr int kRadixBins = 1 << kRadixBits;
constexpr int kRadixItems = 32;                  // 32-element steps per warp tile
constexpr int kRadixTile = 32 * kRadixItems;     // 1024 elements per warp

// ---------------------------------------------------------------- validation

__global__ void validate_csr_kernel(const int32_t *__restrict__ indptr,
                                    const int32_t *__restrict__ indices, int64_t N, int64_t E,
                                    int32_t *err) {
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
        int32_t j = indices[e];
        if (j < 0 || (int64_t)j >= N) bits |= 8;
    }
    if (bits) atomicOr(err, bits);
}

// ---------------------------------------------------------------------- scan

__device__ __forceinline__ int32_t warp_incl_scan(int32_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t u = __shfl_up_sync(SGA_FULL_MASK, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Block-wide exclusive scan of one value per thread; returns the prefix and
// writes the block total to *total.
__device__ int32_t block_excl_scan(int32_t v, int32_t *total) {
    __shared__ int32_t warp_sums[kScanThreads / 32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int32_t inc = warp_incl_scan(v);
    if (lane == 31) warp_sums[w] = inc;
    __syncthreads();
    if (w == 0) {
        int32_t s = (lane < kScanThreads / 32) ? warp_sums[lane] : 0;
        s = warp_incl_scan(s);
        if (lane < kScanThreads / 32) warp_sums[lane] = s;
    }
    __syncthreads();
    int32_t before = (w > 0) ? warp_sums[w - 1] : 0;
    *total = warp_sums[kScanThreads / 32 - 1];
    __syncthreads();
    return before + inc - v;
}

__global__ void __launch_bounds__(kScanThreads)
scan_reduce_kernel(const int32_t *__restrict__ in, int64_t n, int32_t *__restrict__ sums) {
    const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
    int32_t v = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k)
        if (base + k < n) v += in[base + k];
    int32_t total;
    block_excl_scan(v, &total);
    if (threadIdx.x == 0) sums[blockIdx.x] = total;
}

// Exclusive scan of each 4096-element tile plus the tile's offset.  `out`
// may alias `in`: each thread reads its elements before writing them.
__global__ void __launch_bounds__(kScanThreads)
scan_apply_kernel(const int32_t *in, int32_t *out, int64_t n, const int32_t *__restrict__ offsets) {
    const int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
    int32_t x[kScanItems];
    int32_t v = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        x[k] = (base + k < n) ? in[base + k] : 0;
        v += x[k];
    }
    int32_t total;
    int32_t run = block_excl_scan(v, &total) + (offsets ? offsets[blockIdx.x] : 0);
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        if (base + k < n) out[base + k] = run;
        run += x[k];
    }
}

}  // namespace

int64_t scan_tmp_elems(int64_t n) {
    int64_t t = 0;
    while (n > kScanTile) {
        n = (n + kScanTile - 1) / kScanTile;
        t += 2 * n;
    }
    return t + 1;
}

// Exclusive prefix sum of n int32 (out may alias in).  tmp: scan_tmp_elems(n).
cudaError_t exclusive_scan(const int32_t *in, int32_t *out, int64_t n, int32_t *tmp,
                           cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t nb = (n + kScanTile - 1) / kScanTile;
    if (nb == 1) {
        scan_apply_kernel<<<1, kScanThreads, 0, s>>>(in, out, n, nullptr);
        return cudaGetLastError();
    }
    int32_t *sums = tmp, *offs = tmp + nb;
    scan_reduce_kernel<<<(unsigned)nb, kScanThreads, 0, s>>>(in, n, sums);
    cudaError_t e = exclusive_scan(sums, offs, nb, tmp + 2 * nb, s);
    if (e != cudaSuccess) return e;
    scan_apply_kernel<<<(unsigned)nb, kScanThreads, 0, s>>>(in, out, n, offs);
    return cudaGetLastError();
}

namespace {

// ------------------------------------------------------------- radix sort

__global__ void edge_rows_kernel(const int32_t *__restrict__ indptr, int64_t N,
                                 int32_t *__restrict__ rows) {
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (warp >= N) return;
    const int32_t b = indptr[warp], e = indptr[warp + 1];
    for (int32_t x = b + lane; x < e; x += 32) rows[x] = (int32_t)warp;
}

// Per-warp-tile digit histogram, stored digit-major: hist[d * n_tiles + tile].
__global__ void radix_hist_kernel(const int32_t *__restrict__ keys, int64_t n, int shift,
                                  int64_t n_tiles, int32_t *__restrict__ hist) {
    __shared__ int32_t h[kWarpsPerBlock][kRadixBins];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tile = (int64_t)blockIdx.x * kWarpsPerBlock + w;
    for (int d = lane; d < kRadixBins; d += 32) h[w][d] = 0;
    __syncwarp();
    if (tile < n_tiles) {
        const int64_t base = tile * kRadixTile;
        for (int it = 0; it < kRadixItems; ++it) {
            int64_t e = base + it * 32 + lane;
            if (e < n) atomicAdd(&h[w][(keys[e] >> shift) & (kRadixBins - 1)], 1);
        }
    }
    __syncwarp();
    if (tile < n_tiles)
        for (int d = lane; d < kRadixBins; d += 32) hist[(int64_t)d * n_tiles + tile] = h[w][d];
}

// Stable scatter: a warp walks its tile in order, 32 keys at a time; equal
// digits within a step are ranked by lane, and each digit's cursor advances
// by its count, so the input order is preserved within every digit.
__global__ void radix_scatter_kernel(const int32_t *__restrict__ keys,
                                     const int32_t *__restrict__ vals, int64_t n, int shift,
                                     int64_t n_tiles, const int32_t *__restrict__ offsets,
                                     int32_t *__restrict__ keys_out,
                                     int32_t *__restrict__ vals_out) {
    __shared__ int32_t cur[kWarpsPerBlock][kRadixBins];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tile = (int64_t)blockIdx.x * kWarpsPerBlock + w;
    if (tile >= n_tiles) return;  // whole warp leaves together
    for (int d = lane; d < kRadixBins; d += 32) cur[w][d] = offsets[(int64_t)d * n_tiles + tile];
    __syncwarp();
    const unsigned lt = (1u << lane) - 1u;
    const int64_t base = tile * kRadixTile;
    for (int it = 0; it < kRadixItems; ++it) {
        const int64_t e = base + it * 32 + lane;
        const bool valid = e < n;
        const int32_t k = valid ? keys[e] : 0;
        const int32_t v = valid ? vals[e] : 0;
        const int d = valid ? ((k >> shift) & (kRadixBins - 1)) : kRadixBins;
        const unsigned peers = __match_any_sync(SGA_FULL_MASK, d);
        const int rank = __popc(peers & lt);
        int32_t pos = 0;
        if (valid) pos = cur[w][d] + rank;
        __syncwarp();
        if (valid) {
            keys_out[pos] = k;
            vals_out[pos] = v;
            if (rank == 0) cur[w][d] = pos + __popc(peers);
        }
        __syncwarp();
    }
}

__global__ void iota_edges_kernel(int32_t *__restrict__ x, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += stride) x[e] = (int32_t)e;
}

// t_dst[te] = row of CSR edge t_eid[te]
__global__ void gather_rows_kernel(const int32_t *__restrict__ rows, const int32_t *__restrict__ t_eid,
                                   int64_t n, int32_t *__restrict__ t_dst) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t te = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; te < n; te += stride)
        t_dst[te] = rows[t_eid[te]];
}

// Sort keys of the walking order, value = row: descending degree
// (key = maxdeg - degree), or split rows first then ascending id (key = 0 for
// rows above the threshold, 1 for the others).
__global__ void order_keys_kernel(const int32_t *__restrict__ ptr, int64_t N, int32_t maxdeg, int threshold,
                                  bool by_degree, int32_t *__restrict__ key, int32_t *__restrict__ val) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N; i += stride) {
        const int32_t deg = ptr[i + 1] - ptr[i];
        key[i] = by_degree ? maxdeg - deg : (deg > threshold ? 0 : 1);
        val[i] = (int32_t)i;
    }
}

// item list entries of the rows order[0 .. n)
__global__ void item_fill_kernel(const int32_t *__restrict__ ptr, const int32_t *__restrict__ order, int64_t n,
                                 int4 *__restrict__ items) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += stride) {
        const int32_t r = order[x];
        items[x] = make_int4(r, ptr[r], ptr[r + 1], 0);
    }
}

// item list entries of the chunks of split rows
__global__ void chunk_items_kernel(const int32_t *__restrict__ row, const int32_t *__restrict__ beg,
                                   const int32_t *__restrict__ end, int64_t n, int4 *__restrict__ items) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += stride)
        items[x] = make_int4(row[x], beg[x], end[x], 0);
}

__global__ void count_sources_kernel(const int32_t *__restrict__ indices, int64_t E,
                                     int32_t *__restrict__ counts) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < E; e += stride)
        atomicAdd(&counts[indices[e]], 1);
}

// ------------------------------------------------------------- partition

__global__ void part_count_kernel(const int32_t *__restrict__ ptr, int64_t N, int T, int C,
                                  int32_t *__restrict__ flag, int32_t *__restrict__ nch) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i <= N; i += stride) {
        if (i == N) {
            flag[i] = 0;
            nch[i] = 0;
            continue;
        }
        const int32_t deg = ptr[i + 1] - ptr[i];
        const bool split = deg > T;
        flag[i] = split ? 1 : 0;
        nch[i] = split ? (deg + C - 1) / C : 0;
    }
}

__global__ void part_fill_kernel(const int32_t *__restrict__ ptr, int64_t N, int T, int C,
                                 const int32_t *__restrict__ sflag,
                                 const int32_t *__restrict__ snch, Partition p) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < N; i += stride) {
        const int32_t b = ptr[i], e = ptr[i + 1];
        if (e - b <= T) continue;
        const int32_t s = sflag[i];
        int32_t c = snch[i];
        p.split_rows[s] = (int32_t)i;
        p.chunk_ptr[s] = c;
        for (int32_t x = b; x < e; x += C, ++c) {
            p.chunk_row[c] = (int32_t)i;
            p.chunk_split[c] = s;
            p.chunk_beg[c] = x;
            p.chunk_end[c] = min(x + C, e);
        }
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) p.chunk_ptr[p.n_split] = p.n_chunks;
}

unsigned grid_for(int64_t n, int threads, int cap) {
    int64_t g = (n + threads - 1) / threads;
    if (g < 1) g = 1;
    if (g > cap) g = cap;
    return (unsigned)g;
}

struct DevAlloc {
    std::vector<void *> ptrs;
    int64_t bytes = 0;
    cudaError_t err = cudaSuccess;
    template <typename T> T *get(int64_t count) {
        if (err != cudaSuccess) return nullptr;
        void *p = nullptr;
        size_t b = (size_t)std::max<int64_t>(count, 1) * sizeof(T);
        err = cudaMalloc(&p, b);
        if (err != cudaSuccess) return nullptr;
        ptrs.push_back(p);
        bytes += (int64_t)b;
        return static_cast<T *>(p);
    }
    void release() {
        for (void *p : ptrs) cudaFree(p);
        ptrs.clear();
    }
};

#define SGA_TRY(x)                                  \
    do {                                            \
        cudaError_t _e = (x);                       \
        if (_e != cudaSuccess) {                    \
            set_cuda_error(_e);                     \
            tmp.release();                          \
            return SGA_ECUDA;                       \
        }                                           \
    } while (0)

// Build one partition of the CSR `ptr` into plan-owned arrays.
sga_status build_partition(const int32_t *ptr, int64_t N, int T, int C, Partition &out,
                           DevAlloc &own, DevAlloc &tmp, int32_t *scan_tmp, cudaStream_t s) {
    int32_t *flag = tmp.get<int32_t>(N + 1);
    int32_t *nch = tmp.get<int32_t>(N + 1);
    SGA_TRY(tmp.err);
    part_count_kernel<<<grid_for(N + 1, 256, 65535), 256, 0, s>>>(ptr, N, T, C, flag, nch);
    SGA_TRY(cudaGetLastError());
    SGA_TRY(exclusive_scan(flag, flag, N + 1, scan_tmp, s));
    SGA_TRY(exclusive_scan(nch, nch, N + 1, scan_tmp, s));
    int32_t totals[2];
    SGA_TRY(cudaMemcpyAsync(&totals[0], flag + N, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    SGA_TRY(cudaMemcpyAsync(&totals[1], nch + N, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    SGA_TRY(cudaStreamSynchronize(s));
    out.n_split = totals[0];
    out.n_chunks = totals[1];
    out.split_rows = own.get<int32_t>(out.n_split);
    out.chunk_ptr = own.get<int32_t>(out.n_split + 1);
    out.chunk_row = own.get<int32_t>(out.n_chunks);
    out.chunk_beg = own.get<int32_t>(out.n_chunks);
    out.chunk_end = own.get<int32_t>(out.n_chunks);
    out.chunk_split = own.get<int32_t>(out.n_chunks);
    out.arrive = own.get<int32_t>(out.n_split);
    out.next = own.get<int32_t>(1);
    SGA_TRY(own.err);
    if (out.n_split > 0) SGA_TRY(cudaMemsetAsync(out.arrive, 0, sizeof(int32_t) * (size_t)out.n_split, s));
    part_fill_kernel<<<grid_for(N, 256, 65535), 256, 0, s>>>(ptr, N, T, C, flag, nch, out);
    SGA_TRY(cudaGetLastError());
    return SGA_OK;
}

}  // namespace

sga_status plan_build(sga_plan *p, cudaStream_t s) {
    DevAlloc own, tmp;
    const int64_t N = p->N, E = p->E;
    p->d_err = own.get<int32_t>(1);
    p->t_indptr = own.get<int32_t>(N + 1);
    p->t_dst = own.get<int32_t>(E);
    if (p->keep_eid) p->t_eid = own.get<int32_t>(E);
    if (own.err != cudaSuccess) {
        set_cuda_error(own.err);
        own.release();
        return SGA_ECUDA;
    }
#undef SGA_TRY
#define SGA_TRY(x)                                  \
    do {                                            \
        cudaError_t _e = (x);                       \
        if (_e != cudaSuccess) {                    \
            set_cuda_error(_e);                     \
            tmp.release();                          \
            own.release();                          \
            return SGA_ECUDA;                       \
        }                                           \
    } while (0)

    // (1) validation
    SGA_TRY(cudaMemsetAsync(p->d_err, 0, sizeof(int32_t), s));
    validate_csr_kernel<<<grid_for(std::max(N, E), 256, 4096), 256, 0, s>>>(p->indptr, p->indices,
                                                                          N, E, p->d_err);
    SGA_TRY(cudaGetLastError());
    int32_t bad = 0;
    SGA_TRY(cudaMemcpyAsync(&bad, p->d_err, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    SGA_TRY(cudaStreamSynchronize(s));
    if (bad) {
        tmp.release();
        own.release();
        return SGA_EINVAL;
    }

    // (2) transposed CSR: stable radix sort of (source, destination) by source
    const int64_t n_tiles = (E + kRadixTile - 1) / kRadixTile;
    const int64_t hist_n = (int64_t)kRadixBins * std::max<int64_t>(n_tiles, 1);
    int32_t *scan_tmp = tmp.get<int32_t>(scan_tmp_elems(std::max(hist_n, N + 1)));
    int32_t *ka = tmp.get<int32_t>(E), *kb = tmp.get<int32_t>(E);
    int32_t *va = tmp.get<int32_t>(E), *vb = tmp.get<int32_t>(E);
    int32_t *hist = tmp.get<int32_t>(hist_n);
    // the item-list sorts need N-long key/value buffers
    if (N > E) {
        ka = tmp.get<int32_t>(N); kb = tmp.get<int32_t>(N);
        va = tmp.get<int32_t>(N); vb = tmp.get<int32_t>(N);
    }
    int32_t *hist_o = tmp.get<int32_t>(radix_hist_elems(N));
    SGA_TRY(tmp.err);
    if (E > 0) {
        SGA_TRY(cudaMemcpyAsync(ka, p->indices, sizeof(int32_t) * E, cudaMemcpyDeviceToDevice, s));
        // values: the destination of every edge, or (edge-bias plans) the
        // edge itself, whose destination is looked up after the sort
        if (p->keep_eid)
            iota_edges_kernel<<<grid_for(E, 256, 8192), 256, 0, s>>>(va, E);
        else
            edge_rows_kernel<<<grid_for(N * 32, 256, INT32_MAX), 256, 0, s>>>(p->indptr, N, va);
        SGA_TRY(cudaGetLastError());
        int bits = 1;
        while (bits < 31 && ((int64_t)1 << bits) < N) ++bits;
        const unsigned blocks = (unsigned)((n_tiles + kWarpsPerBlock - 1) / kWarpsPerBlock);
        for (int shift = 0; shift < bits; shift += kRadixBits) {
            radix_hist_kernel<<<blocks, 32 * kWarpsPerBlock, 0, s>>>(ka, E, shift, n_tiles, hist);
            SGA_TRY(cudaGetLastError());
            SGA_TRY(exclusive_scan(hist, hist, hist_n, scan_tmp, s));
            radix_scatter_kernel<<<blocks, 32 * kWarpsPerBlock, 0, s>>>(ka, va, E, shift, n_tiles,
                                                                      hist, kb, vb);
            SGA_TRY(cudaGetLastError());
            std::swap(ka, kb);
            std::swap(va, vb);
        }
        if (p->keep_eid) {
            SGA_TRY(cudaMemcpyAsync(p->t_eid, va, sizeof(int32_t) * E, cudaMemcpyDeviceToDevice, s));
            edge_rows_kernel<<<grid_for(N * 32, 256, INT32_MAX), 256, 0, s>>>(p->indptr, N, kb);
            gather_rows_kernel<<<grid_for(E, 256, 8192), 256, 0, s>>>(kb, va, E, p->t_dst);
            SGA_TRY(cudaGetLastError());
        } else {
            SGA_TRY(cudaMemcpyAsync(p->t_dst, va, sizeof(int32_t) * E, cudaMemcpyDeviceToDevice, s));
        }
    }
    SGA_TRY(cudaMemsetAsync(p->t_indptr, 0, sizeof(int32_t) * (N + 1), s));
    if (E > 0) {
        count_sources_kernel<<<grid_for(E, 256, 8192), 256, 0, s>>>(p->indices, E, p->t_indptr);
        SGA_TRY(cudaGetLastError());
    }
    SGA_TRY(exclusive_scan(p->t_indptr, p->t_indptr, N + 1, scan_tmp, s));

    // (3) degree partitions of both CSRs
    sga_status st = build_partition(p->indptr, N, p->split_threshold, p->chunk_len, p->rows, own,
                                    tmp, scan_tmp, s);
    if (st != SGA_OK) { own.release(); return st; }
    st = build_partition(p->t_indptr, N, p->split_threshold, p->chunk_len, p->cols, own, tmp,
                         scan_tmp, s);
    if (st != SGA_OK) { own.release(); return st; }
    // (4) item lists: the chunks of split rows (chunk order), then the other
    // rows in walking order -- by descending degree (ties by id: long rows
    // first, which balances the persistent warps' round-robin share of
    // work), or by ascending id.  Sorting all rows by descending degree puts
    // the split rows (degree > threshold) first, so the others are the tail;
    // for the ascending walk the key is "split" then the id.
    for (int w = 0; w < 2 && N > 0; ++w) {
        const int32_t *ptr = w == 0 ? p->indptr : p->t_indptr;
        Partition &P = w == 0 ? p->rows : p->cols;
        P.n_items = (int64_t)P.n_chunks + (N - P.n_split);
        const int64_t per_warp = E / (16 * (int64_t)std::max(1, p->num_sms));   // 16 resident warps per SM
        P.batch = 1;
        while (P.batch < 64 && (int64_t)P.batch * 2 * std::max(1, p->chunk_len) * 4 <= per_warp * 3) P.batch *= 2;
        P.items = own.get<int4>(P.n_items);
        if (p->row_order == 1) P.order = own.get<int32_t>(N);
        SGA_TRY(own.err);
        if (P.n_chunks > 0) {
            chunk_items_kernel<<<grid_for(P.n_chunks, 256, 65535), 256, 0, s>>>(P.chunk_row, P.chunk_beg,
                                                                                P.chunk_end, P.n_chunks, P.items);
            SGA_TRY(cudaGetLastError());
        }
        int32_t *k1 = ka, *v1 = va, *k2 = kb, *v2 = vb;
        const int32_t maxdeg = (int32_t)std::min<int64_t>(E, INT32_MAX - 1);
        order_keys_kernel<<<grid_for(N, 256, 65535), 256, 0, s>>>(ptr, N, maxdeg, p->split_threshold,
                                                                  p->row_order == 1, k1, v1);
        SGA_TRY(cudaGetLastError());
        int bits = 1;
        if (p->row_order == 1)
            while (bits < 31 && ((int64_t)1 << bits) <= maxdeg) ++bits;
        SGA_TRY(radix_sort_pairs(&k1, &v1, &k2, &v2, N, bits, hist_o, scan_tmp, s));
        if (P.order) SGA_TRY(cudaMemcpyAsync(P.order, v1, 4 * (size_t)N, cudaMemcpyDeviceToDevice, s));
        item_fill_kernel<<<grid_for(N, 256, 65535), 256, 0, s>>>(ptr, v1 + P.n_split, N - P.n_split,
                                                                 P.items + P.n_chunks);
        SGA_TRY(cudaGetLastError());
    }
    SGA_TRY(cudaStreamSynchronize(s));
    tmp.release();
    p->device_bytes = own.bytes;
    p->owned = std::move(own.ptrs);
    return SGA_OK;
}

void plan_free(sga_plan *p) {
    for (void *x : p->owned) cudaFree(x);
    p->owned.clear();
}


int64_t radix_hist_elems(int64_t n) {
    const int64_t n_tiles = (n + kRadixTile - 1) / kRadixTile;
    return (int64_t)kRadixBins * std::max<int64_t>(n_tiles, 1);
}

// Stable LSD radix sort of n (key, value) pairs by the low `bits` bits of the
// non-negative keys, 8 bits per pass.  (*ka, *va) hold the input, (*kb, *vb)
// scratch of n each; hist holds radix_hist_elems(n) and scan_tmp
// scan_tmp_elems(radix_hist_elems(n)) int32.  The sorted pairs end in
// (*ka, *va): the buffer pointers are swapped as the passes alternate.
cudaError_t radix_sort_pairs(int32_t **ka, int32_t **va, int32_t **kb, int32_t **vb, int64_t n,
                             int bits, int32_t *hist, int32_t *scan_tmp, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t n_tiles = (n + kRadixTile - 1) / kRadixTile;
    const int64_t hist_n = (int64_t)kRadixBins * n_tiles;
    const unsigned blocks = (unsigned)((n_tiles + kWarpsPerBlock - 1) / kWarpsPerBlock);
    for (int shift = 0; shift < bits; shift += kRadixBits) {
        radix_hist_kernel<<<blocks, 32 * kWarpsPerBlock, 0, s>>>(*ka, n, shift, n_tiles, hist);
        cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess) e = exclusive_scan(hist, hist, hist_n, scan_tmp, s);
        if (e != cudaSuccess) return e;
        radix_scatter_kernel<<<blocks, 32 * kWarpsPerBlock, 0, s>>>(*ka, *va, n, shift, n_tiles, hist,
                                                                  *kb, *vb);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        std::swap(*ka, *kb);
        std::swap(*va, *vb);
    }
    return cudaSuccess;
}

}  // namespace sga
