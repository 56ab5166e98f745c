// Block-sparse split of a destination-sorted CSR for the tensor-core
// forward: the "block-sparse graph representation that enables the use of
// tensor cores" of the IO-aware layers blog post ("Attention-based layers"
// paragraph), which pays off on locally dense graphs.
//
// Rows form panels of 128 destinations, sources form column tiles of 16.  A
// (panel, tile) pair holding at least min_nnz edges is kept: its column index
// and one 16-bit source mask per panel row are stored.  All other edges stay
// in a residual CSR, in their original order.  One CTA per panel counts the
// edges per column tile in a shared-memory histogram (16-bit counts packed in
// pairs); kept tiles are listed in column order.  Everything is determined by
// the graph and min_nnz: the arrays are bit-exact.
#include <algorithm>
#include <vector>

#include "common.cuh"
#include "plan.h"

namespace sga {
namespace {

constexpr int kPanel = 128, kWidth = 16, kThreads = 256;

__device__ __forceinline__ uint32_t bin_count(const uint32_t *h, int b) {
    return (h[b >> 1] >> ((b & 1) * 16)) & 0xffffu;
}

__device__ void panel_histogram(const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices,
                                int64_t N, int p, uint32_t *h, int words) {
    for (int w = threadIdx.x; w < words; w += blockDim.x) h[w] = 0;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = (int64_t)p * kPanel;
    for (int rr = warp; rr < kPanel && r0 + rr < N; rr += blockDim.x >> 5) {
        const int32_t b = indptr[r0 + rr], e = indptr[r0 + rr + 1];
        for (int32_t x = b + lane; x < e; x += 32) {
            const int bin = indices[x] / kWidth;
            atomicAdd(&h[bin >> 1], 1u << ((bin & 1) * 16));
        }
    }
    __syncthreads();
}

// Kept tiles per panel and residual edges per row.
__global__ void __launch_bounds__(kThreads)
bsr_count_kernel(const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices, int64_t N,
                 int n_bins, int min_nnz, int32_t *__restrict__ kept, int32_t *__restrict__ r_count) {
    extern __shared__ uint32_t h[];
    __shared__ int32_t red[kThreads / 32];
    const int p = blockIdx.x, words = (n_bins + 1) / 2;
    panel_histogram(indptr, indices, N, p, h, words);
    int c = 0;
    for (int b = threadIdx.x; b < n_bins; b += blockDim.x) c += bin_count(h, b) >= (uint32_t)min_nnz;
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(SGA_FULL_MASK, c, o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) red[warp] = c;
    __syncthreads();
    if (threadIdx.x == 0) {
        int t = 0;
        for (int w = 0; w < kThreads / 32; ++w) t += red[w];
        kept[p] = t;
    }
    const int64_t r0 = (int64_t)p * kPanel;
    for (int rr = warp; rr < kPanel && r0 + rr < N; rr += kThreads / 32) {
        const int32_t b = indptr[r0 + rr], e = indptr[r0 + rr + 1];
        int n = 0;
        for (int32_t x = b + lane; x < e; x += 32) n += bin_count(h, indices[x] / kWidth) < (uint32_t)min_nnz;
        for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(SGA_FULL_MASK, n, o);
        if (lane == 0) r_count[r0 + rr] = n;
    }
}

// Tile columns (in column order), tile masks, residual indices (in order).
__global__ void __launch_bounds__(kThreads)
bsr_fill_kernel(const int32_t *__restrict__ indptr, const int32_t *__restrict__ indices, int64_t N,
                int n_bins, int min_nnz, const int32_t *__restrict__ tile_ptr,
                int32_t *__restrict__ tile_col, uint32_t *__restrict__ tile_bits32,
                const int32_t *__restrict__ r_indptr, int32_t *__restrict__ r_indices,
                int32_t *__restrict__ dup) {
    extern __shared__ uint32_t h[];
    __shared__ int32_t scan[kThreads];
    const int p = blockIdx.x, words = (n_bins + 1) / 2, tid = threadIdx.x;
    panel_histogram(indptr, indices, N, p, h, words);
    // kept bins of this thread's contiguous range, then a block prefix sum
    const int per = (n_bins + kThreads - 1) / kThreads;
    const int b0 = min(n_bins, tid * per), b1 = min(n_bins, b0 + per);
    int c = 0;
    for (int b = b0; b < b1; ++b) c += bin_count(h, b) >= (uint32_t)min_nnz;
    scan[tid] = c;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int t = 0; t < kThreads; ++t) {
            const int v = scan[t];
            scan[t] = run;
            run += v;
        }
    }
    __syncthreads();
    // list kept bins; turn the histogram into a map bin -> local tile index (0xffff: not kept)
    int loc = scan[tid];
    const int base = tile_ptr[p];
    uint16_t idx[64];
    int ni = 0;
    for (int b = b0; b < b1; ++b) {
        const bool k = bin_count(h, b) >= (uint32_t)min_nnz;
        if (k) tile_col[base + loc] = b;
        if (ni < 64) idx[ni++] = k ? (uint16_t)loc : (uint16_t)0xffff;
        loc += k;
    }
    __syncthreads();
    uint16_t *map = reinterpret_cast<uint16_t *>(h);
    for (int b = b0, i = 0; b < b1 && i < 64; ++b, ++i) map[b] = idx[i];
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t r0 = (int64_t)p * kPanel;
    for (int rr = warp; rr < kPanel && r0 + rr < N; rr += kThreads / 32) {
        const int32_t b = indptr[r0 + rr], e = indptr[r0 + rr + 1];
        int32_t out = r_indptr[r0 + rr];
        for (int32_t x0 = b; x0 < e; x0 += 32) {
            const int32_t x = x0 + lane;
            const bool in = x < e;
            const int32_t j = in ? indices[x] : 0;
            const uint16_t t = in ? map[j / kWidth] : (uint16_t)0xffff;
            if (in && t != 0xffff) {
                const int64_t word = ((int64_t)(base + t) * kPanel + rr) >> 1;
                const uint32_t bit = (1u << (j % kWidth)) << ((rr & 1) * 16);
                if (atomicOr(&tile_bits32[word], bit) & bit) *dup = 1;   // a repeated edge
            }
            const unsigned res = __ballot_sync(SGA_FULL_MASK, in && t == 0xffff);
            if (in && t == 0xffff) r_indices[out + __popc(res & ((1u << lane) - 1))] = j;
            out += __popc(res);
        }
    }
}

}  // namespace

sga_status bsr_build(sga_plan *p, cudaStream_t s) {
    TileSet &T = p->tiles;
    const int64_t N = p->N;
    const int n_bins = (int)((N + kWidth - 1) / kWidth);
    const size_t hist_bytes = (size_t)((n_bins + 1) / 2) * 4;
    // the histogram and the per-thread bin ranges must fit (bins per thread <= 64)
    if (hist_bytes > 200 * 1024 || (n_bins + kThreads - 1) / kThreads > 64) return SGA_EUNSUPPORTED;
    T.n_panels = (int32_t)((N + kPanel - 1) / kPanel);
    std::vector<void *> tmp;
    auto fail = [&](cudaError_t e) {
        for (void *x : tmp) cudaFree(x);
        set_cuda_error(e);
        return SGA_ECUDA;
    };
    auto alloc = [&](void **ptr, size_t bytes, bool own) -> cudaError_t {
        cudaError_t e = cudaMalloc(ptr, std::max<size_t>(bytes, 4));
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
    int32_t *kept = nullptr, *scan_tmp = nullptr, *dup = nullptr;
    cudaError_t e;
    if ((e = alloc((void **)&kept, sizeof(int32_t) * (T.n_panels + 1), false)) != cudaSuccess) return fail(e);
    if ((e = alloc((void **)&dup, sizeof(int32_t), false)) != cudaSuccess) return fail(e);
    if ((e = alloc((void **)&T.tile_ptr, sizeof(int32_t) * (T.n_panels + 1), true)) != cudaSuccess) return fail(e);
    if ((e = alloc((void **)&T.r_indptr, sizeof(int32_t) * (N + 1), true)) != cudaSuccess) return fail(e);
    if ((e = alloc((void **)&scan_tmp, sizeof(int32_t) * scan_tmp_elems(std::max<int64_t>(N + 1, T.n_panels + 1)),
                   false)) != cudaSuccess)
        return fail(e);
    if (hist_bytes > 48 * 1024) {
        if ((e = cudaFuncSetAttribute(bsr_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)hist_bytes)) != cudaSuccess)
            return fail(e);
        if ((e = cudaFuncSetAttribute(bsr_fill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)hist_bytes)) != cudaSuccess)
            return fail(e);
    }
    if ((e = cudaMemsetAsync(kept, 0, sizeof(int32_t) * (T.n_panels + 1), s)) != cudaSuccess) return fail(e);
    if ((e = cudaMemsetAsync(dup, 0, sizeof(int32_t), s)) != cudaSuccess) return fail(e);
    if ((e = cudaMemsetAsync(T.r_indptr, 0, sizeof(int32_t) * (N + 1), s)) != cudaSuccess) return fail(e);
    if (T.n_panels > 0) {
        bsr_count_kernel<<<T.n_panels, kThreads, hist_bytes, s>>>(p->indptr, p->indices, N, n_bins,
                                                                  T.min_nnz, kept, T.r_indptr);
        if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
    }
    if ((e = exclusive_scan(kept, T.tile_ptr, T.n_panels + 1, scan_tmp, s)) != cudaSuccess) return fail(e);
    if ((e = exclusive_scan(T.r_indptr, T.r_indptr, N + 1, scan_tmp, s)) != cudaSuccess) return fail(e);
    int32_t tot[2] = {0, 0};
    if ((e = cudaMemcpyAsync(&tot[0], T.tile_ptr + T.n_panels, 4, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return fail(e);
    if ((e = cudaMemcpyAsync(&tot[1], T.r_indptr + N, 4, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return fail(e);
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail(e);
    T.n_tiles = tot[0];
    T.E_res = tot[1];
    if ((e = alloc((void **)&T.tile_col, sizeof(int32_t) * (size_t)T.n_tiles, true)) != cudaSuccess) return fail(e);
    if ((e = alloc((void **)&T.tile_bits, sizeof(uint16_t) * kPanel * (size_t)T.n_tiles, true)) != cudaSuccess)
        return fail(e);
    if ((e = alloc((void **)&T.r_indices, sizeof(int32_t) * (size_t)T.E_res, true)) != cudaSuccess) return fail(e);
    if (T.n_tiles > 0 &&
        (e = cudaMemsetAsync(T.tile_bits, 0, sizeof(uint16_t) * kPanel * (size_t)T.n_tiles, s)) != cudaSuccess)
        return fail(e);
    if (T.n_panels > 0) {
        bsr_fill_kernel<<<T.n_panels, kThreads, hist_bytes, s>>>(
            p->indptr, p->indices, N, n_bins, T.min_nnz, T.tile_ptr, T.tile_col,
            reinterpret_cast<uint32_t *>(T.tile_bits), T.r_indptr, T.r_indices, dup);
        if ((e = cudaGetLastError()) != cudaSuccess) return fail(e);
    }
    int32_t repeated = 0;
    if ((e = cudaMemcpyAsync(&repeated, dup, 4, cudaMemcpyDeviceToHost, s)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamSynchronize(s)) != cudaSuccess) return fail(e);
    for (void *x : tmp) cudaFree(x);
    tmp.clear();
    // a tile mask holds an edge once: repeated edges inside kept tiles cannot be represented
    if (repeated) return SGA_EINVAL;

    // column view (host, O(tiles)): entries (row panel, column panel of 8 tile
    // columns) in column-panel order, row panels ascending within each
    std::vector<int32_t> h_ptr(T.n_panels + 1), h_col(T.n_tiles);
    if ((e = cudaMemcpy(h_ptr.data(), T.tile_ptr, sizeof(int32_t) * (T.n_panels + 1), cudaMemcpyDeviceToHost)) !=
        cudaSuccess)
        return fail(e);
    if (T.n_tiles > 0 &&
        (e = cudaMemcpy(h_col.data(), T.tile_col, sizeof(int32_t) * T.n_tiles, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return fail(e);
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
    if ((e = alloc((void **)&T.ct_ptr, sizeof(int32_t) * (T.n_cpanels + 1), true)) != cudaSuccess) return fail(e);
    if ((e = alloc((void **)&T.ct_panel, sizeof(int32_t) * T.n_entries, true)) != cudaSuccess) return fail(e);
    if ((e = alloc((void **)&T.ct_tile, sizeof(int32_t) * 8 * (size_t)T.n_entries, true)) != cudaSuccess)
        return fail(e);
    if ((e = cudaMemcpy(T.ct_ptr, c_ptr.data(), sizeof(int32_t) * (T.n_cpanels + 1), cudaMemcpyHostToDevice)) !=
        cudaSuccess)
        return fail(e);
    if (T.n_entries > 0) {
        if ((e = cudaMemcpy(T.ct_panel, c_panel.data(), sizeof(int32_t) * T.n_entries, cudaMemcpyHostToDevice)) !=
            cudaSuccess)
            return fail(e);
        if ((e = cudaMemcpy(T.ct_tile, c_tile.data(), sizeof(int32_t) * 8 * (size_t)T.n_entries,
                            cudaMemcpyHostToDevice)) != cudaSuccess)
            return fail(e);
    }
    return SGA_OK;
}

}  // namespace sga
