// Degree-aware min / max neighbourhood aggregation over the destination CSR:
// out_i[f] = max_j X_j[f] (or min) over the sources j of row i, with the
// winning source of every element (first edge of the row on ties), and the
// backward pass that routes dOut_i[f] to that source.
//
// Method ("On Efficient Scaling of GNNs via IO-Aware Layers Implementations":
// the arXiv abstract's degree-aware reduction kernels, and the Yandex
// Research blog post's "Aggregation layers" paragraph, which answers
// heavy-tailed degrees with degree-aware tiling and extra parallelism for
// high-degree nodes).  The forward is the attention layers' gather schedule
// with a different combine: the persistent edge stream gathers neighbour
// rows (16-byte chunks, one warp-wide load per chunk) and each lane keeps the
// running extreme of its elements and the row-local position of the edge
// that holds it; rows above the split threshold are cut into chunks whose
// partial extremes are merged in chunk order.  min and max are exact, so the
// values are bit-identical to any correct implementation, and positions make
// the winner independent of the order in which edge groups and chunks are
// combined.
#include <algorithm>

#include "common.cuh"
#include "gt.cuh"
#include "plan.h"

namespace sga {

// gathered X rows; no own rows or scalars
template <int NC, int G> using AggStream = RingCfg<NC, G, 1, 0, 0, 0, 2, 4>;

template <bool MAX> __device__ __forceinline__ bool better(float v, float b) {
    return MAX ? v > b : v < b;
}

template <typename T, bool MAX, int NC, int G>
__global__ void __launch_bounds__(256, 2) agg_fwd_kernel(AggArgs a) {
    using C = AggStream<NC, G>;
    constexpr int EL = Elt<T>::EL, U = C::U, NG = C::NG, STEP = C::STEP;
    extern __shared__ __align__(16) unsigned char dsmem[];
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.HD / EL;
    StreamArrays arr{};
    arr.rows[0] = static_cast<const uint4 *>(a.X);
    EdgeStream<C> st;
    st.init(dsmem + (threadIdx.x >> 5) * C::BYTES, arr, a.rows, a.indptr, a.indices, a.N, 1, R, 1,
            a.split_threshold, a.d_err);
    const float init = MAX ? -INFINITY : INFINITY;
    StreamItem it;
    while (st.next_item(it)) {
        float best[NC][EL];
        int32_t pos[NC][EL];   // row-local edge offset of the winner (INT32_MAX: none yet)
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int x = 0; x < EL; ++x) {
                best[k][x] = init;
                pos[k][x] = INT32_MAX;
            }
        for (int step = 0; step < it.nsteps; ++step) {
            st.wait_step();
#pragma unroll
            for (int u = 0; u < U; ++u) {
                // a group takes its edges in ascending order and keeps the
                // first of equal values (strict comparison; the first edge is
                // taken whatever its value, so infinities are handled too)
                const bool ok = st.valid(u);
                const int32_t off = step * STEP + g + NG * u;
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    float v[EL];
                    unpack<T>(st.row(u, 0, k), v);
#pragma unroll
                    for (int x = 0; x < EL; ++x)
                        if (ok && (pos[k][x] == INT32_MAX || better<MAX>(v[x], best[k][x]))) {
                            best[k][x] = v[x];
                            pos[k][x] = off;
                        }
                }
            }
            st.release_step();
        }
        // merge the edge groups: the better value wins, the earlier edge on ties
#pragma unroll
        for (int o = G; o < 32; o <<= 1)
#pragma unroll
            for (int k = 0; k < NC; ++k)
#pragma unroll
                for (int x = 0; x < EL; ++x) {
                    const float bo = __shfl_xor_sync(SGA_FULL_MASK, best[k][x], o);
                    const int32_t po = __shfl_xor_sync(SGA_FULL_MASK, pos[k][x], o);
                    if (po != INT32_MAX &&
                        (pos[k][x] == INT32_MAX || better<MAX>(bo, best[k][x]) ||
                         (bo == best[k][x] && po < pos[k][x]))) {
                        best[k][x] = bo;
                        pos[k][x] = po;
                    }
                }
        if (g == 0) {
            const int32_t beg = it.partial ? __ldg(a.rows.chunk_beg + it.item) : __ldg(a.indptr + it.row);
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                const int c = gl + G * k;
                if (c >= R) continue;
                if (it.partial) {
                    float4 *dv = reinterpret_cast<float4 *>(a.ws_val + (size_t)it.item * a.HD + c * EL);
                    int4 *dp = reinterpret_cast<int4 *>(a.ws_pos + (size_t)it.item * a.HD + c * EL);
#pragma unroll
                    for (int x = 0; x < EL; x += 4) {
                        dv[x / 4] = make_float4(best[k][x], best[k][x + 1], best[k][x + 2], best[k][x + 3]);
                        int4 p4;
                        p4.x = pos[k][x] == INT32_MAX ? INT32_MAX : beg + pos[k][x];
                        p4.y = pos[k][x + 1] == INT32_MAX ? INT32_MAX : beg + pos[k][x + 1];
                        p4.z = pos[k][x + 2] == INT32_MAX ? INT32_MAX : beg + pos[k][x + 2];
                        p4.w = pos[k][x + 3] == INT32_MAX ? INT32_MAX : beg + pos[k][x + 3];
                        dp[x / 4] = p4;
                    }
                } else {
                    float o[EL];
                    int32_t j[EL];
#pragma unroll
                    for (int x = 0; x < EL; ++x) {
                        const bool has = pos[k][x] != INT32_MAX;
                        o[x] = has ? best[k][x] : 0.0f;
                        j[x] = has ? __ldg(a.indices + beg + pos[k][x]) : -1;
                    }
                    reinterpret_cast<uint4 *>(a.out)[(size_t)it.row * R + c] = pack<T>(o);
                    int4 *da = reinterpret_cast<int4 *>(a.arg + (size_t)it.row * a.HD + c * EL);
#pragma unroll
                    for (int x = 0; x < EL; x += 4) da[x / 4] = make_int4(j[x], j[x + 1], j[x + 2], j[x + 3]);
                }
            }
        }
        st.finish_item();
    }
    st.drain();
}

// Split rows: one block per row, threads over the elements; chunks are taken
// in order with a strict comparison, so the earliest chunk (the earliest
// edge) wins ties.
template <typename T, bool MAX>
__global__ void __launch_bounds__(256) agg_fwd_merge_kernel(AggArgs a) {
    const int64_t s = blockIdx.x;
    if (s >= a.rows.n_split) return;
    const int32_t row = a.rows.split_rows[s];
    const int32_t c0 = a.rows.chunk_ptr[s], c1 = a.rows.chunk_ptr[s + 1];
    T *out = static_cast<T *>(a.out);
    for (int f = threadIdx.x; f < a.HD; f += blockDim.x) {
        float b = MAX ? -INFINITY : INFINITY;
        int32_t p = INT32_MAX;
        for (int32_t ch = c0; ch < c1; ++ch) {
            const float v = a.ws_val[(size_t)ch * a.HD + f];
            const int32_t q = a.ws_pos[(size_t)ch * a.HD + f];
            if (q != INT32_MAX && (p == INT32_MAX || better<MAX>(v, b))) {
                b = v;
                p = q;
            }
        }
        const bool has = p != INT32_MAX;
        out[(size_t)row * a.HD + f] = from_f32<T>(has ? b : 0.0f);
        a.arg[(size_t)row * a.HD + f] = has ? __ldg(a.indices + p) : -1;
    }
}

// Backward: dX_j[f] = sum over the destinations i whose element f was won by
// j of dOut_i[f].  Each (i, f) sends one value, so the pass is a scatter of
// N x HD elements with fp32 atomic adds into acc (which the caller zeroed);
// only the summation order of several contributions to one element varies.
template <typename T>
__global__ void __launch_bounds__(256) agg_bwd_scatter_kernel(const int32_t *__restrict__ arg,
                                                              const T *__restrict__ dOut, int64_t N,
                                                              int HD, float *acc, int32_t *err) {
    const int64_t n = N * HD;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * 4;
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4; t < n; t += stride) {
        const int4 j4 = __ldg(reinterpret_cast<const int4 *>(arg + t));
        const int f = (int)(t % HD);
        float d[4];
        if constexpr (sizeof(T) == 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(dOut + t));
            d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
        } else {
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(dOut + t));
            d[0] = __uint_as_float(v.x << 16);
            d[1] = __uint_as_float(v.x & 0xffff0000u);
            d[2] = __uint_as_float(v.y << 16);
            d[3] = __uint_as_float(v.y & 0xffff0000u);
        }
        const int32_t j[4] = {j4.x, j4.y, j4.z, j4.w};
#pragma unroll
        for (int x = 0; x < 4; ++x) {
            if (j[x] < 0) continue;   // empty row: no source
            if ((int64_t)j[x] >= N) {
                atomicOr(err, kErrIndexRange);
                continue;
            }
            atomicAdd(acc + (size_t)j[x] * HD + f + x, d[x]);
        }
    }
}

__global__ void __launch_bounds__(256) agg_cast_kernel(const float *__restrict__ acc, int64_t n,
                                                       __nv_bfloat16 *__restrict__ out) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * 8;
    for (int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8; t < n; t += stride) {
        const float4 a0 = __ldg(reinterpret_cast<const float4 *>(acc + t));
        const float4 a1 = __ldg(reinterpret_cast<const float4 *>(acc + t + 4));
        const float v[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        *reinterpret_cast<uint4 *>(out + t) = pack<__nv_bfloat16>(v);
    }
}

namespace {

unsigned stride_grid(int64_t n, int per_thread, int num_sms) {
    const int64_t want = (n / per_thread + 255) / 256;
    const int64_t cap = (int64_t)num_sms * 8;
    return (unsigned)std::max<int64_t>(1, std::min(want, cap));
}

template <typename T, bool MAX> cudaError_t agg_fwd_op(const AggArgs &a, cudaStream_t s) {
    const int R = a.HD / Elt<T>::EL;
    const int64_t items = (int64_t)a.rows.n_chunks + a.N;
    cudaError_t e = dispatch_shape<1, max_nc<T>()>(R, [&]<int NC, int G>() -> cudaError_t {
        if (items == 0) return cudaSuccess;
        note_launch(SGA_KERN_AGG_FWD, s, false);
        const cudaError_t e = launch_streamed<AggStream<NC, G>, agg_fwd_kernel<T, MAX, NC, G>>(items, s, a);
        note_launch(SGA_KERN_AGG_FWD, s, true);
        return e;
    });
    if (e != cudaSuccess || a.rows.n_split == 0) return e;
    note_launch(SGA_KERN_AGG_FWD_MERGE, s, false);
    agg_fwd_merge_kernel<T, MAX><<<(unsigned)a.rows.n_split, 256, 0, s>>>(a);
    note_launch(SGA_KERN_AGG_FWD_MERGE, s, true);
    return cudaGetLastError();
}

}  // namespace

template <typename T> cudaError_t agg_fwd_t(const AggArgs &a, bool is_max, cudaStream_t s) {
    return is_max ? agg_fwd_op<T, true>(a, s) : agg_fwd_op<T, false>(a, s);
}

template <typename T> cudaError_t agg_bwd_t(const AggArgs &a, cudaStream_t s) {
    const int64_t n = a.N * (int64_t)a.HD;
    if (n == 0) return cudaSuccess;
    float *acc = sizeof(T) == 4 ? static_cast<float *>(a.dX) : a.ws_acc;
    cudaError_t e = cudaMemsetAsync(acc, 0, sizeof(float) * (size_t)n, s);
    if (e != cudaSuccess) return e;
    note_launch(SGA_KERN_AGG_BWD, s, false);
    agg_bwd_scatter_kernel<T><<<stride_grid(n, 4, a.num_sms), 256, 0, s>>>(
        a.arg, static_cast<const T *>(a.dOut), a.N, a.HD, acc, a.d_err);
    note_launch(SGA_KERN_AGG_BWD, s, true);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if constexpr (sizeof(T) == 2) {
        note_launch(SGA_KERN_AGG_BWD_CAST, s, false);
        agg_cast_kernel<<<stride_grid(n, 8, a.num_sms), 256, 0, s>>>(acc, n, static_cast<__nv_bfloat16 *>(a.dX));
        note_launch(SGA_KERN_AGG_BWD_CAST, s, true);
        e = cudaGetLastError();
    }
    return e;
}

template cudaError_t agg_fwd_t<float>(const AggArgs &, bool, cudaStream_t);
template cudaError_t agg_fwd_t<__nv_bfloat16>(const AggArgs &, bool, cudaStream_t);
template cudaError_t agg_bwd_t<float>(const AggArgs &, cudaStream_t);
template cudaError_t agg_bwd_t<__nv_bfloat16>(const AggArgs &, cudaStream_t);

}  // namespace sga
