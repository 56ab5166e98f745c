// Degree-aware min / max neighbourhood aggregation over the destination CSR:
// out_i[f] = max_j X_j[f] (or min) over the sources j of row i, with the
// winning source of every element (first edge of the row on ties) and a win
// mask per edge (one byte per 16-byte chunk of the row: the bits of the
// chunk's elements that edge won), and the backward pass that gathers
// dOut_i[f] into the winning source over the transposed CSR.
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
template <int NC, int G> using AggStream = RingCfg<NC, G, 1, 0, 0, 0, 2, 4, 0, true, false, true>;

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
#pragma unroll
                    for (int x = 0; x < EL; ++x) o[x] = pos[k][x] != INT32_MAX ? best[k][x] : 0.0f;
                    reinterpret_cast<uint4 *>(a.out)[(size_t)it.row * R + c] = pack<T>(o);
                    if (a.arg) {
                        int32_t j[EL];
#pragma unroll
                        for (int x = 0; x < EL; ++x)
                            j[x] = pos[k][x] != INT32_MAX ? __ldg(a.indices + beg + pos[k][x]) : -1;
                        int4 *da = reinterpret_cast<int4 *>(a.arg + (size_t)it.row * a.HD + c * EL);
#pragma unroll
                        for (int x = 0; x < EL; x += 4) da[x / 4] = make_int4(j[x], j[x + 1], j[x + 2], j[x + 3]);
                    }
                    if (a.mask) {
                        // win mask: the byte of (winning edge, this chunk) gets the bits
                        // of the chunk's elements that edge won (bytes start cleared)
#pragma unroll
                        for (int x = 0; x < EL; ++x) {
                            if (pos[k][x] == INT32_MAX) continue;
                            bool first = true;
                            uint32_t bits = 0;
#pragma unroll
                            for (int y = 0; y < EL; ++y) {
                                if (pos[k][y] != pos[k][x]) continue;
                                if (y < x) first = false;
                                bits |= 1u << y;
                            }
                            if (first) a.mask[(size_t)(beg + pos[k][x]) * R + c] = (uint8_t)bits;
                        }
                    }
                }
            }
        }
        st.finish_item();
    }
    st.drain();
}

// Split rows: one block per row, a thread per element (coalesced reads of
// the chunk partials).  The order (better value, then earlier edge) is a
// total order on the candidates, so the result does not depend on the order
// in which chunks are combined.  The win-mask byte of a 16-byte chunk is
// built from the EL consecutive lanes that hold its elements: lanes with the
// same winning edge share the byte, and the first of them writes it.
template <typename T, bool MAX>
__global__ void __launch_bounds__(256) agg_fwd_merge_kernel(AggArgs a) {
    constexpr int EL = Elt<T>::EL;
    const int64_t s = blockIdx.x;
    if (s >= a.rows.n_split) return;
    const int32_t row = a.rows.split_rows[s];
    const int32_t c0 = a.rows.chunk_ptr[s], c1 = a.rows.chunk_ptr[s + 1];
    const int R = a.HD / EL, lane = threadIdx.x & 31, g0 = lane & ~(EL - 1);
    T *out = static_cast<T *>(a.out);
    // HD is a multiple of 32: a warp is either wholly inside the loop or out
    for (int f = threadIdx.x; f < a.HD; f += blockDim.x) {
        float b = MAX ? -INFINITY : INFINITY;
        int32_t p = INT32_MAX;
#pragma unroll 4
        for (int32_t ch = c0; ch < c1; ++ch) {
            const float v = a.ws_val[(size_t)ch * a.HD + f];
            const int32_t q = a.ws_pos[(size_t)ch * a.HD + f];
            if (q != INT32_MAX && (p == INT32_MAX || better<MAX>(v, b) || (v == b && q < p))) {
                b = v;
                p = q;
            }
        }
        const bool has = p != INT32_MAX;
        out[(size_t)row * a.HD + f] = from_f32<T>(has ? b : 0.0f);
        if (a.arg) a.arg[(size_t)row * a.HD + f] = has ? __ldg(a.indices + p) : -1;
        if (a.mask) {
            const uint32_t bits = (__match_any_sync(SGA_FULL_MASK, p) >> g0) & ((1u << EL) - 1u);
            if (has && lane - g0 == __ffs(bits) - 1) a.mask[(size_t)p * R + f / EL] = (uint8_t)bits;
        }
    }
}

// Backward: dX_j[f] = sum of dOut_i[f] over the destinations i of j whose
// element f the edge (i <- j) won.  A warp per work item of the transposed
// CSR (a source, or a chunk of a high-degree source), lanes across the row's
// 16-byte chunks.  The item's edges are taken 32 at a time (t_eid maps a
// transposed entry to its CSR edge, t_dst gives its destination), and UN of
// them at once per lane chunk: the UN win-mask bytes are loaded together,
// then the dOut chunks of the set bytes only, so that each lane has UN
// independent loads in flight instead of a chain of dependent ones.  No
// atomics: every sum runs in transposed-edge order (reproducible).
template <typename T, int NC>
__global__ void __launch_bounds__(256) agg_bwd_gather_kernel(AggArgs a) {
    constexpr int EL = Elt<T>::EL;
    constexpr int UN = NC >= 8 ? 2 : NC >= 4 ? 4 : 8;   // divides 32
    const int lane = threadIdx.x & 31;
    const int R = a.HD / EL;
    const uint4 *dO = static_cast<const uint4 *>(a.dOut);
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < a.cols.n_items;
         item += stride) {
        const int4 t = __ldg(a.cols.items + item);
        float acc[NC][EL];
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int x = 0; x < EL; ++x) acc[k][x] = 0.f;
        for (int32_t e0 = t.y; e0 < t.z; e0 += 32) {
            const int cnt = min(32, t.z - e0);
            const int32_t eid = lane < cnt ? __ldg(a.t_eid + e0 + lane) : 0;
            int32_t dst = lane < cnt ? __ldg(a.t_dst + e0 + lane) : -1;
            if (lane < cnt && (uint32_t)dst >= (uint32_t)a.N) {
                atomicOr(a.d_err, kErrIndexRange);
                dst = -1;
            }
            for (int u0 = 0; u0 < cnt; u0 += UN) {   // u0 + q <= 31: lanes past cnt carry dst = -1
                int32_t e[UN], i[UN];
#pragma unroll
                for (int q = 0; q < UN; ++q) {
                    e[q] = __shfl_sync(SGA_FULL_MASK, eid, u0 + q);
                    i[q] = __shfl_sync(SGA_FULL_MASK, dst, u0 + q);
                }
                uint32_t m[UN][NC];
#pragma unroll
                for (int q = 0; q < UN; ++q)
#pragma unroll
                    for (int k = 0; k < NC; ++k) {
                        const int c = lane + 32 * k;
                        m[q][k] = i[q] >= 0 && c < R ? (uint32_t)__ldg(a.mask + (size_t)e[q] * R + c) : 0u;
                    }
                uint4 v[UN][NC];
#pragma unroll
                for (int q = 0; q < UN; ++q)
#pragma unroll
                    for (int k = 0; k < NC; ++k)
                        v[q][k] = m[q][k] ? ldg16(dO + (size_t)i[q] * R + lane + 32 * k) : make_uint4(0, 0, 0, 0);
#pragma unroll
                for (int q = 0; q < UN; ++q)
#pragma unroll
                    for (int k = 0; k < NC; ++k) {
                        float x8[EL];
                        unpack<T>(v[q][k], x8);
#pragma unroll
                        for (int x = 0; x < EL; ++x)
                            if ((m[q][k] >> x) & 1u) acc[k][x] += x8[x];
                    }
            }
        }
#pragma unroll
        for (int k = 0; k < NC; ++k) {
            const int c = lane + 32 * k;
            if (c >= R) continue;
            if (item < a.cols.n_chunks) {
                float4 *dst = reinterpret_cast<float4 *>(a.ws_val + (size_t)item * a.HD + c * EL);
#pragma unroll
                for (int x = 0; x < EL; x += 4) dst[x / 4] = make_float4(acc[k][x], acc[k][x + 1], acc[k][x + 2], acc[k][x + 3]);
            } else {
                reinterpret_cast<uint4 *>(a.dX)[(size_t)t.x * R + c] = pack<T>(acc[k]);
            }
        }
    }
}

// Split sources: dX is the sum of the chunks' partial sums, in chunk order.
template <typename T>
__global__ void __launch_bounds__(256) agg_bwd_merge_kernel(AggArgs a) {
    const int64_t s = blockIdx.x;
    if (s >= a.cols.n_split) return;
    const int32_t row = a.cols.split_rows[s];
    const int32_t c0 = a.cols.chunk_ptr[s], c1 = a.cols.chunk_ptr[s + 1];
    T *dX = static_cast<T *>(a.dX);
    for (int f = threadIdx.x; f < a.HD; f += blockDim.x) {
        float v = 0.f;
        for (int32_t ch = c0; ch < c1; ++ch) v += a.ws_val[(size_t)ch * a.HD + f];
        dX[(size_t)row * a.HD + f] = from_f32<T>(v);
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
    if (a.mask && a.E > 0) {   // win-mask bytes start cleared; the forward sets the winners'
        const cudaError_t e0 = cudaMemsetAsync(a.mask, 0, (size_t)a.E * R, s);
        if (e0 != cudaSuccess) return e0;
    }
    cudaError_t e = dispatch_shape<1, max_nc<T>()>(R, [&]<int NC, int G>() -> cudaError_t {
        if (items == 0) return cudaSuccess;
        if (reset_items<AggStream<NC, G>>(a.rows, s) != cudaSuccess) return cudaGetLastError();
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
    if (a.N == 0) return cudaSuccess;
    const int R = a.HD / Elt<T>::EL;
    const int64_t items = a.cols.n_items;
    cudaError_t e = cudaSuccess;
    if (items > 0) {
        note_launch(SGA_KERN_AGG_BWD, s, false);
        auto go = [&]<int NC>() {
            agg_bwd_gather_kernel<T, NC><<<persistent_blocks<agg_bwd_gather_kernel<T, NC>>(items), 256, 0, s>>>(a);
        };
        if (R <= 32) go.template operator()<1>();
        else if (R <= 64) go.template operator()<2>();
        else if (R <= 128) go.template operator()<4>();
        else go.template operator()<8>();
        note_launch(SGA_KERN_AGG_BWD, s, true);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (a.cols.n_split > 0) {
        note_launch(SGA_KERN_AGG_BWD_MERGE, s, false);
        agg_bwd_merge_kernel<T><<<(unsigned)a.cols.n_split, 256, 0, s>>>(a);
        note_launch(SGA_KERN_AGG_BWD_MERGE, s, true);
        e = cudaGetLastError();
    }
    return e;
}

template cudaError_t agg_fwd_t<float>(const AggArgs &, bool, cudaStream_t);
template cudaError_t agg_fwd_t<__nv_bfloat16>(const AggArgs &, bool, cudaStream_t);
template cudaError_t agg_bwd_t<float>(const AggArgs &, cudaStream_t);
template cudaError_t agg_bwd_t<__nv_bfloat16>(const AggArgs &, cudaStream_t);

}  // namespace sga
