// Graph Transformer edge attention: fused forward (online softmax) and the
// recompute-from-lse backward, as templates instantiated per dtype.
//
// Method ("On Efficient Scaling of GNNs via IO-Aware Layers Implementations",
// Yandex Research blog post, "Attention-based layers" paragraph): the edge
// scores s_ij = q_i . k_j / sqrt(D) are produced and consumed on chip by an
// online softmax and never stored; the backward pass rebuilds the weights
// p_ij = exp(s_ij - lse_i) from the saved per-row log-sum-exp, following
// FlashAttention-2.
//
// Schedule (sm_103a).  One warp owns one work item: a whole destination row,
// or one fixed-length chunk of a split (high-degree) row.  A row of H*D
// elements is viewed as R = H*D*sizeof(T)/16 sixteen-byte chunks; lane l of a
// G-lane edge group holds chunks l, l+G, ...  (NC per lane), so one warp-wide
// 16-byte load per chunk gathers a neighbour row coalesced.  When R < 32 the
// warp splits into 32/G groups that take alternate edges and merge at the
// end.  Each head spans LH = D*sizeof(T)/16 adjacent lanes; its dot product
// is a log2(LH)-step xor-shuffle reduction.  U neighbours are loaded before
// any is used, so every lane keeps U*NC*2 sixteen-byte gathers in flight.
#pragma once

#include "common.cuh"
#include "plan.h"

namespace sga {

template <typename T, int D, int NC, int G> struct GtShape {
    static constexpr int EL = Elt<T>::EL;                     // elements per 16-byte chunk
    static constexpr int LH = D * (int)sizeof(T) / 16;        // lanes per head
    static constexpr int NG = 32 / G;                         // edge groups per warp
    static constexpr int U = NC >= 4 ? 1 : 4 / NC;            // neighbours in flight per group
    static_assert(LH <= G, "a head must fit in one edge group");
};

struct ItemRange {
    int32_t row, beg, end;
    bool partial;
};

// Work item w of a launch: chunks of split rows first, then every row (rows
// above the split threshold are skipped; their chunks cover them).
__device__ __forceinline__ bool decode_item(int64_t item, const Partition &P,
                                            const int32_t *__restrict__ ptr, int64_t N,
                                            int threshold, ItemRange &r) {
    if (item < P.n_chunks) {
        r.row = P.chunk_row[item];
        r.beg = P.chunk_beg[item];
        r.end = P.chunk_end[item];
        r.partial = true;
        return true;
    }
    const int64_t i = item - P.n_chunks;
    if (i >= N) return false;
    r.row = (int32_t)i;
    r.beg = ptr[i];
    r.end = ptr[i + 1];
    r.partial = false;
    return r.end - r.beg <= threshold;
}

// Fetch the 32 node ids of edges [e0, e0 + cnt) into one register per lane,
// range-checked against N (an out-of-range id becomes -1 and flags the plan).
__device__ __forceinline__ int32_t load_ids(const int32_t *__restrict__ ids, int32_t e0, int cnt,
                                            int64_t N, int32_t *err) {
    const int lane = threadIdx.x & 31;
    int32_t j = -1;
    if (lane < cnt) {
        j = __ldg(ids + e0 + lane);
        if ((uint32_t)j >= (uint32_t)N) {
            atomicOr(err, kErrIndexRange);
            j = -1;
        }
    }
    return j;
}

// Persistent warps walk the items w, w + S, w + 2S, ... (S = warps in the
// grid) through a three-stage pipeline: while item k runs, the metadata of
// item k + 2S (chunk descriptor or indptr pair) and the first 32 node ids of
// item k + S are already in flight, so a short row costs one gather latency
// instead of three dependent ones.
struct ItemMeta {
    int32_t row, beg, end;   // raw loads; row < 0 past the last item
};

__device__ __forceinline__ void meta_issue(int64_t item, const Partition &P,
                                           const int32_t *__restrict__ ptr, int64_t N,
                                           ItemMeta &m) {
    if (item < P.n_chunks) {
        m.row = __ldg(P.chunk_row + item);
        m.beg = __ldg(P.chunk_beg + item);
        m.end = __ldg(P.chunk_end + item);
    } else if (item - P.n_chunks < N) {
        const int64_t i = item - P.n_chunks;
        m.row = (int32_t)i;
        m.beg = __ldg(ptr + i);
        m.end = __ldg(ptr + i + 1);
    } else {
        m.row = -1;
        m.beg = m.end = 0;
    }
}

// True when the item is to be processed here (not past the end, and not a row
// above the split threshold, whose chunks are separate items).
__device__ __forceinline__ bool meta_eval(int64_t item, const ItemMeta &m, const Partition &P,
                                          int threshold, ItemRange &r) {
    r.row = m.row;
    r.beg = m.beg;
    r.end = m.end;
    r.partial = item < P.n_chunks;
    return m.row >= 0 && (r.partial || m.end - m.beg <= threshold);
}

// First batch of node ids of an item (lanes past the item's edges read nothing).
__device__ __forceinline__ int32_t first_ids(const int32_t *__restrict__ ids, const ItemRange &r,
                                             bool valid) {
    const int lane = threadIdx.x & 31;
    return (valid && lane < r.end - r.beg) ? __ldg(ids + r.beg + lane) : 0;
}

// Node ids of edges [e0, e0 + cnt), range-checked like load_ids: the
// prefetched batch for the item's first 32 edges, a fresh load after that.
__device__ __forceinline__ int32_t batch_ids(const int32_t *__restrict__ ids, int32_t e0, int cnt,
                                             const ItemRange &r, int32_t id0, int64_t N,
                                             int32_t *err) {
    if (e0 != r.beg) return load_ids(ids, e0, cnt, N, err);
    const int lane = threadIdx.x & 31;
    if (lane >= cnt) return -1;
    if ((uint32_t)id0 >= (uint32_t)N) {
        atomicOr(err, kErrIndexRange);
        return -1;
    }
    return id0;
}

// ------------------------------------------------------------------ forward

template <typename T, int D, int NC, int G>
__global__ void __launch_bounds__(256, 2)
gt_fwd_kernel(GtArgs a, float scale2) {
    using S = GtShape<T, D, NC, G>;
    constexpr int EL = S::EL, LH = S::LH, NG = S::NG, U = S::U;
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    const uint4 *__restrict__ Qc = static_cast<const uint4 *>(a.Q);
    const uint4 *__restrict__ Kc = static_cast<const uint4 *>(a.K);
    const uint4 *__restrict__ Vc = static_cast<const uint4 *>(a.V);
    const int64_t n_items = (int64_t)a.rows.n_chunks + a.N;
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerBlock;
    int64_t item = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);

    ItemMeta mn, mnn;
    meta_issue(item, a.rows, a.indptr, a.N, mn);
    ItemRange it;
    bool valid = meta_eval(item, mn, a.rows, a.split_threshold, it);
    int32_t id0 = first_ids(a.indices, it, valid);
    meta_issue(item + stride, a.rows, a.indptr, a.N, mn);
    for (; item < n_items; item += stride) {
        meta_issue(item + 2 * stride, a.rows, a.indptr, a.N, mnn);
        ItemRange itn;
        const bool validn = meta_eval(item + stride, mn, a.rows, a.split_threshold, itn);
        const int32_t id1 = first_ids(a.indices, itn, validn);
        if (valid) {
            float q[NC][EL], acc[NC][EL], m[NC], l[NC];
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                const int c = gl + G * k;
                if (c < R) unpack<T>(ldg16(Qc + (size_t)it.row * R + c), q[k]);
                else
#pragma unroll
                    for (int x = 0; x < EL; ++x) q[k][x] = 0.f;
#pragma unroll
                for (int x = 0; x < EL; ++x) acc[k][x] = 0.f;
                m[k] = -INFINITY;
                l[k] = 0.f;
            }
            for (int32_t e0 = it.beg; e0 < it.end; e0 += 32) {
                const int cnt = min(32, it.end - e0);
                const int32_t myj = batch_ids(a.indices, e0, cnt, it, id0, a.N, a.d_err);
                for (int t0 = 0; t0 < cnt; t0 += NG * U) {
                    uint4 kr[U][NC], vr[U][NC];
                    bool ok[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int t = t0 + g + NG * u;
                        const int32_t j = __shfl_sync(SGA_FULL_MASK, myj, t & 31);
                        ok[u] = (t < cnt) && (j >= 0);
#pragma unroll
                        for (int k = 0; k < NC; ++k) {
                            const int c = gl + G * k;
                            if (ok[u] && c < R) {
                                kr[u][k] = ldg16_stream(Kc + (size_t)j * R + c);
                                vr[u][k] = ldg16_stream(Vc + (size_t)j * R + c);
                            } else {
                                kr[u][k] = make_uint4(0, 0, 0, 0);
                                vr[u][k] = make_uint4(0, 0, 0, 0);
                            }
                        }
                    }
                    float sc[U][NC];
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int k = 0; k < NC; ++k) {
                            float kf[EL];
                            unpack<T>(kr[u][k], kf);
                            float dot = 0.f;
#pragma unroll
                            for (int x = 0; x < EL; ++x) dot = fmaf(q[k][x], kf[x], dot);
                            dot = group_sum<LH>(dot);
                            sc[u][k] = ok[u] ? dot * scale2 : -INFINITY;
                        }
#pragma unroll
                    for (int k = 0; k < NC; ++k) {
                        float mx = m[k];
#pragma unroll
                        for (int u = 0; u < U; ++u) mx = fmaxf(mx, sc[u][k]);
                        if (mx == -INFINITY) continue;
                        const float alpha = exp2_diff(m[k], mx);
                        l[k] *= alpha;
#pragma unroll
                        for (int x = 0; x < EL; ++x) acc[k][x] *= alpha;
#pragma unroll
                        for (int u = 0; u < U; ++u) {
                            const float p = exp2_diff(sc[u][k], mx);
                            l[k] += p;
                            float vf[EL];
                            unpack<T>(vr[u][k], vf);
#pragma unroll
                            for (int x = 0; x < EL; ++x) acc[k][x] = fmaf(p, vf[x], acc[k][x]);
                        }
                        m[k] = mx;
                    }
                }
            }
            // merge the edge groups of the warp (they saw disjoint edges)
#pragma unroll
            for (int off = G; off < 32; off <<= 1)
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    const float mo = __shfl_xor_sync(SGA_FULL_MASK, m[k], off);
                    const float lo = __shfl_xor_sync(SGA_FULL_MASK, l[k], off);
                    const float mx = fmaxf(m[k], mo);
                    const float a1 = exp2_diff(m[k], mx), a2 = exp2_diff(mo, mx);
                    l[k] = l[k] * a1 + lo * a2;
#pragma unroll
                    for (int x = 0; x < EL; ++x) {
                        const float ao = __shfl_xor_sync(SGA_FULL_MASK, acc[k][x], off);
                        acc[k][x] = acc[k][x] * a1 + ao * a2;
                    }
                    m[k] = mx;
                }
            if (g == 0) {
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    const int c = gl + G * k;
                    if (c >= R) continue;
                    const int h = c / LH;
                    if (it.partial) {
                        float4 *dst = reinterpret_cast<float4 *>(a.ws_acc + (size_t)item * HD + c * EL);
#pragma unroll
                        for (int x = 0; x < EL; x += 4)
                            dst[x / 4] = make_float4(acc[k][x], acc[k][x + 1], acc[k][x + 2], acc[k][x + 3]);
                        if (c % LH == 0) {
                            a.ws_ml[((size_t)item * a.H + h) * 2 + 0] = m[k];
                            a.ws_ml[((size_t)item * a.H + h) * 2 + 1] = l[k];
                        }
                    } else {
                        const float inv = l[k] > 0.f ? 1.f / l[k] : 0.f;
                        float o[EL];
#pragma unroll
                        for (int x = 0; x < EL; ++x) o[x] = acc[k][x] * inv;
                        reinterpret_cast<uint4 *>(a.out_w)[(size_t)it.row * R + c] = pack<T>(o);
                        if (c % LH == 0)
                            a.lse_w[(size_t)it.row * a.H + h] =
                                l[k] > 0.f ? (m[k] + log2f(l[k])) * kLn2 : -INFINITY;
                    }
                }
            }
        }
        it = itn;
        valid = validn;
        id0 = id1;
        mn = mnn;
    }
}

// Merge the chunk partials of each split row: one block per split row, warp
// w folds chunks w, w+8, ... with the online rule (m = max, l and acc
// rescaled by 2^(m_c - m)), then the 8 warp results are folded in warp order.
// The order is fixed, so results are reproducible.
template <typename T, int D, typename A>
__global__ void __launch_bounds__(256) gt_fwd_merge_kernel(A a) {
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16;
    __shared__ float m_sh[kWarpsPerBlock][32], l_sh[kWarpsPerBlock][32];
    __shared__ float acc_sh[kWarpsPerBlock][32 * EL];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t s = blockIdx.x;
    if (s >= a.rows.n_split) return;
    const int32_t row = a.rows.split_rows[s];
    const int32_t c0 = a.rows.chunk_ptr[s], c1 = a.rows.chunk_ptr[s + 1];
    const int R = a.H * D / EL, HD = a.H * D;
    for (int cb = 0; cb < R; cb += 32) {
        const int c = cb + lane;
        const int h = c / LH;
        float m = -INFINITY, l = 0.f, acc[EL];
#pragma unroll
        for (int x = 0; x < EL; ++x) acc[x] = 0.f;
        if (c < R) {
            for (int32_t ch = c0 + w; ch < c1; ch += kWarpsPerBlock) {
                const float mc = a.ws_ml[((size_t)ch * a.H + h) * 2];
                const float lc = a.ws_ml[((size_t)ch * a.H + h) * 2 + 1];
                const float mx = fmaxf(m, mc);
                const float a1 = exp2_diff(m, mx), a2 = exp2_diff(mc, mx);
                const float4 *src = reinterpret_cast<const float4 *>(a.ws_acc + (size_t)ch * HD + c * EL);
#pragma unroll
                for (int x = 0; x < EL; x += 4) {
                    const float4 v = src[x / 4];
                    acc[x] = acc[x] * a1 + v.x * a2;
                    acc[x + 1] = acc[x + 1] * a1 + v.y * a2;
                    acc[x + 2] = acc[x + 2] * a1 + v.z * a2;
                    acc[x + 3] = acc[x + 3] * a1 + v.w * a2;
                }
                l = l * a1 + lc * a2;
                m = mx;
            }
        }
        m_sh[w][lane] = m;
        l_sh[w][lane] = l;
#pragma unroll
        for (int x = 0; x < EL; ++x) acc_sh[w][lane * EL + x] = acc[x];
        __syncthreads();
        if (w == 0 && c < R) {
            float M = -INFINITY;
            for (int v = 0; v < kWarpsPerBlock; ++v) M = fmaxf(M, m_sh[v][lane]);
            float L = 0.f, o[EL];
#pragma unroll
            for (int x = 0; x < EL; ++x) o[x] = 0.f;
            for (int v = 0; v < kWarpsPerBlock; ++v) {
                const float wt = exp2_diff(m_sh[v][lane], M);
                L += l_sh[v][lane] * wt;
#pragma unroll
                for (int x = 0; x < EL; ++x) o[x] = fmaf(acc_sh[v][lane * EL + x], wt, o[x]);
            }
            const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
            for (int x = 0; x < EL; ++x) o[x] *= inv;
            reinterpret_cast<uint4 *>(a.out_w)[(size_t)row * R + c] = pack<T>(o);
            if (c % LH == 0)
                a.lse_w[(size_t)row * a.H + h] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
        __syncthreads();
    }
}

// Sum of chunk partials for one split row, block-cooperatively: warp w adds
// chunks w, w+8, ... of `NCOMP` HD-wide components (component q of chunk ch at
// part[(ch * stride_c + q) * HD]) and, if `parts_c`, the per-head scalars;
// the 8 warp sums are then added in warp order into sum[q][x] / csum for
// lane-chunk c of the current batch (valid in warp 0).
template <int EL, int NCOMP>
__device__ __forceinline__ void block_sum_chunks(const float *__restrict__ part, int stride_c, int HD,
                                                 const float *__restrict__ parts_c, int H, int LH,
                                                 int32_t c0, int32_t c1, int c, bool active,
                                                 float (*sh)[NCOMP][32 * EL], float (*shc)[32],
                                                 float (&sum)[NCOMP][EL], float &csum) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float x[NCOMP][EL], xc = 0.f;
#pragma unroll
    for (int q = 0; q < NCOMP; ++q)
#pragma unroll
        for (int e = 0; e < EL; ++e) x[q][e] = 0.f;
    if (active) {
        for (int32_t ch = c0 + w; ch < c1; ch += kWarpsPerBlock) {
#pragma unroll
            for (int q = 0; q < NCOMP; ++q) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    part + ((size_t)ch * stride_c + q) * HD + c * EL);
#pragma unroll
                for (int e = 0; e < EL; e += 4) {
                    const float4 v = src[e / 4];
                    x[q][e] += v.x; x[q][e + 1] += v.y; x[q][e + 2] += v.z; x[q][e + 3] += v.w;
                }
            }
            if (parts_c) xc += parts_c[(size_t)ch * H + c / LH];
        }
    }
#pragma unroll
    for (int q = 0; q < NCOMP; ++q)
#pragma unroll
        for (int e = 0; e < EL; ++e) sh[w][q][lane * EL + e] = x[q][e];
    shc[w][lane] = xc;
    __syncthreads();
    if (w == 0) {
#pragma unroll
        for (int q = 0; q < NCOMP; ++q)
#pragma unroll
            for (int e = 0; e < EL; ++e) sum[q][e] = 0.f;
        csum = 0.f;
        for (int v = 0; v < kWarpsPerBlock; ++v) {
#pragma unroll
            for (int q = 0; q < NCOMP; ++q)
#pragma unroll
                for (int e = 0; e < EL; ++e) sum[q][e] += sh[v][q][lane * EL + e];
            csum += shc[v][lane];
        }
    }
}

// ---------------------------------------------------------- backward: dQ

// Per destination row i and edge j: p = 2^(s2 - lse2_i), dP = dOut_i . v_j.
// With Delta_i = sum_j p dP (the exact row term; equal to dOut_i . out_i
// before out is rounded to the storage dtype), dS = p (dP - Delta_i) and
// dQ_i = sum_j dS k_j / sqrt(D) = (A - Delta_i B) / sqrt(D) where
// A = sum_j p dP k_j and B = sum_j p k_j; A, B and Delta_i are accumulated in
// the same pass over the edges.  Split-row chunks write A, B and their part
// of Delta; the merge kernel finishes them in chunk order.
template <typename T, int D, int NC, int G>
__global__ void __launch_bounds__(256, 2)
gt_bwd_dq_kernel(GtArgs a, float scale2, float scale) {
    using S = GtShape<T, D, NC, G>;
    constexpr int EL = S::EL, LH = S::LH, NG = S::NG, U = S::U;
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    const uint4 *__restrict__ Kc = static_cast<const uint4 *>(a.K);
    const uint4 *__restrict__ Vc = static_cast<const uint4 *>(a.V);
    const int64_t n_items = (int64_t)a.rows.n_chunks + a.N;
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerBlock;
    int64_t item = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);

    ItemMeta mn, mnn;
    meta_issue(item, a.rows, a.indptr, a.N, mn);
    ItemRange it;
    bool valid = meta_eval(item, mn, a.rows, a.split_threshold, it);
    int32_t id0 = first_ids(a.indices, it, valid);
    meta_issue(item + stride, a.rows, a.indptr, a.N, mn);
    for (; item < n_items; item += stride) {
        meta_issue(item + 2 * stride, a.rows, a.indptr, a.N, mnn);
        ItemRange itn;
        const bool validn = meta_eval(item + stride, mn, a.rows, a.split_threshold, itn);
        const int32_t id1 = first_ids(a.indices, itn, validn);
        if (valid) {
            float q[NC][EL], go[NC][EL], A[NC][EL], B[NC][EL], c[NC], lse2[NC];
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                const int ch = gl + G * k;
                if (ch < R) {
                    const size_t off = (size_t)it.row * R + ch;
                    unpack<T>(ldg16(static_cast<const uint4 *>(a.Q) + off), q[k]);
                    unpack<T>(ldg16(static_cast<const uint4 *>(a.dOut) + off), go[k]);
                    lse2[k] = __ldg(a.lse + (size_t)it.row * a.H + ch / LH) * kLog2e;
                } else {
#pragma unroll
                    for (int x = 0; x < EL; ++x) q[k][x] = go[k][x] = 0.f;
                    lse2[k] = 0.f;
                }
#pragma unroll
                for (int x = 0; x < EL; ++x) A[k][x] = B[k][x] = 0.f;
                c[k] = 0.f;
            }
            for (int32_t e0 = it.beg; e0 < it.end; e0 += 32) {
                const int cnt = min(32, it.end - e0);
                const int32_t myj = batch_ids(a.indices, e0, cnt, it, id0, a.N, a.d_err);
                for (int t0 = 0; t0 < cnt; t0 += NG * U) {
                    uint4 kr[U][NC], vr[U][NC];
                    bool ok[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int t = t0 + g + NG * u;
                        const int32_t j = __shfl_sync(SGA_FULL_MASK, myj, t & 31);
                        ok[u] = (t < cnt) && (j >= 0);
#pragma unroll
                        for (int k = 0; k < NC; ++k) {
                            const int ch = gl + G * k;
                            if (ok[u] && ch < R) {
                                kr[u][k] = ldg16_stream(Kc + (size_t)j * R + ch);
                                vr[u][k] = ldg16_stream(Vc + (size_t)j * R + ch);
                            } else {
                                kr[u][k] = make_uint4(0, 0, 0, 0);
                                vr[u][k] = make_uint4(0, 0, 0, 0);
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int k = 0; k < NC; ++k) {
                            float kf[EL], vf[EL];
                            unpack<T>(kr[u][k], kf);
                            unpack<T>(vr[u][k], vf);
                            float sdot = 0.f, dp = 0.f;
#pragma unroll
                            for (int x = 0; x < EL; ++x) {
                                sdot = fmaf(q[k][x], kf[x], sdot);
                                dp = fmaf(go[k][x], vf[x], dp);
                            }
                            group_sum2<LH>(sdot, dp);
                            const float p = ok[u] ? exp2f(sdot * scale2 - lse2[k]) : 0.f;
                            const float pdp = p * dp;
                            c[k] += pdp;
#pragma unroll
                            for (int x = 0; x < EL; ++x) {
                                A[k][x] = fmaf(pdp, kf[x], A[k][x]);
                                B[k][x] = fmaf(p, kf[x], B[k][x]);
                            }
                        }
                }
            }
#pragma unroll
            for (int off = G; off < 32; off <<= 1)
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    c[k] += __shfl_xor_sync(SGA_FULL_MASK, c[k], off);
#pragma unroll
                    for (int x = 0; x < EL; ++x) {
                        A[k][x] += __shfl_xor_sync(SGA_FULL_MASK, A[k][x], off);
                        B[k][x] += __shfl_xor_sync(SGA_FULL_MASK, B[k][x], off);
                    }
                }
            if (g == 0) {
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    const int ch = gl + G * k;
                    if (ch >= R) continue;
                    const int h = ch / LH;
                    if (it.partial) {
                        float4 *dA = reinterpret_cast<float4 *>(a.ws_row + (size_t)item * 2 * HD + ch * EL);
                        float4 *dB = reinterpret_cast<float4 *>(a.ws_row + (size_t)item * 2 * HD + HD + ch * EL);
#pragma unroll
                        for (int x = 0; x < EL; x += 4) {
                            dA[x / 4] = make_float4(A[k][x], A[k][x + 1], A[k][x + 2], A[k][x + 3]);
                            dB[x / 4] = make_float4(B[k][x], B[k][x + 1], B[k][x + 2], B[k][x + 3]);
                        }
                        if (ch % LH == 0) a.ws_rowc[(size_t)item * a.H + h] = c[k];
                    } else {
                        const float dl = c[k] + (a.delta_in ? a.delta_in[(size_t)it.row * a.H + h] : 0.f);
                        float o[EL];
#pragma unroll
                        for (int x = 0; x < EL; ++x) o[x] = (A[k][x] - dl * B[k][x]) * scale;
                        reinterpret_cast<uint4 *>(a.dQ)[(size_t)it.row * R + ch] = pack<T>(o);
                        if (ch % LH == 0) a.ws_delta[(size_t)it.row * a.H + h] = dl;
                    }
                }
            }
        }
        it = itn;
        valid = validn;
        id0 = id1;
        mn = mnn;
    }
}

// ------------------------------------------------------- backward: dK, dV

// Per source j over its destinations i (transposed CSR):
// p = 2^(s2 - lse2_i), dS = p (dOut_i . v_j - Delta_i),
// dV_j += p dOut_i, dK_j += dS q_i.
template <typename T, int D, int NC, int G>
__global__ void __launch_bounds__(256, 2)
gt_bwd_dkdv_kernel(GtArgs a, float scale2, float scale) {
    using S = GtShape<T, D, NC, G>;
    constexpr int EL = S::EL, LH = S::LH, NG = S::NG, U = S::U;
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    const uint4 *__restrict__ Qc = static_cast<const uint4 *>(a.Q);
    const uint4 *__restrict__ Gc = static_cast<const uint4 *>(a.dOut);
    const int64_t n_items = (int64_t)a.cols.n_chunks + a.N;
    const int64_t stride = (int64_t)gridDim.x * kWarpsPerBlock;
    int64_t item = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);

    ItemMeta mn, mnn;
    meta_issue(item, a.cols, a.t_indptr, a.N, mn);
    ItemRange it;
    bool valid = meta_eval(item, mn, a.cols, a.split_threshold, it);
    int32_t id0 = first_ids(a.t_dst, it, valid);
    meta_issue(item + stride, a.cols, a.t_indptr, a.N, mn);
    for (; item < n_items; item += stride) {
        meta_issue(item + 2 * stride, a.cols, a.t_indptr, a.N, mnn);
        ItemRange itn;
        const bool validn = meta_eval(item + stride, mn, a.cols, a.split_threshold, itn);
        const int32_t id1 = first_ids(a.t_dst, itn, validn);
        if (valid) {
            float kj[NC][EL], vj[NC][EL], dk[NC][EL], dv[NC][EL];
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                const int c = gl + G * k;
                if (c < R) {
                    const size_t off = (size_t)it.row * R + c;
                    unpack<T>(ldg16(static_cast<const uint4 *>(a.K) + off), kj[k]);
                    unpack<T>(ldg16(static_cast<const uint4 *>(a.V) + off), vj[k]);
                } else {
#pragma unroll
                    for (int x = 0; x < EL; ++x) kj[k][x] = vj[k][x] = 0.f;
                }
#pragma unroll
                for (int x = 0; x < EL; ++x) dk[k][x] = dv[k][x] = 0.f;
            }
            for (int32_t e0 = it.beg; e0 < it.end; e0 += 32) {
                const int cnt = min(32, it.end - e0);
                const int32_t myi = batch_ids(a.t_dst, e0, cnt, it, id0, a.N, a.d_err);
                for (int t0 = 0; t0 < cnt; t0 += NG * U) {
                    uint4 qr[U][NC], gr[U][NC];
                    float l2[U][NC], dl[U][NC];
                    bool ok[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int t = t0 + g + NG * u;
                        const int32_t i = __shfl_sync(SGA_FULL_MASK, myi, t & 31);
                        ok[u] = (t < cnt) && (i >= 0);
#pragma unroll
                        for (int k = 0; k < NC; ++k) {
                            const int c = gl + G * k;
                            if (ok[u] && c < R) {
                                qr[u][k] = ldg16_stream(Qc + (size_t)i * R + c);
                                gr[u][k] = ldg16_stream(Gc + (size_t)i * R + c);
                                l2[u][k] = __ldg(a.lse + (size_t)i * a.H + c / LH);
                                dl[u][k] = a.ws_delta[(size_t)i * a.H + c / LH];
                            } else {
                                qr[u][k] = make_uint4(0, 0, 0, 0);
                                gr[u][k] = make_uint4(0, 0, 0, 0);
                                l2[u][k] = 0.f;
                                dl[u][k] = 0.f;
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u)
#pragma unroll
                        for (int k = 0; k < NC; ++k) {
                            float qf[EL], gf[EL];
                            unpack<T>(qr[u][k], qf);
                            unpack<T>(gr[u][k], gf);
                            float sdot = 0.f, dp = 0.f;
#pragma unroll
                            for (int x = 0; x < EL; ++x) {
                                sdot = fmaf(qf[x], kj[k][x], sdot);
                                dp = fmaf(gf[x], vj[k][x], dp);
                            }
                            group_sum2<LH>(sdot, dp);
                            const float p = ok[u] ? exp2f(sdot * scale2 - l2[u][k] * kLog2e) : 0.f;
                            const float ds = p * (dp - dl[u][k]);
#pragma unroll
                            for (int x = 0; x < EL; ++x) {
                                dv[k][x] = fmaf(p, gf[x], dv[k][x]);
                                dk[k][x] = fmaf(ds, qf[x], dk[k][x]);
                            }
                        }
                }
            }
#pragma unroll
            for (int off = G; off < 32; off <<= 1)
#pragma unroll
                for (int k = 0; k < NC; ++k)
#pragma unroll
                    for (int x = 0; x < EL; ++x) {
                        dk[k][x] += __shfl_xor_sync(SGA_FULL_MASK, dk[k][x], off);
                        dv[k][x] += __shfl_xor_sync(SGA_FULL_MASK, dv[k][x], off);
                    }
            if (g == 0) {
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    const int c = gl + G * k;
                    if (c >= R) continue;
                    if (it.partial) {
                        float4 *dk_dst = reinterpret_cast<float4 *>(a.ws_col + (size_t)item * 2 * HD + c * EL);
                        float4 *dv_dst = reinterpret_cast<float4 *>(a.ws_col + (size_t)item * 2 * HD + HD + c * EL);
#pragma unroll
                        for (int x = 0; x < EL; x += 4) {
                            dk_dst[x / 4] = make_float4(dk[k][x], dk[k][x + 1], dk[k][x + 2], dk[k][x + 3]);
                            dv_dst[x / 4] = make_float4(dv[k][x], dv[k][x + 1], dv[k][x + 2], dv[k][x + 3]);
                        }
                    } else {
                        float o[EL];
#pragma unroll
                        for (int x = 0; x < EL; ++x) o[x] = dk[k][x] * scale;
                        reinterpret_cast<uint4 *>(a.dK)[(size_t)it.row * R + c] = pack<T>(o);
                        reinterpret_cast<uint4 *>(a.dV)[(size_t)it.row * R + c] = pack<T>(dv[k]);
                    }
                }
            }
        }
        it = itn;
        valid = validn;
        id0 = id1;
        mn = mnn;
    }
}

// Finish split rows, one block each.  which == 0: dQ rows (Delta = sum of
// the chunk parts, dQ = (sum A - Delta sum B) / sqrt(D), Delta stored for the
// dK/dV pass).  which == 1: dK, dV of split sources (plain sums).
template <typename T, int D>
__global__ void __launch_bounds__(256) gt_bwd_merge_kernel(GtArgs a, float scale, int which) {
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16;
    __shared__ float sh[kWarpsPerBlock][2][32 * EL];
    __shared__ float shc[kWarpsPerBlock][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t s = blockIdx.x;
    const Partition &P = which == 0 ? a.rows : a.cols;
    if (s >= P.n_split) return;
    const int32_t row = P.split_rows[s];
    const int32_t c0 = P.chunk_ptr[s], c1 = P.chunk_ptr[s + 1];
    const int R = a.H * D / EL, HD = a.H * D;
    for (int cb = 0; cb < R; cb += 32) {
        const int c = cb + lane;
        float sum[2][EL], delta;
        block_sum_chunks<EL, 2>(which == 0 ? a.ws_row : a.ws_col, 2, HD,
                                which == 0 ? a.ws_rowc : nullptr, a.H, LH, c0, c1, c, c < R, sh,
                                shc, sum, delta);
        if (w == 0 && c < R) {
            if (which == 0) {
                if (a.delta_in) delta += a.delta_in[(size_t)row * a.H + c / LH];
                float o[EL];
#pragma unroll
                for (int x = 0; x < EL; ++x) o[x] = (sum[0][x] - delta * sum[1][x]) * scale;
                reinterpret_cast<uint4 *>(a.dQ)[(size_t)row * R + c] = pack<T>(o);
                if (c % LH == 0) a.ws_delta[(size_t)row * a.H + c / LH] = delta;
            } else {
#pragma unroll
                for (int x = 0; x < EL; ++x) sum[0][x] *= scale;
                reinterpret_cast<uint4 *>(a.dK)[(size_t)row * R + c] = pack<T>(sum[0]);
                reinterpret_cast<uint4 *>(a.dV)[(size_t)row * R + c] = pack<T>(sum[1]);
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------ launch

inline unsigned blocks_for_warps(int64_t warps) {
    return (unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
}

// Grid of a persistent edge kernel: every block resident at once (occupancy
// times the SM count), or fewer when there are fewer items than warps.
template <auto Kernel> unsigned persistent_blocks(int64_t items) {
    static int per_sm = -1;   // one cache per kernel instantiation
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (per_sm < 0) {
        int nb = 1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, Kernel, 256, 0) != cudaSuccess) nb = 1;
        per_sm = nb > 0 ? nb : 1;
    }
    const int64_t full = (int64_t)per_sm * (sms > 0 ? sms : 1);
    const int64_t need = (items + kWarpsPerBlock - 1) / kWarpsPerBlock;
    return (unsigned)(need < full ? (need > 0 ? need : 1) : full);
}

// Calls F.template operator()<NC, G>() for the edge-group shape of a row of
// R sixteen-byte chunks: G = 32 lanes and NC = ceil(R/32) chunks per lane,
// or one chunk per lane in groups of G = next power of two >= R when R < 32.
// Shapes a head of LH lanes cannot use (LH > G) or that exceed MAXNC chunks
// per lane are never instantiated; R >= LH always holds at run time.
template <int LH, int MAXNC, typename F> cudaError_t dispatch_shape(int R, F &&f) {
    if (R > 64) {
        if constexpr (MAXNC >= 8) {
            if (R > 128) return f.template operator()<8, 32>();
        }
        return f.template operator()<4, 32>();
    }
    if (R > 32) return f.template operator()<2, 32>();
    if constexpr (LH <= 16) {
        if (R <= 16) {
            if constexpr (LH <= 8) {
                if (R <= 8) {
                    if constexpr (LH <= 4) {
                        if (R <= 4) return f.template operator()<1, 4>();
                    }
                    return f.template operator()<1, 8>();
                }
            }
            return f.template operator()<1, 16>();
        }
    }
    return f.template operator()<1, 32>();
}

template <typename T> constexpr int max_nc() { return sizeof(T) == 4 ? 8 : 4; }

template <typename T, int D> cudaError_t gt_fwd_d(const GtArgs &a, cudaStream_t s) {
    constexpr int LH = D * (int)sizeof(T) / 16;
    const int R = a.H * D / Elt<T>::EL;
    const float scale2 = kLog2e / sqrtf((float)D);
    const int64_t items = (int64_t)a.rows.n_chunks + a.N;
    cudaError_t e = dispatch_shape<LH, max_nc<T>()>(R, [&]<int NC, int G>() -> cudaError_t {
        if (items == 0) return cudaSuccess;
        note_launch(SGA_KERN_GT_FWD, s, false);
        gt_fwd_kernel<T, D, NC, G>
            <<<persistent_blocks<gt_fwd_kernel<T, D, NC, G>>(items), 256, 0, s>>>(a, scale2);
        note_launch(SGA_KERN_GT_FWD, s, true);
        return cudaGetLastError();
    });
    if (e != cudaSuccess || a.rows.n_split == 0) return e;
    note_launch(SGA_KERN_GT_FWD_MERGE, s, false);
    gt_fwd_merge_kernel<T, D, GtArgs><<<(unsigned)a.rows.n_split, 256, 0, s>>>(a);
    note_launch(SGA_KERN_GT_FWD_MERGE, s, true);
    return cudaGetLastError();
}

template <typename T, int D> cudaError_t gt_bwd_d(const GtArgs &a, cudaStream_t s) {
    constexpr int LH = D * (int)sizeof(T) / 16;
    const int R = a.H * D / Elt<T>::EL;
    const float scale = 1.0f / sqrtf((float)D);
    const float scale2 = kLog2e * scale;
    return dispatch_shape<LH, max_nc<T>()>(R, [&]<int NC, int G>() -> cudaError_t {
        const int64_t items_r = (int64_t)a.rows.n_chunks + a.N;
        const int64_t items_c = (int64_t)a.cols.n_chunks + a.N;
        if (items_r == 0) return cudaSuccess;
        note_launch(SGA_KERN_GT_BWD_DQ, s, false);
        gt_bwd_dq_kernel<T, D, NC, G>
            <<<persistent_blocks<gt_bwd_dq_kernel<T, D, NC, G>>(items_r), 256, 0, s>>>(a, scale2, scale);
        note_launch(SGA_KERN_GT_BWD_DQ, s, true);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (a.rows.n_split > 0) {   // Delta of split rows is needed by the dK/dV pass
            note_launch(SGA_KERN_GT_BWD_MERGE, s, false);
            gt_bwd_merge_kernel<T, D><<<(unsigned)a.rows.n_split, 256, 0, s>>>(a, scale, 0);
            note_launch(SGA_KERN_GT_BWD_MERGE, s, true);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        note_launch(SGA_KERN_GT_BWD_DKDV, s, false);
        gt_bwd_dkdv_kernel<T, D, NC, G>
            <<<persistent_blocks<gt_bwd_dkdv_kernel<T, D, NC, G>>(items_c), 256, 0, s>>>(a, scale2, scale);
        note_launch(SGA_KERN_GT_BWD_DKDV, s, true);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if (a.cols.n_split > 0) {
            note_launch(SGA_KERN_GT_BWD_MERGE, s, false);
            gt_bwd_merge_kernel<T, D><<<(unsigned)a.cols.n_split, 256, 0, s>>>(a, scale, 1);
            note_launch(SGA_KERN_GT_BWD_MERGE, s, true);
            e = cudaGetLastError();
        }
        return e;
    });
}

template <typename T> cudaError_t gt_fwd_t(const GtArgs &a, cudaStream_t s) {
    switch (a.D) {
        case 32: return gt_fwd_d<T, 32>(a, s);
        case 64: return gt_fwd_d<T, 64>(a, s);
        case 128: return gt_fwd_d<T, 128>(a, s);
    }
    return cudaErrorInvalidValue;
}

template <typename T> cudaError_t gt_bwd_t(const GtArgs &a, cudaStream_t s) {
    switch (a.D) {
        case 32: return gt_bwd_d<T, 32>(a, s);
        case 64: return gt_bwd_d<T, 64>(a, s);
        case 128: return gt_bwd_d<T, 128>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sga
