// GAT edge attention (the original graph attention score) over the
// destination CSR: e_ij = LeakyReLU(el_i + er_j) per head, softmax over the
// row, out_i = sum_j p_ij Fv_j, where Fv are the projected node features and
// el_i = a_l . Fv_i, er_j = a_r . Fv_j the two halves of the attention score
// (computed by the caller as two dense per-node dots).  GAT and the Graph
// Transformer are the attention GNNs DF-GNN's abstract names; the IO-aware
// layers blog post ("Attention-based layers" paragraph) fuses such layers so
// that edge scores never reach device memory.
//
// The kernels run on the edge stream of gt.cuh (stream.cuh):
//  - forward: gathered Fv rows and er scalars, the row's own el; online
//    softmax with the lazily moved maximum; split rows write partials that
//    gt_fwd_merge_kernel finishes;
//  - backward destination pass: per row and head, C = sum p dp, Z = sum p,
//    A = sum p dp l', B = sum p l' (dp = dOut_i . Fv_j, l' = LeakyReLU'), so
//    del_i = (A - Delta B) / Z with Delta = C / Z (weights normalised by Z,
//    gt.cuh RowNorm); Delta and lse + ln Z are stored for the source pass;
//  - backward source pass (transposed CSR): per source j over its
//    destinations, dFv_j = sum p dOut_i (the value path) and
//    der_j = sum p (dp - Delta_i) l'.
// Layer gradients (dFL = dFv + a_l del + a_r der, then the projection) are
// the caller's dense chain rule.
#pragma once

#include "gt.cuh"

namespace sga {

// gathered Fv, er; own el
template <int NC, int G> using GatFwdStream = RingCfg<NC, G, 1, 1, 0, 1, 2, 4>;
// gathered Fv, er; own dOut row, own el and lse
template <int NC, int G> using GatDstStream = RingCfg<NC, G, 1, 1, 1, 2, 2, 4>;
// gathered dOut rows and lse + ln Z, Delta, el of the destinations; own Fv row, own er
template <int NC, int G> using GatSrcStream = RingCfg<NC, G, 1, 3, 1, 1, 1, 4>;

__device__ __forceinline__ float lrelu_f(float z, float slope) { return z > 0.f ? z : slope * z; }

template <typename T, int D, int NC, int G>
__global__ void __launch_bounds__(256, 2) gat_fwd_kernel(GatArgs a) {
    using C = GatFwdStream<NC, G>;
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16, U = C::U;
    extern __shared__ __align__(16) unsigned char dsmem[];
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    StreamArrays arr{};
    arr.rows[0] = static_cast<const uint4 *>(a.Fv);
    arr.sc[0] = a.er;
    arr.osc[0] = a.el;
    EdgeStream<C> st;
    st.init(dsmem + (threadIdx.x >> 5) * C::BYTES, arr, a.rows, a.indptr, a.indices, a.N, a.H, R, LH,
            a.split_threshold, a.d_err);
    StreamItem it;
    while (st.next_item(it)) {
        float acc[NC][EL], m[NC], l[NC], el[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
#pragma unroll
            for (int x = 0; x < EL; ++x) acc[k][x] = 0.f;
            m[k] = -INFINITY;
            l[k] = el[k] = 0.f;
        }
        for (int step = 0; step < it.nsteps; ++step) {
            st.wait_step();
            if (step == 0)
#pragma unroll
                for (int k = 0; k < NC; ++k) el[k] = st.own_scalar(0, (gl + G * k) / LH);
            float sc[U][NC];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ok = st.valid(u);
#pragma unroll
                for (int k = 0; k < NC; ++k)
                    sc[u][k] = ok ? lrelu_f(el[k] + st.scalar(u, 0, (gl + G * k) / LH), a.slope) * kLog2e
                                  : -INFINITY;
            }
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                float mx = sc[0][k];
#pragma unroll
                for (int u = 1; u < U; ++u) mx = fmaxf(mx, sc[u][k]);
                if (mx > m[k] + kLazyLog2) {
                    const float alpha = exp2_diff(m[k], mx);
                    l[k] *= alpha;
#pragma unroll
                    for (int x = 0; x < EL; ++x) acc[k][x] *= alpha;
                    m[k] = mx;
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float p = exp2_diff(sc[u][k], m[k]);
                    l[k] += p;
                    float vf[EL];
                    unpack<T>(st.row(u, 0, k), vf);
                    axpy2<EL>(acc[k], p, vf);
                }
            }
            st.release_step();
        }
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
                    float4 *dst = reinterpret_cast<float4 *>(a.ws_acc + (size_t)it.item * HD + c * EL);
#pragma unroll
                    for (int x = 0; x < EL; x += 4)
                        dst[x / 4] = make_float4(acc[k][x], acc[k][x + 1], acc[k][x + 2], acc[k][x + 3]);
                    if (c % LH == 0) {
                        a.ws_ml[((size_t)it.item * a.H + h) * 2 + 0] = m[k];
                        a.ws_ml[((size_t)it.item * a.H + h) * 2 + 1] = l[k];
                    }
                } else {
                    const float inv = l[k] > 0.f ? 1.f / l[k] : 0.f;
                    float o[EL];
#pragma unroll
                    for (int x = 0; x < EL; ++x) o[x] = acc[k][x] * inv;
                    reinterpret_cast<uint4 *>(a.out_w)[(size_t)it.row * R + c] = pack<T>(o);
                    if (c % LH == 0)
                        a.lse_w[(size_t)it.row * a.H + h] = l[k] > 0.f ? (m[k] + log2f(l[k])) * kLn2 : -INFINITY;
                }
            }
        }
        st.finish_item();
    }
    st.drain();
}

// ---- backward: destination pass (per-head scalars only)

template <typename T, int D, int NC, int G>
__global__ void __launch_bounds__(256, 2) gat_bwd_dst_kernel(GatArgs a) {
    using C = GatDstStream<NC, G>;
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16, U = C::U;
    extern __shared__ __align__(16) unsigned char dsmem[];
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL;
    StreamArrays arr{};
    arr.rows[0] = static_cast<const uint4 *>(a.Fv);
    arr.sc[0] = a.er;
    arr.own[0] = static_cast<const uint4 *>(a.dOut);
    arr.osc[0] = a.el;
    arr.osc[1] = a.lse;
    EdgeStream<C> st;
    st.init(dsmem + (threadIdx.x >> 5) * C::BYTES, arr, a.rows, a.indptr, a.indices, a.N, a.H, R, LH,
            a.split_threshold, a.d_err);
    StreamItem it;
    while (st.next_item(it)) {
        float go[NC][EL], el[NC], lse2[NC], c[NC], z[NC], sA[NC], sB[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
#pragma unroll
            for (int x = 0; x < EL; ++x) go[k][x] = 0.f;
            el[k] = lse2[k] = c[k] = z[k] = sA[k] = sB[k] = 0.f;
        }
        for (int step = 0; step < it.nsteps; ++step) {
            st.wait_step();
            if (step == 0)
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    unpack<T>(st.own_row(0, k), go[k]);
                    const int h = (gl + G * k) / LH;
                    el[k] = st.own_scalar(0, h);
                    lse2[k] = st.own_scalar(1, h) * kLog2e;
                }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ok = st.valid(u);
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    float vf[EL];
                    unpack<T>(st.row(u, 0, k), vf);
                    const float dp = group_sum<LH>(dot2<EL>(go[k], vf));
                    const float zz = el[k] + st.scalar(u, 0, (gl + G * k) / LH);
                    const float lp = zz > 0.f ? 1.f : a.slope;
                    const float p = ok ? fast_exp2(lrelu_f(zz, a.slope) * kLog2e - lse2[k]) : 0.f;
                    const float pdp = p * dp;
                    c[k] += pdp;
                    z[k] += p;
                    sA[k] = fmaf(pdp, lp, sA[k]);
                    sB[k] = fmaf(p, lp, sB[k]);
                }
            }
            st.release_step();
        }
#pragma unroll
        for (int off = G; off < 32; off <<= 1)
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                c[k] += __shfl_xor_sync(SGA_FULL_MASK, c[k], off);
                z[k] += __shfl_xor_sync(SGA_FULL_MASK, z[k], off);
                sA[k] += __shfl_xor_sync(SGA_FULL_MASK, sA[k], off);
                sB[k] += __shfl_xor_sync(SGA_FULL_MASK, sB[k], off);
            }
        if (g == 0) {
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                const int ch = gl + G * k;
                if (ch >= R || ch % LH != 0) continue;
                const int h = ch / LH;
                if (it.partial) {
                    float4 *dst = reinterpret_cast<float4 *>(a.ws_rowc + ((size_t)it.item * a.H + h) * 4);
                    *dst = make_float4(c[k], z[k], sA[k], sB[k]);
                } else {
                    const size_t rh = (size_t)it.row * a.H + h;
                    const RowNorm nrm(c[k], z[k]);
                    a.del[rh] = (sA[k] - nrm.delta * sB[k]) * nrm.inv_z;
                    a.ws_delta[rh] = nrm.delta;
                    a.ws_lse[rh] = a.lse[rh] + nrm.lse_shift;
                }
            }
        }
        st.finish_item();
    }
    st.drain();
}

// Split destination rows: sum the chunks' (C, Z, A, B) in chunk order.
__global__ void __launch_bounds__(256) gat_bwd_dst_merge_kernel(GatArgs a) {
    const int64_t s = blockIdx.x;
    if (s >= a.rows.n_split) return;
    const int32_t row = a.rows.split_rows[s];
    const int32_t c0 = a.rows.chunk_ptr[s], c1 = a.rows.chunk_ptr[s + 1];
    for (int h = threadIdx.x; h < a.H; h += blockDim.x) {
        float c = 0.f, z = 0.f, sA = 0.f, sB = 0.f;
        for (int32_t ch = c0; ch < c1; ++ch) {
            const float4 v = *reinterpret_cast<const float4 *>(a.ws_rowc + ((size_t)ch * a.H + h) * 4);
            c += v.x;
            z += v.y;
            sA += v.z;
            sB += v.w;
        }
        const size_t rh = (size_t)row * a.H + h;
        const RowNorm nrm(c, z);
        a.del[rh] = (sA - nrm.delta * sB) * nrm.inv_z;
        a.ws_delta[rh] = nrm.delta;
        a.ws_lse[rh] = a.lse[rh] + nrm.lse_shift;
    }
}

// ---- backward: source pass

template <typename T, int D, int NC, int G>
__global__ void __launch_bounds__(256, 2) gat_bwd_src_kernel(GatArgs a) {
    using C = GatSrcStream<NC, G>;
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16, U = C::U;
    extern __shared__ __align__(16) unsigned char dsmem[];
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    StreamArrays arr{};
    arr.rows[0] = static_cast<const uint4 *>(a.dOut);
    arr.sc[0] = a.ws_lse;
    arr.sc[1] = a.ws_delta;
    arr.sc[2] = a.el;
    arr.own[0] = static_cast<const uint4 *>(a.Fv);
    arr.osc[0] = a.er;
    EdgeStream<C> st;
    st.init(dsmem + (threadIdx.x >> 5) * C::BYTES, arr, a.cols, a.t_indptr, a.t_dst, a.N, a.H, R, LH,
            a.split_threshold, a.d_err);
    StreamItem it;
    while (st.next_item(it)) {
        float fv[NC][EL], dfv[NC][EL], er[NC], der[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
#pragma unroll
            for (int x = 0; x < EL; ++x) fv[k][x] = dfv[k][x] = 0.f;
            er[k] = der[k] = 0.f;
        }
        for (int step = 0; step < it.nsteps; ++step) {
            st.wait_step();
            if (step == 0)
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    unpack<T>(st.own_row(0, k), fv[k]);
                    er[k] = st.own_scalar(0, (gl + G * k) / LH);
                }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ok = st.valid(u);
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    const int h = (gl + G * k) / LH;
                    float gf[EL];
                    unpack<T>(st.row(u, 0, k), gf);
                    const float dp = group_sum<LH>(dot2<EL>(gf, fv[k]));
                    const float zz = st.scalar(u, 2, h) + er[k];
                    const float lp = zz > 0.f ? 1.f : a.slope;
                    const float p = ok ? fast_exp2((lrelu_f(zz, a.slope) - st.scalar(u, 0, h)) * kLog2e) : 0.f;
                    der[k] = fmaf(p * (dp - st.scalar(u, 1, h)), lp, der[k]);
                    axpy2<EL>(dfv[k], p, gf);
                }
            }
            st.release_step();
        }
#pragma unroll
        for (int off = G; off < 32; off <<= 1)
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                der[k] += __shfl_xor_sync(SGA_FULL_MASK, der[k], off);
#pragma unroll
                for (int x = 0; x < EL; ++x) dfv[k][x] += __shfl_xor_sync(SGA_FULL_MASK, dfv[k][x], off);
            }
        if (g == 0) {
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                const int c = gl + G * k;
                if (c >= R) continue;
                const int h = c / LH;
                if (it.partial) {
                    float4 *dst = reinterpret_cast<float4 *>(a.ws_col + (size_t)it.item * HD + c * EL);
#pragma unroll
                    for (int x = 0; x < EL; x += 4)
                        dst[x / 4] = make_float4(dfv[k][x], dfv[k][x + 1], dfv[k][x + 2], dfv[k][x + 3]);
                    if (c % LH == 0) a.ws_colc[(size_t)it.item * a.H + h] = der[k];
                } else {
                    reinterpret_cast<uint4 *>(a.dFv)[(size_t)it.row * R + c] = pack<T>(dfv[k]);
                    if (c % LH == 0) a.der[(size_t)it.row * a.H + h] = der[k];
                }
            }
        }
        st.finish_item();
    }
    st.drain();
}

// Split sources: dFv and der are the sums of the chunk partials (chunk order).
template <typename T, int D>
__global__ void __launch_bounds__(256) gat_bwd_src_merge_kernel(GatArgs a) {
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16;
    __shared__ float sh[kWarpsPerBlock][1][32 * EL];
    __shared__ float shc[kWarpsPerBlock][1][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t s = blockIdx.x;
    if (s >= a.cols.n_split) return;
    const int32_t row = a.cols.split_rows[s];
    const int32_t c0 = a.cols.chunk_ptr[s], c1 = a.cols.chunk_ptr[s + 1];
    const int R = a.H * D / EL, HD = a.H * D;
    for (int cb = 0; cb < R; cb += 32) {
        const int c = cb + lane;
        float sum[1][EL], csum[1];
        block_sum_chunks<EL, 1, 1>(a.ws_col, 1, HD, a.ws_colc, a.H, LH, c0, c1, c, c < R, sh, shc, sum, csum);
        if (w == 0 && c < R) {
            reinterpret_cast<uint4 *>(a.dFv)[(size_t)row * R + c] = pack<T>(sum[0]);
            if (c % LH == 0) a.der[(size_t)row * a.H + c / LH] = csum[0];
        }
        __syncthreads();
    }
}

template <typename T, int D> cudaError_t gat_fwd_d(const GatArgs &a, cudaStream_t s) {
    constexpr int LH = D * (int)sizeof(T) / 16;
    const int R = a.H * D / Elt<T>::EL;
    const int64_t items = (int64_t)a.rows.n_chunks + a.N;
    cudaError_t e = dispatch_shape<LH, max_nc<T>()>(R, [&]<int NC, int G>() -> cudaError_t {
        if (items == 0) return cudaSuccess;
        note_launch(SGA_KERN_GAT_FWD, s, false);
        const cudaError_t e = launch_streamed<GatFwdStream<NC, G>, gat_fwd_kernel<T, D, NC, G>>(items, s, a);
        note_launch(SGA_KERN_GAT_FWD, s, true);
        return e;
    });
    if (e != cudaSuccess || a.rows.n_split == 0) return e;
    note_launch(SGA_KERN_GAT_FWD, s, false);
    gt_fwd_merge_kernel<T, D, GatArgs><<<(unsigned)a.rows.n_split, 256, 0, s>>>(a);
    note_launch(SGA_KERN_GAT_FWD, s, true);
    return cudaGetLastError();
}

template <typename T, int D> cudaError_t gat_bwd_d(const GatArgs &a, cudaStream_t s) {
    constexpr int LH = D * (int)sizeof(T) / 16;
    const int R = a.H * D / Elt<T>::EL;
    return dispatch_shape<LH, max_nc<T>()>(R, [&]<int NC, int G>() -> cudaError_t {
        const int64_t items_r = (int64_t)a.rows.n_chunks + a.N;
        const int64_t items_c = (int64_t)a.cols.n_chunks + a.N;
        if (items_r == 0) return cudaSuccess;
        note_launch(SGA_KERN_GAT_BWD_DST, s, false);
        cudaError_t e = launch_streamed<GatDstStream<NC, G>, gat_bwd_dst_kernel<T, D, NC, G>>(items_r, s, a);
        note_launch(SGA_KERN_GAT_BWD_DST, s, true);
        if (e != cudaSuccess) return e;
        if (a.rows.n_split > 0) {
            gat_bwd_dst_merge_kernel<<<(unsigned)a.rows.n_split, 32, 0, s>>>(a);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        note_launch(SGA_KERN_GAT_BWD_SRC, s, false);
        e = launch_streamed<GatSrcStream<NC, G>, gat_bwd_src_kernel<T, D, NC, G>>(items_c, s, a);
        note_launch(SGA_KERN_GAT_BWD_SRC, s, true);
        if (e != cudaSuccess) return e;
        if (a.cols.n_split > 0) {
            gat_bwd_src_merge_kernel<T, D><<<(unsigned)a.cols.n_split, 256, 0, s>>>(a);
            e = cudaGetLastError();
        }
        return e;
    });
}

template <typename T> cudaError_t gat_fwd_t(const GatArgs &a, cudaStream_t s) {
    switch (a.D) {
        case 32: return gat_fwd_d<T, 32>(a, s);
        case 64: return gat_fwd_d<T, 64>(a, s);
        case 128: return gat_fwd_d<T, 128>(a, s);
    }
    return cudaErrorInvalidValue;
}

template <typename T> cudaError_t gat_bwd_t(const GatArgs &a, cudaStream_t s) {
    switch (a.D) {
        case 32: return gat_bwd_d<T, 32>(a, s);
        case 64: return gat_bwd_d<T, 64>(a, s);
        case 128: return gat_bwd_d<T, 128>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sga
