// GATv2 edge attention: projections, fused edge forward, and the backward
// pass (destination pass for dFL and da, transposed source pass for dFR,
// then the projection gradients).
//
// Method: the GATv2 score e_ij = sum_d a[h,d] LeakyReLU(FL[i,h,d] + FR[j,h,d])
// with FL = X W_l and FR = X W_r ("How Attentive are Graph Attention
// Networks?", cited by both pages) inside the fused online-softmax edge
// kernel of "On Efficient Scaling of GNNs via IO-Aware Layers
// Implementations" (Yandex Research blog post, "Attention-based layers"
// paragraph).  FR_j is both the score operand and the aggregated value, so
// the forward gathers one neighbour row per edge.  The backward recomputes
// the weights from the saved log-sum-exp.
//
// The edge kernels share the Graph Transformer's lane layout (gt.cuh): one
// warp per row or split-row chunk, 16-byte chunks per lane, heads reduced by
// xor shuffles.
#pragma once

#include "gemm.cuh"
#include "gt.cuh"
#include "tc_dx.cuh"
#include "tc_proj.cuh"

namespace sga {

// The projection gradients dFL, dFR are kept per node row in the workspace:
// fp32 [N][HD] for fp32 layers; for bf16 layers a bf16 pair per value,
// row = [hi(0..HD) | lo(0..HD)] with hi = bf16(x), lo = bf16(x - hi) (about 16
// significant bits, the split the tensor-core GEMMs consume), the same 4
// bytes per value.
template <typename T, int EL>
__device__ __forceinline__ void store_dF(float *ws, int64_t row, int HD, int c, const float *v) {
    if constexpr (sizeof(T) == 4) {
        float4 *dst = reinterpret_cast<float4 *>(ws + (size_t)row * HD + c * EL);
#pragma unroll
        for (int x = 0; x < EL; x += 4) dst[x / 4] = make_float4(v[x], v[x + 1], v[x + 2], v[x + 3]);
    } else {
        float h[EL], l[EL];
#pragma unroll
        for (int x = 0; x < EL; ++x) {
            h[x] = __bfloat162float(__float2bfloat16_rn(v[x]));
            l[x] = v[x] - h[x];
        }
        __nv_bfloat16 *base = reinterpret_cast<__nv_bfloat16 *>(ws) + (size_t)row * 2 * HD + c * EL;
        *reinterpret_cast<uint4 *>(base) = pack<__nv_bfloat16>(h);
        *reinterpret_cast<uint4 *>(base + HD) = pack<__nv_bfloat16>(l);
    }
}

// --------------------------------------------------------------- edge fwd

// gathered FR; own FL
// (items taken dynamically in the plan's batches, at most eight: workload of
// 1.7M edges, batches of four, 0.779 -> 0.773 ms a step; a fixed batch of
// eight gave the warps that took the first chunks more than their share of
// the edges, 0.157 -> 0.225 ms for this pass; the source pass keeps the
// fixed share, which measured faster there)
template <typename T, int D, int NC, int G> using Gatv2FwdStream = RingCfg<NC, G, 1, 0, 1, 0, 1, 2, 0, true, false, 8>;
// gathered FR; own FL, dOut, lse
// (a fixed share of items: each block's da partial must sum the same rows in
// every launch for da to be reproducible)
template <typename T, int D, int NC, int G> using Gatv2DstStream = RingCfg<NC, G, 1, 0, 2, 1>;
// gathered FL, dOut, lse, Delta (transposed CSR); own FR
template <typename T, int D, int NC, int G> using Gatv2SrcStream = RingCfg<NC, G, 2, 2, 1, 0>;

// LeakyReLU of z = fl + fr over one chunk and its slope factor d (1 or
// slope): lz = z d.
template <int EL>
__device__ __forceinline__ void lrelu_chunk(const float *fl, const float *fr, float slope, float *lz, float *d) {
#pragma unroll
    for (int x = 0; x < EL; x += 2) {
        const float2 z = fadd2(make_float2(fl[x], fl[x + 1]), make_float2(fr[x], fr[x + 1]));
        d[x] = z.x > 0.f ? 1.f : slope;
        d[x + 1] = z.y > 0.f ? 1.f : slope;
        const float2 l = fmul2(z, make_float2(d[x], d[x + 1]));
        lz[x] = l.x;
        lz[x + 1] = l.y;
    }
}
// LeakyReLU alone, as h z + k |z| with h = (1 + slope) / 2, k = (1 - slope) / 2
// (fma-pipe arithmetic only; within an ulp of the select form).
template <int EL>
__device__ __forceinline__ void lrelu_fma(const float *fl, const float *fr, float h, float k, float *lz) {
#pragma unroll
    for (int x = 0; x < EL; ++x) {
        const float z = fl[x] + fr[x];
        lz[x] = fmaf(k, fabsf(z), h * z);
    }
}

template <typename T, int D, int NC, int G>
__global__ void __launch_bounds__(256, 2)
gatv2_fwd_kernel(Gatv2Args a) {
    using S = GtShape<T, D, NC, G>;
    using C = Gatv2FwdStream<T, D, NC, G>;
    constexpr int EL = S::EL, LH = S::LH, U = C::U;
    extern __shared__ __align__(16) unsigned char dsmem[];
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    const float lr_h = 0.5f * (1.f + a.slope), lr_k = 0.5f * (1.f - a.slope);
    float att[NC][EL];   // a, in log2 units: scores come out in log2 units
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        const int c = gl + G * k;
        if (c < R) unpack<T>(ldg16(static_cast<const uint4 *>(a.a) + c), att[k]);
        else
#pragma unroll
            for (int x = 0; x < EL; ++x) att[k][x] = 0.f;
#pragma unroll
        for (int x = 0; x < EL; ++x) att[k][x] *= kLog2e;
    }
    StreamArrays arr{};
    arr.rows[0] = static_cast<const uint4 *>(a.FR);
    arr.own[0] = static_cast<const uint4 *>(a.FL);
    EdgeStream<C> st;
    st.init(dsmem + (threadIdx.x >> 5) * C::BYTES, arr, a.rows, a.indptr, a.indices, a.N, a.H, R, LH,
            a.split_threshold, a.d_err);
    StreamItem it;
    while (st.next_item(it)) {
        float fl[NC][EL], acc[NC][EL], m[NC], l[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
#pragma unroll
            for (int x = 0; x < EL; ++x) fl[k][x] = acc[k][x] = 0.f;
            m[k] = -INFINITY;
            l[k] = 0.f;
        }
        for (int step = 0; step < it.nsteps; ++step) {
            st.wait_step();
            if (step == 0)
#pragma unroll
                for (int k = 0; k < NC; ++k) unpack<T>(st.own_row(0, k), fl[k]);
            float sc[U][NC];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ok = st.valid(u);
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    float f[EL], lz[EL];
                    unpack<T>(st.row(u, 0, k), f);
                    lrelu_fma<EL>(fl[k], f, lr_h, lr_k, lz);
                    const float e = group_sum<LH>(dot2<EL>(att[k], lz));
                    sc[u][k] = ok ? e : -INFINITY;
                }
            }
            // lazily rescaled online softmax (see the Graph Transformer forward)
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
                    float f[EL];
                    unpack<T>(st.row(u, 0, k), f);
                    axpy2<EL>(acc[k], p, f);
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
                        a.lse_w[(size_t)it.row * a.H + h] =
                            l[k] > 0.f ? (m[k] + log2f(l[k])) * kLn2 : -INFINITY;
                }
            }
        }
        // the last chunk of a split row merges the row
        if (it.partial && last_chunk(a.rows, it.item)) fwd_merge_row<T, D>(a, __ldg(a.rows.chunk_split + it.item));
        st.finish_item();
    }
    st.drain();
}

// Finish split row s in one warp (chunk order).  which == 0 (destination
// rows): C and Z are the sums of the chunk parts, normalised as in the
// destination pass (Delta = C / Z): dFL = (sum fA - Delta sum fB) / Z, and
// the row's da contribution (sum gA - Delta sum gB) / Z goes to its own slot;
// Delta and lse + ln Z are stored for the source pass.  which == 1
// (sources): dFR is the plain sum of the chunk partials.
template <typename T, int D>
__device__ __noinline__ void gatv2_bwd_merge_row(const Gatv2Args &a, int which, int32_t s) {
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16;
    const Partition &P = which == 0 ? a.rows : a.cols;
    const int32_t row = __ldg(P.split_rows + s);
    const int32_t c0 = __ldg(P.chunk_ptr + s), c1 = __ldg(P.chunk_ptr + s + 1);
    const int R = a.H * D / EL, HD = a.H * D;
    for (int c = threadIdx.x & 31; c < R; c += 32) {
        const int h = c / LH;
        if (which == 1) {
            float sum[1][EL], unused[1];
            warp_sum_chunks<EL, 1, 1>(a.ws_col, 1, HD, nullptr, a.H, h, c0, c1, c, sum, unused);
            store_dF<T, EL>(a.ws_dfr, row, HD, c, sum[0]);
        } else {
            float sum[4][EL], cz[2];
            warp_sum_chunks<EL, 4, 2>(a.ws_row, 4, HD, a.ws_rowc, a.H, h, c0, c1, c, sum, cz);
            const RowNorm nrm(cz[0], cz[1]);
            float v[EL];
#pragma unroll
            for (int x = 0; x < EL; ++x) {
                v[x] = (sum[0][x] - nrm.delta * sum[1][x]) * nrm.inv_z;
                a.ws_da_split[(size_t)s * HD + c * EL + x] = (sum[2][x] - nrm.delta * sum[3][x]) * nrm.inv_z;
            }
            store_dF<T, EL>(a.ws_dfl, row, HD, c, v);
            if (c % LH == 0) {
                const size_t rh = (size_t)row * a.H + h;
                a.ws_delta[rh] = nrm.delta;
                a.ws_lse[rh] = a.lse[rh] + nrm.lse_shift;
            }
        }
    }
}

// ---------------------------------------------------- backward: dst pass

// Per destination row i, for each edge (j):
//   z = fl_i + fr_j, e = a . LReLU(z), p = exp(e - lse_i), dp = dOut_i . fr_j,
//   de = p (dp - Delta_i), dFL_i += de a * LReLU'(z), da += de LReLU(z).
// C_i = sum_j p dp and Z_i = sum_j p are accumulated in the same pass, so
// each de-weighted sum is kept as (sum p dp x) - Delta_i (sum p x), with the
// weights normalised by Z at the end of the row (RowNorm, gt.cuh: Delta =
// C / Z, sums / Z, lse + ln Z stored for the source pass).  Warps stride over
// work items; each block leaves one fp32 partial of da.  Split-row chunks
// write their four partial sums and their parts of C and Z for the merge
// kernel.
template <typename T, int D, int NC, int G>
__global__ void __launch_bounds__(256, 2)
gatv2_bwd_dst_kernel(Gatv2Args a) {
    using S = GtShape<T, D, NC, G>;
    using C = Gatv2DstStream<T, D, NC, G>;
    constexpr int EL = S::EL, LH = S::LH, U = C::U;
    __shared__ float da_sh[1024];
    extern __shared__ __align__(16) unsigned char dsmem[];
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    const float slope = a.slope;

    for (int x = threadIdx.x; x < HD; x += blockDim.x) da_sh[x] = 0.f;

    float att[NC][EL], dacc[NC][EL];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        const int c = gl + G * k;
        if (c < R) unpack<T>(ldg16(static_cast<const uint4 *>(a.a) + c), att[k]);
        else
#pragma unroll
            for (int x = 0; x < EL; ++x) att[k][x] = 0.f;
#pragma unroll
        for (int x = 0; x < EL; ++x) dacc[k][x] = 0.f;
    }
    StreamArrays arr{};
    arr.rows[0] = static_cast<const uint4 *>(a.FR);
    arr.own[0] = static_cast<const uint4 *>(a.FL);
    arr.own[1] = static_cast<const uint4 *>(a.dOut);
    arr.osc[0] = a.lse;
    EdgeStream<C> st;
    st.init(dsmem + (threadIdx.x >> 5) * C::BYTES, arr, a.rows, a.indptr, a.indices, a.N, a.H, R, LH,
            a.split_threshold, a.d_err);
    StreamItem it;
    while (st.next_item(it)) {
        // fA/fB: dFL sums (of LReLU'(z), times a after the row), gA/gB: da sums
        // (A weighted by p dp, B by p), c: Delta part
        float fl[NC][EL], go[NC][EL], fA[NC][EL], fB[NC][EL], gA[NC][EL], gB[NC][EL];
        float c[NC], z[NC], lse2[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
#pragma unroll
            for (int x = 0; x < EL; ++x) fl[k][x] = go[k][x] = fA[k][x] = fB[k][x] = gA[k][x] = gB[k][x] = 0.f;
            c[k] = z[k] = 0.f;
            lse2[k] = 0.f;
        }
        for (int step = 0; step < it.nsteps; ++step) {
            st.wait_step();
            if (step == 0)
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    unpack<T>(st.own_row(0, k), fl[k]);
                    unpack<T>(st.own_row(1, k), go[k]);
                    lse2[k] = st.own_scalar(0, (gl + G * k) / LH) * kLog2e;
                }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ok = st.valid(u);
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    float f[EL], lz[EL], dz[EL];
                    unpack<T>(st.row(u, 0, k), f);
                    lrelu_chunk<EL>(fl[k], f, slope, lz, dz);
                    float e = dot2<EL>(att[k], lz), dp = dot2<EL>(go[k], f);
                    group_sum2<LH>(e, dp);
                    const float p = ok ? fast_exp2(e * kLog2e - lse2[k]) : 0.f;
                    const float pdp = p * dp;
                    c[k] += pdp;
                    z[k] += p;
                    axpy2<EL>(fA[k], pdp, dz);
                    axpy2<EL>(fB[k], p, dz);
                    axpy2<EL>(gA[k], pdp, lz);
                    axpy2<EL>(gB[k], p, lz);
                }
            }
            st.release_step();
        }
        // a is constant over the row: the dFL sums take it once
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int x = 0; x < EL; x += 2) {
                const float2 ax = make_float2(att[k][x], att[k][x + 1]);
                const float2 ra = fmul2(ax, make_float2(fA[k][x], fA[k][x + 1]));
                const float2 rb = fmul2(ax, make_float2(fB[k][x], fB[k][x + 1]));
                fA[k][x] = ra.x;
                fA[k][x + 1] = ra.y;
                fB[k][x] = rb.x;
                fB[k][x + 1] = rb.y;
            }
        // Delta and the dFL sums over the whole warp (all edge groups)
#pragma unroll
        for (int off = G; off < 32; off <<= 1)
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                c[k] += __shfl_xor_sync(SGA_FULL_MASK, c[k], off);
                z[k] += __shfl_xor_sync(SGA_FULL_MASK, z[k], off);
#pragma unroll
                for (int x = 0; x < EL; ++x) {
                    fA[k][x] += __shfl_xor_sync(SGA_FULL_MASK, fA[k][x], off);
                    fB[k][x] += __shfl_xor_sync(SGA_FULL_MASK, fB[k][x], off);
                }
            }
        if (it.partial) {
            // da sums of this chunk, combined over the groups, go to the merge kernel
#pragma unroll
            for (int off = G; off < 32; off <<= 1)
#pragma unroll
                for (int k = 0; k < NC; ++k)
#pragma unroll
                    for (int x = 0; x < EL; ++x) {
                        gA[k][x] += __shfl_xor_sync(SGA_FULL_MASK, gA[k][x], off);
                        gB[k][x] += __shfl_xor_sync(SGA_FULL_MASK, gB[k][x], off);
                    }
            if (g == 0) {
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    const int ch = gl + G * k;
                    if (ch >= R) continue;
                    float *base = a.ws_row + (size_t)it.item * 4 * HD + ch * EL;
#pragma unroll
                    for (int x = 0; x < EL; x += 4) {
                        *reinterpret_cast<float4 *>(base + x) =
                            make_float4(fA[k][x], fA[k][x + 1], fA[k][x + 2], fA[k][x + 3]);
                        *reinterpret_cast<float4 *>(base + HD + x) =
                            make_float4(fB[k][x], fB[k][x + 1], fB[k][x + 2], fB[k][x + 3]);
                        *reinterpret_cast<float4 *>(base + 2 * HD + x) =
                            make_float4(gA[k][x], gA[k][x + 1], gA[k][x + 2], gA[k][x + 3]);
                        *reinterpret_cast<float4 *>(base + 3 * HD + x) =
                            make_float4(gB[k][x], gB[k][x + 1], gB[k][x + 2], gB[k][x + 3]);
                    }
                    if (ch % LH == 0) {
                        a.ws_rowc[((size_t)it.item * a.H + ch / LH) * 2] = c[k];
                        a.ws_rowc[((size_t)it.item * a.H + ch / LH) * 2 + 1] = z[k];
                    }
                }
            }
        } else {
            // normalised weights p / Z (RowNorm): Delta = C / Z, sums / Z
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                const RowNorm nrm(c[k], z[k]);
#pragma unroll
                for (int x = 0; x < EL; ++x) dacc[k][x] += (gA[k][x] - nrm.delta * gB[k][x]) * nrm.inv_z;
            }
            if (g == 0) {
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    const int ch = gl + G * k;
                    if (ch >= R) continue;
                    const RowNorm nrm(c[k], z[k]);
                    float v[EL];
#pragma unroll
                    for (int x = 0; x < EL; ++x) v[x] = (fA[k][x] - nrm.delta * fB[k][x]) * nrm.inv_z;
                    store_dF<T, EL>(a.ws_dfl, it.row, HD, ch, v);
                    if (ch % LH == 0) {
                        const size_t rh = (size_t)it.row * a.H + ch / LH;
                        a.ws_delta[rh] = nrm.delta;
                        a.ws_lse[rh] = a.lse[rh] + nrm.lse_shift;
                    }
                }
            }
        }
        if (it.partial && last_chunk(a.rows, it.item)) gatv2_bwd_merge_row<T, D>(a, 0, __ldg(a.rows.chunk_split + it.item));
        st.finish_item();
    }
    st.drain();
    // da: groups -> lanes of group 0, warps -> shared memory in warp order
#pragma unroll
    for (int off = G; off < 32; off <<= 1)
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int x = 0; x < EL; ++x) dacc[k][x] += __shfl_xor_sync(SGA_FULL_MASK, dacc[k][x], off);
    __syncthreads();
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
        if ((threadIdx.x >> 5) == w && g == 0) {
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                const int c = gl + G * k;
                if (c < R)
#pragma unroll
                    for (int x = 0; x < EL; ++x) da_sh[c * EL + x] += dacc[k][x];
            }
        }
        __syncthreads();
    }
    for (int x = threadIdx.x; x < HD; x += blockDim.x)
        a.ws_da[(size_t)blockIdx.x * HD + x] = da_sh[x];
}

// ---------------------------------------------------- backward: src pass

// Per source j over its destinations i (transposed CSR):
//   dFR_j += p dOut_i + de a * LReLU'(z).
template <typename T, int D, int NC, int G>
__global__ void __launch_bounds__(256, 2)
gatv2_bwd_src_kernel(Gatv2Args a) {
    using S = GtShape<T, D, NC, G>;
    using C = Gatv2SrcStream<T, D, NC, G>;
    constexpr int EL = S::EL, LH = S::LH, U = C::U;
    extern __shared__ __align__(16) unsigned char dsmem[];
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    const float slope = a.slope;
    float att[NC][EL];
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        const int c = gl + G * k;
        if (c < R) unpack<T>(ldg16(static_cast<const uint4 *>(a.a) + c), att[k]);
        else
#pragma unroll
            for (int x = 0; x < EL; ++x) att[k][x] = 0.f;
    }
    StreamArrays arr{};
    arr.rows[0] = static_cast<const uint4 *>(a.FL);
    arr.rows[1] = static_cast<const uint4 *>(a.dOut);
    arr.sc[0] = a.ws_lse;     // lse + ln Z of each destination (normalised weights)
    arr.sc[1] = a.ws_delta;
    arr.own[0] = static_cast<const uint4 *>(a.FR);
    EdgeStream<C> st;
    st.init(dsmem + (threadIdx.x >> 5) * C::BYTES, arr, a.cols, a.t_indptr, a.t_dst, a.N, a.H, R, LH,
            a.split_threshold, a.d_err);
    StreamItem it;
    while (st.next_item(it)) {
        // dfr: sum of p dOut_i; dfw: sum of de LReLU'(z), times a after the
        // column (up to two chunks per lane; wider rows lack the registers and
        // weight each edge's term by a directly)
        constexpr bool kFactorA = NC <= 2;
        float frj[NC][EL], dfr[NC][EL], dfw[NC][EL];
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int x = 0; x < EL; ++x) frj[k][x] = dfr[k][x] = dfw[k][x] = 0.f;
        for (int step = 0; step < it.nsteps; ++step) {
            st.wait_step();
            if (step == 0)
#pragma unroll
                for (int k = 0; k < NC; ++k) unpack<T>(st.own_row(0, k), frj[k]);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ok = st.valid(u);
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    float f[EL], gf[EL], lz[EL], dz[EL];
                    unpack<T>(st.row(u, 0, k), f);
                    unpack<T>(st.row(u, 1, k), gf);
                    lrelu_chunk<EL>(f, frj[k], slope, lz, dz);
                    float e = dot2<EL>(att[k], lz), dp = dot2<EL>(gf, frj[k]);
                    group_sum2<LH>(e, dp);
                    const int h = (gl + G * k) / LH;
                    const float p = ok ? fast_exp2((e - st.scalar(u, 0, h)) * kLog2e) : 0.f;
                    const float de = p * (dp - st.scalar(u, 1, h));
                    axpy2<EL>(dfr[k], p, gf);
                    if constexpr (kFactorA) {
                        axpy2<EL>(dfw[k], de, dz);
                    } else {
                        float w[EL];
#pragma unroll
                        for (int x = 0; x < EL; ++x) w[x] = att[k][x] * dz[x];
                        axpy2<EL>(dfr[k], de, w);
                    }
                }
            }
            st.release_step();
        }
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int x = 0; x < EL && kFactorA; x += 2) {
                const float2 r = ffma2(make_float2(att[k][x], att[k][x + 1]), make_float2(dfw[k][x], dfw[k][x + 1]),
                                       make_float2(dfr[k][x], dfr[k][x + 1]));
                dfr[k][x] = r.x;
                dfr[k][x + 1] = r.y;
            }
#pragma unroll
        for (int off = G; off < 32; off <<= 1)
#pragma unroll
            for (int k = 0; k < NC; ++k)
#pragma unroll
                for (int x = 0; x < EL; ++x) dfr[k][x] += __shfl_xor_sync(SGA_FULL_MASK, dfr[k][x], off);
        if (g == 0) {
#pragma unroll
            for (int k = 0; k < NC; ++k) {
                const int c = gl + G * k;
                if (c >= R) continue;
                if (it.partial) {
                    float4 *dst = reinterpret_cast<float4 *>(a.ws_col + (size_t)it.item * HD + c * EL);
#pragma unroll
                    for (int x = 0; x < EL; x += 4)
                        dst[x / 4] = make_float4(dfr[k][x], dfr[k][x + 1], dfr[k][x + 2], dfr[k][x + 3]);
                } else {
                    store_dF<T, EL>(a.ws_dfr, it.row, HD, c, dfr[k]);
                }
            }
        }
        if (it.partial && last_chunk(a.cols, it.item)) gatv2_bwd_merge_row<T, D>(a, 1, __ldg(a.cols.chunk_split + it.item));
        st.finish_item();
    }
    st.drain();
}

// ------------------------------------------------------------ dense GEMMs

// C = sum over pairs p of op(A_p) op(B_p) with fp32 accumulation (SIMT),
// used for float layers, whose fp32 tolerance the bf16 tensor cores miss.
//   A: [M, K] row-major, or [K, M] row-major when TA (then op(A) = A^T).
//   B: [K, N] row-major, or [N, K] row-major when TB.
// Tiles 64 x 64 x 16, 256 threads, 4 x 4 outputs per thread.  Rows [k0, k1)
// of the K range are used (split-K slabs); blockIdx.z selects the slab.
// The result goes to C (dtype T) or, when Cpart is set, to the fp32 partial
// Cpart[slab][M][N].
template <typename TA_, typename TB_, typename T, bool TA, bool TB> struct GemmArgs {
    const TA_ *A[2];
    const TB_ *B[2];
    int pairs;
    int64_t M, N, K;
    int64_t k_per_slab;
    T *C;
    float *Cpart;
};

template <typename TA_, typename TB_, typename T, bool TA, bool TB>
__global__ void __launch_bounds__(256) gemm_simt_kernel(GemmArgs<TA_, TB_, T, TA, TB> g) {
    constexpr int BM = 64, BN = 64, BK = 16;
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    const int64_t k_lo = (int64_t)blockIdx.z * g.k_per_slab;
    const int64_t k_hi = min(g.K, k_lo + g.k_per_slab);
    float acc[4][4] = {};
    for (int p = 0; p < g.pairs; ++p) {
        const TA_ *A = g.A[p];
        const TB_ *B = g.B[p];
        for (int64_t kb = k_lo; kb < k_hi; kb += BK) {
            for (int idx = threadIdx.x; idx < BM * BK; idx += 256) {
                int mm, kk;
                if (TA) { mm = idx % BM; kk = idx / BM; } else { kk = idx % BK; mm = idx / BK; }
                const int64_t gm = m0 + mm, gk = kb + kk;
                float v = 0.f;
                if (gm < g.M && gk < k_hi)
                    v = to_f32<TA_>(TA ? A[gk * g.M + gm] : A[gm * g.K + gk]);
                As[kk][mm] = v;
            }
            for (int idx = threadIdx.x; idx < BN * BK; idx += 256) {
                int nn, kk;
                if (TB) { kk = idx % BK; nn = idx / BK; } else { nn = idx % BN; kk = idx / BN; }
                const int64_t gn = n0 + nn, gk = kb + kk;
                float v = 0.f;
                if (gn < g.N && gk < k_hi)
                    v = to_f32<TB_>(TB ? B[gn * g.K + gk] : B[gk * g.N + gn]);
                Bs[kk][nn] = v;
            }
            __syncthreads();
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                float av[4], bv[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) av[r] = As[kk][ty * 4 + r];
#pragma unroll
                for (int c = 0; c < 4; ++c) bv[c] = Bs[kk][tx * 4 + c];
#pragma unroll
                for (int r = 0; r < 4; ++r)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
            }
            __syncthreads();
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int64_t gm = m0 + ty * 4 + r;
        if (gm >= g.M) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int64_t gn = n0 + tx * 4 + c;
            if (gn >= g.N) continue;
            if (g.Cpart) g.Cpart[((int64_t)blockIdx.z * g.M + gm) * g.N + gn] = acc[r][c];
            else g.C[gm * g.N + gn] = from_f32<T>(acc[r][c]);
        }
    }
}

// dW_l, dW_r = sum of the slab partials [2][slab][F*HD]; da = sum of the
// per-block partials followed by the split rows' contributions.  A block of
// 32 outputs x 8 lanes of partials: lane group r adds partials r, r + 8, ...
// in increasing order, then group 0 adds the eight sums in order, so the
// result is independent of scheduling.
constexpr int kRedOut = 32, kRedGroups = 8;
template <typename T>
__global__ void __launch_bounds__(kRedOut * kRedGroups)
gatv2_reduce_kernel(const float *__restrict__ dw_part, int slabs, int64_t FHD, T *dWl, T *dWr,
                    const float *__restrict__ da_part, int blocks, const float *__restrict__ da_split,
                    int n_split, int HD, T *da) {
    __shared__ float sh[kRedGroups][kRedOut];
    const int o = threadIdx.x % kRedOut, r = threadIdx.x / kRedOut;
    const int64_t t = (int64_t)blockIdx.x * kRedOut + o;
    // partials r, r + 8, r + 16, ... are fetched sixteen at a time
    // (independent loads in flight) and added in increasing order
    constexpr int kBatch = 16;
    float sum = 0.f;
    if (t < 2 * FHD) {
        const int which = (int)(t / FHD);
        const float *base = dw_part + (int64_t)which * slabs * FHD + t % FHD;
        for (int k0 = r; k0 < slabs; k0 += kRedGroups * kBatch) {
            float v[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int k = k0 + j * kRedGroups;
                v[j] = k < slabs ? base[(int64_t)k * FHD] : 0.f;
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) sum += v[j];
        }
    } else if (t < 2 * FHD + HD) {
        const int x = (int)(t - 2 * FHD), n = blocks + n_split;
        for (int k0 = r; k0 < n; k0 += kRedGroups * kBatch) {
            float v[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                const int k = k0 + j * kRedGroups;
                v[j] = k < blocks ? da_part[(int64_t)k * HD + x]
                                  : (k < n ? da_split[(int64_t)(k - blocks) * HD + x] : 0.f);
            }
#pragma unroll
            for (int j = 0; j < kBatch; ++j) sum += v[j];
        }
    }
    sh[r][o] = sum;
    __syncthreads();
    if (r == 0) {
        float tot = 0.f;
#pragma unroll
        for (int q = 0; q < kRedGroups; ++q) tot += sh[q][o];
        if (t < 2 * FHD) {
            const int which = (int)(t / FHD);
            (which ? dWr : dWl)[t % FHD] = from_f32<T>(tot);
        } else if (t < 2 * FHD + HD) {
            da[t - 2 * FHD] = from_f32<T>(tot);
        }
    }
}

template <typename TA_, typename TB_, typename T, bool TA, bool TB>
cudaError_t gemm(const GemmArgs<TA_, TB_, T, TA, TB> &g, int slabs, sga_kernel_id kid, cudaStream_t s) {
    dim3 grid((unsigned)((g.N + 63) / 64), (unsigned)((g.M + 63) / 64), (unsigned)slabs);
    note_launch(kid, s, false);
    gemm_simt_kernel<TA_, TB_, T, TA, TB><<<grid, 256, 0, s>>>(g);
    note_launch(kid, s, true);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ launch

template <typename T, int D> cudaError_t gatv2_fwd_d(const Gatv2Args &a, cudaStream_t s) {
    constexpr int LH = D * (int)sizeof(T) / 16;
    const int R = a.H * D / Elt<T>::EL;
    const int HD = a.H * D;
    // projections FL = X W_l, FR = X W_r (bf16: tensor cores, correctly rounded)
    if constexpr (sizeof(T) == 2) {
        if (a.N > 0 && tc_proj_supported(a.F, HD)) {   // tcgen05 path
            TcProj tp{};
            tp.X = static_cast<const __nv_bfloat16 *>(a.X);
            tp.Wl = static_cast<const __nv_bfloat16 *>(a.Wl);
            tp.Wr = static_cast<const __nv_bfloat16 *>(a.Wr);
            tp.FL = static_cast<__nv_bfloat16 *>(a.FL_w);
            tp.FR = static_cast<__nv_bfloat16 *>(a.FR_w);
            tp.M = a.N;
            tp.K = a.F;
            tp.HD = HD;
            tp.err = a.d_err;
            cudaError_t e = tc_proj(tp, s);
            if (e != cudaSuccess) return e;
        } else if (a.N > 0) {
            cudaError_t e = cudaMemsetAsync(a.ws_fix_count, 0, sizeof(int32_t), s);
            for (int w = 0; w < 2 && e == cudaSuccess; ++w) {
                MmaGemm<T, T, T, false, true, 0> g{};
                g.A[0] = static_cast<const T *>(a.X);
                g.B[0] = static_cast<const T *>(w ? a.Wr : a.Wl);
                g.pairs = 1;
                g.M = a.N; g.N = HD; g.K = a.F; g.k_per_slab = a.F;
                g.C = static_cast<T *>(w ? a.FR_w : a.FL_w);
                g.fix_count = a.ws_fix_count;
                g.fix_list = a.ws_fix_list;
                g.fix_cap = a.fix_cap;
                g.fix_tag = w;
                e = mma_gemm(g, 1, SGA_KERN_GATV2_PROJ, s);
            }
            if (e != cudaSuccess) return e;
            if (a.F > 2 * mm::BK) {   // k range too long for in-block rounding
                ExactRound r{};
                r.X = static_cast<const __nv_bfloat16 *>(a.X);
                r.W[0] = static_cast<const __nv_bfloat16 *>(a.Wl);
                r.W[1] = static_cast<const __nv_bfloat16 *>(a.Wr);
                r.C[0] = static_cast<__nv_bfloat16 *>(a.FL_w);
                r.C[1] = static_cast<__nv_bfloat16 *>(a.FR_w);
                r.M = a.N; r.N = HD; r.K = a.F;
                r.count = a.ws_fix_count;
                r.list = a.ws_fix_list;
                r.cap = a.fix_cap;
                note_launch(SGA_KERN_GATV2_PROJ, s, false);
                exact_round_kernel<<<persistent_blocks<exact_round_kernel>(1 << 30), 256, 0, s>>>(r);
                note_launch(SGA_KERN_GATV2_PROJ, s, true);
                if ((e = cudaGetLastError()) != cudaSuccess) return e;
            }
        }
    } else {
        for (int w = 0; w < 2 && a.N > 0; ++w) {
            GemmArgs<T, T, T, false, false> g{};
            g.A[0] = static_cast<const T *>(a.X);
            g.B[0] = static_cast<const T *>(w ? a.Wr : a.Wl);
            g.pairs = 1;
            g.M = a.N; g.N = HD; g.K = a.F; g.k_per_slab = a.F;
            g.C = static_cast<T *>(w ? a.FR_w : a.FL_w);
            g.Cpart = nullptr;
            cudaError_t e = gemm(g, 1, SGA_KERN_GATV2_PROJ, s);
            if (e != cudaSuccess) return e;
        }
    }
    Gatv2Args b = a;
    b.FL = a.FL_w;
    b.FR = a.FR_w;
    const int64_t items = (int64_t)a.rows.n_chunks + a.N;
    cudaError_t e = dispatch_shape<LH, max_nc<T>()>(R, [&]<int NC, int G>() -> cudaError_t {
        if (items == 0) return cudaSuccess;
        if (reset_items<Gatv2FwdStream<T, D, NC, G>>(a.rows, s) != cudaSuccess) return cudaGetLastError();
        note_launch(SGA_KERN_GATV2_FWD, s, false);
        const cudaError_t e2 =
            launch_streamed<Gatv2FwdStream<T, D, NC, G>, gatv2_fwd_kernel<T, D, NC, G>>(items, s, b);
        note_launch(SGA_KERN_GATV2_FWD, s, true);
        return e2;
    });
    return e;   // (split rows are merged by their last chunk inside the edge kernel)
}

template <typename T, int D> cudaError_t gatv2_bwd_d(const Gatv2Args &a, cudaStream_t s) {
    constexpr int LH = D * (int)sizeof(T) / 16;
    const int R = a.H * D / Elt<T>::EL;
    const int HD = a.H * D;
    cudaError_t e = dispatch_shape<LH, max_nc<T>()>(R, [&]<int NC, int G>() -> cudaError_t {
        if (reset_items<Gatv2DstStream<T, D, NC, G>>(a.rows, s) != cudaSuccess) return cudaGetLastError();
        note_launch(SGA_KERN_GATV2_BWD_DST, s, false);
        // one da partial per block: exactly da_blocks blocks
        cudaError_t e2 = launch_streamed_grid<Gatv2DstStream<T, D, NC, G>, gatv2_bwd_dst_kernel<T, D, NC, G>,
                                              4096>(a.da_blocks, s, a);
        note_launch(SGA_KERN_GATV2_BWD_DST, s, true);
        if (e2 != cudaSuccess) return e2;
        // (split rows are merged by their last chunk inside each pass; the
        // destination pass's merges leave Delta for the source pass)
        const int64_t items_c = (int64_t)a.cols.n_chunks + a.N;
        if (items_c == 0) return cudaSuccess;
        if (reset_items<Gatv2SrcStream<T, D, NC, G>>(a.cols, s) != cudaSuccess) return cudaGetLastError();
        note_launch(SGA_KERN_GATV2_BWD_SRC, s, false);
        e2 = launch_streamed<Gatv2SrcStream<T, D, NC, G>, gatv2_bwd_src_kernel<T, D, NC, G>>(items_c, s, a);
        note_launch(SGA_KERN_GATV2_BWD_SRC, s, true);
        return e2;
    });
    if (e != cudaSuccess) return e;
    // dX = dFL W_l^T + dFR W_r^T
    const int64_t per = (a.N + a.dw_slabs - 1) / a.dw_slabs;
    int dw_slabs_used = 0;   // slabs the tensor-core dW wrote (0: the GEMM below wrote dw_slabs)
    const int64_t FHD = (int64_t)a.F * HD;
    if (a.N > 0) {
        if constexpr (sizeof(T) == 2) {
          if (tc_dx_supported(a.F, HD, a.N)) {   // tcgen05 + TMA
            TcDx t{};
            t.dfl = reinterpret_cast<const __nv_bfloat16 *>(a.ws_dfl);
            t.dfr = reinterpret_cast<const __nv_bfloat16 *>(a.ws_dfr);
            t.Wl = static_cast<const __nv_bfloat16 *>(a.Wl);
            t.Wr = static_cast<const __nv_bfloat16 *>(a.Wr);
            t.dX = static_cast<__nv_bfloat16 *>(a.dX);
            t.M = a.N;
            t.F = a.F;
            t.HD = HD;
            t.err = a.d_err;
            note_launch(SGA_KERN_GATV2_BWD_DX, s, false);
            e = tc_dx(t, s);
            note_launch(SGA_KERN_GATV2_BWD_DX, s, true);
            if (e != cudaSuccess) return e;
          } else {
            // four bf16 pairs: dFL hi, dFL lo, dFR hi, dFR lo against W_l, W_l, W_r, W_r
            MmaGemm<T, T, T, false, false, 1> g{};
            const T *dfl = reinterpret_cast<const T *>(a.ws_dfl), *dfr = reinterpret_cast<const T *>(a.ws_dfr);
            g.A[0] = dfl;
            g.A[1] = dfl + HD;
            g.A[2] = dfr;
            g.A[3] = dfr + HD;
            g.B[0] = g.B[1] = static_cast<const T *>(a.Wl);
            g.B[2] = g.B[3] = static_cast<const T *>(a.Wr);
            g.pairs = 4;
            g.lda = 2 * HD;
            g.M = a.N; g.N = a.F; g.K = HD; g.k_per_slab = HD;
            g.C = static_cast<T *>(a.dX);
            if ((e = mma_gemm(g, 1, SGA_KERN_GATV2_BWD_DX, s)) != cudaSuccess) return e;
          }
        } else {
            GemmArgs<float, T, T, false, true> g{};
            g.A[0] = a.ws_dfl;
            g.B[0] = static_cast<const T *>(a.Wl);
            g.A[1] = a.ws_dfr;
            g.B[1] = static_cast<const T *>(a.Wr);
            g.pairs = 2;
            g.M = a.N; g.N = a.F; g.K = HD; g.k_per_slab = HD;
            g.C = static_cast<T *>(a.dX);
            if ((e = gemm(g, 1, SGA_KERN_GATV2_BWD_DX, s)) != cudaSuccess) return e;
        }
        // dW = X^T dF over node slabs: fp32 partials [2][slab][F][HD]
        if constexpr (sizeof(T) == 2) {
            if (tc_dw_supported(a.F, HD, a.N)) {   // tcgen05 + TMA, both matrices in one pass
                int dev = 0, sms = 1;
                cudaGetDevice(&dev);
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
                TcDw t{};
                t.X = static_cast<const __nv_bfloat16 *>(a.X);
                t.dfl = reinterpret_cast<const __nv_bfloat16 *>(a.ws_dfl);
                t.dfr = reinterpret_cast<const __nv_bfloat16 *>(a.ws_dfr);
                t.part = a.ws_dw;
                t.M = a.N;
                t.F = a.F;
                t.HD = HD;
                t.slab_rows = dw_slab_rows(a.N, sms);
                t.slabs = (int)((a.N + t.slab_rows - 1) / t.slab_rows);
                t.err = a.d_err;
                if (t.slabs > a.dw_slabs) return cudaErrorInvalidValue;   // the workspace holds dw_slabs
                note_launch(SGA_KERN_GATV2_BWD_DW, s, false);
                e = tc_dw(t, s);
                note_launch(SGA_KERN_GATV2_BWD_DW, s, true);
                if (e != cudaSuccess) return e;
                dw_slabs_used = t.slabs;
            }
        }
        for (int w = 0; w < 2 && dw_slabs_used == 0; ++w) {
            if constexpr (sizeof(T) == 2) {
                MmaGemm<T, T, float, true, true, 2> g{};   // X^T (dF hi) + X^T (dF lo)
                const T *df = reinterpret_cast<const T *>(w ? a.ws_dfr : a.ws_dfl);
                g.A[0] = g.A[1] = static_cast<const T *>(a.X);
                g.B[0] = df;
                g.B[1] = df + HD;
                g.pairs = 2;
                g.ldb = 2 * HD;
                g.M = a.F; g.N = HD; g.K = a.N; g.k_per_slab = per;
                g.Cpart = a.ws_dw + (size_t)w * FHD * a.dw_slabs;
                if ((e = mma_gemm(g, a.dw_slabs, SGA_KERN_GATV2_BWD_DW, s)) != cudaSuccess) return e;
            } else {
                GemmArgs<T, float, T, true, false> g{};
                g.A[0] = static_cast<const T *>(a.X);
                g.B[0] = w ? a.ws_dfr : a.ws_dfl;
                g.pairs = 1;
                g.M = a.F; g.N = HD; g.K = a.N; g.k_per_slab = per;
                g.C = nullptr;
                g.Cpart = a.ws_dw + (size_t)w * FHD * a.dw_slabs;
                if ((e = gemm(g, a.dw_slabs, SGA_KERN_GATV2_BWD_DW, s)) != cudaSuccess) return e;
            }
        }
    }
    const int64_t total = 2 * FHD + HD;
    note_launch(SGA_KERN_GATV2_BWD_REDUCE, s, false);
    gatv2_reduce_kernel<T><<<(unsigned)((total + kRedOut - 1) / kRedOut), kRedOut * kRedGroups, 0, s>>>(
        a.ws_dw, dw_slabs_used ? dw_slabs_used : a.dw_slabs, FHD, static_cast<T *>(a.dWl), static_cast<T *>(a.dWr),
        a.ws_da,
        a.da_blocks, a.ws_da_split, a.rows.n_split, HD, static_cast<T *>(a.da));
    note_launch(SGA_KERN_GATV2_BWD_REDUCE, s, true);
    return cudaGetLastError();
}

template <typename T> cudaError_t gatv2_fwd_t(const Gatv2Args &a, cudaStream_t s) {
    switch (a.D) {
        case 32: return gatv2_fwd_d<T, 32>(a, s);
        case 64: return gatv2_fwd_d<T, 64>(a, s);
        case 128: return gatv2_fwd_d<T, 128>(a, s);
    }
    return cudaErrorInvalidValue;
}

template <typename T> cudaError_t gatv2_bwd_t(const Gatv2Args &a, cudaStream_t s) {
    switch (a.D) {
        case 32: return gatv2_bwd_d<T, 32>(a, s);
        case 64: return gatv2_bwd_d<T, 64>(a, s);
        case 128: return gatv2_bwd_d<T, 128>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace sga
