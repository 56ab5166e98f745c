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

#include <algorithm>

#include "common.cuh"
#include "items.cuh"
#include "plan.h"
#include "stream.cuh"

namespace sga {

template <typename T, int D, int NC, int G> struct GtShape {
    static constexpr int EL = Elt<T>::EL;                     // elements per 16-byte chunk
    static constexpr int LH = D * (int)sizeof(T) / 16;        // lanes per head
    static constexpr int NG = 32 / G;                         // edge groups per warp
    static constexpr int U = NC >= 4 ? 1 : 4 / NC;            // neighbours in flight per group
    static_assert(LH <= G, "a head must fit in one edge group");
};

// Head sums of two value pairs per lane, (s0, t0) of its first chunk and
// (s1, t1) of its second, when both chunks' heads span the same LH lanes
// (two chunks per lane, LH >= 2): the lanes whose bit LH/2 is clear finish the
// first chunk's sums and the others the second's, so one exchange halves the
// work before the usual butterfly.  Returns whether this lane finished the
// second chunk; (s, t) are its head sums.
template <int LH>
__device__ __forceinline__ bool head_sums_split(float s0, float t0, float s1, float t1, float &s, float &t) {
    static_assert(LH >= 2, "a head spans at least two lanes");
    const bool hi = (threadIdx.x & (LH / 2)) != 0;
    s = (hi ? s1 : s0) + __shfl_xor_sync(SGA_FULL_MASK, hi ? s0 : s1, LH / 2);
    t = (hi ? t1 : t0) + __shfl_xor_sync(SGA_FULL_MASK, hi ? t0 : t1, LH / 2);
#pragma unroll
    for (int o = LH / 4; o > 0; o >>= 1) {
        s += __shfl_xor_sync(SGA_FULL_MASK, s, o);
        t += __shfl_xor_sync(SGA_FULL_MASK, t, o);
    }
    return hi;
}

// ------------------------------------------------------------------ forward

// Stream shape of a kernel with NROW gathered row arrays: U neighbours per
// group and step, and a ring of about 10 KB per warp (2 to 8 steps).  Rows of
// one chunk per lane take 4 neighbours a step when groups are narrower than a
// warp, else U1; rows of two chunks per lane take U2; wider rows take 1.  More
// neighbours a step spread the per-step bookkeeping (queue, masks, waits) over
// more edges but leave fewer steps in flight and hold more registers, so each
// kernel takes the largest counts that keep its registers.
template <int NC, int NROW, int NSC = 0, int NOWN = 1, int NOSC = 0, int G = 32, int U2 = 1, int U1 = 2>
struct RingDims {
    static constexpr int U0 = NC >= 2 ? (NC == 2 ? U2 : 1) : (G < 32 ? 4 : U1);
    static constexpr int OWN_BYTES = NC * 32 * (NOWN * 16 + NOSC * 4);
    static constexpr int QD = 3 * OWN_BYTES > 4096 ? 2 : 3;
    // a step of U0 neighbours that leaves room for fewer than two steps
    // (several gathered scalars per neighbour) takes two neighbours instead
    static constexpr int U = (U0 > 2 && (13312 - QD * OWN_BYTES) / (U0 * NC * 32 * (NROW * 16 + NSC * 4)) < 2)
                                 ? 2 : U0;
    static constexpr int STEP_BYTES = U * NC * 32 * (NROW * 16 + NSC * 4);
    static constexpr int FIT = (13312 - QD * OWN_BYTES) / STEP_BYTES;
    static_assert(U <= 2 || FIT >= 2, "two steps of several neighbours must fit the ring");
    static constexpr int DEPTH = FIT < 2 ? 2 : (FIT > 8 ? 8 : FIT);
};
template <int NC, int G, int NROW, int NSC, int NOWN, int NOSC, int U2 = 1, int U1 = 2, int ESC = 0,
          bool LIST = true, bool W32 = false, int DYN = 0>
using RingCfg = StreamCfg<NC, G, RingDims<NC, NROW, NSC, NOWN, NOSC, G, U2, U1>::U, NROW, NSC, NOWN, NOSC,
                          RingDims<NC, NROW, NSC, NOWN, NOSC, G, U2, U1>::DEPTH,
                          RingDims<NC, NROW, NSC, NOWN, NOSC, G, U2, U1>::QD, ESC, LIST, W32, DYN>;

// Dynamic items of the GT passes: the plan's batch, at most eight, on
// one-chunk rows (R-MAT step 12.84 -> 12.47 ms against single items); single
// items on wider rows, where batches lost (SBM forward 2.28 -> 2.84 ms with
// batches of four).
template <int NC> constexpr int gt_batch() { return NC == 1 ? 8 : 1; }

// gathered K, V (and the edge's score bias); own Q.  LIST = false: no item
// list (the no-allocation forward, which has no plan)
template <typename T, int D, int NC, int G, bool BIAS = false, bool LIST = true>
using GtFwdStream = RingCfg<NC, G, 2, BIAS ? 1 : 0, 1, 0, 2, 4, BIAS ? 1 : 0, LIST, true, LIST ? gt_batch<NC>() : 0>;
// gathered K, V (and the edge's score bias); own Q, dOut, lse
template <typename T, int D, int NC, int G, bool BIAS = false>
using GtDqStream = RingCfg<NC, G, 2, BIAS ? 1 : 0, 2, 1, 2, 4, BIAS ? 1 : 0, true, true, gt_batch<NC>()>;
// gathered Q, dOut, lse, Delta (over the transposed CSR; and the edge's score
// bias in transposed order); own K, V
template <typename T, int D, int NC, int G, bool BIAS = false>
using GtDkdvStream = RingCfg<NC, G, 2, BIAS ? 3 : 2, 2, 0, 1, 4, BIAS ? 4 : 0, true, true, gt_batch<NC>()>;

// ---- split rows merged by their last chunk ----------------------------------
//
// The Graph Transformer passes merge this way on rows of two or more chunks
// per lane; on one-chunk rows the merge call cost the main loop more than
// the separate merge kernels cost (workload 4), so those keep the kernels.
template <int NC> constexpr bool gt_fold() { return NC >= 2; }
//
// A chunk of a split row writes its partial and then counts itself in
// P.arrive[split]; the warp whose arrival completes the row merges all of the
// row's partials in chunk order (so the result does not depend on which chunk
// finished last) and sets the count back to 0 for the next launch.  The
// partials of other SMs are read past L1.  (The split index is looked up from
// the chunk index here rather than carried by the edge stream, whose state is
// at the register limit in the Graph Transformer passes.)
__device__ __forceinline__ bool last_chunk(const Partition &P, int32_t chunk) {
    __threadfence();   // this warp's partial before its arrival
    __syncwarp();
    int32_t last = 0;
    if ((threadIdx.x & 31) == 0) {
        const int32_t s = __ldg(P.chunk_split + chunk);
        const int32_t k = __ldg(P.chunk_ptr + s + 1) - __ldg(P.chunk_ptr + s);
        last = atomicAdd(P.arrive + s, 1) + 1 == k ? 1 : 0;
        if (last) P.arrive[s] = 0;   // (every chunk of the row has arrived)
    }
    last = __shfl_sync(SGA_FULL_MASK, last, 0);
    if (last) __threadfence();   // the other chunks' partials after their arrivals
    return last != 0;
}

// Forward: fold the chunk partials of split row s with the online rule
// (m = max, l and acc rescaled by 2^(m_c - m)) in chunk order; one warp,
// lane-chunks lane, lane + 32, ...; out = acc / l, lse = (m + log2 l) ln 2.
template <typename T, int D, typename A> __device__ __noinline__ void fwd_merge_row(const A &a, int32_t s) {
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16;
    const int32_t row = __ldg(a.rows.split_rows + s);
    const int32_t c0 = __ldg(a.rows.chunk_ptr + s), c1 = __ldg(a.rows.chunk_ptr + s + 1);
    const int R = a.H * D / EL, HD = a.H * D;
    for (int c = threadIdx.x & 31; c < R; c += 32) {
        const int h = c / LH;
        float m = -INFINITY, l = 0.f, acc[EL];
#pragma unroll
        for (int x = 0; x < EL; ++x) acc[x] = 0.f;
#pragma unroll 4
        for (int32_t ch = c0; ch < c1; ++ch) {
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.ws_ml + ((size_t)ch * a.H + h) * 2));
            const float mx = fmaxf(m, ml.x);
            const float a1 = exp2_diff(m, mx), a2 = exp2_diff(ml.x, mx);
            const float4 *src = reinterpret_cast<const float4 *>(a.ws_acc + (size_t)ch * HD + c * EL);
#pragma unroll
            for (int x = 0; x < EL; x += 4) {
                const float4 v = __ldcg(src + x / 4);
                acc[x] = acc[x] * a1 + v.x * a2;
                acc[x + 1] = acc[x + 1] * a1 + v.y * a2;
                acc[x + 2] = acc[x + 2] * a1 + v.z * a2;
                acc[x + 3] = acc[x + 3] * a1 + v.w * a2;
            }
            l = l * a1 + ml.y * a2;
            m = mx;
        }
        const float inv = l > 0.f ? 1.f / l : 0.f;
        float o[EL];
#pragma unroll
        for (int x = 0; x < EL; ++x) o[x] = acc[x] * inv;
        reinterpret_cast<uint4 *>(a.out_w)[(size_t)row * R + c] = pack<T>(o);
        if (c % LH == 0) a.lse_w[(size_t)row * a.H + h] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
    }
}

// Sums over chunks c0 .. c1 - 1 (chunk order) of NCOMP [HD] partial rows
// (component q of chunk ch at part[(ch * stride_c + q) * HD]) and of NSC
// per-head scalars (parts_c[(ch * H + h) * NSC + t]), for lane-chunk c.
template <int EL, int NCOMP, int NSC>
__device__ __forceinline__ void warp_sum_chunks(const float *part, int stride_c, int HD, const float *parts_c,
                                                int H, int h, int32_t c0, int32_t c1, int c,
                                                float (&sum)[NCOMP][EL], float (&csum)[NSC]) {
#pragma unroll
    for (int q = 0; q < NCOMP; ++q)
#pragma unroll
        for (int x = 0; x < EL; ++x) sum[q][x] = 0.f;
#pragma unroll
    for (int t = 0; t < NSC; ++t) csum[t] = 0.f;
#pragma unroll 2
    for (int32_t ch = c0; ch < c1; ++ch) {
#pragma unroll
        for (int q = 0; q < NCOMP; ++q) {
            const float4 *src = reinterpret_cast<const float4 *>(part + ((size_t)ch * stride_c + q) * HD + c * EL);
#pragma unroll
            for (int x = 0; x < EL; x += 4) {
                const float4 v = __ldcg(src + x / 4);
                sum[q][x] += v.x;
                sum[q][x + 1] += v.y;
                sum[q][x + 2] += v.z;
                sum[q][x + 3] += v.w;
            }
        }
        if (parts_c)
#pragma unroll
            for (int t = 0; t < NSC; ++t) csum[t] += __ldcg(parts_c + ((size_t)ch * H + h) * NSC + t);
    }
}

// With BIAS, each edge's score gains a per-head term b[e, h] (fp32, [E, H] in
// CSR edge order): s_ij = q_i . k_j / sqrt(D) + b_eh.
template <typename T, int D, int NC, int G, bool BIAS, bool LIST>
__global__ void __launch_bounds__(256, 2)
gt_fwd_kernel(GtArgs a, float scale2) {
    using S = GtShape<T, D, NC, G>;
    using C = GtFwdStream<T, D, NC, G, BIAS, LIST>;
    constexpr int EL = S::EL, LH = S::LH, U = C::U;
    extern __shared__ __align__(16) unsigned char dsmem[];
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    StreamArrays arr{};
    arr.rows[0] = static_cast<const uint4 *>(a.K);
    arr.rows[1] = static_cast<const uint4 *>(a.V);
    arr.own[0] = static_cast<const uint4 *>(a.Q);
    if (BIAS) arr.sc[0] = a.bias;
    EdgeStream<C> st;
    st.init(dsmem + (threadIdx.x >> 5) * C::BYTES, arr, a.rows, a.indptr, a.indices, a.N, a.H, R, LH,
            a.split_threshold, a.d_err);
    StreamItem it;
    while (st.next_item(it)) {
        float q[NC][EL], acc[NC][EL], m[NC], l[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
#pragma unroll
            for (int x = 0; x < EL; ++x) q[k][x] = acc[k][x] = 0.f;
            m[k] = -INFINITY;
            l[k] = 0.f;
        }
        for (int step = 0; step < it.nsteps; ++step) {
            st.wait_step();
            if (step == 0)
#pragma unroll
                for (int k = 0; k < NC; ++k) unpack<T>(st.own_row(0, k), q[k]);
            float sc[U][NC];
            bool ok[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                ok[u] = st.valid(u);
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    float kf[EL];
                    unpack<T>(st.row(u, 0, k), kf);
                    const float dot = group_sum<LH>(dot2<EL>(q[k], kf));
                    if constexpr (BIAS)
                        sc[u][k] = ok[u] ? dot * scale2 + st.scalar(u, 0, (gl + G * k) / LH) * kLog2e : -INFINITY;
                    else
                        sc[u][k] = ok[u] ? dot * scale2 : -INFINITY;
                }
            }
            // online softmax with a lazily moved maximum: the accumulator is
            // rescaled only when a score exceeds the running maximum by more
            // than 2^kLazyLog2, so weights stay below 2^kLazyLog2
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
                    unpack<T>(st.row(u, 1, k), vf);
                    axpy2<EL>(acc[k], p, vf);
                }
            }
            st.release_step();
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
        if constexpr (LIST && gt_fold<NC>()) {   // the last chunk of a split row merges the row
            if (it.partial && last_chunk(a.rows, it.item)) fwd_merge_row<T, D>(a, __ldg(a.rows.chunk_split + it.item));
        }
        st.finish_item();
    }
    st.drain();
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
// part[(ch * stride_c + q) * HD]) and, if `parts_c`, NSC per-head scalars
// (scalar t of chunk ch, head h at parts_c[(ch * H + h) * NSC + t]); the 8
// warp sums are then added in warp order into sum[q][x] / csum[t] for
// lane-chunk c of the current batch (valid in warp 0).
template <int EL, int NCOMP, int NSC = 1>
__device__ __forceinline__ void block_sum_chunks(const float *__restrict__ part, int stride_c, int HD,
                                                 const float *__restrict__ parts_c, int H, int LH,
                                                 int32_t c0, int32_t c1, int c, bool active,
                                                 float (*sh)[NCOMP][32 * EL], float (*shc)[NSC][32],
                                                 float (&sum)[NCOMP][EL], float (&csum)[NSC]) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    float x[NCOMP][EL], xc[NSC];
#pragma unroll
    for (int q = 0; q < NCOMP; ++q)
#pragma unroll
        for (int e = 0; e < EL; ++e) x[q][e] = 0.f;
#pragma unroll
    for (int t = 0; t < NSC; ++t) xc[t] = 0.f;
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
            if (parts_c)
#pragma unroll
                for (int t = 0; t < NSC; ++t) xc[t] += parts_c[((size_t)ch * H + c / LH) * NSC + t];
        }
    }
#pragma unroll
    for (int q = 0; q < NCOMP; ++q)
#pragma unroll
        for (int e = 0; e < EL; ++e) sh[w][q][lane * EL + e] = x[q][e];
#pragma unroll
    for (int t = 0; t < NSC; ++t) shc[w][t][lane] = xc[t];
    __syncthreads();
    if (w == 0) {
#pragma unroll
        for (int q = 0; q < NCOMP; ++q)
#pragma unroll
            for (int e = 0; e < EL; ++e) sum[q][e] = 0.f;
#pragma unroll
        for (int t = 0; t < NSC; ++t) csum[t] = 0.f;
        for (int v = 0; v < kWarpsPerBlock; ++v) {
#pragma unroll
            for (int q = 0; q < NCOMP; ++q)
#pragma unroll
                for (int e = 0; e < EL; ++e) sum[q][e] += sh[v][q][lane * EL + e];
#pragma unroll
            for (int t = 0; t < NSC; ++t) csum[t] += shc[v][t][lane];
        }
    }
}

// Row normalisation of the backward pass.  The weights are recomputed as
// p = 2^(s2 - lse2) from the forward's fp32 lse, whose rounding scales a
// whole row's weights by one factor (1 + eps), so they sum to Z = 1 + eps
// rather than 1; left alone, that error reaches the gradients through
// Delta times sum_j p x_j, which does not cancel.  The passes therefore also
// sum Z = sum_j p and use the normalised weights p / Z: Delta = C / Z (C =
// sum p dP), the row sums divided by Z, and lse + ln Z stored for the
// transposed pass, whose recomputed weights are then normalised as well.
struct RowNorm {
    float inv_z, delta, lse_shift;   // 1/Z, C/Z, ln Z
    __device__ __forceinline__ RowNorm(float c, float z) {
        inv_z = z > 0.f ? 1.f / z : 0.f;
        delta = c * inv_z;
        lse_shift = z > 0.f ? logf(z) : 0.f;
    }
};

// Backward: finish split row s in one warp (chunk order).  which == 0: dQ
// rows (C and Z are the sums of the chunk parts, normalised as in the dQ
// pass; Delta and lse + ln Z stored for the dK/dV pass).  which == 1: dK, dV
// of split sources (plain sums).
template <typename T, int D>
__device__ __noinline__ void gt_bwd_merge_row(const GtArgs &a, float scale, int which, int32_t s) {
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16;
    const Partition &P = which == 0 ? a.rows : a.cols;
    const int32_t row = __ldg(P.split_rows + s);
    const int32_t c0 = __ldg(P.chunk_ptr + s), c1 = __ldg(P.chunk_ptr + s + 1);
    const int R = a.H * D / EL, HD = a.H * D;
    for (int c = threadIdx.x & 31; c < R; c += 32) {
        const int h = c / LH;
        float sum[2][EL], cz[2];
        warp_sum_chunks<EL, 2, 2>(which == 0 ? a.ws_row : a.ws_col, 2, HD, which == 0 ? a.ws_rowc : nullptr,
                                  a.H, h, c0, c1, c, sum, cz);
        if (which == 0) {
            const size_t rh = (size_t)row * a.H + h;
            const RowNorm nrm(cz[0] + (a.delta_in ? a.delta_in[rh] : 0.f), cz[1] + (a.z_in ? a.z_in[rh] : 0.f));
            const float sc = scale * nrm.inv_z;
            float o[EL];
#pragma unroll
            for (int x = 0; x < EL; ++x) o[x] = (sum[0][x] - nrm.delta * sum[1][x]) * sc;
            reinterpret_cast<uint4 *>(a.dQ)[(size_t)row * R + c] = pack<T>(o);
            if (c % LH == 0) {
                a.ws_delta[rh] = nrm.delta;
                a.ws_lse[rh] = a.lse[rh] + nrm.lse_shift;
            }
        } else {
#pragma unroll
            for (int x = 0; x < EL; ++x) sum[0][x] *= scale;
            reinterpret_cast<uint4 *>(a.dK)[(size_t)row * R + c] = pack<T>(sum[0]);
            reinterpret_cast<uint4 *>(a.dV)[(size_t)row * R + c] = pack<T>(sum[1]);
        }
    }
}

// ---------------------------------------------------------- backward: dQ

// Per destination row i and edge j: p = 2^(s2 - lse2_i), dP = dOut_i . v_j.
// With Delta_i = sum_j p dP (the exact row term; equal to dOut_i . out_i
// before out is rounded to the storage dtype), dS = p (dP - Delta_i) and
// dQ_i = sum_j dS k_j / sqrt(D) = (A - Delta_i B) / sqrt(D) where
// A = sum_j p dP k_j and B = sum_j p k_j; A, B, C = sum_j p dP and Z =
// sum_j p are accumulated in the same pass over the edges and the weights
// normalised by Z at the end (RowNorm).  Split-row chunks write A, B and
// their parts of C and Z; the merge kernel finishes them in chunk order.
template <typename T, int D, int NC, int G, bool BIAS>
__global__ void __launch_bounds__(256, 2)
gt_bwd_dq_kernel(GtArgs a, float scale2, float scale) {
    using S = GtShape<T, D, NC, G>;
    using C = GtDqStream<T, D, NC, G, BIAS>;
    constexpr int EL = S::EL, LH = S::LH, U = C::U;
    extern __shared__ __align__(16) unsigned char dsmem[];
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    StreamArrays arr{};
    arr.rows[0] = static_cast<const uint4 *>(a.K);
    arr.rows[1] = static_cast<const uint4 *>(a.V);
    arr.own[0] = static_cast<const uint4 *>(a.Q);
    arr.own[1] = static_cast<const uint4 *>(a.dOut);
    arr.osc[0] = a.lse;
    if (BIAS) arr.sc[0] = a.bias;
    EdgeStream<C> st;
    st.init(dsmem + (threadIdx.x >> 5) * C::BYTES, arr, a.rows, a.indptr, a.indices, a.N, a.H, R, LH,
            a.split_threshold, a.d_err);
    StreamItem it;
    while (st.next_item(it)) {
        float q[NC][EL], go[NC][EL], A[NC][EL], B[NC][EL], c[NC], z[NC], lse2[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
#pragma unroll
            for (int x = 0; x < EL; ++x) q[k][x] = go[k][x] = A[k][x] = B[k][x] = 0.f;
            c[k] = z[k] = 0.f;
            lse2[k] = 0.f;
        }
        for (int step = 0; step < it.nsteps; ++step) {
            st.wait_step();
            if (step == 0)
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    unpack<T>(st.own_row(0, k), q[k]);
                    unpack<T>(st.own_row(1, k), go[k]);
                    lse2[k] = st.own_scalar(0, (gl + G * k) / LH) * kLog2e;
                }
            // two-chunk rows take their two neighbours one after the other
            // (unrolled, the pair needs more registers than a thread has)
#pragma unroll(NC >= 2 ? 1 : U)
            for (int u = 0; u < U; ++u) {
                const bool ok = st.valid(u);
                if constexpr (NC == 2) {
                    // the two chunks' head sums split across lane pairs: one
                    // weight per lane, exchanged afterwards
                    float kf[2][EL], sd[2], dv[2];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        float vf[EL];
                        unpack<T>(st.row(u, 0, k), kf[k]);
                        unpack<T>(st.row(u, 1, k), vf);
                        sd[k] = dot2<EL>(q[k], kf[k]);
                        dv[k] = dot2<EL>(go[k], vf);
                    }
                    float sdot, dp;
                    const bool hi = head_sums_split<LH>(sd[0], dv[0], sd[1], dv[1], sdot, dp);
                    float p;
                    if constexpr (BIAS)
                        p = ok ? fast_exp2(sdot * scale2 - (hi ? lse2[1] : lse2[0]) +
                                       st.scalar(u, 0, (gl + G * (hi ? 1 : 0)) / LH) * kLog2e)
                               : 0.f;
                    else
                        p = ok ? fast_exp2(sdot * scale2 - (hi ? lse2[1] : lse2[0])) : 0.f;
                    const float pdp = p * dp;
                    const float po = __shfl_xor_sync(SGA_FULL_MASK, p, LH / 2);
                    const float pdpo = __shfl_xor_sync(SGA_FULL_MASK, pdp, LH / 2);
                    const float p0 = hi ? po : p, p1 = hi ? p : po, d0 = hi ? pdpo : pdp, d1 = hi ? pdp : pdpo;
                    c[0] += d0;
                    c[1] += d1;
                    z[0] += p0;
                    z[1] += p1;
                    axpy2<EL>(A[0], d0, kf[0]);
                    axpy2<EL>(B[0], p0, kf[0]);
                    axpy2<EL>(A[1], d1, kf[1]);
                    axpy2<EL>(B[1], p1, kf[1]);
                } else {
#pragma unroll
                    for (int k = 0; k < NC; ++k) {
                        float kf[EL], vf[EL];
                        unpack<T>(st.row(u, 0, k), kf);
                        unpack<T>(st.row(u, 1, k), vf);
                        float sdot = dot2<EL>(q[k], kf), dp = dot2<EL>(go[k], vf);
                        group_sum2<LH>(sdot, dp);
                        float p;
                        if constexpr (BIAS)
                            p = ok ? fast_exp2(sdot * scale2 - lse2[k] + st.scalar(u, 0, (gl + G * k) / LH) * kLog2e)
                                   : 0.f;
                        else
                            p = ok ? fast_exp2(sdot * scale2 - lse2[k]) : 0.f;
                        const float pdp = p * dp;
                        c[k] += pdp;
                        z[k] += p;
                        axpy2<EL>(A[k], pdp, kf);
                        axpy2<EL>(B[k], p, kf);
                    }
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
                    float4 *dA = reinterpret_cast<float4 *>(a.ws_row + (size_t)it.item * 2 * HD + ch * EL);
                    float4 *dB = reinterpret_cast<float4 *>(a.ws_row + (size_t)it.item * 2 * HD + HD + ch * EL);
#pragma unroll
                    for (int x = 0; x < EL; x += 4) {
                        dA[x / 4] = make_float4(A[k][x], A[k][x + 1], A[k][x + 2], A[k][x + 3]);
                        dB[x / 4] = make_float4(B[k][x], B[k][x + 1], B[k][x + 2], B[k][x + 3]);
                    }
                    if (ch % LH == 0) {
                        a.ws_rowc[((size_t)it.item * a.H + h) * 2] = c[k];
                        a.ws_rowc[((size_t)it.item * a.H + h) * 2 + 1] = z[k];
                    }
                } else {
                    const size_t rh = (size_t)it.row * a.H + h;
                    const RowNorm nrm(c[k] + (a.delta_in ? a.delta_in[rh] : 0.f),
                                      z[k] + (a.z_in ? a.z_in[rh] : 0.f));
                    const float sc = scale * nrm.inv_z;
                    float o[EL];
#pragma unroll
                    for (int x = 0; x < EL; ++x) o[x] = (A[k][x] - nrm.delta * B[k][x]) * sc;
                    reinterpret_cast<uint4 *>(a.dQ)[(size_t)it.row * R + ch] = pack<T>(o);
                    if (ch % LH == 0) {
                        a.ws_delta[rh] = nrm.delta;
                        a.ws_lse[rh] = a.lse[rh] + nrm.lse_shift;
                    }
                }
            }
        }
        if constexpr (gt_fold<NC>()) {
            if (it.partial && last_chunk(a.rows, it.item))
                gt_bwd_merge_row<T, D>(a, scale, 0, __ldg(a.rows.chunk_split + it.item));
        }
        st.finish_item();
    }
    st.drain();
}

// ------------------------------------------------------- backward: dK, dV

// Per source j over its destinations i (transposed CSR):
// p = 2^(s2 - lse2_i), dS = p (dOut_i . v_j - Delta_i),
// dV_j += p dOut_i, dK_j += dS q_i, with the dQ pass's normalised lse_i
// (lse_i + ln Z_i) and Delta_i.
template <typename T, int D, int NC, int G, bool BIAS>
__global__ void __launch_bounds__(256, 2)
gt_bwd_dkdv_kernel(GtArgs a, float scale2, float scale) {
    using S = GtShape<T, D, NC, G>;
    using C = GtDkdvStream<T, D, NC, G, BIAS>;
    constexpr int NG = C::NG, STEP = C::STEP;
    constexpr int EL = S::EL, LH = S::LH, U = C::U;
    extern __shared__ __align__(16) unsigned char dsmem[];
    const int lane = threadIdx.x & 31, g = lane / G, gl = lane % G;
    const int R = a.H * D / EL, HD = a.H * D;
    StreamArrays arr{};
    arr.rows[0] = static_cast<const uint4 *>(a.Q);
    arr.rows[1] = static_cast<const uint4 *>(a.dOut);
    arr.sc[0] = a.ws_lse;     // lse + ln Z of each destination (normalised weights)
    arr.sc[1] = a.ws_delta;
    arr.own[0] = static_cast<const uint4 *>(a.K);
    arr.own[1] = static_cast<const uint4 *>(a.V);
    if (BIAS) arr.sc[2] = a.bias_t;   // the bias in transposed-CSR order
    EdgeStream<C> st;
    st.init(dsmem + (threadIdx.x >> 5) * C::BYTES, arr, a.cols, a.t_indptr, a.t_dst, a.N, a.H, R, LH,
            a.split_threshold, a.d_err);
    StreamItem it;
    while (st.next_item(it)) {
        float kj[NC][EL], vj[NC][EL], dk[NC][EL], dv[NC][EL];
        // transposed position of the item's first edge (bias gradient output)
        int32_t tbeg = 0;
        if (BIAS) tbeg = it.partial ? __ldg(a.cols.chunk_beg + it.item) : __ldg(a.t_indptr + it.row);
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int x = 0; x < EL; ++x) kj[k][x] = vj[k][x] = dk[k][x] = dv[k][x] = 0.f;
        for (int step = 0; step < it.nsteps; ++step) {
            st.wait_step();
            if (step == 0)
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    unpack<T>(st.own_row(0, k), kj[k]);
                    unpack<T>(st.own_row(1, k), vj[k]);
                }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const bool ok = st.valid(u);
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    float qf[EL], gf[EL];
                    unpack<T>(st.row(u, 0, k), qf);
                    unpack<T>(st.row(u, 1, k), gf);
                    float sdot = dot2<EL>(qf, kj[k]), dp = dot2<EL>(gf, vj[k]);
                    group_sum2<LH>(sdot, dp);
                    const int h = (gl + G * k) / LH;
                    float p;
                    if constexpr (BIAS)
                        p = ok ? fast_exp2(sdot * scale2 + (st.scalar(u, 2, h) - st.scalar(u, 0, h)) * kLog2e) : 0.f;
                    else
                        p = ok ? fast_exp2(sdot * scale2 - st.scalar(u, 0, h) * kLog2e) : 0.f;
                    const float ds = p * (dp - st.scalar(u, 1, h));
                    axpy2<EL>(dv[k], p, gf);
                    axpy2<EL>(dk[k], ds, qf);
                    if (BIAS && ok && (gl + G * k) % LH == 0 && gl + G * k < R) {
                        // dL/db = dS, at the edge's position in CSR order
                        const int32_t te = tbeg + step * STEP + g + NG * u;
                        a.dbias[(size_t)__ldg(a.t_eid + te) * a.H + h] = ds;
                    }
                }
            }
            st.release_step();
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
                    float4 *dk_dst = reinterpret_cast<float4 *>(a.ws_col + (size_t)it.item * 2 * HD + c * EL);
                    float4 *dv_dst = reinterpret_cast<float4 *>(a.ws_col + (size_t)it.item * 2 * HD + HD + c * EL);
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
        if constexpr (gt_fold<NC>()) {
            if (it.partial && last_chunk(a.cols, it.item))
                gt_bwd_merge_row<T, D>(a, scale, 1, __ldg(a.cols.chunk_split + it.item));
        }
        st.finish_item();
    }
    st.drain();
}

// Finish split rows, one block each.  which == 0: dQ rows (C and Z = sums of
// the chunk parts, normalised as in the dQ pass, Delta and lse + ln Z stored
// for the dK/dV pass).  which == 1: dK, dV of split sources (plain sums).
template <typename T, int D>
__global__ void __launch_bounds__(256) gt_bwd_merge_kernel(GtArgs a, float scale, int which) {
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16;
    __shared__ float sh[kWarpsPerBlock][2][32 * EL];
    __shared__ float shc[kWarpsPerBlock][2][32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t s = blockIdx.x;
    const Partition &P = which == 0 ? a.rows : a.cols;
    if (s >= P.n_split) return;
    const int32_t row = P.split_rows[s];
    const int32_t c0 = P.chunk_ptr[s], c1 = P.chunk_ptr[s + 1];
    const int R = a.H * D / EL, HD = a.H * D;
    for (int cb = 0; cb < R; cb += 32) {
        const int c = cb + lane;
        float sum[2][EL], cz[2];
        block_sum_chunks<EL, 2, 2>(which == 0 ? a.ws_row : a.ws_col, 2, HD,
                                   which == 0 ? a.ws_rowc : nullptr, a.H, LH, c0, c1, c, c < R, sh,
                                   shc, sum, cz);
        if (w == 0 && c < R) {
            if (which == 0) {
                const size_t rh = (size_t)row * a.H + c / LH;
                const RowNorm nrm(cz[0] + (a.delta_in ? a.delta_in[rh] : 0.f),
                                  cz[1] + (a.z_in ? a.z_in[rh] : 0.f));
                const float sc = scale * nrm.inv_z;
                float o[EL];
#pragma unroll
                for (int x = 0; x < EL; ++x) o[x] = (sum[0][x] - nrm.delta * sum[1][x]) * sc;
                reinterpret_cast<uint4 *>(a.dQ)[(size_t)row * R + c] = pack<T>(o);
                if (c % LH == 0) {
                    a.ws_delta[rh] = nrm.delta;
                    a.ws_lse[rh] = a.lse[rh] + nrm.lse_shift;
                }
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
template <auto Kernel> unsigned persistent_blocks(int64_t items, size_t smem = 0, int warps = kWarpsPerBlock) {
    static int per_sm = -1;   // one cache per kernel instantiation
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (per_sm < 0) {
        if (smem > 48 * 1024)
            cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        int nb = 1;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, Kernel, warps * 32, smem) != cudaSuccess) nb = 1;
        per_sm = nb > 0 ? nb : 1;
    }
    const int64_t full = (int64_t)per_sm * (sms > 0 ? sms : 1);
    const int64_t need = (items + warps - 1) / warps;
    return (unsigned)(need < full ? (need > 0 ? need : 1) : full);
}

// Warps per block of a streamed kernel: eight, fewer when eight rings (and
// the kernel's STATIC bytes of static shared memory) would not fit the 227 KB
// a block may use.
template <typename C, int STATIC = 0> constexpr int stream_warps() {
    constexpr int fit = (227 * 1024 - STATIC) / C::BYTES;
    return fit >= kWarpsPerBlock ? kWarpsPerBlock : (fit > 0 ? fit : 1);
}

// Zero the partition's item counter before a launch whose stream takes its
// items dynamically (StreamCfg::DYN).
template <typename C> cudaError_t reset_items(const Partition &P, cudaStream_t s) {
    if constexpr (C::DYN) return cudaMemsetAsync(P.next, 0, sizeof(int32_t), s);
    return cudaSuccess;
}

// Launch a persistent streamed kernel over `items` work items.
template <typename C, auto Kernel, typename... Args>
cudaError_t launch_streamed(int64_t items, cudaStream_t s, Args... args) {
    constexpr int warps = stream_warps<C>();
    static_assert((size_t)C::BYTES * warps <= 227 * 1024, "one warp's ring must fit a block");
    constexpr size_t smem = (size_t)C::BYTES * warps;
    Kernel<<<persistent_blocks<Kernel>(items, smem, warps), warps * 32, smem, s>>>(args...);
    return cudaGetLastError();
}

// The same with a fixed grid (kernels that leave one partial per block).
template <typename C, auto Kernel, int STATIC, typename... Args>
cudaError_t launch_streamed_grid(unsigned grid, cudaStream_t s, Args... args) {
    constexpr int warps = stream_warps<C, STATIC>();
    static_assert((size_t)C::BYTES * warps + STATIC <= 227 * 1024, "one warp's ring must fit a block");
    constexpr size_t smem = (size_t)C::BYTES * warps;
    static bool configured = false;
    if (!configured) {
        if (smem > 48 * 1024) {
            const cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
        }
        configured = true;
    }
    Kernel<<<grid, warps * 32, smem, s>>>(args...);
    return cudaGetLastError();
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

template <typename T, int D, bool BIAS, bool LIST> cudaError_t gt_fwd_db(const GtArgs &a, cudaStream_t s) {
    constexpr int LH = D * (int)sizeof(T) / 16;
    const int R = a.H * D / Elt<T>::EL;
    const float scale2 = kLog2e / sqrtf((float)D);
    const int64_t items = (int64_t)a.rows.n_chunks + a.N;
    bool folded = false;   // the edge kernel merges the split rows itself
    cudaError_t e = dispatch_shape<LH, max_nc<T>()>(R, [&]<int NC, int G>() -> cudaError_t {
        folded = LIST && gt_fold<NC>();
        if (items == 0) return cudaSuccess;
        if (reset_items<GtFwdStream<T, D, NC, G, BIAS, LIST>>(a.rows, s) != cudaSuccess) return cudaGetLastError();
        note_launch(SGA_KERN_GT_FWD, s, false);
        const cudaError_t e =
            launch_streamed<GtFwdStream<T, D, NC, G, BIAS, LIST>, gt_fwd_kernel<T, D, NC, G, BIAS, LIST>>(
                items, s, a, scale2);
        note_launch(SGA_KERN_GT_FWD, s, true);
        return e;
    });
    if (e != cudaSuccess || a.rows.n_split == 0 || folded) return e;
    note_launch(SGA_KERN_GT_FWD_MERGE, s, false);
    gt_fwd_merge_kernel<T, D, GtArgs><<<(unsigned)a.rows.n_split, 256, 0, s>>>(a);
    note_launch(SGA_KERN_GT_FWD_MERGE, s, true);
    return cudaGetLastError();
}

template <typename T, int D> cudaError_t gt_fwd_d(const GtArgs &a, cudaStream_t s) {
    if (!a.rows.items) return gt_fwd_db<T, D, false, false>(a, s);   // no plan: no bias either
    return a.bias ? gt_fwd_db<T, D, true, true>(a, s) : gt_fwd_db<T, D, false, true>(a, s);
}

// bias_t[te, h] = bias[t_eid[te], h]: the score bias in transposed-CSR order
static __global__ void bias_transpose_kernel(const float *__restrict__ bias, const int32_t *__restrict__ t_eid,
                                      int64_t E, int H, float *__restrict__ bias_t) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t n = E * H;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += stride) {
        const int64_t te = x / H;
        bias_t[x] = bias[(size_t)__ldg(t_eid + te) * H + (x - te * H)];
    }
}

template <typename T, int D, bool BIAS> cudaError_t gt_bwd_db(const GtArgs &a, cudaStream_t s) {
    constexpr int LH = D * (int)sizeof(T) / 16;
    const int R = a.H * D / Elt<T>::EL;
    const float scale = 1.0f / sqrtf((float)D);
    const float scale2 = kLog2e * scale;
    return dispatch_shape<LH, max_nc<T>()>(R, [&]<int NC, int G>() -> cudaError_t {
        const int64_t items_r = (int64_t)a.rows.n_chunks + a.N;
        const int64_t items_c = (int64_t)a.cols.n_chunks + a.N;
        if (items_r == 0) return cudaSuccess;
        if (BIAS) {
            const int64_t n = a.E * a.H;
            if (n > 0) {
                const unsigned g = (unsigned)std::min<int64_t>((n + 255) / 256, 8192);
                bias_transpose_kernel<<<g, 256, 0, s>>>(a.bias, a.t_eid, a.E, a.H, a.bias_t);
                const cudaError_t e0 = cudaGetLastError();
                if (e0 != cudaSuccess) return e0;
            }
        }
        if (reset_items<GtDqStream<T, D, NC, G, BIAS>>(a.rows, s) != cudaSuccess) return cudaGetLastError();
        note_launch(SGA_KERN_GT_BWD_DQ, s, false);
        cudaError_t e = launch_streamed<GtDqStream<T, D, NC, G, BIAS>, gt_bwd_dq_kernel<T, D, NC, G, BIAS>>(
            items_r, s, a, scale2, scale);
        note_launch(SGA_KERN_GT_BWD_DQ, s, true);
        if (e != cudaSuccess) return e;
        if (!gt_fold<NC>() && a.rows.n_split > 0) {   // Delta of split rows is needed by the dK/dV pass
            note_launch(SGA_KERN_GT_BWD_MERGE, s, false);
            gt_bwd_merge_kernel<T, D><<<(unsigned)a.rows.n_split, 256, 0, s>>>(a, scale, 0);
            note_launch(SGA_KERN_GT_BWD_MERGE, s, true);
            if ((e = cudaGetLastError()) != cudaSuccess) return e;
        }
        if (reset_items<GtDkdvStream<T, D, NC, G, BIAS>>(a.cols, s) != cudaSuccess) return cudaGetLastError();
        note_launch(SGA_KERN_GT_BWD_DKDV, s, false);
        e = launch_streamed<GtDkdvStream<T, D, NC, G, BIAS>, gt_bwd_dkdv_kernel<T, D, NC, G, BIAS>>(
            items_c, s, a, scale2, scale);
        note_launch(SGA_KERN_GT_BWD_DKDV, s, true);
        if (e != cudaSuccess) return e;
        if (!gt_fold<NC>() && a.cols.n_split > 0) {
            note_launch(SGA_KERN_GT_BWD_MERGE, s, false);
            gt_bwd_merge_kernel<T, D><<<(unsigned)a.cols.n_split, 256, 0, s>>>(a, scale, 1);
            note_launch(SGA_KERN_GT_BWD_MERGE, s, true);
            e = cudaGetLastError();
        }
        return e;
    });
}

template <typename T, int D> cudaError_t gt_bwd_d(const GtArgs &a, cudaStream_t s) {
    return a.bias ? gt_bwd_db<T, D, true>(a, s) : gt_bwd_db<T, D, false>(a, s);
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
