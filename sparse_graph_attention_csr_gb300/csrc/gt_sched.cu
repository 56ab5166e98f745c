// Alternative thread mappings of the Graph Transformer forward, kept as
// measured comparison points for the default edge stream (gt.cuh).
//
// The pages contrast neighbour-parallel and feature-parallel designs ("On
// Efficient Scaling of GNNs via IO-Aware Layers Implementations", arXiv
// abstract: graph reordering "benefits neighbor-parallel (gather-dominated)
// kernels more consistently than feature-parallel designs"), and DF-GNN's
// abstract schedules the score stage and the aggregation stage of an
// attention layer with different thread mappings ("bi-level thread
// scheduling").  Two such mappings are written here:
//
//  - SGA_SCHED_FEATURE: one warp per work item, lanes across the row's
//    features (16-byte chunks of H*D), neighbours taken one at a time with
//    direct loads: the dot product is a shuffle reduction over the lanes of a
//    head, the softmax is updated every edge, and the value row is loaded
//    right after the key row.  No shared-memory staging.
//  - SGA_SCHED_BILEVEL: scores edge-parallel, aggregation feature-parallel.
//    The item's query row is staged in shared memory; lane l takes edge l of
//    a batch of 32 and computes all H scores of its edge alone (reading its
//    own key row in 16-byte pieces); the batch maximum and sum per head are
//    warp reductions; the weights go to shared memory; then lanes switch to
//    features and accumulate the batch's value rows (one coalesced load per
//    edge and chunk).
//
// Both walk the same work items as the edge stream (chunks of split rows
// first, then every row of degree <= the split threshold) and write the same
// chunk partials (running maximum and sum in log2 units, unnormalised
// accumulator), so the split-row merge kernel finishes them unchanged.
#include "common.cuh"
#include "gt.cuh"
#include "items.cuh"
#include "plan.h"

namespace sga {
namespace {

// Finish one item: normalised output and lse for a whole row, or the chunk
// partial for a chunk of a split row.  Lane chunk c of the row holds acc[k]
// for c = lane + 32 k; (m, l) are the head's running max and sum (log2).
template <typename T, int NC>
__device__ __forceinline__ void finish_item(const GtArgs &a, const ItemRange &r, int64_t item, int R, int LH,
                                            const float (&acc)[NC][Elt<T>::EL], const float (&m)[NC],
                                            const float (&l)[NC]) {
    constexpr int EL = Elt<T>::EL;
    const int lane = threadIdx.x & 31, HD = R * EL;
#pragma unroll
    for (int k = 0; k < NC; ++k) {
        const int c = lane + 32 * k;
        if (c >= R) continue;
        const int h = c / LH;
        if (r.partial) {
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
            reinterpret_cast<uint4 *>(a.out_w)[(size_t)r.row * R + c] = pack<T>(o);
            if (c % LH == 0)
                a.lse_w[(size_t)r.row * a.H + h] = l[k] > 0.f ? (m[k] + log2f(l[k])) * kLn2 : -INFINITY;
        }
    }
}

// ---------------------------------------------------------- feature-parallel

template <typename T, int D, int NC>
__global__ void __launch_bounds__(256) gt_fwd_feature_kernel(GtArgs a, float scale2) {
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16;
    const int lane = threadIdx.x & 31;
    const int R = a.H * D / EL;
    const uint4 *Kr = static_cast<const uint4 *>(a.K);
    const uint4 *Vr = static_cast<const uint4 *>(a.V);
    const uint4 *Qr = static_cast<const uint4 *>(a.Q);
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t n_items = (int64_t)a.rows.n_chunks + a.N;
    for (int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); item < n_items;
         item += stride) {
        ItemRange r;
        if (!decode_item(item, a.rows, a.indptr, a.N, a.split_threshold, r)) continue;
        float q[NC][EL], acc[NC][EL], m[NC], l[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
            const int c = lane + 32 * k;
            if (c < R) unpack<T>(ldg16(Qr + (size_t)r.row * R + c), q[k]);
            else
#pragma unroll
                for (int x = 0; x < EL; ++x) q[k][x] = 0.f;
#pragma unroll
            for (int x = 0; x < EL; ++x) acc[k][x] = 0.f;
            m[k] = -INFINITY;
            l[k] = 0.f;
        }
        for (int32_t e0 = r.beg; e0 < r.end; e0 += 32) {
            const int cnt = min(32, r.end - e0);
            const int32_t ids = load_ids(a.indices, e0, cnt, a.N, a.d_err);
            for (int t = 0; t < cnt; ++t) {
                const int32_t j = __shfl_sync(SGA_FULL_MASK, ids, t);
                if (j < 0) continue;   // out-of-range id: skipped and flagged
                uint4 kr[NC], vr[NC];
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    const int c = lane + 32 * k;
                    const bool ok = c < R;
                    kr[k] = ok ? ldg16_stream(Kr + (size_t)j * R + c) : make_uint4(0, 0, 0, 0);
                    vr[k] = ok ? ldg16_stream(Vr + (size_t)j * R + c) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    float kf[EL], vf[EL];
                    unpack<T>(kr[k], kf);
                    unpack<T>(vr[k], vf);
                    const float s = group_sum<LH>(dot2<EL>(q[k], kf)) * scale2;
                    const float mn = fmaxf(m[k], s);
                    const float alpha = exp2_diff(m[k], mn), p = fast_exp2(s - mn);
                    l[k] = l[k] * alpha + p;
#pragma unroll
                    for (int x = 0; x < EL; ++x) acc[k][x] = fmaf(p, vf[x], acc[k][x] * alpha);
                    m[k] = mn;
                }
            }
        }
        finish_item<T, NC>(a, r, item, R, LH, acc, m, l);
    }
}

// ------------------------------------------------------------------ bi-level

constexpr int kMaxHeads = 32;   // H <= 1024 / 32

template <typename T, int D, int NC>
__global__ void __launch_bounds__(256) gt_fwd_bilevel_kernel(GtArgs a, float scale2) {
    constexpr int EL = Elt<T>::EL, LH = D * (int)sizeof(T) / 16, DC = D / EL;
    // per warp: query row (H*D fp32), batch weights [32 edges][H], head max / sum
    extern __shared__ __align__(16) float sm_f[];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int H = a.H, R = H * DC, HD = H * D;
    float *q_s = sm_f + (size_t)w * (HD + 32 * H + 2 * kMaxHeads);
    float *p_s = q_s + HD;
    float *m_s = p_s + 32 * H, *l_s = m_s + kMaxHeads;
    const uint4 *Kr = static_cast<const uint4 *>(a.K);
    const uint4 *Vr = static_cast<const uint4 *>(a.V);
    const uint4 *Qr = static_cast<const uint4 *>(a.Q);
    const int64_t stride = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t n_items = (int64_t)a.rows.n_chunks + a.N;
    for (int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + w; item < n_items; item += stride) {
        ItemRange r;
        if (!decode_item(item, a.rows, a.indptr, a.N, a.split_threshold, r)) continue;
        __syncwarp();
        for (int c = lane; c < R; c += 32) {
            float qf[EL];
            unpack<T>(ldg16(Qr + (size_t)r.row * R + c), qf);
#pragma unroll
            for (int x = 0; x < EL; ++x) q_s[c * EL + x] = qf[x] * scale2;
        }
        for (int h = lane; h < H; h += 32) {
            m_s[h] = -INFINITY;
            l_s[h] = 0.f;
        }
        float acc[NC][EL];
#pragma unroll
        for (int k = 0; k < NC; ++k)
#pragma unroll
            for (int x = 0; x < EL; ++x) acc[k][x] = 0.f;
        __syncwarp();
        for (int32_t e0 = r.beg; e0 < r.end; e0 += 32) {
            const int cnt = min(32, r.end - e0);
            const int32_t j = load_ids(a.indices, e0, cnt, a.N, a.d_err);
            // (1) scores, one edge per lane, all heads; log2 units
            for (int h = 0; h < H; ++h) {
                float s = -INFINITY;
                if (j >= 0) {
                    float acc_s = 0.f;
#pragma unroll 4
                    for (int c = 0; c < DC; ++c) {
                        float kf[EL];
                        unpack<T>(ldg16(Kr + (size_t)j * R + h * DC + c), kf);
                        acc_s += dot2<EL>(q_s + h * D + c * EL, kf);
                    }
                    s = acc_s;
                }
                // (2) batch softmax statistics of head h (warp reductions)
                float mx = s;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(SGA_FULL_MASK, mx, o));
                const float m_old = m_s[h];
                const float m_new = fmaxf(m_old, mx);
                const float p = exp2_diff(s, m_new);
                float ps = p;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(SGA_FULL_MASK, ps, o);
                p_s[lane * H + h] = p;
                __syncwarp();
                if (lane == 0) {
                    l_s[h] = l_s[h] * exp2_diff(m_old, m_new) + ps;
                    m_s[h] = m_new;
                }
                // rescale this head's accumulator chunks
                const float alpha = exp2_diff(m_old, m_new);
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    const int c = lane + 32 * k;
                    if (c < R && c / LH == h)
#pragma unroll
                        for (int x = 0; x < EL; ++x) acc[k][x] *= alpha;
                }
            }
            __syncwarp();
            // (3) aggregation, lanes across features, one edge after another
            for (int t = 0; t < cnt; ++t) {
                const int32_t jt = __shfl_sync(SGA_FULL_MASK, j, t);
                if (jt < 0) continue;
#pragma unroll
                for (int k = 0; k < NC; ++k) {
                    const int c = lane + 32 * k;
                    if (c >= R) continue;
                    const float p = p_s[t * H + c / LH];
                    float vf[EL];
                    unpack<T>(ldg16_stream(Vr + (size_t)jt * R + c), vf);
                    axpy2<EL>(acc[k], p, vf);
                }
            }
            __syncwarp();
        }
        float m[NC], l[NC];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
            const int c = lane + 32 * k;
            const int h = c < R ? c / LH : 0;
            m[k] = m_s[h];
            l[k] = l_s[h];
        }
        finish_item<T, NC>(a, r, item, R, LH, acc, m, l);
    }
}

template <auto Kernel> unsigned grid_of(int64_t items, size_t smem) {
    return persistent_blocks<Kernel>(items, smem, kWarpsPerBlock);
}

}  // namespace

template <typename T, int D> cudaError_t gt_fwd_sched_d(const GtArgs &a, int schedule, cudaStream_t s) {
    const int R = a.H * D / Elt<T>::EL;
    const float scale2 = kLog2e / sqrtf((float)D);
    const int64_t items = (int64_t)a.rows.n_chunks + a.N;
    cudaError_t e = cudaSuccess;
    if (items > 0) {
        note_launch(SGA_KERN_GT_FWD, s, false);
        auto go = [&]<int NC>() {
            if (schedule == SGA_SCHED_FEATURE) {
                gt_fwd_feature_kernel<T, D, NC><<<grid_of<gt_fwd_feature_kernel<T, D, NC>>(items, 0), 256, 0, s>>>(
                    a, scale2);
            } else {
                const size_t smem = (size_t)kWarpsPerBlock * 4 * (a.H * D + 32 * a.H + 2 * kMaxHeads);
                static bool configured = false;
                if (!configured) {
                    cudaFuncSetAttribute(gt_fwd_bilevel_kernel<T, D, NC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
                    configured = true;
                }
                gt_fwd_bilevel_kernel<T, D, NC>
                    <<<grid_of<gt_fwd_bilevel_kernel<T, D, NC>>(items, smem), 256, smem, s>>>(a, scale2);
            }
        };
        // lanes across features: NC = ceil(R / 32) chunks per lane
        if (R <= 32) go.template operator()<1>();
        else if (R <= 64) go.template operator()<2>();
        else if (R <= 128) go.template operator()<4>();
        else go.template operator()<8>();
        e = cudaGetLastError();
        note_launch(SGA_KERN_GT_FWD, s, true);
    }
    if (e != cudaSuccess || a.rows.n_split == 0) return e;
    note_launch(SGA_KERN_GT_FWD_MERGE, s, false);
    gt_fwd_merge_kernel<T, D, GtArgs><<<(unsigned)a.rows.n_split, 256, 0, s>>>(a);
    note_launch(SGA_KERN_GT_FWD_MERGE, s, true);
    return cudaGetLastError();
}

template <typename T> cudaError_t gt_fwd_sched_t(const GtArgs &a, int schedule, cudaStream_t s) {
    switch (a.D) {
        case 32: return gt_fwd_sched_d<T, 32>(a, schedule, s);
        case 64: return gt_fwd_sched_d<T, 64>(a, schedule, s);
        case 128: return gt_fwd_sched_d<T, 128>(a, schedule, s);
    }
    return cudaErrorInvalidValue;
}

template cudaError_t gt_fwd_sched_t<float>(const GtArgs &, int, cudaStream_t);
template cudaError_t gt_fwd_sched_t<__nv_bfloat16>(const GtArgs &, int, cudaStream_t);

}  // namespace sga
