// Block-sparse Graph Transformer backward on the tcgen05 tensor cores, the
// FlashAttention-2 style backward that the IO-aware layers blog post
// ("Attention-based layers" paragraph) pairs with the block-sparse tensor-core
// variant.  For a kept tile edge (i, j), with s = q_i . k_j / sqrt(D):
//   p = exp(s - lse_i),  dP = dOut_i . v_j,  dS = p (dP - Delta_i),
//   dQ_i += dS k_j / sqrt(D),  dK_j += dS q_i / sqrt(D),  dV_j += p dOut_i,
// with Delta_i = sum over all edges of row i of p dP.  The weights are
// normalised to sum to one per row (the residual CSR pass divides by
// Z = sum p over all of the row's edges and stores lse + ln Z, which the dQ and
// dK/dV passes here use): the Delta pass returns the tile parts of
// sum p dP and of Z.
//
// Three passes, each one CTA of 4 warps per (panel, head); all products on
// the tensor cores with fp32 accumulators in TMEM:
//   Delta pass (per row panel, groups of four kept tiles = 64 sources):
//     S = Q K^T, dP = dOut V^T, the row sums of p dP and of p over tile edges;
//   dQ pass (same loop, Delta known): dS to shared memory as a pair of bf16
//     tiles (hi = bf16(dS), lo = bf16(dS - hi): about 16 significant bits),
//     dQ += dS_hi K + dS_lo K;
//   dK/dV pass (per column panel of 128 sources, over the row panels that
//     keep one of its tiles, 64 rows at a time):
//     S^T = K Q^T, dP^T = V dOut^T, P^T and the dS^T pair to shared memory,
//     dV += P^T dOut, dK += dS^T_hi Q + dS^T_lo Q.
// dS is split because it cancels: a row's dS sum to zero, so a single bf16
// rounding of every term (2^-9 relative) leaves dQ and dK errors of 2^-9 times
// the sum of |dS k| terms, which is far larger than the result where scores
// or dP are large.  P (non-negative) and the node rows stay single bf16.
// Node rows are staged once, 128-byte swizzled with 64-wide column atoms: the
// K-major operand over D of the S and dP products, and as they stand the
// MN-major operand over D of the dQ, dV and dK products (no transposes).
// The residual CSR passes run in between (their Delta includes the tile part), so
// each pass here adds its tile part to gradients already stored.  No atomics:
// every output row is owned by one CTA, and the results are deterministic.
#include "common.cuh"
#include "plan.h"
#include "tc.cuh"

namespace sga {
namespace {

constexpr int kThreads = 128;
constexpr int kGroup = 64;   // sources per group of the row passes (four tiles)

// Rows row0 .. row0 + R - 1 of head h of a [N, H, D] bf16 tensor into a
// swizzled K-major tile of R rows (zero rows past N).
template <int D>
__device__ __forceinline__ void load_rows(uint32_t dst, const __nv_bfloat16 *X, int64_t row0, int R,
                                          int64_t N, int H, int h) {
    constexpr int DC = D / 8;
    for (int idx = threadIdx.x; idx < R * DC; idx += kThreads) {
        const int rr = idx / DC, c = idx % DC;
        const bool ok = row0 + rr < N;
        tc::cp16(dst + tc::sw128_offset(rr, c * 8, R), ok ? X + ((row0 + rr) * H + h) * D + c * 8 : X, ok);
    }
}

// The 64 source rows of kept tiles t .. t + 3 (rows of missing tiles and
// sources past N are zero).
template <int D>
__device__ __forceinline__ void load_tile_rows(uint32_t dst, const __nv_bfloat16 *X, const int32_t *tile_col,
                                               int32_t t, int32_t t_end, int64_t N, int H, int h) {
    constexpr int DC = D / 8;
    for (int idx = threadIdx.x; idx < kGroup * DC; idx += kThreads) {
        const int jr = idx / DC, c = idx % DC;
        const int32_t ti = t + jr / 16;
        const int64_t j = ti < t_end ? (int64_t)tile_col[ti] * 16 + (jr % 16) : -1;
        const bool ok = j >= 0 && j < N;
        tc::cp16(dst + tc::sw128_offset(jr, c * 8, kGroup), ok ? X + (j * H + h) * D + c * 8 : X, ok);
    }
}

// Four k-steps over 64 node rows (K = 64): A K-major (one 64-wide atom of the
// A tile), B the 64 node rows x N columns as an MN-major operand.
__device__ __forceinline__ void mma_rows64(uint32_t tmem, uint32_t a, uint32_t b_rows, uint32_t idesc, bool first) {
    for (int kk = 0; kk < 4; ++kk)
        tc::mma_bf16_ss(tmem, tc::desc_sw128(a + kk * 32), tc::desc_sw128_mn(b_rows + kk * 2048, 64 * 128), idesc,
                        (!first || kk > 0) ? 1u : 0u);
}

// D/16 k-steps of a 128 x N product with both operands K-major over D
// (A: 128 rows, B: RB rows).
__device__ __forceinline__ void mma_over_d(uint32_t tmem, uint32_t a, uint32_t b, int RB, int D,
                                           uint32_t idesc) {
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ao = (uint32_t)((kk >> 2) * 128 * 128 + (kk & 3) * 32);
        const uint32_t bo = (uint32_t)((kk >> 2) * RB * 128 + (kk & 3) * 32);
        tc::mma_bf16_ss(tmem, tc::desc_sw128(a + ao), tc::desc_sw128(b + bo), idesc, kk > 0);
    }
}

// Eight fp32 values as a bf16 pair: hi = the nearest bf16, lo = the nearest
// bf16 of the remainder (x - hi is exact in fp32).
__device__ __forceinline__ void split_bf16x8(const float *x, uint4 &hi, uint4 &lo) {
    float h[8], r[8];
    hi = pack<__nv_bfloat16>(x);
    unpack<__nv_bfloat16>(hi, h);
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = x[i] - h[i];
    lo = pack<__nv_bfloat16>(r);
}

// Add an fp32 row (from TMEM, times `scale`) to a bf16 row of D values.
template <int D>
__device__ __forceinline__ void add_row_from_tmem(uint32_t taddr, __nv_bfloat16 *dst, float scale, bool has) {
    for (int cb = 0; cb < D; cb += 32) {
        uint32_t u[32];
        tc::tmem_ld32(taddr + cb, u);   // warp-collective: every lane takes part
        if (!has) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float o[8], x[8];
            unpack<__nv_bfloat16>(*reinterpret_cast<const uint4 *>(dst + cb + 8 * q), x);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = x[i] + scale * __uint_as_float(u[8 * q + i]);
            *reinterpret_cast<uint4 *>(dst + cb + 8 * q) = pack<__nv_bfloat16>(o);
        }
    }
}

// ------------------------------------------------------------ row passes

// The Delta pass keeps one K/V buffer (the next group loads once the S and dP
// products have consumed it), so that two of its CTAs share an SM; the dQ
// pass, above half an SM's shared memory either way, keeps two.
__host__ __device__ constexpr int row_buffers(int mode) { return mode == 0 ? 1 : 2; }

struct RowLayout {   // byte offsets in dynamic shared memory (1024-aligned base)
    uint32_t q, g, k[2], v[2], ds, ds_lo, total;
    __host__ __device__ RowLayout(int D, int mode) {
        const uint32_t DA = (uint32_t)D / 64, NB = (uint32_t)row_buffers(mode);
        q = 0;
        g = q + DA * 128 * 128;
        k[0] = g + DA * 128 * 128;
        k[1] = k[0] + (NB - 1) * DA * kGroup * 128;
        v[0] = k[1] + DA * kGroup * 128;
        v[1] = v[0] + (NB - 1) * DA * kGroup * 128;
        ds = v[1] + DA * kGroup * 128;
        ds_lo = ds + (mode == 1 ? 128 * 128 : 0);
        total = ds_lo + (mode == 1 ? 128 * 128 : 0);
    }
};

// MODE 0: Delta pass (writes delta_t, z_t).  MODE 1: dQ pass (adds to dQ).
template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1) bsr_bwd_row_kernel(BsrBwdArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t mbar_s, mbar_o;
    __shared__ uint32_t tmem_base;
    const RowLayout L(D, MODE);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int panel = blockIdx.x, h = blockIdx.y, H = a.H;
    const int32_t t0 = a.tile_ptr[panel], t1 = a.tile_ptr[panel + 1];
    const int ng = (t1 - t0 + 3) / 4;
    if (ng == 0) return;   // whole CTA: no kept tile

    const int64_t r0 = (int64_t)panel * 128, row = r0 + tid;
    const bool in = row < a.N;
    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(a.Q);
    const __nv_bfloat16 *K = static_cast<const __nv_bfloat16 *>(a.K);
    const __nv_bfloat16 *V = static_cast<const __nv_bfloat16 *>(a.V);
    const __nv_bfloat16 *G = static_cast<const __nv_bfloat16 *>(a.dOut);
    const uint32_t sbase = tc::smem_u32(smem);

    if (warp == 0) tc::tmem_alloc(&tmem_base, 256);
    if (tid == 0) {
        tc::mbar_init(&mbar_s, 1);
        tc::mbar_init(&mbar_o, 1);
    }
    load_rows<D>(sbase + L.q, Q, r0, 128, a.N, H, h);
    load_rows<D>(sbase + L.g, G, r0, 128, a.N, H, h);
    load_tile_rows<D>(sbase + L.k[0], K, a.tile_col, t0, t1, a.N, H, h);
    load_tile_rows<D>(sbase + L.v[0], V, a.tile_col, t0, t1, a.N, H, h);
    tc::cp_commit();
    // the Delta pass uses the forward's lse and sums C and Z of its tile edges;
    // the dQ pass uses the normalised lse + ln Z and Delta = C / Z of the row
    const float lse2 = in ? (MODE == 0 ? a.lse : a.lse_n)[row * H + h] * kLog2e : 0.f;
    const float dl = (MODE == 1 && in) ? a.delta[row * H + h] : 0.f;
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tS = tmem_base, tP = tmem_base + 64, tQ = tmem_base + 128;
    const uint32_t tlane = (uint32_t)(warp * 32) << 16;
    const uint32_t idesc_s = tc::idesc_bf16(128, kGroup), idesc_q = tc::idesc_bf16(128, D) | tc::kMajorMnB;
    const float scale2 = kLog2e * rsqrtf((float)D);

    float dsum = 0.f, zsum = 0.f;
    bool failed = false;
    int n_o = 0;   // dQ products issued (uniform over the CTA)
    constexpr int NB = row_buffers(MODE);
    for (int g = 0; g < ng; ++g) {
        const int b = NB == 2 ? (g & 1) : 0;
        // the previous dS K product reads dS and the other K buffer: it must be done first
        if (MODE == 1 && g > 0 && !tc::mbar_wait(&mbar_o, (g - 1) & 1, tc::kWaitLimit)) failed = true;
        if (__syncthreads_or(failed)) break;
        if (NB == 2 && g + 1 < ng) {
            load_tile_rows<D>(sbase + L.k[b ^ 1], K, a.tile_col, t0 + 4 * (g + 1), t1, a.N, H, h);
            load_tile_rows<D>(sbase + L.v[b ^ 1], V, a.tile_col, t0 + 4 * (g + 1), t1, a.N, H, h);
            tc::cp_commit();
            tc::cp_wait<1>();
        } else {
            tc::cp_wait<0>();
        }
        tc::fence_after_sync();
        tc::fence_proxy_async();
        __syncthreads();
        if (tid == 0) {   // S = Q K^T, dP = dOut V^T
            tc::fence_after_sync();
            mma_over_d(tS, sbase + L.q, sbase + L.k[b], kGroup, D, idesc_s);
            mma_over_d(tP, sbase + L.g, sbase + L.v[b], kGroup, D, idesc_s);
            tc::mma_commit(&mbar_s);
        }
        if (!tc::mbar_wait(&mbar_s, g & 1, tc::kWaitLimit)) failed = true;
        if (__syncthreads_or(failed)) break;
        tc::fence_after_sync();
        if (NB == 1 && g + 1 < ng) {   // K and V consumed: the next group loads during the softmax
            load_tile_rows<D>(sbase + L.k[0], K, a.tile_col, t0 + 4 * (g + 1), t1, a.N, H, h);
            load_tile_rows<D>(sbase + L.v[0], V, a.tile_col, t0 + 4 * (g + 1), t1, a.N, H, h);
            tc::cp_commit();
        }

        uint32_t bits[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int32_t ti = t0 + 4 * g + q;
            bits[q] = (ti < t1 && in) ? a.tile_bits[(size_t)ti * 128 + tid] : 0u;
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t us[32], up[32];
            tc::tmem_ld32(tS + tlane + half * 32, us);
            tc::tmem_ld32(tP + tlane + half * 32, up);
            float ds[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int c = half * 32 + i;
                const bool on = (bits[c >> 4] >> (c & 15)) & 1u;
                const float p = on ? exp2f(__uint_as_float(us[i]) * scale2 - lse2) : 0.f;
                const float dp = __uint_as_float(up[i]);
                if (MODE == 0) {
                    dsum = fmaf(p, dp, dsum);
                    zsum += p;
                }
                ds[i] = p * (dp - dl);
            }
            if (MODE == 1) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t o = tc::sw128_offset(tid, half * 32 + c * 8, 128);
                    uint4 hi, lo;
                    split_bf16x8(ds + 8 * c, hi, lo);
                    *reinterpret_cast<uint4 *>(smem + L.ds + o) = hi;
                    *reinterpret_cast<uint4 *>(smem + L.ds_lo + o) = lo;
                }
            }
        }
        tc::fence_before_sync();
        if (MODE == 1) {
            tc::fence_proxy_async();
            __syncthreads();
            if (tid == 0) {   // dQ += dS_hi K + dS_lo K
                tc::fence_after_sync();
                mma_rows64(tQ, sbase + L.ds, sbase + L.k[b], idesc_q, g == 0);
                mma_rows64(tQ, sbase + L.ds_lo, sbase + L.k[b], idesc_q, false);
                tc::mma_commit(&mbar_o);
            }
            ++n_o;
        }
    }
    tc::cp_wait<0>();
    if (MODE == 1 && !failed && !tc::mbar_wait(&mbar_o, (ng - 1) & 1, tc::kWaitLimit)) failed = true;
    failed = __syncthreads_or(failed);
    if (failed) {
        if (tid == 0) atomicOr(a.d_err, tc::kErrMmaTimeout);
        if (MODE == 1 && n_o > 0) tc::mbar_wait(&mbar_o, (n_o - 1) & 1, tc::kWaitLimit);
    } else if (MODE == 0) {
        if (in) {
            a.delta_t[row * H + h] = dsum;
            a.z_t[row * H + h] = zsum;
        }
    } else {
        tc::fence_after_sync();
        __nv_bfloat16 *dq = static_cast<__nv_bfloat16 *>(a.dQ) + (row * H + h) * D;
        add_row_from_tmem<D>(tQ + tlane, dq, rsqrtf((float)D), in);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem_base, 256);
}

// ----------------------------------------------------------- column pass

struct ColLayout {   // byte offsets in dynamic shared memory (1024-aligned base)
    uint32_t kc, vc, qh[2], gh[2], p, ds, ds_lo, bits[2], lse[2], dl[2], total;
    __host__ __device__ ColLayout(int D) {
        const uint32_t DA = (uint32_t)D / 64;
        kc = 0;
        vc = kc + DA * 128 * 128;
        qh[0] = vc + DA * 128 * 128;
        qh[1] = qh[0] + DA * 64 * 128;
        gh[0] = qh[1] + DA * 64 * 128;
        gh[1] = gh[0] + DA * 64 * 128;
        p = gh[1] + DA * 64 * 128;
        ds = p + 128 * 128;
        ds_lo = ds + 128 * 128;
        bits[0] = ds_lo + 128 * 128;  // 8 tiles x 64 rows x 16 bits
        bits[1] = bits[0] + 1024;
        lse[0] = bits[1] + 1024;      // 64 fp32
        lse[1] = lse[0] + 256;
        dl[0] = lse[1] + 256;
        dl[1] = dl[0] + 256;
        total = dl[1] + 256;
    }
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) bsr_bwd_col_kernel(BsrBwdArgs a) {
    constexpr uint32_t kCols = D == 128 ? 512 : 256;   // S^T, dP^T (64 each), dV, dK (D each)
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t mbar_s, mbar_o;
    __shared__ uint32_t tmem_base;
    const ColLayout L(D);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int cp = blockIdx.x, h = blockIdx.y, H = a.H;
    const int32_t e0 = a.ct_ptr[cp], e1 = a.ct_ptr[cp + 1];
    const int nu = 2 * (e1 - e0);   // units: (entry, 64-row half)
    if (nu == 0) return;            // whole CTA: no kept tile in these columns

    const int64_t c0 = (int64_t)cp * 128, src = c0 + tid;
    const bool in = src < a.N;
    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(a.Q);
    const __nv_bfloat16 *K = static_cast<const __nv_bfloat16 *>(a.K);
    const __nv_bfloat16 *V = static_cast<const __nv_bfloat16 *>(a.V);
    const __nv_bfloat16 *G = static_cast<const __nv_bfloat16 *>(a.dOut);
    const uint32_t sbase = tc::smem_u32(smem);

    if (warp == 0) tc::tmem_alloc(&tmem_base, kCols);
    if (tid == 0) {
        tc::mbar_init(&mbar_s, 1);
        tc::mbar_init(&mbar_o, 1);
    }
    // rows of one unit: Q and dOut of 64 destinations, their masks, lse, Delta
    auto load_unit = [&](int u, int b) {
        const int32_t e = e0 + u / 2;
        const int hf = u & 1;
        const int64_t row0 = (int64_t)a.ct_panel[e] * 128 + hf * 64;
        load_rows<D>(sbase + L.qh[b], Q, row0, 64, a.N, H, h);
        load_rows<D>(sbase + L.gh[b], G, row0, 64, a.N, H, h);
        if (tid < 64) {   // 8 tiles x 8 chunks of 8 rows
            const int t = tid >> 3, ch = tid & 7;
            const int32_t tile = a.ct_tile[(size_t)e * 8 + t];
            const bool ok = tile >= 0;
            tc::cp16(sbase + L.bits[b] + (uint32_t)(t * 64 + ch * 8) * 2,
                     ok ? a.tile_bits + (size_t)tile * 128 + hf * 64 + ch * 8 : a.tile_bits, ok);
        } else {
            const int i = tid - 64;
            const bool ok = row0 + i < a.N;
            const size_t off = ok ? (size_t)(row0 + i) * H + h : 0;
            tc::cp4(sbase + L.lse[b] + i * 4, a.lse_n + off, ok);
            tc::cp4(sbase + L.dl[b] + i * 4, a.delta + off, ok);
        }
        tc::cp_commit();
    };
    load_rows<D>(sbase + L.kc, K, c0, 128, a.N, H, h);
    load_rows<D>(sbase + L.vc, V, c0, 128, a.N, H, h);
    load_unit(0, 0);   // the column rows travel in the first group
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tS = tmem_base, tP = tmem_base + 64, tV = tmem_base + 128, tK = tmem_base + 128 + D;
    const uint32_t tlane = (uint32_t)(warp * 32) << 16;
    const uint32_t idesc_s = tc::idesc_bf16(128, 64), idesc_d = tc::idesc_bf16(128, D) | tc::kMajorMnB;
    const float scale2 = kLog2e * rsqrtf((float)D);

    bool failed = false;
    int n_o = 0;
    for (int u = 0; u < nu; ++u) {
        const int b = u & 1;
        // the previous dV / dK products read P^T, dS^T and the other unit's dOut and Q rows
        if (u > 0 && !tc::mbar_wait(&mbar_o, (u - 1) & 1, tc::kWaitLimit)) failed = true;
        if (__syncthreads_or(failed)) break;
        if (u + 1 < nu) {
            load_unit(u + 1, b ^ 1);
            tc::cp_wait<1>();
        } else {
            tc::cp_wait<0>();
        }
        tc::fence_after_sync();
        tc::fence_proxy_async();
        __syncthreads();
        if (tid == 0) {   // S^T = K Q^T, dP^T = V dOut^T
            tc::fence_after_sync();
            mma_over_d(tS, sbase + L.kc, sbase + L.qh[b], 64, D, idesc_s);
            mma_over_d(tP, sbase + L.vc, sbase + L.gh[b], 64, D, idesc_s);
            tc::mma_commit(&mbar_s);
        }
        if (!tc::mbar_wait(&mbar_s, u & 1, tc::kWaitLimit)) failed = true;
        if (__syncthreads_or(failed)) break;
        tc::fence_after_sync();

        const uint16_t *bits = reinterpret_cast<const uint16_t *>(smem + L.bits[b]) + (tid >> 4) * 64;
        const float *lse = reinterpret_cast<const float *>(smem + L.lse[b]);
        const float *dl = reinterpret_cast<const float *>(smem + L.dl[b]);
        const int bit = tid & 15;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            uint32_t us[32], up[32];
            tc::tmem_ld32(tS + tlane + half * 32, us);
            tc::tmem_ld32(tP + tlane + half * 32, up);
            float pv[32], ds[32];
#pragma unroll
            for (int ii = 0; ii < 32; ++ii) {
                const int i = half * 32 + ii;
                const bool on = in && ((bits[i] >> bit) & 1u);
                const float p = on ? exp2f(__uint_as_float(us[ii]) * scale2 - lse[i] * kLog2e) : 0.f;
                pv[ii] = p;
                ds[ii] = p * (__uint_as_float(up[ii]) - dl[i]);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t o = tc::sw128_offset(tid, half * 32 + c * 8, 128);
                uint4 hi, lo;
                split_bf16x8(ds + 8 * c, hi, lo);
                *reinterpret_cast<uint4 *>(smem + L.p + o) = pack<__nv_bfloat16>(pv + 8 * c);
                *reinterpret_cast<uint4 *>(smem + L.ds + o) = hi;
                *reinterpret_cast<uint4 *>(smem + L.ds_lo + o) = lo;
            }
        }
        tc::fence_before_sync();
        tc::fence_proxy_async();
        __syncthreads();
        if (tid == 0) {   // dV += P^T dOut, dK += dS^T_hi Q + dS^T_lo Q
            tc::fence_after_sync();
            mma_rows64(tV, sbase + L.p, sbase + L.gh[b], idesc_d, u == 0);
            mma_rows64(tK, sbase + L.ds, sbase + L.qh[b], idesc_d, u == 0);
            mma_rows64(tK, sbase + L.ds_lo, sbase + L.qh[b], idesc_d, false);
            tc::mma_commit(&mbar_o);
        }
        ++n_o;
    }
    tc::cp_wait<0>();
    if (!failed && !tc::mbar_wait(&mbar_o, (nu - 1) & 1, tc::kWaitLimit)) failed = true;
    failed = __syncthreads_or(failed);
    if (failed) {
        if (tid == 0) atomicOr(a.d_err, tc::kErrMmaTimeout);
        if (n_o > 0) tc::mbar_wait(&mbar_o, (n_o - 1) & 1, tc::kWaitLimit);
    } else {
        tc::fence_after_sync();
        const size_t off = ((size_t)src * H + h) * D;
        add_row_from_tmem<D>(tK + tlane, static_cast<__nv_bfloat16 *>(a.dK) + (in ? off : 0),
                             rsqrtf((float)D), in);
        add_row_from_tmem<D>(tV + tlane, static_cast<__nv_bfloat16 *>(a.dV) + (in ? off : 0), 1.f, in);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem_base, kCols);
}

// ---------------------------------------------------------------- launch

// At least 100 KB of shared memory per CTA: at most two CTAs (two 256-column
// TMEM allocations) share an SM; the 512-column dK/dV CTA needs more than
// half of the SM's shared memory, so it runs alone.
template <auto Kernel>
cudaError_t launch(const BsrBwdArgs &a, dim3 grid, size_t bytes, sga_kernel_id id, cudaStream_t s) {
    const size_t smem = bytes + 1024 > 100 * 1024 ? bytes + 1024 : 100 * 1024;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    note_launch(id, s, false);
    Kernel<<<grid, kThreads, smem, s>>>(a);
    note_launch(id, s, true);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bsr_bwd_delta(const BsrBwdArgs &a, cudaStream_t s) {
    if (a.n_panels == 0) return cudaSuccess;
    const dim3 grid((unsigned)a.n_panels, (unsigned)a.H);
    const size_t bytes = RowLayout(a.D, 0).total;
    return a.D == 128 ? launch<bsr_bwd_row_kernel<128, 0>>(a, grid, bytes, SGA_KERN_BSR_BWD_DELTA, s)
                      : launch<bsr_bwd_row_kernel<64, 0>>(a, grid, bytes, SGA_KERN_BSR_BWD_DELTA, s);
}

cudaError_t launch_bsr_bwd_dq(const BsrBwdArgs &a, cudaStream_t s) {
    if (a.n_panels == 0) return cudaSuccess;
    const dim3 grid((unsigned)a.n_panels, (unsigned)a.H);
    const size_t bytes = RowLayout(a.D, 1).total;
    return a.D == 128 ? launch<bsr_bwd_row_kernel<128, 1>>(a, grid, bytes, SGA_KERN_BSR_BWD_DQ, s)
                      : launch<bsr_bwd_row_kernel<64, 1>>(a, grid, bytes, SGA_KERN_BSR_BWD_DQ, s);
}

cudaError_t launch_bsr_bwd_dkdv(const BsrBwdArgs &a, cudaStream_t s) {
    if (a.n_cpanels == 0) return cudaSuccess;
    const dim3 grid((unsigned)a.n_cpanels, (unsigned)a.H);
    const size_t bytes = ColLayout(a.D).total;
    return a.D == 128 ? launch<bsr_bwd_col_kernel<128>>(a, grid, bytes, SGA_KERN_BSR_BWD_DKDV, s)
                      : launch<bsr_bwd_col_kernel<64>>(a, grid, bytes, SGA_KERN_BSR_BWD_DKDV, s);
}

}  // namespace sga
