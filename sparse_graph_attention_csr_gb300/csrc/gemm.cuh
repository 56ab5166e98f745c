// Dense GEMMs of the GATv2 layer on the tensor cores (bf16 mma.sync, fp32
// accumulate): the projections FL = X W_l, FR = X W_r, the input gradient
// dX = dFL W_l^T + dFR W_r^T and the weight gradients dW = X^T dF (split-K
// over node slabs, fp32 partials reduced in a fixed order).
//
// Operands are staged through shared memory in their global layout and read
// with ldmatrix (.trans for M- or N-major tiles).  fp32 operands (dFL, dFR)
// are split into bf16 hi + lo parts (hi = bf16(x), lo = bf16(x - hi)), so each
// product keeps about 16 significant bits; the two parts take two MMAs.
//
// Exact projections: FL/FR are stored in bf16 and decide LeakyReLU branches
// downstream, so they are rounded correctly.  The fp32 accumulation of a
// k-term dot product x . w differs from the exact value by a small multiple
// of 2^-24 |x||w| (measured: at most 0.6 for sequential fp32 sums of the
// GATv2 workload).  When every value within B = 2 * 2^-24 |x||w| + ulp of the
// fp32 result rounds to the same bf16 number, that number is correct;
// otherwise (about 0.35% of elements for unit-scale data) the dot product is
// recomputed with error-free transformations in fp32 -- by one warp per
// element from the shared-memory tiles when k <= 128, else by
// exact_round_kernel from a workspace list: bf16 x bf16 products
// are exact in fp32 and a TwoSum cascade carries the rounding error of every
// addition, so hi + lo equals the exact sum to far below bf16 resolution.
// The result is rounded to float, then to bf16 (ties to even).
#pragma once

#include "common.cuh"

namespace sga {

namespace mm {

constexpr int BM = 128, BN = 128, BK = 64, THREADS = 256;
constexpr int PAD = 8;   // bf16 elements of row padding: conflict-free ldmatrix

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// 16-byte global -> shared copy that bypasses registers; `ok` false zero-fills.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool ok) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src),
                 "r"(ok ? 16 : 0));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N));
}

// bf16 hi part and remainder of 8 floats.
__device__ __forceinline__ void split8(const uint4 &u0, const uint4 &u1, uint4 &hi, uint4 &lo) {
    float x[8], h[8], l[8];
    unpack<float>(u0, x);
    unpack<float>(u1, x + 4);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        h[i] = __bfloat162float(__float2bfloat16_rn(x[i]));
        l[i] = x[i] - h[i];
    }
    hi = pack<__nv_bfloat16>(h);
    lo = pack<__nv_bfloat16>(l);
}

}  // namespace mm

// C = sum_p op(A_p) op(B_p).  AM: A stored [K][M] (else [M][K]); BN_MAJOR: B
// stored [K][N] (else [N][K]).  MODE 0: bf16 C, correctly rounded (one pair,
// bf16 operands); MODE 1: C in TC rounded to nearest; MODE 2: fp32 partial
// Cpart[slab][M][N] over the K rows of slab blockIdx.z.
template <typename TA, typename TB, typename TC, bool AM, bool BN_MAJOR, int MODE>
struct MmaGemm {
    const TA *A[4];
    const TB *B[4];
    int pairs;                // 1 .. 4
    int64_t M, N, K, k_per_slab;
    int64_t lda, ldb;         // leading dimensions (elements); 0: packed (M or K, N or K)
    TC *C;
    float *Cpart;
    // MODE 0: elements whose rounding the fp32 sum leaves open are listed here
    // (row, column | tag << 16) for exact_round_kernel; tag names the output.
    int32_t *fix_count;
    int2 *fix_list;
    int32_t fix_cap, fix_tag;
};

// Exact fp32 sum of the products x_k w_k of bf16 inputs (each product is exact
// in fp32) for k = k0, k0 + step, ...: TwoSum keeps every addition's rounding
// error in `lo`, so hi + lo is the sum to about 2^-48 relative.
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// One operand tile of one k chunk: 1024 chunks of 8 elements, 4 per thread.
// MAJ (the tile's rows are k) selects [BK][BX+PAD]; else [BX][BK+PAD].
template <bool MAJ, int BX> struct TileMap {
    __device__ static void at(int c, int &r, int &col) {   // chunk c -> (smem row, col)
        if (MAJ) { r = c / (BX / 8); col = (c % (BX / 8)) * 8; }
        else     { r = c / (mm::BK / 8); col = (c % (mm::BK / 8)) * 8; }
    }
    static constexpr int LD = MAJ ? BX + mm::PAD : mm::BK + mm::PAD;
    static constexpr int ELEMS = MAJ ? mm::BK * (BX + mm::PAD) : BX * (mm::BK + mm::PAD);
};

template <typename TA, typename TB, typename TC, bool AM, bool BN_MAJOR, int MODE>
__global__ void __launch_bounds__(mm::THREADS, MODE == 0 ? 1 : 2)
mma_gemm_kernel(MmaGemm<TA, TB, TC, AM, BN_MAJOR, MODE> g) {
    using namespace mm;
    constexpr bool SA = sizeof(TA) == 4, SB = sizeof(TB) == 4;   // fp32 operands split hi/lo
    constexpr int NA = SA ? 2 : 1, NB = SB ? 2 : 1;
    using MA = TileMap<AM, BM>;
    using MB = TileMap<BN_MAJOR, BN>;
    constexpr int STAGE = NA * MA::ELEMS + NB * MB::ELEMS;   // bf16 elements per stage
    extern __shared__ __align__(16) __nv_bfloat16 smem[];
    __shared__ float rnorm[BM], cnorm[BN];
    constexpr int kFixSh = 512;
    __shared__ int2 fix_sh[MODE == 0 ? kFixSh : 1];
    __shared__ int fix_n, fix_base;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp & 3, wn = warp >> 2;          // warp tile 32 x 64
    if (MODE == 0 && tid == 0) fix_n = 0;
    const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * BN;
    const int64_t k_lo = (int64_t)blockIdx.z * g.k_per_slab;
    const int64_t k_hi = min(g.K, k_lo + g.k_per_slab);
    const int per_pair = k_hi > k_lo ? (int)((k_hi - k_lo + BK - 1) / BK) : 0;
    const int n_chunks = per_pair * g.pairs;

    const int64_t lda = g.lda ? g.lda : (AM ? g.M : g.K), ldb = g.ldb ? g.ldb : (BN_MAJOR ? g.N : g.K);
    // global element (row-of-tile, col-of-tile) of chunk c of the current k chunk
    auto a_src = [&](int p, int64_t kb, int c, bool &ok) -> const TA * {
        int r, col;
        MA::at(c, r, col);
        int64_t gm, gk;
        if (AM) { gk = kb + r; gm = m0 + col; } else { gm = m0 + r; gk = kb + col; }
        ok = gm < g.M && gk < k_hi;
        return ok ? g.A[p] + (AM ? gk * lda + gm : gm * lda + gk) : g.A[p];
    };
    auto b_src = [&](int p, int64_t kb, int c, bool &ok) -> const TB * {
        int r, col;
        MB::at(c, r, col);
        int64_t gn, gk;
        if (BN_MAJOR) { gk = kb + r; gn = n0 + col; } else { gn = n0 + r; gk = kb + col; }
        ok = gn < g.N && gk < k_hi;
        return ok ? g.B[p] + (BN_MAJOR ? gk * ldb + gn : gn * ldb + gk) : g.B[p];
    };
    __nv_bfloat16 *stage_base[2] = {smem, smem + STAGE};
    // fp32 operand chunks held in registers between load and store
    uint4 ra[SA ? 8 : 1], rb[SB ? 8 : 1];

    auto issue = [&](int chunk, int st) {   // start loading chunk into stage st
        const int p = chunk / per_pair;
        const int64_t kb = k_lo + (int64_t)(chunk % per_pair) * BK;
        __nv_bfloat16 *As = stage_base[st], *Bs = stage_base[st] + NA * MA::ELEMS;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = tid + i * THREADS;
            int r, col;
            bool ok;
            MA::at(c, r, col);
            const TA *src = a_src(p, kb, c, ok);
            if constexpr (SA) {
                ra[2 * i] = ok ? ldg16(src) : make_uint4(0, 0, 0, 0);
                ra[2 * i + 1] = ok ? ldg16(src + 4) : make_uint4(0, 0, 0, 0);
            } else {
                cp_async16(&As[r * MA::LD + col], src, ok);
            }
            MB::at(c, r, col);
            const TB *srcb = b_src(p, kb, c, ok);
            if constexpr (SB) {
                rb[2 * i] = ok ? ldg16(srcb) : make_uint4(0, 0, 0, 0);
                rb[2 * i + 1] = ok ? ldg16(srcb + 4) : make_uint4(0, 0, 0, 0);
            } else {
                cp_async16(&Bs[r * MB::LD + col], srcb, ok);
            }
        }
        cp_async_commit();
    };
    auto store_regs = [&](int st) {          // fp32 chunks: split and store
        __nv_bfloat16 *As = stage_base[st], *Bs = stage_base[st] + NA * MA::ELEMS;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int c = tid + i * THREADS;
            int r, col;
            if constexpr (SA) {
                MA::at(c, r, col);
                uint4 hi, lo;
                split8(ra[2 * i], ra[2 * i + 1], hi, lo);
                *reinterpret_cast<uint4 *>(&As[r * MA::LD + col]) = hi;
                *reinterpret_cast<uint4 *>(&As[MA::ELEMS + r * MA::LD + col]) = lo;
            }
            if constexpr (SB) {
                MB::at(c, r, col);
                uint4 hi, lo;
                split8(rb[2 * i], rb[2 * i + 1], hi, lo);
                *reinterpret_cast<uint4 *>(&Bs[r * MB::LD + col]) = hi;
                *reinterpret_cast<uint4 *>(&Bs[MB::ELEMS + r * MB::LD + col]) = lo;
            }
        }
    };

    float acc[2][8][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[i][j][r] = 0.f;
    float rsq = 0.f, csq = 0.f;   // MODE 0: squared norms (row tid/2, column tid%128)

    if (n_chunks > 0) {
        issue(0, 0);
        if (SA || SB) store_regs(0);
    }
    for (int ch = 0; ch < n_chunks; ++ch) {
        const int cur = ch & 1;
        const bool more = ch + 1 < n_chunks;
        if (more) issue(ch + 1, cur ^ 1);
        if (more) cp_async_wait<1>(); else cp_async_wait<0>();
        __syncthreads();
        const __nv_bfloat16 *As = stage_base[cur], *Bs = stage_base[cur] + NA * MA::ELEMS;
        if (MODE == 0) {   // squared norms of the A rows and B columns, k in order
            if (!AM) {
                const __nv_bfloat16 *row = &As[(tid >> 1) * MA::LD + (tid & 1) * 32];
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    const float v = __bfloat162float(row[x]);
                    rsq = fmaf(v, v, rsq);
                }
            }
            if (BN_MAJOR) {
                const int col = tid & 127, k0 = (tid >> 7) * 32;
#pragma unroll
                for (int x = 0; x < 32; ++x) {
                    const float v = __bfloat162float(Bs[(k0 + x) * MB::LD + col]);
                    csq = fmaf(v, v, csq);
                }
            }
        }
#pragma unroll
        for (int ks = 0; ks < BK; ks += 16) {
#pragma unroll
            for (int ia = 0; ia < NA; ++ia)
#pragma unroll
                for (int ib = 0; ib < NB; ++ib) {
                    const __nv_bfloat16 *Ai = As + ia * MA::ELEMS, *Bi = Bs + ib * MB::ELEMS;
                    uint32_t af[2][4];
#pragma unroll
                    for (int mi = 0; mi < 2; ++mi) {
                        const int mb = wm * 32 + mi * 16;
                        if (AM) {
                            const int kr = ks + (lane & 7) + ((lane >> 4) << 3);
                            const int mc = mb + (((lane >> 3) & 1) << 3);
                            ldsm_x4_t(af[mi], &Ai[kr * MA::LD + mc]);
                        } else {
                            const int mr = mb + (lane & 15);
                            const int kc = ks + ((lane >> 4) << 3);
                            ldsm_x4(af[mi], &Ai[mr * MA::LD + kc]);
                        }
                    }
#pragma unroll
                    for (int nj = 0; nj < 8; nj += 2) {
                        const int nb = wn * 64 + nj * 8;
                        uint32_t bf[4];
                        if (BN_MAJOR) {
                            const int kr = ks + (lane & 7) + (((lane >> 3) & 1) << 3);
                            const int nc = nb + ((lane >> 4) << 3);
                            ldsm_x4_t(bf, &Bi[kr * MB::LD + nc]);
                        } else {
                            const int nr = nb + (lane & 7) + ((lane >> 4) << 3);
                            const int kc = ks + (((lane >> 3) & 1) << 3);
                            ldsm_x4(bf, &Bi[nr * MB::LD + kc]);
                        }
#pragma unroll
                        for (int mi = 0; mi < 2; ++mi) {
                            mma_bf16(acc[mi][nj], af[mi], bf[0], bf[1]);
                            mma_bf16(acc[mi][nj + 1], af[mi], bf[2], bf[3]);
                        }
                    }
                }
        }
        __syncthreads();
        if (more && (SA || SB)) store_regs(cur ^ 1);
    }

    if (MODE == 0) {
        rsq += __shfl_xor_sync(SGA_FULL_MASK, rsq, 1);
        if ((tid & 1) == 0) rnorm[tid >> 1] = rsq;
        if (tid >= 128) cnorm[tid & 127] = csq;
        __syncthreads();
        if (tid < 128) cnorm[tid] = sqrtf(cnorm[tid] + csq);
        if (tid < 128) rnorm[tid] = sqrtf(rnorm[tid]);
        __syncthreads();
    }

    // ---- epilogue: thread holds rows (lane/4, +8), columns 2*(lane%4) + {0,1}
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            const int lr = wm * 32 + mi * 16 + (lane >> 2) + hr * 8;
            const int64_t gm = m0 + lr;
            if (gm >= g.M) continue;
#pragma unroll
            for (int nj = 0; nj < 8; ++nj) {
                const int lc = wn * 64 + nj * 8 + (lane & 3) * 2;
                const int64_t gn = n0 + lc;
                if (gn >= g.N) continue;   // N is a multiple of 8: both columns valid
                float v0 = acc[mi][nj][hr * 2], v1 = acc[mi][nj][hr * 2 + 1];
                if (MODE == 2) {
                    *reinterpret_cast<float2 *>(&g.Cpart[((int64_t)blockIdx.z * g.M + gm) * g.N + gn]) =
                        make_float2(v0, v1);
                    continue;
                }
                if (MODE == 0) {   // flag sums whose bf16 rounding is open (see header)
                    const float rn = rnorm[lr] * (2.0f * 5.9604645e-8f);
                    const float vv[2] = {v0, v1};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const float bound = rn * cnorm[lc + e] + fabsf(vv[e]) * 1.2e-7f;
                        if (__float2bfloat16_rn(vv[e] - bound) != __float2bfloat16_rn(vv[e] + bound)) {
                            const int slot = atomicAdd(&fix_n, 1);
                            if (slot < kFixSh) {
                                fix_sh[slot] = make_int2(lr, lc + e);
                            } else {   // shared list full (not expected): exact sum in place
                                float sh = 0.f, sl = 0.f;
                                for (int64_t k = 0; k < g.K; ++k) {
                                    const float x = to_f32<TA>(g.A[0][gm * g.K + k]);
                                    const float w = to_f32<TB>(g.B[0][k * g.N + gn + e]);
                                    float t, err;
                                    two_sum(sh, __fmul_rn(x, w), t, err);
                                    sh = t;
                                    sl = __fadd_rn(sl, err);
                                }
                                (e == 0 ? v0 : v1) = __fadd_rn(sh, sl);
                            }
                        }
                    }
                }
                TC *dst = g.C + gm * g.N + gn;
                dst[0] = from_f32<TC>(v0);
                dst[1] = from_f32<TC>(v1);
            }
        }
    if (MODE == 0) {   // exact recompute of the flagged elements
        static_assert(MODE != 0 || (!AM && BN_MAJOR), "projection layout: X [M][K], W [K][N]");
        __syncthreads();
        const int n = min(fix_n, kFixSh);
        if (g.K <= 2 * BK && g.pairs == 1) {
            // the whole k range is still in the two stages: one warp per element
            for (int i = warp; i < n; i += THREADS / 32) {
                const int lr = fix_sh[i].x, lc = fix_sh[i].y;
                float hi = 0.f, lo = 0.f;
                for (int k = lane; k < g.K; k += 32) {
                    const __nv_bfloat16 *As = stage_base[k / BK];
                    const __nv_bfloat16 *Bs = stage_base[k / BK] + NA * MA::ELEMS;
                    const float x = __bfloat162float(As[lr * MA::LD + (k % BK)]);
                    const float w = __bfloat162float(Bs[(k % BK) * MB::LD + lc]);
                    float t, err;
                    two_sum(hi, __fmul_rn(x, w), t, err);
                    hi = t;
                    lo = __fadd_rn(lo, err);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ho = __shfl_xor_sync(SGA_FULL_MASK, hi, o);
                    const float lo2 = __shfl_xor_sync(SGA_FULL_MASK, lo, o);
                    float t, err;
                    two_sum(hi, ho, t, err);
                    hi = t;
                    lo = __fadd_rn(__fadd_rn(lo, lo2), err);
                }
                if (lane == 0) g.C[(m0 + lr) * g.N + n0 + lc] = from_f32<TC>(__fadd_rn(hi, lo));
            }
        } else {
            // k range too long for shared memory (or list overflow): exact_round_kernel
            if (tid == 0) fix_base = n ? atomicAdd(g.fix_count, n) : 0;
            __syncthreads();
            for (int i = tid; i < n; i += THREADS) {
                const int2 f = fix_sh[i];
                const int at = fix_base + i;
                const int64_t gm = m0 + f.x, gn = n0 + f.y;
                if (at < g.fix_cap) {
                    g.fix_list[at] = make_int2((int)gm, (int)gn | (g.fix_tag << 16));
                } else {   // list full (not expected): exact sum in place
                    float sh = 0.f, sl = 0.f;
                    for (int64_t k = 0; k < g.K; ++k) {
                        const float x = to_f32<TA>(g.A[0][gm * g.K + k]);
                        const float w = to_f32<TB>(g.B[0][k * g.N + gn]);
                        float t, err;
                        two_sum(sh, __fmul_rn(x, w), t, err);
                        sh = t;
                        sl = __fadd_rn(sl, err);
                    }
                    g.C[gm * g.N + gn] = from_f32<TC>(__fadd_rn(sh, sl));
                }
            }
        }
    }
}

// Recompute the listed elements exactly, one warp each: lanes split k, each
// keeps an error-free (hi, lo) sum, and the lane sums are combined with
// TwoSum as well.  X [M][K]; W_t [K][N] for tag t; C_t [M][N] bf16.
struct ExactRound {
    const __nv_bfloat16 *X;
    const __nv_bfloat16 *W[2];
    __nv_bfloat16 *C[2];
    int64_t M, N, K;
    const int32_t *count;
    const int2 *list;
    int32_t cap;
};

static __global__ void __launch_bounds__(256) exact_round_kernel(ExactRound r) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int n = min(*r.count, r.cap);
    for (int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < n; i += nw) {
        const int2 f = r.list[i];
        const int64_t m = f.x, col = f.y & 0xffff;
        const int t = f.y >> 16;
        float hi = 0.f, lo = 0.f;
        for (int64_t k = lane; k < r.K; k += 32) {
            const float x = __bfloat162float(r.X[m * r.K + k]);
            const float w = __bfloat162float(r.W[t][k * r.N + col]);
            float s, e;
            two_sum(hi, __fmul_rn(x, w), s, e);
            hi = s;
            lo = __fadd_rn(lo, e);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ho = __shfl_xor_sync(SGA_FULL_MASK, hi, o);
            const float lo2 = __shfl_xor_sync(SGA_FULL_MASK, lo, o);
            float s, e;
            two_sum(hi, ho, s, e);
            hi = s;
            lo = __fadd_rn(__fadd_rn(lo, lo2), e);
        }
        if (lane == 0) r.C[t][m * r.N + col] = __float2bfloat16_rn(__fadd_rn(hi, lo));
    }
}

template <typename TA, typename TB, typename TC, bool AM, bool BN_MAJOR, int MODE>
cudaError_t mma_gemm(const MmaGemm<TA, TB, TC, AM, BN_MAJOR, MODE> &g, int slabs,
                     sga_kernel_id kid, cudaStream_t s) {
    constexpr int NA = sizeof(TA) == 4 ? 2 : 1, NB = sizeof(TB) == 4 ? 2 : 1;
    constexpr size_t smem = 2 * sizeof(__nv_bfloat16) *
                            (NA * TileMap<AM, mm::BM>::ELEMS + NB * TileMap<BN_MAJOR, mm::BN>::ELEMS);
    static bool configured = false;   // one per instantiation
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(mma_gemm_kernel<TA, TB, TC, AM, BN_MAJOR, MODE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid((unsigned)((g.N + mm::BN - 1) / mm::BN), (unsigned)((g.M + mm::BM - 1) / mm::BM),
              (unsigned)slabs);
    note_launch(kid, s, false);
    mma_gemm_kernel<TA, TB, TC, AM, BN_MAJOR, MODE><<<grid, mm::THREADS, smem, s>>>(g);
    note_launch(kid, s, true);
    return cudaGetLastError();
}

}  // namespace sga
