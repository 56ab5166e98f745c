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
// Three passes, each a persistent kernel (one CTA per SM) with the same
// roles as the forward: warp 0 one lane issues TMA loads into a ring of
// stages, warp 1 one lane issues the MMAs (fp32 accumulators in TMEM), warps
// 2-9 (thread = TMEM lane, two warps per lane quarter, each taking half of a
// group's columns) turn the products into weights and gradients; every
// handoff is an mbarrier and every wait is bounded.
//   Delta pass (units: row panel x head, groups of four kept tiles = 64
//     sources): S = Q K^T, dP = dOut V^T into two TMEM buffers (the next
//     group's products run while the current one is reduced); the row sums
//     of p dP and of p over tile edges;
//   dQ pass (same loop, Delta known): dS to shared memory as a pair of bf16
//     tiles (hi = bf16(dS), lo = bf16(dS - hi): about 16 significant bits),
//     dQ += dS_hi K + dS_lo K in TMEM, issued after the next group's S and dP;
//   dK/dV pass (units: column panel of 128 sources x head, over the row
//     panels that keep one of its tiles, 64 rows at a time):
//     S^T = K Q^T, dP^T = V dOut^T, P^T and the dS^T pair to shared memory,
//     dV += P^T dOut, dK += dS^T_hi Q + dS^T_lo Q.
// dS is split because it cancels: a row's dS sum to zero, so a single bf16
// rounding of every term (2^-9 relative) leaves dQ and dK errors of 2^-9 times
// the sum of |dS k| terms, which is far larger than the result where scores
// or dP are large.  P (non-negative) and the node rows stay single bf16.
// Node rows are staged by TMA, 128-byte swizzled with 64-wide column atoms:
// the K-major operand over D of the S and dP products, and as they stand the
// MN-major operand over D of the dQ, dV and dK products (no transposes).
// The residual CSR passes run in between (their Delta includes the tile part), so
// each pass here adds its tile part to gradients already stored.  No atomics:
// every output row is owned by one unit, and the results are deterministic.
#include <cuda.h>

#include "common.cuh"
#include "plan.h"
#include "tc.cuh"
#include "tc_dx.cuh"

namespace sga {
namespace {

constexpr int kThreads = 320;   // producer, MMA lane, eight weight warps
constexpr int kSoft = 8;        // weight warps: arrivals per handoff
constexpr int kGroup = 64;      // sources per group of the row passes (four tiles)

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

// Add an fp32 row (from TMEM, times `scale`) to NCOL bf16 values: the row's
// current values are loaded first, all at once (one round trip).
template <int D>
__device__ __forceinline__ void add_row_from_tmem(uint32_t taddr, __nv_bfloat16 *dst, float scale, bool has) {
    uint4 x[D / 8];
    if (has)
#pragma unroll
        for (int c = 0; c < D / 8; ++c) x[c] = *reinterpret_cast<const uint4 *>(dst + 8 * c);
#pragma unroll
    for (int cb = 0; cb < D; cb += 32) {
        uint32_t u[32];
        tc::tmem_ld32(taddr + cb, u);   // warp-collective: every lane takes part
        if (!has) continue;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float o[8], y[8];
            unpack<__nv_bfloat16>(x[cb / 8 + q], y);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = y[i] + scale * __uint_as_float(u[8 * q + i]);
            *reinterpret_cast<uint4 *>(dst + cb + 8 * q) = pack<__nv_bfloat16>(o);
        }
    }
}

// Add an fp32 row (from TMEM, times `scale`) to the NCOL bf16 values of one
// row of a staged TMA box (128-byte rows, 16-byte chunks swizzled by the row
// index mod 8); every lane takes part in the TMEM loads.
template <int NCOL>
__device__ __forceinline__ void add_box_from_tmem(uint32_t taddr, unsigned char *box_row, int row, float scale) {
#pragma unroll
    for (int cb = 0; cb < NCOL; cb += 32) {
        uint32_t u[32];
        tc::tmem_ld32(taddr + cb, u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 *ptr = reinterpret_cast<uint4 *>(box_row + (((cb / 8 + q) ^ (row & 7)) << 4));
            float o[8], y[8];
            unpack<__nv_bfloat16>(*ptr, y);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[i] = y[i] + scale * __uint_as_float(u[8 * q + i]);
            *ptr = pack<__nv_bfloat16>(o);
        }
    }
}

// L2 prefetch of a bf16 row of D values (read again at the end of the unit).
template <int D> __device__ __forceinline__ void prefetch_row(const __nv_bfloat16 *row) {
#pragma unroll
    for (int b = 0; b < D * 2; b += 128) tc::prefetch_l2(reinterpret_cast<const char *>(row) + b);
}

// ------------------------------------------------------------ row passes

template <int D, int MODE> struct RowCfg {
    static constexpr int DA = D / 64;
    static constexpr uint32_t PB = DA * 128 * 128;       // a 128-row panel tile (Q or dOut)
    static constexpr uint32_t KB = DA * kGroup * 128;    // K or V rows of a group
    // panel buffers (two: the next unit's panel loads during this one) and
    // K/V stages, within the shared memory of one SM
    static constexpr int NQ = (D == 64 || MODE == 0) ? 2 : 1;
    static constexpr int NST = D == 64 ? 3 : (MODE == 0 ? 2 : 3);
    static constexpr uint32_t Q0 = 0;                    // buffer b: Q, then dOut
    static constexpr uint32_t ST0 = Q0 + NQ * 2 * PB;    // stage s: K, then V
    static constexpr uint32_t DS0 = ST0 + NST * 2 * KB;  // dQ pass: dS hi, dS lo (128 x 64 bf16 each)
    // dQ pass, D = 128: each weight warp stages its 32 rows x 64 dQ columns
    // (one 128-byte-swizzled TMA box) for a bulk read-modify-write
    static constexpr bool STAGE = MODE == 1 && D == 128;
    static constexpr uint32_t O0 = DS0 + (MODE == 1 ? 2 * 128 * 128 : 0);
    static constexpr uint32_t BYTES = O0 + (STAGE ? 8 * 4096 : 0);
    static constexpr uint32_t TCOLS = MODE == 1 ? 512 : 256;   // S, dP (x2), dQ
};

struct RowParams {
    CUtensorMap tq, tg, tk, tv;   // [N][H*D] bf16: Q, dOut boxes 64 x 128; K, V boxes 64 x 16
    CUtensorMap to;               // dQ [N][H*D] bf16, box 64 x 32 (one weight warp's rows and columns)
    BsrBwdArgs a;
};

// MODE 0: Delta pass (writes delta_t, z_t).  MODE 1: dQ pass (adds to dQ).
template <int D, int MODE>
__global__ void __launch_bounds__(kThreads, 1) bsr_bwd_row_kernel(const __grid_constant__ RowParams prm) {
    using C = RowCfg<D, MODE>;
    const BsrBwdArgs &a = prm.a;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t q_full[2], q_empty[2], kv_full[C::NST], kv_empty[C::NST], s_full[2], s_empty[2], ds_full,
        ds_empty, acc_empty, mma_done, st_full[8];
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t sbase = tc::smem_u32(smem);
    const int H = a.H;
    const int64_t n_units = (int64_t)a.n_active * H;

    if (warp == 0) tc::tmem_alloc(&tmem_base, C::TCOLS);
    if (tid == 32) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&q_full[i], 1);
            tc::mbar_init(&q_empty[i], 1);
            tc::mbar_init(&s_full[i], 1);
            tc::mbar_init(&s_empty[i], kSoft);
        }
        for (int i = 0; i < C::NST; ++i) {
            tc::mbar_init(&kv_full[i], 1);
            tc::mbar_init(&kv_empty[i], 1);
        }
        tc::mbar_init(&ds_full, kSoft);
        tc::mbar_init(&ds_empty, 1);
        tc::mbar_init(&acc_empty, kSoft);
        tc::mbar_init(&mma_done, 1);
        for (int i = 0; i < 8; ++i) tc::mbar_init(&st_full[i], 1);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // TMEM: S and dP of buffer sb at 128 sb, 128 sb + 64; the dQ accumulator at 256
    const uint32_t tbase = tmem_base, tQ = tmem_base + 256;

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------------ TMA producer
            int64_t G = 0, U = 0;
            bool ok = true;
            int4 nfo = tc::unit_info(a.panel_info, blockIdx.x, n_units, H);
            for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++U) {
                const int4 cur = nfo;
                nfo = tc::unit_info(a.panel_info, u + gridDim.x, n_units, H);
                const int32_t panel = cur.x, t0 = cur.y, t1 = cur.z;
                const int h = (int)(u % H);
                const int ng = (t1 - t0 + 3) / 4;
                const int qb = (int)(U % C::NQ);
                const int64_t nq = U / C::NQ;
                if (nq >= 1 && !tc::mbar_wait(&q_empty[qb], (nq - 1) & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                const uint32_t qd = sbase + C::Q0 + qb * 2 * C::PB;
                tc::mbar_expect_tx(&q_full[qb], 2 * C::PB);
                for (int at = 0; at < C::DA; ++at) {
                    tc::tma_load_2d(qd + at * 128 * 128, &prm.tq, h * D + at * 64, panel * 128, &q_full[qb]);
                    tc::tma_load_2d(qd + C::PB + at * 128 * 128, &prm.tg, h * D + at * 64, panel * 128, &q_full[qb]);
                }
                for (int g = 0; g < ng; ++g, ++G) {
                    const int s = (int)(G % C::NST);
                    const int64_t n = G / C::NST;
                    int ys[4];   // first source of each tile (loaded before the wait; past N: zero rows)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int32_t ti = t0 + 4 * g + q;
                        ys[q] = ti < t1 ? __ldg(a.tile_col + ti) * 16 : (int)a.N;
                    }
                    if (n >= 1 && !tc::mbar_wait(&kv_empty[s], (n - 1) & 1, tc::kWaitLimit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + C::ST0 + s * 2 * C::KB;
                    tc::mbar_expect_tx(&kv_full[s], 2 * C::KB);
                    for (int q = 0; q < 4; ++q) {
                        const int y = ys[q];
                        for (int at = 0; at < C::DA; ++at) {
                            const uint32_t off = at * kGroup * 128 + q * 16 * 128;
                            tc::tma_load_2d(st + off, &prm.tk, h * D + at * 64, y, &kv_full[s]);
                            tc::tma_load_2d(st + C::KB + off, &prm.tv, h * D + at * 64, y, &kv_full[s]);
                        }
                    }
                }
            }
            if (!ok) atomicOr(a.d_err, tc::kErrMmaTimeout);
            // loads that no MMA consumed (only after a timeout) land before the CTA ends
            for (int64_t i = G - 1; i >= 0 && i >= G - C::NST; --i)
                tc::mbar_wait(&kv_full[i % C::NST], (i / C::NST) & 1, tc::kWaitLimit);
            for (int64_t i = U - 1; i >= 0 && i >= U - C::NQ; --i)
                tc::mbar_wait(&q_full[i % C::NQ], (i / C::NQ) & 1, tc::kWaitLimit);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ------------------------------------------------ MMA issuer
            const uint32_t idesc_s = tc::idesc_bf16(128, kGroup), idesc_q = tc::idesc_bf16(128, D) | tc::kMajorMnB;
            int64_t G = 0, U = 0;
            bool ok = true;
            // dQ += dS_hi K + dS_lo K of group Gp; the first of unit Up
            // overwrites dQ once the previous unit's epilogue has read it
            auto issue_dq = [&](int64_t Gp, bool first, int64_t Up) -> bool {
                if (!tc::mbar_wait(&ds_full, Gp & 1, tc::kWaitLimit)) return false;
                if (first && Up >= 1 && !tc::mbar_wait(&acc_empty, (Up - 1) & 1, tc::kWaitLimit)) return false;
                tc::fence_after_sync();
                const int s = (int)(Gp % C::NST);
                const uint32_t kr = sbase + C::ST0 + s * 2 * C::KB;
                mma_rows64(tQ, sbase + C::DS0, kr, idesc_q, first);
                mma_rows64(tQ, sbase + C::DS0 + 128 * 128, kr, idesc_q, false);
                tc::mma_commit(&kv_empty[s]);
                tc::mma_commit(&ds_empty);
                return true;
            };
            int64_t pend = -1, pend_u = 0;
            bool pend_first = false;
            int4 nfo = tc::unit_info(a.panel_info, blockIdx.x, n_units, H);
            for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++U) {
                const int4 cur = nfo;
                nfo = tc::unit_info(a.panel_info, u + gridDim.x, n_units, H);
                const int32_t t0 = cur.y, t1 = cur.z;
                const int ng = (t1 - t0 + 3) / 4;
                const int qb = (int)(U % C::NQ);
                if (!tc::mbar_wait(&q_full[qb], (U / C::NQ) & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                const uint32_t qa = sbase + C::Q0 + qb * 2 * C::PB;
                for (int g = 0; g < ng; ++g, ++G) {
                    const int s = (int)(G % C::NST), sb = (int)(G & 1);
                    if (!tc::mbar_wait(&kv_full[s], (G / C::NST) & 1, tc::kWaitLimit) ||
                        (G >= 2 && !tc::mbar_wait(&s_empty[sb], ((G >> 1) - 1) & 1, tc::kWaitLimit))) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t st = sbase + C::ST0 + s * 2 * C::KB;
                    mma_over_d(tbase + sb * 128, qa, st, kGroup, D, idesc_s);                   // S = Q K^T
                    mma_over_d(tbase + sb * 128 + 64, qa + C::PB, st + C::KB, kGroup, D, idesc_s);   // dP = dOut V^T
                    tc::mma_commit(&s_full[sb]);
                    if (MODE == 0) tc::mma_commit(&kv_empty[s]);   // the Delta pass is done with K and V
                    if (g == ng - 1) tc::mma_commit(&q_empty[qb]);
                    if (MODE == 1) {
                        if (pend >= 0 && !issue_dq(pend, pend_first, pend_u)) {
                            ok = false;
                            break;
                        }
                        pend = G;
                        pend_first = g == 0;
                        pend_u = U;
                    }
                }
            }
            if (MODE == 1 && ok && pend >= 0 && !issue_dq(pend, pend_first, pend_u)) ok = false;
            if (!ok) atomicOr(a.d_err, tc::kErrMmaTimeout);
            tc::mma_commit(&mma_done);   // every product issued is complete before TMEM is released
            tc::mbar_wait(&mma_done, 0, tc::kWaitLimit);
        }
    } else {   // ---------------------------------------------------- weights and gradients
        const int quarter = warp & 3, hf = (warp - 2) >> 2, r = quarter * 32 + lane;   // half hf: sources 32 hf ..
        const uint32_t tlane = (uint32_t)(quarter * 32) << 16;
        const float scale2 = kLog2e * rsqrtf((float)D);
        constexpr int DH = D / 2;   // dQ columns this warp adds
        int64_t G = 0, U = 0;
        bool ok = true;
        int4 nfo = tc::unit_info(a.panel_info, blockIdx.x, n_units, H);
        for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++U) {
            const int4 cur = nfo;
            nfo = tc::unit_info(a.panel_info, u + gridDim.x, n_units, H);
            const int32_t panel = cur.x, t0 = cur.y, t1 = cur.z;
            const int h = (int)(u % H);
            const int ng = (t1 - t0 + 3) / 4;
            const int64_t row = (int64_t)panel * 128 + r;
            const bool in = row < a.N;
            // the Delta pass uses the forward's lse and sums C and Z of its tile edges;
            // the dQ pass uses the normalised lse + ln Z and Delta = C / Z of the row
            const float lse2 = in ? (MODE == 0 ? a.lse : a.lse_n)[row * H + h] * kLog2e : 0.f;
            const float dl = (MODE == 1 && in) ? a.delta[row * H + h] : 0.f;
            __nv_bfloat16 *dq = static_cast<__nv_bfloat16 *>(a.dQ) + ((in ? row : 0) * H + h) * D + hf * DH;
            const uint32_t stg = sbase + C::O0 + (warp - 2) * 4096;   // (STAGE) this warp's box
            if constexpr (C::STAGE) {
                if (lane == 0) {
                    if (U >= 1) tc::bulk_wait_read();   // the previous unit's store has read the box
                    tc::mbar_expect_tx(&st_full[warp - 2], 4096);
                    tc::tma_load_2d(stg, &prm.to, h * D + hf * DH, panel * 128 + quarter * 32, &st_full[warp - 2]);
                }
            } else if (MODE == 1 && in) {
                prefetch_row<DH>(dq);
            }
            float ps[2] = {0.f, 0.f}, zs[2] = {0.f, 0.f};
            for (int g = 0; g < ng; ++g, ++G) {
                const int sb = (int)(G & 1);
                uint32_t bits[2];   // this row's source masks of the half's two tiles (zero tile for missing ones)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int32_t ti = t0 + 4 * g + 2 * hf + q;
                    bits[q] = a.tile_bits[(size_t)(ti < t1 ? ti : a.n_tiles) * 128 + r];
                }
                if (!tc::warp_wait(&s_full[sb], (G >> 1) & 1, tc::kWaitLimit) ||
                    (MODE == 1 && G >= 1 && !tc::warp_wait(&ds_empty, (G - 1) & 1, tc::kWaitLimit))) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                uint32_t us[32], up[32];
                tc::tmem_ld32(tbase + sb * 128 + hf * 32 + tlane, us);
                tc::tmem_ld32(tbase + sb * 128 + 64 + hf * 32 + tlane, up);
                float ds[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const bool on = (bits[i >> 4] >> (i & 15)) & 1u;
                    const float p = on ? tc::ex2(__uint_as_float(us[i]) * scale2 - lse2) : 0.f;
                    const float dp = __uint_as_float(up[i]);
                    if (MODE == 0) {
                        ps[i & 1] = fmaf(p, dp, ps[i & 1]);
                        zs[i & 1] += p;
                    }
                    ds[i] = p * (dp - dl);
                }
                if (MODE == 1) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint32_t o = tc::sw128_offset(r, hf * 32 + c * 8, 128);
                        uint4 hi, lo;
                        split_bf16x8(ds + 8 * c, hi, lo);
                        *reinterpret_cast<uint4 *>(smem + C::DS0 + o) = hi;
                        *reinterpret_cast<uint4 *>(smem + C::DS0 + 128 * 128 + o) = lo;
                    }
                }
                tc::fence_before_sync();
                if (MODE == 1) tc::fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&s_empty[sb]);
                    if (MODE == 1) tc::mbar_arrive(&ds_full);
                }
            }
            if (!ok) break;
            if (MODE == 0) {
                // the two halves' sums of the row added to the zeroed outputs: with two
                // terms onto zero, either order rounds to the same fl(a + b)
                if (in) {
                    atomicAdd(a.delta_t + row * H + h, ps[0] + ps[1]);
                    atomicAdd(a.z_t + row * H + h, zs[0] + zs[1]);
                }
            } else {
                // the unit's last dQ product, then add this half of the tile part to dQ
                if (!tc::warp_wait(&ds_empty, (G - 1) & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                if constexpr (C::STAGE) {
                    // the residual dQ values arrived in the staged box (row = lane, 128-byte swizzle)
                    if (!tc::warp_wait(&st_full[warp - 2], U & 1, tc::kWaitLimit)) {
                        ok = false;
                        break;
                    }
                    add_box_from_tmem<DH>(tQ + hf * DH + tlane, smem + C::O0 + (warp - 2) * 4096 + lane * 128, lane,
                                          rsqrtf((float)D));
                    tc::fence_proxy_async();   // the box's new values, for the TMA store
                    __syncwarp();
                    if (lane == 0) {
                        tc::tma_store_2d(&prm.to, h * D + hf * DH, panel * 128 + quarter * 32, stg);
                        tc::bulk_commit();
                    }
                } else {
                    add_row_from_tmem<DH>(tQ + hf * DH + tlane, dq, rsqrtf((float)D), in);
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&acc_empty);
            }
        }
        if (!ok && lane == 0) atomicOr(a.d_err, tc::kErrMmaTimeout);
        if constexpr (C::STAGE) {
            // a staged box whose load was issued but not consumed (only after a
            // timeout, in the unit that failed) lands before the CTA ends; every store completes
            if (lane == 0) {
                if (!ok) tc::mbar_wait(&st_full[warp - 2], U & 1, tc::kWaitLimit);
                tc::bulk_wait_all();
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::tmem_dealloc(tmem_base, C::TCOLS);
    }
}

// ----------------------------------------------------------- column pass

template <int D> struct ColCfg {
    static constexpr int DA = D / 64;
    static constexpr uint32_t CB = DA * 128 * 128;   // K or V of the column panel (128 sources)
    static constexpr uint32_t HB = DA * 64 * 128;    // Q or dOut of a block (64 destinations)
    static constexpr int NST = D == 128 ? 2 : 4;
    static constexpr uint32_t C0 = 0;                // K, then V
    static constexpr uint32_t ST0 = C0 + 2 * CB;     // stage: Q, dOut, masks (8 tiles x 16 sources x 64 bits), lse, Delta
    static constexpr uint32_t TX = 2 * HB + 1024 + 256 + 256;   // bytes a stage receives
    static constexpr uint32_t STB = (TX + 1023) / 1024 * 1024;  // stages 1024-aligned (128-byte swizzle)
    static constexpr uint32_t PD0 = ST0 + NST * STB; // P^T, dS^T hi, dS^T lo (128 x 64 bf16 each)
    // each weight warp stages 32 rows x 64 columns of its gradient (one
    // 128-byte-swizzled TMA box) for a bulk read-modify-write, D / 64 boxes in turn
    static constexpr int NH = D / 64;
    static constexpr uint32_t O0 = PD0 + 3 * 128 * 128;
    static constexpr uint32_t BYTES = O0 + 8 * 4096;
};

static_assert(ColCfg<64>::STB % 1024 == 0 && ColCfg<128>::STB % 1024 == 0, "stage alignment");
static_assert(ColCfg<128>::BYTES + 1024 <= 227 * 1024 && ColCfg<64>::BYTES + 1024 <= 227 * 1024, "shared memory");
static_assert(RowCfg<128, 0>::BYTES + 1024 <= 227 * 1024 && RowCfg<128, 1>::BYTES + 1024 + 1024 <= 227 * 1024 &&
                  RowCfg<64, 0>::BYTES + 1024 <= 227 * 1024 && RowCfg<64, 1>::BYTES + 1024 <= 227 * 1024,
              "shared memory");

struct ColParams {
    CUtensorMap tk, tv, tq, tg;   // [N][H*D] bf16: K, V boxes 64 x 128; Q, dOut boxes 64 x 64
    CUtensorMap tdk, tdv;         // dK, dV [N][H*D] bf16, box 64 x 32 (one weight warp's rows, 64 columns)
    BsrBwdArgs a;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) bsr_bwd_col_kernel(const __grid_constant__ ColParams prm) {
    using C = ColCfg<D>;
    const BsrBwdArgs &a = prm.a;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t c_full, c_empty, kv_full[C::NST], kv_empty[C::NST], s_full[2], s_empty[2], pd_full, pd_empty,
        acc_empty, mma_done, st_full[8];
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t sbase = tc::smem_u32(smem);
    const int H = a.H;
    const int64_t n_units = (int64_t)a.n_cactive * H;

    if (warp == 0) tc::tmem_alloc(&tmem_base, 512);
    if (tid == 32) {
        tc::mbar_init(&c_full, 1);
        tc::mbar_init(&c_empty, 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&s_full[i], 1);
            tc::mbar_init(&s_empty[i], kSoft);
        }
        for (int i = 0; i < C::NST; ++i) {
            tc::mbar_init(&kv_full[i], 1);
            tc::mbar_init(&kv_empty[i], 1);
        }
        tc::mbar_init(&pd_full, kSoft);
        tc::mbar_init(&pd_empty, 1);
        tc::mbar_init(&acc_empty, kSoft);
        tc::mbar_init(&mma_done, 1);
        for (int i = 0; i < 8; ++i) tc::mbar_init(&st_full[i], 1);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // TMEM: S^T and dP^T of buffer sb at 128 sb, 128 sb + 64; dV at 256, dK at 256 + D
    const uint32_t tbase = tmem_base, tV = tmem_base + 256, tK = tmem_base + 256 + D;

    if (warp == 0) {
        if (lane == 0) {   // ------------------------------------------------ TMA producer
            int64_t B = 0, U = 0;
            bool ok = true;
            int4 nfo = tc::unit_info(a.cpanel_info, blockIdx.x, n_units, H);
            for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++U) {
                const int4 cur = nfo;
                nfo = tc::unit_info(a.cpanel_info, u + gridDim.x, n_units, H);
                const int32_t cp = cur.x, e0 = cur.y, e1 = cur.z;
                const int h = (int)(u % H);
                const int nb = 2 * (e1 - e0);   // blocks: (entry, 64-row half)
                if (U >= 1 && !tc::mbar_wait(&c_empty, (U - 1) & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                tc::mbar_expect_tx(&c_full, 2 * C::CB);
                for (int at = 0; at < C::DA; ++at) {
                    tc::tma_load_2d(sbase + C::C0 + at * 128 * 128, &prm.tk, h * D + at * 64, cp * 128, &c_full);
                    tc::tma_load_2d(sbase + C::C0 + C::CB + at * 128 * 128, &prm.tv, h * D + at * 64, cp * 128,
                                    &c_full);
                }
                for (int b = 0; b < nb; ++b, ++B) {
                    const int s = (int)(B % C::NST);
                    const int64_t n = B / C::NST;
                    // the block's row panel and tiles (loaded before the wait)
                    const int32_t e = e0 + b / 2;
                    const int hf = b & 1;
                    const int row0 = __ldg(a.ct_panel + e) * 128 + hf * 64;
                    const int4 ta = __ldg(reinterpret_cast<const int4 *>(a.ct_tile) + 2 * e);
                    const int4 tb = __ldg(reinterpret_cast<const int4 *>(a.ct_tile) + 2 * e + 1);
                    const int32_t tiles[8] = {ta.x, ta.y, ta.z, ta.w, tb.x, tb.y, tb.z, tb.w};
                    if (n >= 1 && !tc::mbar_wait(&kv_empty[s], (n - 1) & 1, tc::kWaitLimit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + C::ST0 + s * C::STB;
                    tc::mbar_expect_tx(&kv_full[s], C::TX);
                    for (int at = 0; at < C::DA; ++at) {
                        tc::tma_load_2d(st + at * 64 * 128, &prm.tq, h * D + at * 64, row0, &kv_full[s]);
                        tc::tma_load_2d(st + C::HB + at * 64 * 128, &prm.tg, h * D + at * 64, row0, &kv_full[s]);
                    }
                    for (int t = 0; t < 8; ++t) {   // the 8 tile columns' masks of the 64 rows, transposed
                        const int32_t tile = tiles[t];
                        tc::bulk_load(st + 2 * C::HB + t * 128,
                                      a.tile_bits_t + ((size_t)(tile >= 0 ? tile : a.n_tiles) * 2 + hf) * 16, 128,
                                      &kv_full[s]);
                    }
                    tc::bulk_load(st + 2 * C::HB + 1024, a.lse_t + (size_t)h * a.N_pad + row0, 256, &kv_full[s]);
                    tc::bulk_load(st + 2 * C::HB + 1280, a.delta_t_hm + (size_t)h * a.N_pad + row0, 256,
                                  &kv_full[s]);
                }
            }
            if (!ok) atomicOr(a.d_err, tc::kErrMmaTimeout);
            for (int64_t i = B - 1; i >= 0 && i >= B - C::NST; --i)
                tc::mbar_wait(&kv_full[i % C::NST], (i / C::NST) & 1, tc::kWaitLimit);
            if (U >= 1) tc::mbar_wait(&c_full, (U - 1) & 1, tc::kWaitLimit);
        }
    } else if (warp == 1) {
        if (lane == 0) {   // ------------------------------------------------ MMA issuer
            const uint32_t idesc_s = tc::idesc_bf16(128, 64), idesc_d = tc::idesc_bf16(128, D) | tc::kMajorMnB;
            int64_t B = 0, U = 0;
            bool ok = true;
            // dV += P^T dOut, dK += dS^T_hi Q + dS^T_lo Q of block Bp; the first
            // of unit Up overwrites dK/dV once the previous unit's epilogue has read them
            auto issue_kv = [&](int64_t Bp, bool first, int64_t Up) -> bool {
                if (!tc::mbar_wait(&pd_full, Bp & 1, tc::kWaitLimit)) return false;
                if (first && Up >= 1 && !tc::mbar_wait(&acc_empty, (Up - 1) & 1, tc::kWaitLimit)) return false;
                tc::fence_after_sync();
                const int s = (int)(Bp % C::NST);
                const uint32_t st = sbase + C::ST0 + s * C::STB;
                mma_rows64(tV, sbase + C::PD0, st + C::HB, idesc_d, first);
                mma_rows64(tK, sbase + C::PD0 + 128 * 128, st, idesc_d, first);
                mma_rows64(tK, sbase + C::PD0 + 2 * 128 * 128, st, idesc_d, false);
                tc::mma_commit(&kv_empty[s]);
                tc::mma_commit(&pd_empty);
                return true;
            };
            int64_t pend = -1, pend_u = 0;
            bool pend_first = false;
            int4 nfo = tc::unit_info(a.cpanel_info, blockIdx.x, n_units, H);
            for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++U) {
                const int4 cur = nfo;
                nfo = tc::unit_info(a.cpanel_info, u + gridDim.x, n_units, H);
                const int nb = 2 * (cur.z - cur.y);
                if (!tc::mbar_wait(&c_full, U & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                for (int b = 0; b < nb; ++b, ++B) {
                    const int s = (int)(B % C::NST), sb = (int)(B & 1);
                    if (!tc::mbar_wait(&kv_full[s], (B / C::NST) & 1, tc::kWaitLimit) ||
                        (B >= 2 && !tc::mbar_wait(&s_empty[sb], ((B >> 1) - 1) & 1, tc::kWaitLimit))) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t st = sbase + C::ST0 + s * C::STB;
                    mma_over_d(tbase + sb * 128, sbase + C::C0, st, 64, D, idesc_s);                   // S^T = K Q^T
                    mma_over_d(tbase + sb * 128 + 64, sbase + C::C0 + C::CB, st + C::HB, 64, D, idesc_s);   // dP^T
                    tc::mma_commit(&s_full[sb]);
                    if (b == nb - 1) tc::mma_commit(&c_empty);
                    if (pend >= 0 && !issue_kv(pend, pend_first, pend_u)) {
                        ok = false;
                        break;
                    }
                    pend = B;
                    pend_first = b == 0;
                    pend_u = U;
                }
            }
            if (ok && pend >= 0 && !issue_kv(pend, pend_first, pend_u)) ok = false;
            if (!ok) atomicOr(a.d_err, tc::kErrMmaTimeout);
            tc::mma_commit(&mma_done);
            tc::mbar_wait(&mma_done, 0, tc::kWaitLimit);
        }
    } else {   // ---------------------------------------------------- weights and gradients
        // thread = source of the column panel (TMEM lane); half hf: destination rows 32 hf ..
        // of each block, and at the end of the unit dK (hf 0) or dV (hf 1)
        const int quarter = warp & 3, hf = (warp - 2) >> 2, r = quarter * 32 + lane;
        const uint32_t tlane = (uint32_t)(quarter * 32) << 16;
        const float scale2 = kLog2e * rsqrtf((float)D);
        int64_t B = 0, U = 0, nld = 0;   // nld: staged box loads issued (lane 0 issues them)
        bool ok = true;
        int4 nfo = tc::unit_info(a.cpanel_info, blockIdx.x, n_units, H);
        for (int64_t u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++U) {
            const int4 cur = nfo;
            nfo = tc::unit_info(a.cpanel_info, u + gridDim.x, n_units, H);
            const int32_t cp = cur.x;
            const int h = (int)(u % H);
            const int nb = 2 * (cur.z - cur.y);
            const int64_t src = (int64_t)cp * 128 + r;
            const bool in = src < a.N;
            // this warp's gradient rows (dK for hf 0, dV for hf 1): the first box loads now
            const CUtensorMap *tg_map = hf == 0 ? &prm.tdk : &prm.tdv;
            const uint32_t stg = sbase + C::O0 + (warp - 2) * 4096;
            if (lane == 0) {
                if (U >= 1) tc::bulk_wait_read();   // the previous unit's last store has read the box
                tc::mbar_expect_tx(&st_full[warp - 2], 4096);
                tc::tma_load_2d(stg, tg_map, h * D, cp * 128 + quarter * 32, &st_full[warp - 2]);
            }
            ++nld;
            for (int b = 0; b < nb; ++b, ++B) {
                const int s = (int)(B % C::NST), sb = (int)(B & 1);
                // products, the stage's masks and row terms, and a free P / dS buffer
                if (!tc::warp_wait(&s_full[sb], (B >> 1) & 1, tc::kWaitLimit) ||
                    !tc::warp_wait(&kv_full[s], (B / C::NST) & 1, tc::kWaitLimit) ||
                    (B >= 1 && !tc::warp_wait(&pd_empty, (B - 1) & 1, tc::kWaitLimit))) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const unsigned char *st = smem + C::ST0 + s * C::STB;
                // this source's bits for the half's 32 rows (transposed masks: word r)
                const uint32_t m32 =
                    in ? (uint32_t)(reinterpret_cast<const uint64_t *>(st + 2 * C::HB)[r] >> (32 * hf)) : 0u;
                const float4 *lse4 = reinterpret_cast<const float4 *>(st + 2 * C::HB + 1024) + hf * 8;
                const float4 *dl4 = reinterpret_cast<const float4 *>(st + 2 * C::HB + 1280) + hf * 8;
                uint32_t us[32], up[32];
                tc::tmem_ld32(tbase + sb * 128 + hf * 32 + tlane, us);
                tc::tmem_ld32(tbase + sb * 128 + 64 + hf * 32 + tlane, up);
                float pv[32], ds[32];
#pragma unroll
                for (int i4 = 0; i4 < 8; ++i4) {
                    const float4 l4 = lse4[i4], d4 = dl4[i4];
                    const float lv[4] = {l4.x, l4.y, l4.z, l4.w}, dv[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int ii = i4 * 4 + k;
                        const bool on = (m32 >> ii) & 1u;
                        const float p = on ? tc::ex2(__uint_as_float(us[ii]) * scale2 - lv[k] * kLog2e) : 0.f;
                        pv[ii] = p;
                        ds[ii] = p * (__uint_as_float(up[ii]) - dv[k]);
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const uint32_t o = tc::sw128_offset(r, hf * 32 + c * 8, 128);
                    uint4 hi, lo;
                    split_bf16x8(ds + 8 * c, hi, lo);
                    *reinterpret_cast<uint4 *>(smem + C::PD0 + o) = pack<__nv_bfloat16>(pv + 8 * c);
                    *reinterpret_cast<uint4 *>(smem + C::PD0 + 128 * 128 + o) = hi;
                    *reinterpret_cast<uint4 *>(smem + C::PD0 + 2 * 128 * 128 + o) = lo;
                }
                tc::fence_before_sync();
                tc::fence_proxy_async();
                __syncwarp();
                if (lane == 0) {
                    tc::mbar_arrive(&s_empty[sb]);
                    tc::mbar_arrive(&pd_full);
                }
            }
            if (!ok) break;
            // the unit's last products, then add the tile part to dK (hf 0) or dV (hf 1)
            if (!tc::warp_wait(&pd_empty, (B - 1) & 1, tc::kWaitLimit)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            // add the accumulator to the staged boxes, 64 columns at a time (row = lane)
            for (int c2 = 0; c2 < C::NH; ++c2) {
                if (c2 > 0 && lane == 0) {   // the box is reloaded once the store has read it
                    tc::bulk_wait_read();
                    tc::mbar_expect_tx(&st_full[warp - 2], 4096);
                    tc::tma_load_2d(stg, tg_map, h * D + c2 * 64, cp * 128 + quarter * 32, &st_full[warp - 2]);
                }
                if (c2 > 0) ++nld;
                if (!tc::warp_wait(&st_full[warp - 2], (U * C::NH + c2) & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                add_box_from_tmem<64>((hf == 0 ? tK : tV) + tlane + c2 * 64,
                                      smem + C::O0 + (warp - 2) * 4096 + lane * 128, lane,
                                      hf == 0 ? rsqrtf((float)D) : 1.f);
                tc::fence_proxy_async();   // the box's new values, for the TMA store
                __syncwarp();
                if (lane == 0) {
                    tc::tma_store_2d(tg_map, h * D + c2 * 64, cp * 128 + quarter * 32, stg);
                    tc::bulk_commit();
                }
            }
            if (!ok) break;
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&acc_empty);
        }
        if (!ok && lane == 0) atomicOr(a.d_err, tc::kErrMmaTimeout);
        if (lane == 0) {
            // after a timeout the box load last issued lands before the CTA ends; every store completes
            if (!ok && nld > 0) tc::mbar_wait(&st_full[warp - 2], (nld - 1) & 1, tc::kWaitLimit);
            tc::bulk_wait_all();
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::tmem_dealloc(tmem_base, 512);
    }
}

// lse + ln Z and Delta in head-major order [H][N_pad] (zero past N), so that
// a block's 64 consecutive rows are one 256-byte bulk copy
__global__ void head_major_kernel(const float *__restrict__ lse_n, const float *__restrict__ delta, int64_t N,
                                  int64_t N_pad, int H, float *__restrict__ lse_t, float *__restrict__ dl_t) {
    const int64_t n = N_pad * H, stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += stride) {
        const int h = (int)(x / N_pad);
        const int64_t i = x % N_pad;
        lse_t[x] = i < N ? lse_n[i * H + h] : 0.f;
        dl_t[x] = i < N ? delta[i * H + h] : 0.f;
    }
}

// ---------------------------------------------------------------- launch

template <auto Kernel, typename P>
cudaError_t launch(const P &prm, int64_t units, int num_sms, size_t bytes, sga_kernel_id id, cudaStream_t s) {
    const size_t smem = bytes + 1024;
    if (cudaError_t e = allow_smem<Kernel>(smem); e != cudaSuccess) return e;
    const unsigned grid = (unsigned)(units < num_sms ? units : num_sms);
    note_launch(id, s, false);
    Kernel<<<grid, kThreads, smem, s>>>(prm);
    note_launch(id, s, true);
    return cudaGetLastError();
}

template <int D> cudaError_t row_pass(const BsrBwdArgs &a, int mode, cudaStream_t s) {
    RowParams prm{};
    prm.a = a;
    const int64_t HD = (int64_t)a.H * D;
    auto bf = [](const void *p) { return static_cast<const __nv_bfloat16 *>(p); };
    cudaError_t e = bf16_tensor_map(&prm.tq, bf(a.Q), a.N, HD, HD, 64, 128);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.tg, bf(a.dOut), a.N, HD, HD, 64, 128);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.tk, bf(a.K), a.N, HD, HD, 64, 16);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.tv, bf(a.V), a.N, HD, HD, 64, 16);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.to, bf(a.dQ), a.N, HD, HD, 64, 32);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.n_active * a.H;
    return mode == 0 ? launch<bsr_bwd_row_kernel<D, 0>>(prm, units, a.num_sms, RowCfg<D, 0>::BYTES,
                                                         SGA_KERN_BSR_BWD_DELTA, s)
                     : launch<bsr_bwd_row_kernel<D, 1>>(prm, units, a.num_sms, RowCfg<D, 1>::BYTES,
                                                        SGA_KERN_BSR_BWD_DQ, s);
}

template <int D> cudaError_t col_pass(const BsrBwdArgs &a, cudaStream_t s) {
    ColParams prm{};
    prm.a = a;
    const int64_t HD = (int64_t)a.H * D;
    auto bf = [](const void *p) { return static_cast<const __nv_bfloat16 *>(p); };
    cudaError_t e = bf16_tensor_map(&prm.tk, bf(a.K), a.N, HD, HD, 64, 128);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.tv, bf(a.V), a.N, HD, HD, 64, 128);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.tq, bf(a.Q), a.N, HD, HD, 64, 64);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.tg, bf(a.dOut), a.N, HD, HD, 64, 64);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.tdk, bf(a.dK), a.N, HD, HD, 64, 32);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.tdv, bf(a.dV), a.N, HD, HD, 64, 32);
    if (e != cudaSuccess) return e;
    const int64_t units = (int64_t)a.n_cactive * a.H;
    return launch<bsr_bwd_col_kernel<D>>(prm, units, a.num_sms, ColCfg<D>::BYTES, SGA_KERN_BSR_BWD_DKDV, s);
}

}  // namespace

cudaError_t launch_bsr_bwd_delta(const BsrBwdArgs &a, cudaStream_t s) {
    if (a.n_active == 0) return cudaSuccess;
    return a.D == 128 ? row_pass<128>(a, 0, s) : row_pass<64>(a, 0, s);
}

cudaError_t launch_bsr_bwd_dq(const BsrBwdArgs &a, cudaStream_t s) {
    if (a.n_active == 0) return cudaSuccess;
    return a.D == 128 ? row_pass<128>(a, 1, s) : row_pass<64>(a, 1, s);
}

cudaError_t launch_bsr_bwd_dkdv(const BsrBwdArgs &a, cudaStream_t s) {
    if (a.n_cactive == 0) return cudaSuccess;
    const int64_t n = a.N_pad * a.H;
    head_major_kernel<<<(unsigned)std::min<int64_t>((n + 255) / 256, 65535), 256, 0, s>>>(
        a.lse_n, a.delta, a.N, a.N_pad, a.H, a.lse_t, a.delta_t_hm);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return a.D == 128 ? col_pass<128>(a, s) : col_pass<64>(a, s);
}

}  // namespace sga
