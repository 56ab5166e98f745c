// Block-sparse Graph Transformer forward on the tcgen05 tensor cores: the
// "Tensor Core (block-sparse) variant" of "On Efficient Scaling of GNNs via
// IO-Aware Layers Implementations" (arXiv abstract; blog post,
// "Attention-based layers" paragraph), which pays off on locally dense graphs.
//
// Persistent CTAs, one per SM, take work units (128-row panel, head) from the
// plan's panel order (most kept tiles first), round robin.  A unit's kept
// column tiles are taken four at a time (64 sources, a "group").  Roles:
//   warp 0, one lane: TMA loads -- the unit's Q panel (two buffers, so the
//     next unit's panel loads during this one) and, for every group, its K
//     and V rows (one 16-row box per tile and 64-wide column atom; missing
//     tiles read rows past N, which TMA fills with zeros) plus the four tiles'
//     source masks (a bulk copy each; a missing tile copies the plan's zero
//     tile), into a ring of stages;
//   warp 1, one lane: the MMAs -- S = Q K^T (128 x 64, K = D) into one of two
//     TMEM score buffers, and O += P V (128 x D, K = 64; V rows are the
//     MN-major B operand as they lie) into the TMEM accumulator, issued in
//     the order S(g), P V(g-1), so the tensor core computes the next scores
//     and the previous product while the softmax runs;
//   warps 2-9 (thread = panel row = TMEM lane; two warps per lane quarter,
//     each taking 32 of a group's 64 sources): the online softmax with a
//     lazily moved maximum (the half's O is rescaled in TMEM only when its
//     maximum grows by more than 2^8, so P stays below 2^8), P to shared
//     memory in bf16, and the epilogue.  Each half keeps its own maximum, sum
//     and accumulator (O_A += P_A V_A, O_B += P_B V_B: two K = 32 products),
//     so the two warps of a row never wait on each other within a unit; the
//     epilogue merges the halves and then the tile result with the residual
//     CSR result already stored in out and lse, by log-sum-exp, each warp
//     writing half of the row.
// Every handoff is an mbarrier (TMA transaction counts, tcgen05.commit, or
// the arrivals of the four softmax warps); every wait is bounded and a
// timeout sets the plan's error word and ends the role.
#include <cuda.h>

#include "common.cuh"
#include "plan.h"
#include "tc.cuh"
#include "tc_dx.cuh"

namespace sga {
namespace {

constexpr int kThreads = 320;   // producer, MMA lane, eight softmax warps
constexpr int kSoft = 8;        // softmax warps: arrivals per handoff
constexpr int kGroup = 64;      // sources per group (four 16-wide tiles)
constexpr float kLazy = 8.0f;

template <int D> struct FwdCfg {
    static constexpr int DA = D / 64;                          // 64-wide column atoms of a head row
    static constexpr uint32_t QB = DA * 128 * 128;             // Q panel (128 rows)
    static constexpr uint32_t KB = DA * kGroup * 128;          // K (or V) rows of a group
    // shared memory goes to K/V stages first (the loads in flight); the Q
    // panel is double-buffered where that still leaves five stages
    static constexpr int NQ = D == 64 ? 2 : 1;
    static constexpr int NST = D == 64 ? 8 : 4;
    // D = 128: each softmax warp stages its 32 rows x 64 output columns (one
    // 128-byte-swizzled TMA box) for a bulk read-modify-write of out
    static constexpr bool STAGE = D == 128;
    static constexpr uint32_t Q0 = 0;                          // Q buffers
    static constexpr uint32_t ST0 = Q0 + NQ * QB;              // stage s: K, then V, then masks
    static constexpr uint32_t STB = 2 * KB + 1024;             //   (masks: 4 tiles x 128 rows x 2 B)
    static constexpr uint32_t P0 = ST0 + NST * STB;            // P (128 x 64 bf16)
    static constexpr uint32_t O0 = P0 + 128 * 128;             // staging: 8 warps x 32 rows x 128 B
    static constexpr uint32_t BYTES = O0 + (STAGE ? 8 * 4096 : 0);
    static constexpr uint32_t TX = 2 * KB + 1024;              // transaction bytes of a stage
};

static_assert(FwdCfg<64>::STB % 1024 == 0 && FwdCfg<128>::STB % 1024 == 0, "stage alignment");
static_assert(FwdCfg<128>::BYTES + 1024 <= 227 * 1024 && FwdCfg<64>::BYTES + 1024 <= 227 * 1024, "shared memory");

struct FwdParams {
    CUtensorMap tq, tk, tv;   // [N][H*D] bf16; boxes 64 x 128 (Q), 64 x 16 (K, V); 128-byte swizzle
    CUtensorMap to;           // out [N][H*D] bf16, box 64 x 32 (one softmax warp's rows and columns)
    BsrArgs a;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 1) bsr_fwd_kernel(const __grid_constant__ FwdParams prm) {
    using C = FwdCfg<D>;
    const BsrArgs &a = prm.a;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t q_full[2], q_empty[2], kv_full[C::NST], kv_empty[C::NST], s_full[2], s_empty[2], p_full,
        pv_done, o_empty, xch_full, mma_done, st_full[8];
    __shared__ uint32_t tmem_base;
    __shared__ float2 xch[2][128];   // per half and row: (maximum, sum) at the end of a unit
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t sbase = tc::smem_u32(smem);
    const int H = a.H;
    const int64_t n_units = (int64_t)a.n_active * H;
    constexpr uint32_t kCols = 4 * D <= 256 ? 256 : 512;   // O_A, O_B (D each), two S buffers (64 each)

    if (warp == 0) tc::tmem_alloc(&tmem_base, kCols);
    if (tid == 32) {
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&q_full[i], 1);
            tc::mbar_init(&q_empty[i], 1);
            tc::mbar_init(&s_full[i], 1);
            tc::mbar_init(&s_empty[i], kSoft);
        }
        tc::mbar_init(&p_full, kSoft);
        tc::mbar_init(&pv_done, 1);
        for (int i = 0; i < C::NST; ++i) {
            tc::mbar_init(&kv_full[i], 1);
            tc::mbar_init(&kv_empty[i], 1);
        }
        tc::mbar_init(&o_empty, kSoft);
        tc::mbar_init(&xch_full, kSoft);
        for (int i = 0; i < 8; ++i) tc::mbar_init(&st_full[i], 1);
        tc::mbar_init(&mma_done, 1);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tO = tmem_base, tS0 = tmem_base + 2 * D;   // O_A, O_B: D columns each; S buffers: 64 each

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
                tc::mbar_expect_tx(&q_full[qb], C::QB);
                for (int at = 0; at < C::DA; ++at)
                    tc::tma_load_2d(sbase + C::Q0 + qb * C::QB + at * 128 * 128, &prm.tq, h * D + at * 64,
                                    panel * 128, &q_full[qb]);
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
                    const uint32_t st = sbase + C::ST0 + s * C::STB;
                    tc::mbar_expect_tx(&kv_full[s], C::TX);
                    for (int q = 0; q < 4; ++q) {
                        const int32_t ti = t0 + 4 * g + q;
                        const int y = ys[q];
                        for (int at = 0; at < C::DA; ++at) {
                            const uint32_t off = at * kGroup * 128 + q * 16 * 128;
                            tc::tma_load_2d(st + off, &prm.tk, h * D + at * 64, y, &kv_full[s]);
                            tc::tma_load_2d(st + C::KB + off, &prm.tv, h * D + at * 64, y, &kv_full[s]);
                        }
                        tc::bulk_load(st + 2 * C::KB + q * 256,
                                      a.tile_bits + (size_t)(ti < t1 ? ti : a.n_tiles) * 128, 256, &kv_full[s]);
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
            const uint32_t idesc_s = tc::idesc_bf16(128, kGroup);
            const uint32_t idesc_o = tc::idesc_bf16(128, D) | tc::kMajorMnB;
            int64_t G = 0, U = 0;
            bool ok = true;
            // O += P(Gp) V(Gp); the first product of unit Up overwrites O, once
            // the previous unit's epilogue has read it
            auto issue_pv = [&](int64_t Gp, bool first, int64_t Up) -> bool {
                const int s = (int)(Gp % C::NST);
                if (!tc::mbar_wait(&p_full, Gp & 1, tc::kWaitLimit)) return false;
                if (first && Up >= 1 && !tc::mbar_wait(&o_empty, (Up - 1) & 1, tc::kWaitLimit)) return false;
                tc::fence_after_sync();
                const uint32_t pa = sbase + C::P0;
                const uint32_t va = sbase + C::ST0 + s * C::STB + C::KB;
                for (int kk = 0; kk < kGroup / 16; ++kk)   // k-steps 0, 1 -> O_A; 2, 3 -> O_B
                    tc::mma_bf16_ss(tO + (kk >> 1) * D, tc::desc_sw128(pa + kk * 32),
                                    tc::desc_sw128_mn(va + kk * 2048, kGroup * 128), idesc_o,
                                    (!first || (kk & 1)) ? 1u : 0u);
                tc::mma_commit(&kv_empty[s]);
                tc::mma_commit(&pv_done);
                return true;
            };
            // issue order S(G), P V(G - 1), across unit boundaries too: the
            // tensor core computes the next scores while the softmax runs
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
                const uint32_t qa = sbase + C::Q0 + qb * C::QB;
                for (int g = 0; g < ng; ++g, ++G) {
                    const int s = (int)(G % C::NST), sb = (int)(G & 1);
                    if (!tc::mbar_wait(&kv_full[s], (G / C::NST) & 1, tc::kWaitLimit) ||
                        (G >= 2 && !tc::mbar_wait(&s_empty[sb], ((G >> 1) - 1) & 1, tc::kWaitLimit))) {
                        ok = false;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t ka = sbase + C::ST0 + s * C::STB;
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t ao = (uint32_t)((kk >> 2) * 128 * 128 + (kk & 3) * 32);
                        const uint32_t bo = (uint32_t)((kk >> 2) * kGroup * 128 + (kk & 3) * 32);
                        tc::mma_bf16_ss(tS0 + sb * kGroup, tc::desc_sw128(qa + ao), tc::desc_sw128(ka + bo), idesc_s,
                                        kk > 0 ? 1u : 0u);
                    }
                    tc::mma_commit(&s_full[sb]);
                    if (g == ng - 1) tc::mma_commit(&q_empty[qb]);
                    if (pend >= 0 && !issue_pv(pend, pend_first, pend_u)) {
                        ok = false;
                        break;
                    }
                    pend = G;
                    pend_first = g == 0;
                    pend_u = U;
                }
            }
            if (ok && pend >= 0 && !issue_pv(pend, pend_first, pend_u)) ok = false;
            if (!ok) atomicOr(a.d_err, tc::kErrMmaTimeout);
            // every product issued is complete before TMEM is released
            tc::mma_commit(&mma_done);
            tc::mbar_wait(&mma_done, 0, tc::kWaitLimit);
        }
    } else {   // ---------------------------------------------------- softmax + epilogue
        const int quarter = warp & 3, hf = (warp - 2) >> 2, r = quarter * 32 + lane;   // TMEM lanes 32 * (warp % 4) ..
        const uint32_t tlane = (uint32_t)(quarter * 32) << 16;
        const float scale2 = kLog2e * rsqrtf((float)D);
        constexpr int DH = D / 2;   // output columns this warp writes
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
            // this warp's half of the residual result of its rows, read back at the end of the unit
            __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + ((in ? row : 0) * H + h) * D + hf * DH;
            const uint32_t stg = sbase + C::O0 + (warp - 2) * 4096;   // (STAGE) this warp's box
            if constexpr (C::STAGE) {
                if (lane == 0) {
                    if (U >= 1) tc::bulk_wait_read();   // the previous unit's store has read the box
                    tc::mbar_expect_tx(&st_full[warp - 2], 4096);
                    tc::tma_load_2d(stg, &prm.to, h * D + hf * DH, panel * 128 + quarter * 32, &st_full[warp - 2]);
                }
            } else if (in) {
#pragma unroll
                for (int b = 0; b < DH * 2; b += 128) tc::prefetch_l2(reinterpret_cast<const char *>(out) + b);
            }
            const float lr = in ? a.lse[row * H + h] : -INFINITY;
            float m = -INFINITY, l = 0.f;
            for (int g = 0; g < ng; ++g, ++G) {
                const int s = (int)(G % C::NST), sb = (int)(G & 1);
                // scores of this group (the stage's masks landed with its rows)
                if (!tc::warp_wait(&s_full[sb], (G >> 1) & 1, tc::kWaitLimit) ||
                    !tc::warp_wait(&kv_full[s], (G / C::NST) & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                float sc[32];
                {
                    uint32_t v[32];
                    tc::tmem_ld32(tS0 + sb * kGroup + hf * 32 + tlane, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) sc[i] = __uint_as_float(v[i]);
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&s_empty[sb]);
                const uint16_t *mk =
                    reinterpret_cast<const uint16_t *>(smem + C::ST0 + s * C::STB + 2 * C::KB) + hf * 2 * 128 + r;
                float mx[2] = {-INFINITY, -INFINITY};   // two independent chains
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const uint32_t bits = mk[q * 128];
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const float x = ((bits >> c) & 1u) ? sc[q * 16 + c] * scale2 : -INFINITY;
                        sc[q * 16 + c] = x;
                        mx[c & 1] = fmaxf(mx[c & 1], x);
                    }
                }
                const float smax = fmaxf(mx[0], mx[1]);
                const bool grow = smax > m + kLazy || (m == -INFINITY && smax > -INFINITY);
                const float m_new = grow ? fmaxf(m, smax) : m;
                const float alpha = tc::ex2_diff(m, m_new);
                // the previous product (which reads P and adds to O) must be done before
                // O is rescaled or P rewritten
                bool prev_done = G == 0;
                if (__any_sync(SGA_FULL_MASK, grow && l > 0.f)) {
                    // rescale this warp's rows of its half's O
                    if (!tc::warp_wait(&pv_done, (G - 1) & 1, tc::kWaitLimit)) {
                        ok = false;
                        break;
                    }
                    prev_done = true;
                    tc::fence_after_sync();
                    const float f = (grow && l > 0.f) ? alpha : 1.f;
                    for (int cb = 0; cb < D; cb += 32) {
                        uint32_t v[32];
                        tc::tmem_ld32(tO + hf * D + tlane + cb, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * f);
                        tc::tmem_st32(tO + hf * D + tlane + cb, v);
                    }
                }
                if (grow) {
                    l *= alpha;
                    m = m_new;
                }
                float pr[32], ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    pr[i] = tc::ex2_diff(sc[i], m);
                    ls[i & 3] += pr[i];
                }
                l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
                if (!prev_done && !tc::warp_wait(&pv_done, (G - 1) & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                unsigned char *prow = smem + C::P0;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    *reinterpret_cast<uint4 *>(prow + tc::sw128_offset(r, hf * 32 + c * 8, 128)) =
                        pack<__nv_bfloat16>(pr + 8 * c);
                tc::fence_proxy_async();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&p_full);
            }
            if (!ok) break;
            // epilogue: the unit's last product, the two halves merged, then the
            // tile result merged with the residual result
            if (!tc::warp_wait(&pv_done, (G - 1) & 1, tc::kWaitLimit)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            // exchange (maximum, sum) with the other half of the row (the slot is
            // rewritten only after the next unit's products, which need both halves)
            xch[hf][r] = make_float2(m, l);
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&xch_full);
            if (!tc::warp_wait(&xch_full, U & 1, tc::kWaitLimit)) {
                ok = false;
                break;
            }
            const float2 ma = xch[0][r], mb = xch[1][r];
            const float M2 = fmaxf(ma.x, mb.x);
            const float fa = tc::ex2_diff(ma.x, M2), fb = tc::ex2_diff(mb.x, M2);
            const float L = ma.y * fa + mb.y * fb;
            const bool has = L > 0.f && in;
            float wt = 0.f, wr = 0.f, lse_new = 0.f;
            if (has) {
                const float lt = (M2 + log2f(L)) * kLn2;
                const float Mx = fmaxf(lt, lr);
                wt = __expf(lt - Mx);
                wr = lr == -INFINITY ? 0.f : __expf(lr - Mx);
                lse_new = Mx + logf(wt + wr);
                const float inv = 1.f / (wt + wr);
                wt *= inv / L;   // weight of the unnormalised tile accumulator
                wr *= inv;
            }
            const float wa = wt * fa, wb = wt * fb;
            if constexpr (C::STAGE) {
                // the residual values arrived in the staged box (row = lane, 128-byte swizzle)
                if (!tc::warp_wait(&st_full[warp - 2], U & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                unsigned char *srow = smem + C::O0 + (warp - 2) * 4096 + lane * 128;
#pragma unroll
                for (int cb = 0; cb < DH; cb += 32) {
                    uint32_t va_[32], vb_[32];
                    tc::tmem_ld32(tO + hf * DH + tlane + cb, va_);   // warp-collective: every lane takes part
                    tc::tmem_ld32(tO + D + hf * DH + tlane + cb, vb_);
                    if (has) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int c = cb / 8 + q;
                            uint4 *ptr = reinterpret_cast<uint4 *>(srow + ((c ^ (lane & 7)) << 4));
                            float o[8], y[8];
                            unpack<__nv_bfloat16>(*ptr, y);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                o[i] = wa * __uint_as_float(va_[8 * q + i]) + wb * __uint_as_float(vb_[8 * q + i]) +
                                       wr * y[i];
                            *ptr = pack<__nv_bfloat16>(o);
                        }
                    }
                }
                tc::fence_proxy_async();   // the box's new values, for the TMA store
                __syncwarp();
                if (lane == 0) {
                    tc::tma_store_2d(&prm.to, h * D + hf * DH, panel * 128 + quarter * 32, stg);
                    tc::bulk_commit();
                }
            } else {
                uint4 x[DH / 8];
                if (has)
#pragma unroll
                    for (int c = 0; c < DH / 8; ++c) x[c] = *reinterpret_cast<const uint4 *>(out + 8 * c);
#pragma unroll
                for (int cb = 0; cb < DH; cb += 32) {
                    uint32_t va_[32], vb_[32];
                    tc::tmem_ld32(tO + hf * DH + tlane + cb, va_);   // warp-collective: every lane takes part
                    tc::tmem_ld32(tO + D + hf * DH + tlane + cb, vb_);
                    if (has) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            float o[8], y[8];
                            unpack<__nv_bfloat16>(x[cb / 8 + q], y);
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                o[i] = wa * __uint_as_float(va_[8 * q + i]) + wb * __uint_as_float(vb_[8 * q + i]) +
                                       wr * y[i];
                            *reinterpret_cast<uint4 *>(out + cb + 8 * q) = pack<__nv_bfloat16>(o);
                        }
                    }
                }
            }
            if (has && hf == 0) a.lse[row * H + h] = lse_new;
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&o_empty);
        }
        if (!ok && lane == 0) atomicOr(a.d_err, tc::kErrMmaTimeout);
        if constexpr (C::STAGE) {
            // a staged box whose load was issued but not consumed (only after a
            // timeout) lands before the CTA ends; every store completes
            if (lane == 0) {
                if (!ok) tc::mbar_wait(&st_full[warp - 2], U & 1, tc::kWaitLimit);   // (the unit that failed)
                tc::bulk_wait_all();
            }
        }
    }
    // the MMA lane waited for all its products; the producer for its loads
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::tmem_dealloc(tmem_base, kCols);
    }
}

template <int D> cudaError_t launch_d(const BsrArgs &a, cudaStream_t s) {
    using C = FwdCfg<D>;
    FwdParams prm{};
    prm.a = a;
    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(a.Q), *K = static_cast<const __nv_bfloat16 *>(a.K),
                        *V = static_cast<const __nv_bfloat16 *>(a.V);
    const int64_t HD = (int64_t)a.H * D;
    cudaError_t e = bf16_tensor_map(&prm.tq, Q, a.N, HD, HD, 64, 128);
    if (e == cudaSuccess)
        e = bf16_tensor_map(&prm.to, static_cast<const __nv_bfloat16 *>(a.out), a.N, HD, HD, 64, 32);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.tk, K, a.N, HD, HD, 64, 16);
    if (e == cudaSuccess) e = bf16_tensor_map(&prm.tv, V, a.N, HD, HD, 64, 16);
    if (e != cudaSuccess) return e;
    const size_t smem = C::BYTES + 1024;
    static bool configured = false;
    if (!configured) {
        e = cudaFuncSetAttribute(bsr_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int64_t units = (int64_t)a.n_active * a.H;
    const unsigned grid = (unsigned)(units < a.num_sms ? units : a.num_sms);
    note_launch(SGA_KERN_BSR_FWD, s, false);
    bsr_fwd_kernel<D><<<grid, kThreads, smem, s>>>(prm);
    note_launch(SGA_KERN_BSR_FWD, s, true);
    return cudaGetLastError();
}

}  // namespace

bool bsr_fwd_supported(sga_dtype dt, int D) { return dt == SGA_BF16 && (D == 64 || D == 128); }

cudaError_t launch_bsr_fwd(const BsrArgs &a, cudaStream_t s) {
    if (a.n_active == 0) return cudaSuccess;
    return a.D == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace sga
