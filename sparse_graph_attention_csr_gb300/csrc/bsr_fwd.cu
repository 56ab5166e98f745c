// Block-sparse Graph Transformer forward on the tcgen05 tensor cores: the
// "Tensor Core (block-sparse) variant" of "On Efficient Scaling of GNNs via
// IO-Aware Layers Implementations" (arXiv abstract; blog post,
// "Attention-based layers" paragraph), which pays off on locally dense graphs.
//
// One CTA (4 warps, thread = panel row) per (128-row panel, head).  The
// panel's kept column tiles are taken four at a time (64 sources).  Per
// group: S = Q_panel K_group^T (128 x 64, K = D) into TMEM; each thread reads
// its row of S, masks it with the tile bitmaps, scales it and runs the online
// softmax with a lazily moved maximum (the accumulator is rescaled only when
// a row's maximum grows by more than 2^8, so P stays below 2^8); P goes to
// shared memory in bf16 and O += P V_group (128 x D, K = 64) accumulates in
// TMEM.  V rows stay in their node-major 128-byte-swizzled layout, which is
// the MN-major B operand of that product (no transpose).  The next group's K
// rows load once S has consumed K, its V rows once the previous P V product
// has consumed the other V buffer; both overlap the softmax.
//
// The residual edges (outside kept tiles) were processed beforehand by the
// CSR forward, whose out/lse sit in the output buffers; each row's tile result
// (O / l, m + log l) is merged with them by log-sum-exp.
#include "common.cuh"
#include "plan.h"
#include "tc.cuh"

namespace sga {
namespace {

constexpr int kBsThreads = 128;
constexpr int kGroup = 64;           // sources per group (four 16-wide tiles)
constexpr float kLazy = 8.0f;        // log2 growth that triggers a rescale

// One K buffer (reloaded once S has consumed it) and two V buffers (the P V
// product reads V directly): under 100 KB, so two CTAs share an SM.
struct BsLayout {   // byte offsets in dynamic shared memory (1024-aligned base)
    uint32_t q, k, v[2], p, total;
    __host__ __device__ BsLayout(int D) {
        const uint32_t DA = (uint32_t)(D + 63) / 64;
        q = 0;
        k = q + DA * 128 * 128;
        v[0] = k + DA * kGroup * 128;
        v[1] = v[0] + DA * kGroup * 128;
        p = v[1] + DA * kGroup * 128;
        total = p + 128 * 128;
    }
};

template <int D>
__global__ void __launch_bounds__(kBsThreads, 1) bsr_fwd_kernel(BsrArgs a) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t mbar_s, mbar_o;
    __shared__ uint32_t tmem_base;
    const BsLayout L(D);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int panel = blockIdx.x, h = blockIdx.y, H = a.H;
    const int32_t t0 = a.tile_ptr[panel], t1 = a.tile_ptr[panel + 1];
    const int ng = (t1 - t0 + 3) / 4;
    if (ng == 0) return;   // whole CTA: no kept tile, the residual result stands

    const int64_t r0 = (int64_t)panel * 128;
    const int r = tid;                       // panel row of this thread (TMEM lane r)
    const int64_t row = r0 + r;
    const __nv_bfloat16 *Q = static_cast<const __nv_bfloat16 *>(a.Q);
    const __nv_bfloat16 *K = static_cast<const __nv_bfloat16 *>(a.K);
    const __nv_bfloat16 *V = static_cast<const __nv_bfloat16 *>(a.V);
    const uint32_t sbase = tc::smem_u32(smem);
    constexpr int DC = D / 8;                // 16-byte chunks per head row

    if (warp == 0) tc::tmem_alloc(&tmem_base, 256);
    if (tid == 0) {
        tc::mbar_init(&mbar_s, 1);
        tc::mbar_init(&mbar_o, 1);
    }
    // Q panel rows, head h (zero rows past N)
    for (int idx = tid; idx < 128 * DC; idx += kBsThreads) {
        const int rr = idx / DC, c = idx % DC;
        const bool ok = r0 + rr < a.N;
        tc::cp16(sbase + L.q + tc::sw128_offset(rr, c * 8, 128),
                 ok ? Q + ((r0 + rr) * H + h) * D + c * 8 : Q, ok);
    }
    // rows of group g's kept tiles (zero past N or past the panel's tiles) of
    // one head of X into the swizzled tile at dst
    auto load_rows = [&](int g, const __nv_bfloat16 *X, uint32_t dst) {
        for (int idx = tid; idx < kGroup * DC; idx += kBsThreads) {
            const int jr = idx / DC, c = idx % DC;
            const int32_t ti = t0 + 4 * g + jr / 16;
            const int64_t j = ti < t1 ? (int64_t)a.tile_col[ti] * 16 + (jr % 16) : -1;
            const bool ok = j >= 0 && j < a.N;
            tc::cp16(dst + tc::sw128_offset(jr, c * 8, kGroup), ok ? X + ((size_t)j * H + h) * D + c * 8 : X, ok);
        }
        tc::cp_commit();
    };
    load_rows(0, K, sbase + L.k);   // Q travels in the same first group
    load_rows(0, V, sbase + L.v[0]);
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tO = tmem_base, tS = tmem_base + D;
    const uint32_t tlane = (uint32_t)(warp * 32) << 16;
    const uint32_t idesc_s = tc::idesc_bf16(128, kGroup), idesc_o = tc::idesc_bf16(128, D) | tc::kMajorMnB;
    const float scale2 = kLog2e * rsqrtf((float)D);

    float m = -INFINITY, l = 0.f;
    bool failed = false;
    int n_o = 0;   // P V products issued (uniform over the CTA)
    for (int g = 0; g < ng; ++g) {
        const int b = g & 1;
        tc::cp_wait<0>();   // this group's K and V rows
        // the previous P V product must be done before P, O and the other V buffer are touched
        if (g > 0 && !tc::mbar_wait(&mbar_o, (g - 1) & 1, tc::kWaitLimit)) failed = true;
        if (__syncthreads_or(failed)) break;
        tc::fence_after_sync();
        if (g + 1 < ng) load_rows(g + 1, V, sbase + L.v[b ^ 1]);   // lands during this group
        tc::fence_proxy_async();
        __syncthreads();
        if (tid == 0) {   // S = Q K^T
            tc::fence_after_sync();
            for (int kk = 0; kk < D / 16; ++kk) {
                const uint32_t ao = (uint32_t)((kk >> 2) * 128 * 128 + (kk & 3) * 32);
                const uint32_t bo = (uint32_t)((kk >> 2) * kGroup * 128 + (kk & 3) * 32);
                tc::mma_bf16_ss(tS, tc::desc_sw128(sbase + L.q + ao), tc::desc_sw128(sbase + L.k + bo),
                                idesc_s, kk > 0);
            }
            tc::mma_commit(&mbar_s);
        }
        if (!tc::mbar_wait(&mbar_s, g & 1, tc::kWaitLimit)) failed = true;
        if (__syncthreads_or(failed)) break;
        tc::fence_after_sync();
        // K is consumed: the next group's K rows load during the softmax
        if (g + 1 < ng) load_rows(g + 1, K, sbase + L.k);

        // masked, scaled scores of row r; lazy online softmax
        float s[kGroup];
        {
            uint32_t u[32];
            tc::tmem_ld32(tS + tlane, u);
#pragma unroll
            for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(u[i]);
            tc::tmem_ld32(tS + tlane + 32, u);
#pragma unroll
            for (int i = 0; i < 32; ++i) s[32 + i] = __uint_as_float(u[i]);
        }
        float smax = -INFINITY;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int32_t ti = t0 + 4 * g + q;
            const uint32_t bits = (ti < t1 && row < a.N) ? a.tile_bits[(size_t)ti * 128 + r] : 0u;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const float v = ((bits >> c) & 1u) ? s[q * 16 + c] * scale2 : -INFINITY;
                s[q * 16 + c] = v;
                smax = fmaxf(smax, v);
            }
        }
        const bool grow = smax > m + kLazy || (m == -INFINITY && smax > -INFINITY);
        const float m_new = grow ? fmaxf(m, smax) : m;
        const float alpha = exp2_diff(m, m_new);
        if (__any_sync(SGA_FULL_MASK, grow && g > 0 && l > 0.f)) {   // rescale O rows of this warp
            const float f = (grow && l > 0.f) ? alpha : 1.f;
            for (int cb = 0; cb < D; cb += 32) {
                uint32_t u[32];
                tc::tmem_ld32(tO + tlane + cb, u);
#pragma unroll
                for (int i = 0; i < 32; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * f);
                tc::tmem_st32(tO + tlane + cb, u);
            }
        }
        if (grow) {
            l *= alpha;
            m = m_new;
        }
        float pr[kGroup];
#pragma unroll
        for (int i = 0; i < kGroup; ++i) {
            pr[i] = exp2_diff(s[i], m);
            l += pr[i];
        }
        // P row -> shared memory (bf16, K-major swizzled, 64 sources = one atom)
#pragma unroll
        for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4 *>(smem + L.p + tc::sw128_offset(r, c * 8, 128)) =
                pack<__nv_bfloat16>(pr + 8 * c);
        tc::fence_before_sync();
        tc::fence_proxy_async();
        __syncthreads();
        if (tid == 0) {   // O += P V
            tc::fence_after_sync();
            // B = V rows as an MN-major operand: D-wide column atoms of 64 rows, 16 rows per k-step
            for (int kk = 0; kk < kGroup / 16; ++kk)
                tc::mma_bf16_ss(tO, tc::desc_sw128(sbase + L.p + kk * 32),
                                tc::desc_sw128_mn(sbase + L.v[b] + kk * 2048, kGroup * 128), idesc_o,
                                (g > 0 || kk > 0));
            tc::mma_commit(&mbar_o);
        }
        ++n_o;
    }
    tc::cp_wait<0>();
    if (!failed && !tc::mbar_wait(&mbar_o, (ng - 1) & 1, tc::kWaitLimit)) failed = true;
    failed = __syncthreads_or(failed);
    if (failed) {
        if (tid == 0) atomicOr(a.d_err, tc::kErrMmaTimeout);
        // let the last product issued finish (bounded) before TMEM is released
        if (n_o > 0) tc::mbar_wait(&mbar_o, (n_o - 1) & 1, tc::kWaitLimit);
    } else {
        tc::fence_after_sync();
        // merge the tile result of row r with the residual result already stored
        const bool has = l > 0.f && row < a.N;
        __nv_bfloat16 *out = static_cast<__nv_bfloat16 *>(a.out) + (row * H + h) * D;
        float wt = 0.f, wr = 0.f, lse_new = 0.f;
        if (has) {
            const float lt = (m + log2f(l)) * kLn2, lr = a.lse[row * H + h];
            const float M = fmaxf(lt, lr);
            wt = __expf(lt - M);
            wr = lr == -INFINITY ? 0.f : __expf(lr - M);
            lse_new = M + logf(wt + wr);
            const float inv = 1.f / (wt + wr);
            wt *= inv / l;        // weight of the unnormalised tile accumulator
            wr *= inv;
        }
        for (int cb = 0; cb < D; cb += 32) {
            uint32_t u[32];
            tc::tmem_ld32(tO + tlane + cb, u);   // warp-collective: every lane takes part
            if (has) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float o[8], x[8];
                    unpack<__nv_bfloat16>(*reinterpret_cast<const uint4 *>(out + cb + 8 * q), x);
#pragma unroll
                    for (int i = 0; i < 8; ++i) o[i] = wt * __uint_as_float(u[8 * q + i]) + wr * x[i];
                    *reinterpret_cast<uint4 *>(out + cb + 8 * q) = pack<__nv_bfloat16>(o);
                }
            }
        }
        if (has) a.lse[row * H + h] = lse_new;
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tmem_base, 256);
}

template <int D> cudaError_t launch_d(const BsrArgs &a, cudaStream_t s) {
    const BsLayout L(D);
    // at least 100 KB: at most two CTAs (2 x 256 TMEM columns) share an SM
    const size_t smem = L.total + 1024 > 100 * 1024 ? L.total + 1024 : 100 * 1024;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(bsr_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    dim3 grid((unsigned)a.n_panels, (unsigned)a.H);
    note_launch(SGA_KERN_BSR_FWD, s, false);
    bsr_fwd_kernel<D><<<grid, kBsThreads, smem, s>>>(a);
    note_launch(SGA_KERN_BSR_FWD, s, true);
    return cudaGetLastError();
}

}  // namespace

bool bsr_fwd_supported(sga_dtype dt, int D) { return dt == SGA_BF16 && (D == 64 || D == 128); }

cudaError_t launch_bsr_fwd(const BsrArgs &a, cudaStream_t s) {
    if (a.n_panels == 0) return cudaSuccess;
    return a.D == 128 ? launch_d<128>(a, s) : launch_d<64>(a, s);
}

}  // namespace sga
