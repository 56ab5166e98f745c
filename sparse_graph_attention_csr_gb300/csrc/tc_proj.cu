// tcgen05 kernel of the GATv2 projections (declared in tc_proj.cuh).
#include "gemm.cuh"
#include "tc.cuh"
#include "tc_proj.cuh"

namespace sga {

// Warps: 4 lane quarters (TMEM lanes 32q .. 32q+31 = tile rows) times
// NT / 64 column groups of 64 accumulator columns each.
constexpr int kTpMaxThreads = 512;
constexpr int kTpFix = 1024;

// A tiles in flight: three when they fit (the next tile's MMA and the load of
// the one after run during an epilogue), else two.
__host__ __device__ inline int tc_proj_abufs(int K, int HD) {
    const int KA = (K + 63) / 64;
    return 1024 + (size_t)KA * 2 * HD * 128 + 3 * (size_t)KA * 128 * 128 <= 227 * 1024 ? 3 : 2;
}
__host__ __device__ inline size_t tc_proj_smem(int K, int HD) {
    const int KA = (K + 63) / 64;
    return 1024 + (size_t)KA * 2 * HD * 128 + tc_proj_abufs(K, HD) * (size_t)KA * 128 * 128;
}

__device__ __forceinline__ float bf16_at(const unsigned char *tile, int row, int k, int R) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + tc::sw128_offset(row, k, R)));
}

// Squared Euclidean norm of row `row` of a swizzled K-major tile (16-byte reads).
__device__ __forceinline__ float row_sq(const unsigned char *tile, int row, int K, int R) {
    float q = 0.f;
    for (int c = 0; c < K / 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4 *>(tile + tc::sw128_offset(row, c * 8, R));
        float x[8];
        unpack<__nv_bfloat16>(u, x);
#pragma unroll
        for (int i = 0; i < 8; ++i) q = fmaf(x[i], x[i], q);
    }
    return q;
}

__global__ void __launch_bounds__(kTpMaxThreads, 1) tc_proj_kernel(TcProj p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ float cnorm[256], rnorm[128];
    __shared__ uint64_t mbar[2];   // MMA completion per TMEM accumulator
    __shared__ uint32_t tmem_base;
    __shared__ int2 fixl[kTpFix];
    __shared__ int fix_n;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nthr = blockDim.x;
    const int K = p.K, HD = p.HD, NT = 2 * HD, KA = (K + 63) / 64, KC = K / 8;
    const int quarter = warp & 3, cgroup = warp >> 2;   // rows 32*quarter.., columns 64*cgroup..
    const int NBUF = tc_proj_abufs(K, HD);
    unsigned char *Bs = smem;
    unsigned char *As[3];
    for (int b = 0; b < 3; ++b) As[b] = Bs + (size_t)KA * NT * 128 + (size_t)(b < NBUF ? b : 0) * KA * 16384;
    const int64_t n_tiles = (p.M + 127) / 128;
    const uint32_t idesc = tc::idesc_bf16(128, NT);
    const uint32_t tcols = NT > 128 ? 512 : 256;   // two accumulators of NT columns

    if (warp == 0) tc::tmem_alloc(&tmem_base, tcols);
    if (tid == 0) {
        tc::mbar_init(&mbar[0], 1);
        tc::mbar_init(&mbar[1], 1);
        fix_n = 0;
    }
    // B = [W_l | W_r]^T, K-major swizzled: row n = output column (loads of
    // several iterations in flight before their stores)
#pragma unroll 4
    for (int idx = tid; idx < K * (NT / 8); idx += nthr) {
        const int k = idx / (NT / 8), n0 = (idx % (NT / 8)) * 8;
        const __nv_bfloat16 *W = n0 < HD ? p.Wl : p.Wr;
        const uint4 u = ldg16(W + (size_t)k * HD + (n0 % HD));
        const __nv_bfloat16 *e = reinterpret_cast<const __nv_bfloat16 *>(&u);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            *reinterpret_cast<__nv_bfloat16 *>(Bs + tc::sw128_offset(n0 + i, k, NT)) = e[i];
    }
    auto load_a = [&](int64_t tile, int st) {
        const int64_t m0 = tile * 128;
        const uint32_t base = tc::smem_u32(As[st]);
        for (int idx = tid; idx < 128 * KC; idx += nthr) {
            const int r = idx / KC, c = idx % KC;
            const bool ok = m0 + r < p.M;
            tc::cp16(base + tc::sw128_offset(r, c * 8, 128), ok ? p.X + (m0 + r) * K + c * 8 : p.X, ok);
        }
        tc::cp_commit();
    };
    const int64_t stride = gridDim.x;
    const int64_t tile0 = blockIdx.x;
    // tiles of this CTA: tile0, tile0 + stride, ...; A of tile j sits in buffer j % NBUF
    if (tile0 < n_tiles) load_a(tile0, 0);
    if (tile0 + stride < n_tiles) load_a(tile0 + stride, 1 % NBUF);
    else tc::cp_commit();
    __syncthreads();
    for (int n = tid; n < NT; n += nthr) cnorm[n] = sqrtf(row_sq(Bs, n, K, NT));   // column norms of W
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = tmem_base;
    // D[acc] = A[buf] B^T, one elected thread
    auto issue_mma = [&](int buf, int acc) {
        tc::fence_after_sync();
        const uint32_t a0 = tc::smem_u32(As[buf]), b0 = tc::smem_u32(Bs), d = tbase + (uint32_t)(acc * NT);
        for (int kk = 0; kk < K / 16; ++kk) {
            const uint32_t ao = (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32);
            const uint32_t bo = (uint32_t)((kk >> 2) * NT * 128 + (kk & 3) * 32);
            tc::mma_bf16_ss(d, tc::desc_sw128(a0 + ao), tc::desc_sw128(b0 + bo), idesc, kk > 0);
        }
        tc::mma_commit(&mbar[acc]);
    };
    if (tile0 < n_tiles) {   // the first tile's product
        tc::cp_wait<1>();
        tc::fence_proxy_async();
        __syncthreads();
        if (tid == 0) issue_mma(0, 0);
    }

    bool failed = false;
    int64_t tile = tile0;
    for (int it = 0; tile < n_tiles; tile += stride, ++it) {
        const int st = it % NBUF, acc = it & 1;
        const bool has_next = tile + stride < n_tiles;
        // with three buffers, the tile after next loads now (its buffer held tile it - 1)
        if (NBUF == 3) {
            if (tile + 2 * stride < n_tiles) load_a(tile + 2 * stride, (it + 2) % 3);
            else tc::cp_commit();
        }
        if (has_next) {   // the next tile's product runs during this epilogue
            if (NBUF == 3) tc::cp_wait<1>();
            else tc::cp_wait<0>();
            tc::fence_proxy_async();
            __syncthreads();
            if (tid == 0) issue_mma((it + 1) % NBUF, acc ^ 1);
        }
        bool ok = tc::mbar_wait(&mbar[acc], (it >> 1) & 1, tc::kWaitLimit);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) atomicOr(p.err, tc::kErrMmaTimeout);
            failed = true;
            tc::mbar_wait(&mbar[acc], (it >> 1) & 1, tc::kWaitLimit);
            if (has_next) tc::mbar_wait(&mbar[acc ^ 1], ((it + 1) >> 1) & 1, tc::kWaitLimit);
            break;
        }
        tc::fence_after_sync();
        const uint32_t tacc = tbase + (uint32_t)(acc * NT);

        // epilogue: thread owns row r of the tile and 64 columns of it
        const int r = quarter * 32 + lane;
        const int64_t m = tile * 128 + r;
        if (cgroup == 0) rnorm[r] = sqrtf(row_sq(As[st], r, K, 128)) * (2.0f * 5.9604645e-8f);
        __syncthreads();
        const float rn = rnorm[r];
#pragma unroll 1
        for (int cc = cgroup * 2; cc < cgroup * 2 + 2; ++cc) {
            uint32_t v[32];
            tc::tmem_ld32(tacc + ((uint32_t)(quarter * 32) << 16) + cc * 32, v);
            float o[32];
            uint32_t overflow = 0;   // flagged elements the list had no room for
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float f = __uint_as_float(v[i]);
                const int col = cc * 32 + i;
                const float bound = fmaf(rn, cnorm[col], fabsf(f) * 1.2e-7f);
                o[i] = f;
                if (__float2bfloat16_rn(f - bound) != __float2bfloat16_rn(f + bound)) {
                    const int slot = atomicAdd(&fix_n, 1);
                    if (slot < kTpFix) fixl[slot] = make_int2(r, col);
                    else overflow |= 1u << i;
                }
            }
            // (not expected: about 0.5% of a tile's elements are flagged) exact sums by this thread
            for (uint32_t ov = overflow; ov; ov &= ov - 1) {
                const int i = __ffs(ov) - 1, col = cc * 32 + i;
                float hi = 0.f, lo = 0.f;
                for (int k = 0; k < K; ++k) {
                    float t, e;
                    two_sum(hi, __fmul_rn(bf16_at(As[st], r, k, 128), bf16_at(Bs, col, k, NT)), t, e);
                    hi = t;
                    lo = __fadd_rn(lo, e);
                }
#pragma unroll
                for (int q = 0; q < 32; ++q)
                    if (q == i) o[q] = __fadd_rn(hi, lo);
            }
            if (m < p.M) {
                const int c0 = cc * 32;
                __nv_bfloat16 *dst = c0 < HD ? p.FL + m * HD + c0 : p.FR + m * HD + (c0 - HD);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    reinterpret_cast<uint4 *>(dst)[q] = pack<__nv_bfloat16>(o + 8 * q);
            }
        }
        tc::fence_before_sync();
        __syncthreads();
        // exact recompute of the flagged elements: a half-warp per element,
        // lane j takes the 16-byte chunks j, j + 16, ... of the row of A and
        // of the column of W (eight exact products each), TwoSum throughout
        const int nf = min(fix_n, kTpFix);
        const int hl = lane & 15;
        for (int i0 = warp * 2; i0 < nf; i0 += nthr / 16) {
            const int i = i0 + (lane >> 4);
            const bool act = i < nf;
            const int fr = act ? fixl[i].x : 0, fc = act ? fixl[i].y : 0;
            float hi = 0.f, lo = 0.f;
            for (int c = hl; c < KC; c += 16) {
                float xa[8], xb[8];
                unpack<__nv_bfloat16>(*reinterpret_cast<const uint4 *>(As[st] + tc::sw128_offset(fr, c * 8, 128)), xa);
                unpack<__nv_bfloat16>(*reinterpret_cast<const uint4 *>(Bs + tc::sw128_offset(fc, c * 8, NT)), xb);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    float t, e;
                    two_sum(hi, __fmul_rn(xa[q], xb[q]), t, e);
                    hi = t;
                    lo = __fadd_rn(lo, e);
                }
            }
#pragma unroll
            for (int o2 = 8; o2 > 0; o2 >>= 1) {
                const float ho = __shfl_xor_sync(SGA_FULL_MASK, hi, o2);
                const float lo2 = __shfl_xor_sync(SGA_FULL_MASK, lo, o2);
                float t, e;
                two_sum(hi, ho, t, e);
                hi = t;
                lo = __fadd_rn(__fadd_rn(lo, lo2), e);
            }
            const int64_t fm = tile * 128 + fr;
            if (act && hl == 0 && fm < p.M) {
                __nv_bfloat16 *dst = fc < HD ? p.FL + fm * HD + fc : p.FR + fm * HD + (fc - HD);
                *dst = __float2bfloat16_rn(__fadd_rn(hi, lo));
            }
        }
        __syncthreads();
        if (tid == 0) fix_n = 0;
        // with two buffers, the tile after next loads into this tile's buffer now
        if (NBUF == 2 && tile + 2 * stride < n_tiles) load_a(tile + 2 * stride, st);
    }
    tc::cp_wait<0>();
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, tcols);
}

cudaError_t tc_proj(const TcProj &p, cudaStream_t s) {
    const size_t smem = tc_proj_smem(p.K, p.HD);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(tc_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem > 200 * 1024 ? (int)smem : 200 * 1024);
        if (e != cudaSuccess) return e;
        configured = true;
    }
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t tiles = (p.M + 127) / 128;
    const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
    note_launch(SGA_KERN_GATV2_PROJ, s, false);
    const int threads = 128 * (2 * p.HD / 64);   // 4 lane quarters x column groups of 64
    tc_proj_kernel<<<grid, threads, smem, s>>>(p);
    note_launch(SGA_KERN_GATV2_PROJ, s, true);
    return cudaGetLastError();
}

}  // namespace sga
