// tcgen05 + TMA kernel of the GATv2 input gradient (declared in tc_dx.cuh).
//
// Persistent CTAs over 128-row tiles, warp-specialised:
//   warp 0, one lane: TMA loads of A atoms (128 rows x 64 bf16 of one of the
//     four K segments) into a ring of kStages shared-memory stages, each
//     signalling a "full" mbarrier with its byte count;
//   warp 1, one lane: for each atom four 128 x F x 16 MMAs into one of two
//     TMEM accumulators; tcgen05.commit frees the stage ("empty") and, after a
//     tile's last atom, hands the accumulator to the epilogue ("tfull");
//   warps 2-5: the epilogue reads the accumulator (warp w owns TMEM lanes
//     32 (w mod 4) ..), rounds to bf16, stores dX rows and frees the
//     accumulator ("tempty").
// The weights are staged once per CTA.  Every wait is bounded: on a timeout
// the role sets the error word and stops; before TMEM is released the MMA
// lane waits for its last products and the TMA lane for its last loads.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "tc.cuh"
#include "tc_dx.cuh"

namespace sga {
namespace {

constexpr int kStages = 8;
constexpr int kThreads = 192;
constexpr uint32_t kAtomBytes = 128 * 128;   // 128 rows x 64 bf16

struct DxParams {
    CUtensorMap ta[2];                       // dFL, dFR as [M][2 HD] bf16, box 64 x 128, 128-byte swizzle
    const __nv_bfloat16 *Wl, *Wr;
    __nv_bfloat16 *dX;
    int64_t M;
    int F, HD;
    int32_t *err;
};

__device__ __forceinline__ void mbar_expect_tx(uint64_t *mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(mbar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(mbar)) : "memory");
}
// 2-D tiled TMA load of the box at (x, y) into shared memory, completing on mbar.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_u32(mbar))
        : "memory");
}

__host__ __device__ inline size_t dx_b_bytes(int F, int HD) { return (size_t)2 * (HD / 64) * F * 128; }
__host__ __device__ inline size_t dx_smem(int F, int HD) { return 1024 + dx_b_bytes(F, HD) + kStages * kAtomBytes; }

__global__ void __launch_bounds__(kThreads, 1) tc_dx_kernel(const __grid_constant__ DxParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[kStages], empty[kStages], tfull[2], tempty[2], done;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int F = p.F, HD = p.HD, AS = HD / 64, NA = 4 * AS;   // atoms per K segment, per tile
    // (F is a multiple of 32: the epilogue's 32-column TMEM loads stay inside one accumulator)
    const int64_t n_tiles = (p.M + 127) / 128;
    const uint32_t sB = tc::smem_u32(smem), sA = sB + (uint32_t)dx_b_bytes(F, HD);
    const uint32_t tcols = 2 * F <= 32 ? 32 : (2 * F <= 64 ? 64 : (2 * F <= 128 ? 128 : (2 * F <= 256 ? 256 : 512)));

    if (warp == 0) tc::tmem_alloc(&tmem_base, tcols);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], 128);
        }
        tc::mbar_init(&done, 1);
    }
    // B: W_l atoms then W_r atoms, rows f (output column), K-major, 128-byte swizzled
    for (int idx = tid; idx < 2 * F * (HD / 8); idx += kThreads) {
        const int x = idx / (F * (HD / 8)), r = idx % (F * (HD / 8));
        const int f = r / (HD / 8), c = r % (HD / 8);
        const __nv_bfloat16 *W = x ? p.Wr : p.Wl;
        tc::cp16(sB + (uint32_t)(x * AS * F * 128) + tc::sw128_offset(f, c * 8, F), W + (size_t)f * HD + c * 8,
                 true);
    }
    tc::cp_commit();
    tc::cp_wait<0>();
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = tmem_base;

    if (warp == 0 && lane == 0) {   // ---------------- TMA producer
        int q = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x)
            for (int j = 0; j < NA; ++j, ++q) {
                const int s = q % kStages, n = q / kStages;
                if (n >= 1 && !tc::mbar_wait(&empty[s], (n - 1) & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                const int seg = j / AS, a = j % AS;   // seg: dFL hi, dFL lo, dFR hi, dFR lo
                mbar_expect_tx(&full[s], kAtomBytes);
                tma_load_2d(sA + (uint32_t)s * kAtomBytes, &p.ta[seg >> 1], (seg & 1) * HD + a * 64, (int)(t * 128),
                            &full[s]);
            }
        if (!ok) atomicOr(p.err, tc::kErrMmaTimeout);
        // loads issued but not consumed (only after a timeout) must land before the CTA ends
        for (int i = q - 1; i >= 0 && i >= q - kStages; --i)
            tc::mbar_wait(&full[i % kStages], (i / kStages) & 1, tc::kWaitLimit);
    } else if (warp == 1 && lane == 0) {   // ---------------- MMA issuer
        const uint32_t idesc = tc::idesc_bf16(128, F);
        int q = 0, tl = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++tl) {
            const int acc = tl & 1, u = tl >> 1;
            if (u >= 1 && !tc::mbar_wait(&tempty[acc], (u - 1) & 1, tc::kWaitLimit)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            const uint32_t d = tbase + (uint32_t)(acc * F);
            for (int j = 0; j < NA; ++j, ++q) {
                const int s = q % kStages, n = q / kStages;
                if (!tc::mbar_wait(&full[s], n & 1, tc::kWaitLimit)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const int seg = j / AS, a = j % AS;
                const uint32_t a0 = sA + (uint32_t)s * kAtomBytes;
                const uint32_t b0 = sB + (uint32_t)(((seg >> 1) * AS + a) * F * 128);
                for (int kk = 0; kk < 4; ++kk)
                    tc::mma_bf16_ss(d, tc::desc_sw128(a0 + kk * 32), tc::desc_sw128(b0 + kk * 32), idesc,
                                    (j > 0 || kk > 0) ? 1u : 0u);
                tc::mma_commit(&empty[s]);
            }
            if (ok) tc::mma_commit(&tfull[acc]);
        }
        if (!ok) atomicOr(p.err, tc::kErrMmaTimeout);
        tc::mma_commit(&done);   // completes when every product issued above has
        tc::mbar_wait(&done, 0, tc::kWaitLimit);
    } else if (warp >= 2) {   // ---------------- epilogue
        const int quarter = warp & 3, r = quarter * 32 + lane;
        int tl = 0;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++tl) {
            const int acc = tl & 1, u = tl >> 1;
            const bool ok = tc::mbar_wait(&tfull[acc], u & 1, tc::kWaitLimit);
            if (__any_sync(SGA_FULL_MASK, !ok)) {
                if (lane == 0) atomicOr(p.err, tc::kErrMmaTimeout);
                break;
            }
            tc::fence_after_sync();
            const int64_t m = t * 128 + r;
            const uint32_t src = tbase + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * F);
            for (int cb = 0; cb < F; cb += 32) {
                uint32_t v[32];
                tc::tmem_ld32(src + cb, v);   // warp-collective
                if (m < p.M) {
                    float o[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __uint_as_float(v[i]);
                    uint4 *dst = reinterpret_cast<uint4 *>(p.dX + m * F + cb);
#pragma unroll
                    for (int qd = 0; qd < 4; ++qd) dst[qd] = pack<__nv_bfloat16>(o + 8 * qd);
                }
            }
            tc::fence_before_sync();
            mbar_arrive(&tempty[acc]);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::tmem_dealloc(tbase, tcols);
    }
}

// ---------------------------------------------------------------- dW

constexpr int kDwThreads = 128;
constexpr uint32_t kBox = 64 * 128;   // TMA box: 64 node rows x 64 bf16 (128 bytes)

struct DwParams {
    CUtensorMap tx;      // X as [M][F], box 64 x 64
    CUtensorMap tf[2];   // dFL, dFR as [M][2 HD], box 64 x 64
    float *part;
    int64_t M;
    int F, HD, slab_rows, slabs;
    int32_t *err;
};

// Per stage: X boxes (F / 64), then dF boxes ordered (w, hi/lo, h block).
__host__ __device__ inline uint32_t dw_stage_bytes(int F, int HD) {
    return (uint32_t)(F / 64 + 4 * (HD / 64)) * kBox;
}
// two stages, plus a pad that keeps every descriptor read inside the allocation
__host__ __device__ inline size_t dw_smem(int F, int HD) { return 1024 + 2 * (size_t)dw_stage_bytes(F, HD) + 16384; }

__global__ void __launch_bounds__(kDwThreads, 1) tc_dw_kernel(const __grid_constant__ DwParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ uint64_t full[2], empty[2], done;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int F = p.F, HD = p.HD, FB = F / 64, AS = HD / 64;
    const uint32_t stage = dw_stage_bytes(F, HD), sbase = tc::smem_u32(smem);
    const int64_t r0 = (int64_t)blockIdx.x * p.slab_rows;
    const int64_t rows = min((int64_t)p.slab_rows, p.M - r0);
    const int nchunks = rows > 0 ? (int)((rows + 63) / 64) : 0;
    const uint32_t tcols = 2 * HD <= 128 ? 128 : 256;   // dW_l then dW_r accumulators, HD columns each

    if (warp == 0) tc::tmem_alloc(&tmem_base, tcols);
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&full[b], 1);
            tc::mbar_init(&empty[b], 1);
        }
        tc::mbar_init(&done, 1);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = tmem_base;
    bool failed = false;

    if (warp == 0 && lane == 0) {   // ---------------- TMA producer
        int c = 0;
        for (; c < nchunks; ++c) {
            const int s = c & 1, n = c >> 1;
            if (n >= 1 && !tc::mbar_wait(&empty[s], (n - 1) & 1, tc::kWaitLimit)) {
                failed = true;
                break;
            }
            const int y = (int)(r0 + 64 * c);
            const uint32_t st = sbase + (uint32_t)s * stage;
            mbar_expect_tx(&full[s], stage);
            for (int fb = 0; fb < FB; ++fb) tma_load_2d(st + fb * kBox, &p.tx, fb * 64, y, &full[s]);
            for (int w = 0; w < 2; ++w)
                for (int part = 0; part < 2; ++part)
                    for (int a = 0; a < AS; ++a)
                        tma_load_2d(st + (uint32_t)(FB + (w * 2 + part) * AS + a) * kBox, &p.tf[w], part * HD + a * 64,
                                    y, &full[s]);
        }
        if (failed) atomicOr(p.err, tc::kErrMmaTimeout);
        for (int i = c - 1; i >= 0 && i >= c - 2; --i)   // issued loads land before the CTA ends
            tc::mbar_wait(&full[i & 1], (i >> 1) & 1, tc::kWaitLimit);
    } else if (warp == 1 && lane == 0) {   // ---------------- MMA issuer
        // M = F (A = X^T, MN-major), N = HD (B = dF^T, MN-major), K = 64 nodes per chunk
        const uint32_t idesc = tc::idesc_bf16(128, HD) | tc::kMajorMnA | tc::kMajorMnB;
        for (int c = 0; c < nchunks; ++c) {
            const int s = c & 1, n = c >> 1;
            if (!tc::mbar_wait(&full[s], n & 1, tc::kWaitLimit)) {
                failed = true;
                break;
            }
            tc::fence_after_sync();
            const uint32_t st = sbase + (uint32_t)s * stage;
            for (int w = 0; w < 2; ++w)
                for (int part = 0; part < 2; ++part) {
                    const uint32_t b0 = st + (uint32_t)(FB + (w * 2 + part) * AS) * kBox;
                    for (int kk = 0; kk < 4; ++kk)   // 16 nodes = two 8-row K groups per step
                        tc::mma_bf16_ss(tbase + (uint32_t)(w * HD), tc::desc_sw128_mn(st + kk * 2048, kBox),
                                        tc::desc_sw128_mn(b0 + kk * 2048, kBox), idesc,
                                        (c > 0 || part > 0 || kk > 0) ? 1u : 0u);
                }
            tc::mma_commit(&empty[s]);
        }
        if (failed) atomicOr(p.err, tc::kErrMmaTimeout);
        tc::mma_commit(&done);
    }
    // ---------------- epilogue (all four warps): TMEM lane f = row f of dW
    const bool ok = nchunks == 0 || tc::mbar_wait(&done, 0, tc::kWaitLimit);
    __syncwarp();   // warps 0 and 1 reconverge before the warp-collective TMEM loads
    tc::fence_after_sync();
    const int f = warp * 32 + lane;
    for (int w = 0; w < 2; ++w)
        for (int cb = 0; cb < HD; cb += 32) {
            uint32_t v[32];
            tc::tmem_ld32(tbase + ((uint32_t)(warp * 32) << 16) + (uint32_t)(w * HD + cb), v);   // warp-collective
            if (f < F && ok) {
                float4 *dst = reinterpret_cast<float4 *>(
                    p.part + (((size_t)w * p.slabs + blockIdx.x) * F + f) * HD + cb);
                if (nchunks == 0) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                             __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
                }
            }
        }
    if (!ok && tid == 0) atomicOr(p.err, tc::kErrMmaTimeout);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::tmem_dealloc(tbase, tcols);
    }
}

}  // namespace

namespace {

// The driver's tensor-map encoder, looked up once through the runtime.
cudaError_t tmap_encoder(PFN_cuTensorMapEncodeTiled_v12000 &out) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    out = encode;
    return cudaSuccess;
}

}  // namespace

cudaError_t bf16_tensor_map(CUtensorMap *m, const __nv_bfloat16 *base, int64_t rows, int64_t cols,
                            int64_t row_elems, uint32_t box_cols, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 encode;
    cudaError_t e = tmap_encoder(encode);
    if (e != cudaSuccess) return e;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_elems * sizeof(__nv_bfloat16)};
    const cuuint32_t box[2] = {box_cols, box_rows}, estr[2] = {1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t tc_dx(const TcDx &p, cudaStream_t s) {
    if (p.M == 0) return cudaSuccess;
    PFN_cuTensorMapEncodeTiled_v12000 encode;
    if (cudaError_t e = tmap_encoder(encode); e != cudaSuccess) return e;
    DxParams dp{};
    const __nv_bfloat16 *src[2] = {p.dfl, p.dfr};
    for (int i = 0; i < 2; ++i) {
        const cuuint64_t dims[2] = {(cuuint64_t)(2 * p.HD), (cuuint64_t)p.M};
        const cuuint64_t strides[1] = {(cuuint64_t)(2 * p.HD) * sizeof(__nv_bfloat16)};
        const cuuint32_t box[2] = {64, 128}, estr[2] = {1, 1};
        const CUresult r = encode(&dp.ta[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(src[i]),
                                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    dp.Wl = p.Wl;
    dp.Wr = p.Wr;
    dp.dX = p.dX;
    dp.M = p.M;
    dp.F = p.F;
    dp.HD = p.HD;
    dp.err = p.err;
    const size_t smem = dx_smem(p.F, p.HD);
    if (cudaError_t e = allow_smem<tc_dx_kernel>(smem); e != cudaSuccess) return e;
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t tiles = (p.M + 127) / 128;
    const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
    tc_dx_kernel<<<grid, kThreads, smem, s>>>(dp);
    return cudaGetLastError();
}

cudaError_t tc_dw(const TcDw &p, cudaStream_t s) {
    if (p.slabs == 0) return cudaSuccess;
    DwParams dp{};
    cudaError_t e = bf16_tensor_map(&dp.tx, p.X, p.M, p.F, p.F, 64, 64);
    if (e == cudaSuccess) e = bf16_tensor_map(&dp.tf[0], p.dfl, p.M, 2 * p.HD, 2 * p.HD, 64, 64);
    if (e == cudaSuccess) e = bf16_tensor_map(&dp.tf[1], p.dfr, p.M, 2 * p.HD, 2 * p.HD, 64, 64);
    if (e != cudaSuccess) return e;
    dp.part = p.part;
    dp.M = p.M;
    dp.F = p.F;
    dp.HD = p.HD;
    dp.slab_rows = p.slab_rows;
    dp.slabs = p.slabs;
    dp.err = p.err;
    const size_t smem = dw_smem(p.F, p.HD);
    if ((e = allow_smem<tc_dw_kernel>(smem)) != cudaSuccess) return e;
    tc_dw_kernel<<<(unsigned)p.slabs, kDwThreads, smem, s>>>(dp);
    return cudaGetLastError();
}

}  // namespace sga
