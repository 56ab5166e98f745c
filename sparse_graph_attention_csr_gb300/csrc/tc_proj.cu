// tcgen05 + TMA kernel of the GATv2 projections (declared in tc_proj.cuh).
//
// Persistent CTAs over 128-row tiles of X, warp-specialised:
//   warp 0, one lane: TMA loads of a tile's X rows (K/64 atoms of 128 rows x
//     64 bf16, 128-byte swizzle) into one of nslot slots ("sfull");
//   warp 1, one lane: the tile's MMAs (128 x 2HD x 16) into one of two TMEM
//     accumulators ("tfull");
//   warps 2-17: the epilogue.  Warp w reads TMEM lanes 32 (w mod 4) .. (tile
//     rows) and every fourth 32-column chunk, checks whether each fp32 value's
//     bf16 rounding is settled (bound 2 * 2^-24 |x||w| + ulp; two values per
//     packed instruction), stores FL/FR,
//     frees the accumulator ("tempty"), then recomputes the flagged elements
//     exactly from the slot's X rows and the staged weights (four lanes per
//     element, TwoSum) and frees the slot ("sempty").
// The weights [W_l | W_r] are transposed into the K-major operand once per
// CTA.  Every mbarrier wait is bounded; the epilogue warps take their
// timeout decision together (barrier reduction), so none is left at a named
// barrier.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "gemm.cuh"
#include "tc.cuh"
#include "tc_dx.cuh"
#include "tc_proj.cuh"

namespace sga {
namespace {

constexpr int kEpiWarps = 16, kEpiThreads = 32 * kEpiWarps, kThreads = 64 + kEpiThreads;
constexpr int kColGroups = kEpiWarps / 4;   // epilogue warps per TMEM lane quarter
constexpr int kTpFix = 1024;
constexpr uint32_t kAtom = 128 * 128;   // 128 rows x 64 bf16

struct ProjParams {
    CUtensorMap tx;   // X as [M][K] bf16, box 64 x 128
    const __nv_bfloat16 *Wl, *Wr;
    __nv_bfloat16 *FL, *FR;
    int64_t M;
    int K, HD, nslot;
    int32_t *err;
};

// static shared memory of the kernel, with room to spare (norms, barriers, fix list)
constexpr size_t kStaticSmem = 16 * 1024;

__host__ __device__ inline size_t proj_b_bytes(int K, int HD) { return (size_t)((K + 63) / 64) * 2 * HD * 128; }
// X slots in flight: three when they fit beside the static arrays, else two
__host__ __device__ inline int proj_slots(int K, int HD) {
    const size_t slot = (size_t)((K + 63) / 64) * kAtom;
    return 1024 + proj_b_bytes(K, HD) + 3 * slot + kStaticSmem <= 227 * 1024 ? 3 : 2;
}
__host__ __device__ inline size_t proj_smem(int K, int HD) {
    return 1024 + proj_b_bytes(K, HD) + (size_t)proj_slots(K, HD) * ((K + 63) / 64) * kAtom;
}

__device__ __forceinline__ void sts16(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// Both fp32 values rounded to bf16 (round to nearest even), packed low = a.
__device__ __forceinline__ uint32_t bf16x2_bits(float a, float b) {
    const __nv_bfloat162 r = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tc::smem_u32(mbar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(mbar)) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint64_t *mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(tc::smem_u32(mbar))
        : "memory");
}
// Named barrier 1 over the epilogue warps.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }
// The same barrier, returning whether any epilogue thread passed `flag`.
__device__ __forceinline__ bool epi_any(bool flag) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbarrier.red.or.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r) : "r"((uint32_t)flag), "n"(kEpiThreads) : "memory");
    return r != 0;
}

__device__ __forceinline__ float bf16_at(uint32_t tile, int row, int k, int R) {
    __nv_bfloat16 v;
    asm volatile("ld.shared.b16 %0, [%1];" : "=h"(*reinterpret_cast<unsigned short *>(&v))
                 : "r"(tile + tc::sw128_offset(row, k, R)));
    return __bfloat162float(v);
}
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
    uint4 u;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w) : "r"(addr));
    return u;
}
// Squared Euclidean norm of row `row` of a swizzled K-major tile of R rows.
__device__ __forceinline__ float row_sq(uint32_t tile, int row, int K, int R) {
    float q = 0.f;
    for (int c = 0; c < K / 8; ++c) {
        float x[8];
        unpack<__nv_bfloat16>(lds16(tile + tc::sw128_offset(row, c * 8, R)), x);
#pragma unroll
        for (int i = 0; i < 8; ++i) q = fmaf(x[i], x[i], q);
    }
    return q;
}

__global__ void __launch_bounds__(kThreads, 1) tc_proj_kernel(const __grid_constant__ ProjParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(16) float cnorm[256];
    __shared__ float rsq[kColGroups][128];   // quarters of each tile row's squared norm
    __shared__ uint64_t sfull[3], sempty[3], tfull[2], tempty[2], done;
    __shared__ uint32_t tmem_base;
    __shared__ int2 fixl[kTpFix];
    __shared__ int fix_n;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int K = p.K, HD = p.HD, NT = 2 * HD, KA = (K + 63) / 64, KC = K / 8, NS = p.nslot;
    const uint32_t sB = tc::smem_u32(smem), sX = sB + (uint32_t)proj_b_bytes(K, HD), slot_bytes = KA * kAtom;
    const int64_t n_tiles = (p.M + 127) / 128;
    const uint32_t tcols = NT > 128 ? 512 : (NT > 64 ? 256 : 128);   // two accumulators of NT columns

    if (warp == 0) tc::tmem_alloc(&tmem_base, tcols);
    if (tid == 0) {
        for (int s = 0; s < 3; ++s) {
            tc::mbar_init(&sfull[s], 1);
            tc::mbar_init(&sempty[s], kEpiThreads);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], kEpiThreads);
        }
        tc::mbar_init(&done, 1);
        fix_n = 0;
    }
    // B = [W_l | W_r]^T, K-major swizzled: row n = output column.  A thread
    // moves one 8 x 8 block (W rows 8 kc .., columns n0 ..): eight 16-byte
    // loads, a transpose in registers, eight 16-byte stores.  k-chunks vary
    // fastest across the warp, so the eight chunks of one B row land in
    // distinct bank groups (no conflicts beyond the four wavefronts of 512 B).
    for (int blk = tid; blk < KC * (NT / 8); blk += kThreads) {
        const int kc = blk % KC, n0 = (blk / KC) * 8;
        const __nv_bfloat16 *W = (n0 < HD ? p.Wl : p.Wr) + (size_t)kc * 8 * HD + (n0 % HD);
        uint4 rw[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) rw[q] = ldg16(W + (size_t)q * HD);
#pragma unroll
        for (int i = 0; i < 8; ++i) {   // column n0 + i: element i of each row, rows in pairs
            const uint32_t sel = (i & 1) ? 0x7632u : 0x5410u;
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t a = (&rw[2 * q].x)[i >> 1], b = (&rw[2 * q + 1].x)[i >> 1];
                w[q] = __byte_perm(a, b, sel);
            }
            sts16(sB + tc::sw128_offset(n0 + i, kc * 8, NT), make_uint4(w[0], w[1], w[2], w[3]));
        }
    }
    __syncthreads();
    for (int n = tid; n < NT; n += kThreads) cnorm[n] = sqrtf(row_sq(sB, n, K, NT));   // column norms of W
    tc::fence_proxy_async();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = tmem_base;

    if (warp == 0 && lane == 0) {   // ---------------- TMA producer
        int it = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
            const int s = it % NS, n = it / NS;
            if (n >= 1 && !tc::mbar_wait(&sempty[s], (n - 1) & 1, tc::kWaitLimit)) {
                ok = false;
                break;
            }
            mbar_expect_tx(&sfull[s], slot_bytes);
            for (int a = 0; a < KA; ++a)
                tma_load_2d(sX + (uint32_t)s * slot_bytes + a * kAtom, &p.tx, a * 64, (int)(t * 128), &sfull[s]);
        }
        if (!ok) atomicOr(p.err, tc::kErrMmaTimeout);
        for (int i = it - 1; i >= 0 && i >= it - NS; --i)   // issued loads land before the CTA ends
            tc::mbar_wait(&sfull[i % NS], (i / NS) & 1, tc::kWaitLimit);
    } else if (warp == 1 && lane == 0) {   // ---------------- MMA issuer
        const uint32_t idesc = tc::idesc_bf16(128, NT);
        int it = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
            const int s = it % NS, n = it / NS, acc = it & 1, u = it >> 1;
            if ((u >= 1 && !tc::mbar_wait(&tempty[acc], (u - 1) & 1, tc::kWaitLimit)) ||
                !tc::mbar_wait(&sfull[s], n & 1, tc::kWaitLimit)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            const uint32_t a0 = sX + (uint32_t)s * slot_bytes, d = tbase + (uint32_t)(acc * NT);
            for (int kk = 0; kk < K / 16; ++kk) {
                const uint32_t ao = (uint32_t)((kk >> 2) * kAtom + (kk & 3) * 32);
                const uint32_t bo = (uint32_t)((kk >> 2) * NT * 128 + (kk & 3) * 32);
                tc::mma_bf16_ss(d, tc::desc_sw128(a0 + ao), tc::desc_sw128(sB + bo), idesc, kk > 0);
            }
            tc::mma_commit(&tfull[acc]);
        }
        if (!ok) atomicOr(p.err, tc::kErrMmaTimeout);
        tc::mma_commit(&done);   // completes when every product issued above has
        tc::mbar_wait(&done, 0, tc::kWaitLimit);
    } else if (warp >= 2) {   // ---------------- epilogue
        const int ew = warp - 2, et = tid - 64, quarter = warp & 3, cgroup = ew >> 2;
        const int r = quarter * 32 + lane;   // tile row = TMEM lane
        int it = 0;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
            const int s = it % NS, acc = it & 1;
            const bool ok = tc::mbar_wait(&tfull[acc], (it >> 1) & 1, tc::kWaitLimit) &&
                            tc::mbar_wait(&sfull[s], (it / NS) & 1, tc::kWaitLimit);   // the X rows, for the norms
            if (epi_any(!ok)) {
                if (et == 0) atomicOr(p.err, tc::kErrMmaTimeout);
                break;
            }
            tc::fence_after_sync();
            const uint32_t xs = sX + (uint32_t)s * slot_bytes;
            const int64_t m = t * 128 + r;
            {   // the lane quarter's four column groups split the row norm's K range
                const int c0 = cgroup * (KC / kColGroups), c1 = c0 + KC / kColGroups;
                float q0 = 0.f, q1 = 0.f;
                for (int c = c0; c < c1; ++c) {
                    float x[8];
                    unpack<__nv_bfloat16>(lds16(xs + tc::sw128_offset(r, c * 8, 128)), x);
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        q0 = fmaf(x[i], x[i], q0);
                        q1 = fmaf(x[i + 1], x[i + 1], q1);
                    }
                }
                rsq[cgroup][r] = q0 + q1;
            }
            epi_sync();   // (the next tile's writes come after this tile's later barriers)
            const float rn = sqrtf(((rsq[0][r] + rsq[1][r]) + rsq[2][r]) + rsq[3][r]) * (2.0f * 5.9604645e-8f);
#pragma unroll 1
            for (int cc = cgroup; cc < NT / 32; cc += kColGroups) {
                uint32_t v[32];
                tc::tmem_ld32(tbase + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * NT + cc * 32), v);
                // two values a step: their bf16 bits, and whether each one's
                // rounding is settled (both ends of [f - bound, f + bound] round
                // to the same bf16)
                uint32_t packed[16], flags = 0, overflow = 0;   // unsettled; those the list had no room for
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float2 f = make_float2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                    const float2 cn = *reinterpret_cast<const float2 *>(cnorm + cc * 32 + 2 * j);
                    const float2 b = ffma2(make_float2(rn, rn), cn,
                                           fmul2(make_float2(fabsf(f.x), fabsf(f.y)), make_float2(1.2e-7f, 1.2e-7f)));
                    const float2 lo = fadd2(f, make_float2(-b.x, -b.y)), hi = fadd2(f, b);
                    packed[j] = bf16x2_bits(f.x, f.y);
                    const uint32_t d = bf16x2_bits(lo.x, lo.y) ^ bf16x2_bits(hi.x, hi.y);
                    flags |= ((d & 0xffffu) != 0u ? 1u : 0u) << (2 * j);
                    flags |= ((d >> 16) != 0u ? 1u : 0u) << (2 * j + 1);
                }
                for (uint32_t fl = flags; fl; fl &= fl - 1) {
                    const int i = __ffs(fl) - 1;
                    const int slot = atomicAdd(&fix_n, 1);
                    if (slot < kTpFix) fixl[slot] = make_int2(r, cc * 32 + i);
                    else overflow |= 1u << i;
                }
                const int c0 = cc * 32;
                __nv_bfloat16 *dst = c0 < HD ? p.FL + m * HD + c0 : p.FR + m * HD + (c0 - HD);
                if (m < p.M) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        reinterpret_cast<uint4 *>(dst)[q] =
                            make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                }
                // (not expected: the list holds about eight times the usual count)
                // exact sums by this thread, stored over the plain values
                for (uint32_t ov = overflow; ov; ov &= ov - 1) {
                    const int i = __ffs(ov) - 1, col = cc * 32 + i;
                    float hi = 0.f, lo = 0.f;
                    for (int k = 0; k < K; ++k) {
                        float tt, e;
                        two_sum(hi, __fmul_rn(bf16_at(xs, r, k, 128), bf16_at(sB, col, k, NT)), tt, e);
                        hi = tt;
                        lo = __fadd_rn(lo, e);
                    }
                    if (m < p.M) dst[i] = __float2bfloat16_rn(__fadd_rn(hi, lo));
                }
            }
            tc::fence_before_sync();
            mbar_arrive(&tempty[acc]);   // the accumulator may take the tile after next
            epi_sync();                  // every flagged element is listed (and its plain value stored)
            // exact recompute: four lanes per element (eight elements a warp),
            // lane j of a group takes 16-byte chunks j, j + 4, ... of the X row
            // and of the W column
            const int nf = min(fix_n, kTpFix), hl = lane & 3;
            for (int i0 = ew * 8; i0 < nf; i0 += 8 * kEpiWarps) {
                const int i = i0 + (lane >> 2);
                const bool act = i < nf;
                const int fr = act ? fixl[i].x : 0, fc = act ? fixl[i].y : 0;
                float hi = 0.f, lo = 0.f;
                for (int c = hl; c < KC; c += 4) {
                    float xa[8], xb[8];
                    unpack<__nv_bfloat16>(lds16(xs + tc::sw128_offset(fr, c * 8, 128)), xa);
                    unpack<__nv_bfloat16>(lds16(sB + tc::sw128_offset(fc, c * 8, NT)), xb);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        float tt, e;
                        two_sum(hi, __fmul_rn(xa[q], xb[q]), tt, e);
                        hi = tt;
                        lo = __fadd_rn(lo, e);
                    }
                }
#pragma unroll
                for (int o2 = 2; o2 > 0; o2 >>= 1) {
                    const float ho = __shfl_xor_sync(SGA_FULL_MASK, hi, o2);
                    const float lo2 = __shfl_xor_sync(SGA_FULL_MASK, lo, o2);
                    float tt, e;
                    two_sum(hi, ho, tt, e);
                    hi = tt;
                    lo = __fadd_rn(__fadd_rn(lo, lo2), e);
                }
                const int64_t fm = t * 128 + fr;
                if (act && hl == 0 && fm < p.M) {
                    __nv_bfloat16 *dst = fc < HD ? p.FL + fm * HD + fc : p.FR + fm * HD + (fc - HD);
                    *dst = __float2bfloat16_rn(__fadd_rn(hi, lo));
                }
            }
            epi_sync();   // the list is consumed
            if (et == 0) fix_n = 0;
            epi_sync();   // the reset is seen before the next tile's flags
            mbar_arrive(&sempty[s]);   // the slot's X rows are no longer read
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        __syncwarp();
        tc::tmem_dealloc(tbase, tcols);
    }
}

}  // namespace

cudaError_t tc_proj(const TcProj &p, cudaStream_t s) {
    if (p.M == 0) return cudaSuccess;
    ProjParams pp{};
    cudaError_t e = bf16_tensor_map(&pp.tx, p.X, p.M, p.K, p.K, 64, 128);
    if (e != cudaSuccess) return e;
    pp.Wl = p.Wl;
    pp.Wr = p.Wr;
    pp.FL = p.FL;
    pp.FR = p.FR;
    pp.M = p.M;
    pp.K = p.K;
    pp.HD = p.HD;
    pp.nslot = proj_slots(p.K, p.HD);
    pp.err = p.err;
    const size_t smem = proj_smem(p.K, p.HD);
    if ((e = allow_smem<tc_proj_kernel>(smem)) != cudaSuccess) return e;
    int dev = 0, sms = 1;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t tiles = (p.M + 127) / 128;
    const unsigned grid = (unsigned)(tiles < sms ? tiles : sms);
    note_launch(SGA_KERN_GATV2_PROJ, s, false);
    tc_proj_kernel<<<grid, kThreads, smem, s>>>(pp);
    note_launch(SGA_KERN_GATV2_PROJ, s, true);
    return cudaGetLastError();
}

}  // namespace sga
