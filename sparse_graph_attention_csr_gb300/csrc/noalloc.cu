// gt_attn_fwd_noalloc: the Graph Transformer forward for callers that cannot
// allocate device memory.  The split-row partition and the chunk partials
// that gt_attn_fwd keeps in its plan and workspace live here in one
// file-scope static device array instead; the caller passes only the graph,
// Q/K/V and the outputs.  The edge kernels are the same as gt_attn_fwd's.
#include <stddef.h>

#include <mutex>

#include "common.cuh"
#include "plan.h"

namespace sga {
namespace {

// Rows of degree > kNaThreshold are split into chunks of kNaChunk edges.
constexpr int kNaThreshold = 1024;
constexpr int kNaChunk = 1024;
constexpr int kNaMaxSplit = 4096;                       // split rows per call
constexpr size_t kNaPartialBytes = size_t(24) << 20;    // chunk partials
constexpr size_t kNaScratchBytes = size_t(32) << 20;    // whole array

// Layout of the scratch array (byte offsets).
struct NaHeader {
    int32_t n_split;    // split rows found (may exceed kNaMaxSplit: then rejected)
    int32_t n_chunks;   // chunks those rows need
    int32_t csr_err;    // CSR validation bits
    int32_t range_err;  // device range-check word of the edge kernels; kept across
                        // calls until sga_noalloc_read_device_error reads and clears it
};
constexpr size_t kOffHeader = 0;
constexpr size_t kOffSplitRows = 256;
constexpr size_t kOffChunkPtr = kOffSplitRows + 4 * kNaMaxSplit;
constexpr size_t kOffChunkRow = kOffChunkPtr + 4 * (kNaMaxSplit + 256);
constexpr size_t kMaxChunksAny = kNaPartialBytes / ((32 + 2) * 4);   // smallest row: H*D = 32
constexpr size_t kOffChunkBeg = kOffChunkRow + 4 * kMaxChunksAny;
constexpr size_t kOffChunkEnd = kOffChunkBeg + 4 * kMaxChunksAny;
constexpr size_t kOffPartials = (kOffChunkEnd + 4 * kMaxChunksAny + 255) & ~size_t(255);
static_assert(kOffPartials + kNaPartialBytes <= kNaScratchBytes, "scratch layout overflow");

static __device__ __align__(256) unsigned char g_na_scratch[kNaScratchBytes];

// Device address of g_na_scratch per device, looked up once per device.
std::mutex g_na_mu;
void *g_na_ptr[64] = {};

cudaError_t scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_na_mu);
    if (!g_na_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_na_scratch);
        if (e != cudaSuccess) return e;
        g_na_ptr[dev] = p;
    }
    *out = g_na_ptr[dev];
    return cudaSuccess;
}

// Validate the CSR (as plan creation does) and collect the split rows in
// arbitrary order with their chunk count.
__global__ void na_collect_kernel(const int32_t *__restrict__ indptr,
                                  const int32_t *__restrict__ indices, int64_t N, int64_t E,
                                  unsigned char *scratch) {
    NaHeader *hdr = reinterpret_cast<NaHeader *>(scratch + kOffHeader);
    int32_t *split = reinterpret_cast<int32_t *>(scratch + kOffSplitRows);
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    int bits = 0;
    if (t0 == 0) {
        if (indptr[0] != 0) bits |= 1;
        if ((int64_t)indptr[N] != E) bits |= 4;
    }
    for (int64_t i = t0; i < N; i += stride) {
        const int32_t b = indptr[i], e = indptr[i + 1];
        if (b > e) {
            bits |= 2;
            continue;
        }
        if (e - b > kNaThreshold) {
            const int32_t s = atomicAdd(&hdr->n_split, 1);
            if (s < kNaMaxSplit) split[s] = (int32_t)i;
            atomicAdd(&hdr->n_chunks, (e - b + kNaChunk - 1) / kNaChunk);
        }
    }
    for (int64_t e = t0; e < E; e += stride) {
        const int32_t j = indices[e];
        if (j < 0 || (int64_t)j >= N) bits |= 8;
    }
    if (bits) atomicOr(&hdr->csr_err, bits);
}

// One block: sort the split rows ascending (bitonic, in shared memory), then
// lay out their chunks in that order.
__global__ void __launch_bounds__(1024)
na_partition_kernel(const int32_t *__restrict__ indptr, int32_t n_split, unsigned char *scratch) {
    __shared__ int32_t key[kNaMaxSplit];
    __shared__ int32_t cnt[kNaMaxSplit];
    int32_t *split = reinterpret_cast<int32_t *>(scratch + kOffSplitRows);
    int32_t *cptr = reinterpret_cast<int32_t *>(scratch + kOffChunkPtr);
    int32_t *crow = reinterpret_cast<int32_t *>(scratch + kOffChunkRow);
    int32_t *cbeg = reinterpret_cast<int32_t *>(scratch + kOffChunkBeg);
    int32_t *cend = reinterpret_cast<int32_t *>(scratch + kOffChunkEnd);
    int n2 = 1;
    while (n2 < n_split) n2 <<= 1;
    for (int x = threadIdx.x; x < n2; x += blockDim.x) key[x] = x < n_split ? split[x] : INT32_MAX;
    __syncthreads();
    for (int k = 2; k <= n2; k <<= 1)
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int x = threadIdx.x; x < n2; x += blockDim.x) {
                const int y = x ^ j;
                if (y > x) {
                    const bool up = (x & k) == 0;
                    const int32_t a = key[x], b = key[y];
                    if ((a > b) == up) {
                        key[x] = b;
                        key[y] = a;
                    }
                }
            }
            __syncthreads();
        }
    for (int x = threadIdx.x; x < n_split; x += blockDim.x) {
        const int32_t r = key[x];
        cnt[x] = (indptr[r + 1] - indptr[r] + kNaChunk - 1) / kNaChunk;
        split[x] = r;
    }
    __syncthreads();
    if (threadIdx.x == 0) {   // serial prefix over at most kNaMaxSplit rows
        int32_t run = 0;
        for (int x = 0; x < n_split; ++x) {
            const int32_t c = cnt[x];
            cnt[x] = run;
            run += c;
        }
        cptr[n_split] = run;
    }
    __syncthreads();
    for (int x = threadIdx.x; x < n_split; x += blockDim.x) {
        const int32_t r = key[x];
        int32_t c = cnt[x];
        cptr[x] = c;
        const int32_t b = indptr[r], e = indptr[r + 1];
        for (int32_t y = b; y < e; y += kNaChunk, ++c) {
            crow[c] = r;
            cbeg[c] = y;
            cend[c] = min(y + kNaChunk, e);
        }
    }
}

}  // namespace
}  // namespace sga

using namespace sga;

extern "C" size_t sga_noalloc_scratch_bytes(void) { return kNaScratchBytes; }

extern "C" sga_status gt_attn_fwd_noalloc(const int32_t *indptr, const int32_t *indices,
                                          const void *Q, const void *K, const void *V, int64_t N,
                                          int64_t E, int H, int D, sga_dtype dt, void *out,
                                          float *lse, void *stream) {
    if (!indptr || (reinterpret_cast<uintptr_t>(indptr) % 4) != 0) return SGA_EINVAL;
    if (E > 0 && (!indices || (reinterpret_cast<uintptr_t>(indices) % 4) != 0)) return SGA_EINVAL;
    if (N < 0 || E < 0 || N >= INT32_MAX || E >= INT32_MAX) return SGA_EINVAL;
    if (dt != SGA_F32 && dt != SGA_BF16) return SGA_EUNSUPPORTED;
    if (!(D == 32 || D == 64 || D == 128) || H < 1 || (int64_t)H * D > 1024) return SGA_EUNSUPPORTED;
    if (N > 0)
        for (const void *q : {Q, K, V, (const void *)out, (const void *)lse})
            if (!q || (reinterpret_cast<uintptr_t>(q) % 16) != 0) return SGA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *base = nullptr;
    cudaError_t ce = scratch_address(&base);
    if (ce != cudaSuccess) {
        set_cuda_error(ce);
        return SGA_ECUDA;
    }
    unsigned char *scratch = static_cast<unsigned char *>(base);
    // every call starts from cleared split counts and CSR bits (the array keeps
    // the last call's contents); the range-check word is left for the caller to
    // read with sga_noalloc_read_device_error
    ce = cudaMemsetAsync(scratch + kOffHeader, 0, offsetof(NaHeader, range_err), s);
    if (ce == cudaSuccess && (N > 0 || E > 0)) {
        int64_t work = N > E ? N : E;
        unsigned blocks = (unsigned)((work + 255) / 256);
        if (blocks > 4096) blocks = 4096;
        if (blocks == 0) blocks = 1;
        na_collect_kernel<<<blocks, 256, 0, s>>>(indptr, indices, N, E, scratch);
        ce = cudaGetLastError();
    }
    NaHeader hdr{};
    if (ce == cudaSuccess)
        ce = cudaMemcpyAsync(&hdr, scratch + kOffHeader, sizeof(hdr), cudaMemcpyDeviceToHost, s);
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
    if (ce != cudaSuccess) {
        set_cuda_error(ce);
        return SGA_ECUDA;
    }
    if (hdr.csr_err) return SGA_EINVAL;
    const size_t HD = (size_t)H * D;
    const size_t max_chunks = kNaPartialBytes / ((HD + 2 * (size_t)H) * 4);
    if (hdr.n_split > kNaMaxSplit || (size_t)hdr.n_chunks > max_chunks) return SGA_ELIMIT;
    if (hdr.n_split > 0) {
        na_partition_kernel<<<1, 1024, 0, s>>>(indptr, hdr.n_split, scratch);
        if ((ce = cudaGetLastError()) != cudaSuccess) {
            set_cuda_error(ce);
            return SGA_ECUDA;
        }
    }
    GtArgs a{};
    a.indptr = indptr;
    a.indices = indices;
    a.Q = Q;
    a.K = K;
    a.V = V;
    a.out_w = out;
    a.lse_w = lse;
    a.N = N;
    a.H = H;
    a.D = D;
    a.split_threshold = kNaThreshold;
    a.rows.n_split = hdr.n_split;
    a.rows.n_chunks = hdr.n_chunks;
    a.rows.split_rows = reinterpret_cast<int32_t *>(scratch + kOffSplitRows);
    a.rows.chunk_ptr = reinterpret_cast<int32_t *>(scratch + kOffChunkPtr);
    a.rows.chunk_row = reinterpret_cast<int32_t *>(scratch + kOffChunkRow);
    a.rows.chunk_beg = reinterpret_cast<int32_t *>(scratch + kOffChunkBeg);
    a.rows.chunk_end = reinterpret_cast<int32_t *>(scratch + kOffChunkEnd);
    a.ws_ml = reinterpret_cast<float *>(scratch + kOffPartials);
    a.ws_acc = a.ws_ml + (((size_t)hdr.n_chunks * H * 2 + 63) & ~size_t(63));
    a.d_err = &reinterpret_cast<NaHeader *>(scratch + kOffHeader)->range_err;
    ce = dt == SGA_F32 ? gt_fwd_t<float>(a, s) : gt_fwd_t<__nv_bfloat16>(a, s);
    if (ce != cudaSuccess) {
        set_cuda_error(ce);
        return SGA_ECUDA;
    }
    return SGA_OK;
}

extern "C" sga_status sga_noalloc_read_device_error(void *stream, int32_t *code) {
    if (!code) return SGA_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    void *base = nullptr;
    cudaError_t ce = scratch_address(&base);
    int32_t *word = &reinterpret_cast<NaHeader *>(static_cast<unsigned char *>(base) + kOffHeader)->range_err;
    int32_t v = 0;
    if (ce == cudaSuccess) ce = cudaMemcpyAsync(&v, word, sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (ce == cudaSuccess) ce = cudaMemsetAsync(word, 0, sizeof(int32_t), s);
    if (ce == cudaSuccess) ce = cudaStreamSynchronize(s);
    if (ce != cudaSuccess) {
        set_cuda_error(ce);
        return SGA_ECUDA;
    }
    *code = v;
    return v ? SGA_EDEVICE_CHECK : SGA_OK;
}
