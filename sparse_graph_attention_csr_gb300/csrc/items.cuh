// Work items of the persistent edge kernels: whole destination (or source)
// rows, and fixed-length chunks of split rows, with the pipelined loads of
// their descriptors and first node ids.
#pragma once

#include "common.cuh"
#include "plan.h"

namespace sga {

struct ItemRange {
    int32_t row, beg, end;
    bool partial;
};

// Work item w of a launch: the plan's item list (chunks of split rows, then
// the other rows in walking order), or without one chunks first, then every
// row by id (rows above the split threshold are skipped; their chunks cover
// them).
__device__ __forceinline__ bool decode_item(int64_t item, const Partition &P,
                                            const int32_t *__restrict__ ptr, int64_t N,
                                            int threshold, ItemRange &r) {
    if (P.items) {   // the plan's item list
        if (item >= P.n_items) return false;
        const int4 t = __ldg(P.items + item);
        r.row = t.x;
        r.beg = t.y;
        r.end = t.z;
        r.partial = item < P.n_chunks;
        return true;
    }
    if (item < P.n_chunks) {
        r.row = P.chunk_row[item];
        r.beg = P.chunk_beg[item];
        r.end = P.chunk_end[item];
        r.partial = true;
        return true;
    }
    const int64_t i = item - P.n_chunks;
    if (i >= N) return false;
    r.row = (int32_t)i;
    r.beg = ptr[i];
    r.end = ptr[i + 1];
    r.partial = false;
    return r.end - r.beg <= threshold;
}

// Fetch the 32 node ids of edges [e0, e0 + cnt) into one register per lane,
// range-checked against N (an out-of-range id becomes -1 and flags the plan).
__device__ __forceinline__ int32_t load_ids(const int32_t *__restrict__ ids, int32_t e0, int cnt,
                                            int64_t N, int32_t *err) {
    const int lane = threadIdx.x & 31;
    int32_t j = -1;
    if (lane < cnt) {
        j = __ldg(ids + e0 + lane);
        if ((uint32_t)j >= (uint32_t)N) {
            atomicOr(err, kErrIndexRange);
            j = -1;
        }
    }
    return j;
}

// Persistent warps walk the items w, w + S, w + 2S, ... (S = warps in the
// grid) through a three-stage pipeline: while item k runs, the metadata of
// item k + 2S (chunk descriptor or indptr pair) and the first 32 node ids of
// item k + S are already in flight, so a short row costs one gather latency
// instead of three dependent ones.
struct ItemMeta {
    int32_t row, beg, end;   // raw loads; row < 0 past the last item
};

// LIST: the partition's item list (one load path, no skipped rows);
// otherwise chunks, then every row by id.
template <bool LIST>
__device__ __forceinline__ void meta_issue(int64_t item, const Partition &P,
                                           const int32_t *__restrict__ ptr, int64_t N,
                                           ItemMeta &m) {
    if constexpr (LIST) {
        if (item < P.n_items) {
            const int4 t = __ldg(P.items + item);
            m.row = t.x;
            m.beg = t.y;
            m.end = t.z;
        } else {
            m.row = -1;
            m.beg = m.end = 0;
        }
        return;
    }
    if (item < P.n_chunks) {
        m.row = __ldg(P.chunk_row + item);
        m.beg = __ldg(P.chunk_beg + item);
        m.end = __ldg(P.chunk_end + item);
    } else if (item - P.n_chunks < N) {
        const int64_t i = item - P.n_chunks;
        m.row = (int32_t)i;
        m.beg = __ldg(ptr + i);
        m.end = __ldg(ptr + i + 1);
    } else {
        m.row = -1;
        m.beg = m.end = 0;
    }
}

// True when the item is to be processed here (not past the end, and not a row
// above the split threshold, whose chunks are separate items).
template <bool LIST>
__device__ __forceinline__ bool meta_eval(int64_t item, const ItemMeta &m, const Partition &P,
                                          int threshold, ItemRange &r) {
    r.row = m.row;
    r.beg = m.beg;
    r.end = m.end;
    r.partial = item < P.n_chunks;
    if constexpr (LIST) return m.row >= 0;
    return m.row >= 0 && (r.partial || m.end - m.beg <= threshold);
}

// First batch of node ids of an item (lanes past the item's edges read nothing).
__device__ __forceinline__ int32_t first_ids(const int32_t *__restrict__ ids, const ItemRange &r,
                                             bool valid) {
    const int lane = threadIdx.x & 31;
    return (valid && lane < r.end - r.beg) ? __ldg(ids + r.beg + lane) : 0;
}

// Node ids of edges [e0, e0 + cnt), range-checked like load_ids: the
// prefetched batch for the item's first 32 edges, a fresh load after that.
__device__ __forceinline__ int32_t batch_ids(const int32_t *__restrict__ ids, int32_t e0, int cnt,
                                             const ItemRange &r, int32_t id0, int64_t N,
                                             int32_t *err) {
    if (e0 != r.beg) return load_ids(ids, e0, cnt, N, err);
    const int lane = threadIdx.x & 31;
    if (lane >= cnt) return -1;
    if ((uint32_t)id0 >= (uint32_t)N) {
        atomicOr(err, kErrIndexRange);
        return -1;
    }
    return id0;
}

}  // namespace sga
