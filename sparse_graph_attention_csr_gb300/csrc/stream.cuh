// Edge stream: the gather side of the persistent edge kernels, decoupled from
// their arithmetic by a per-warp ring in shared memory.
//
// A warp walks its work items (w, w + S, w + 2S, ...; S = warps in the grid).
// An item is a whole row or one chunk of a split row; its edges are consumed
// in steps of STEP = NG * U edges (U per edge group of G lanes, NG groups per
// warp).  For every step the warp's "producer" copies, with cp.async, the
// gathered rows of the step's neighbours (NROW arrays of R sixteen-byte
// chunks per node; lane l of a group copies chunks l, l + G, ...) and their
// per-head scalars (NSC arrays of [N, H] fp32, or [E, H] indexed by the edge's
// CSR position; lane h < H of a group copies head h) into a ring of DEPTH step
// slots; the "consumer" (the same warp, later) computes on slot t while the
// copies of steps t+1 .. t+DEPTH-1 are in flight.  An item's own rows (NOWN
// arrays) and own scalars (NOSC) are copied when the item is queued, so the
// next items' first loads overlap the tail of the current one.  Items wait in
// a small queue (QD entries) in shared memory.
//
// The ring is private to its warp: lanes read the chunks they copied
// themselves and the per-head scalars of their own head; lane 0 writes the
// per-step validity masks and queue entries.  All of it is read after the
// wait and a __syncwarp.  Each step
// records the commit group that carried it; the consumer waits for exactly
// that group, so steps may lag groups (the producer commits an empty group
// when it has nothing to issue) without breaking the pipeline.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "items.cuh"
#include "plan.h"

namespace sga {

__device__ __forceinline__ void cp16_async(uint32_t dst, const void *src, bool ok) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(ok ? 16 : 0));
}
// The same with the source size given (16 copies, 0 fills zeros and reads nothing).
__device__ __forceinline__ void cp16_async_sz(uint32_t dst, const void *src, uint32_t sz) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(sz));
}
__device__ __forceinline__ void cp4_async(uint32_t dst, const void *src, bool ok) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(ok ? 4 : 0));
}
__device__ __forceinline__ void cp_commit_group() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_wait_group() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Wait until at most n of this thread's most recent groups are pending.
__device__ __forceinline__ void cp_wait_newer(int n) {
    switch (n < 0 ? 0 : n) {
        case 0: cp_wait_group<0>(); break;
        case 1: cp_wait_group<1>(); break;
        case 2: cp_wait_group<2>(); break;
        case 3: cp_wait_group<3>(); break;
        case 4: cp_wait_group<4>(); break;
        case 5: cp_wait_group<5>(); break;
        case 6: cp_wait_group<6>(); break;
        default: cp_wait_group<7>(); break;
    }
}

template <int NC_, int G_, int U_, int NROW_, int NSC_, int NOWN_, int NOSC_, int DEPTH_, int QD_,
          int ESC_ = 0, bool LIST_ = true, bool W32_ = false, int DYN_ = 0>
struct StreamCfg {
    // W32: the row copies take 32-bit byte offsets from the array bases when
    // every gathered row array is below 4 GB (checked at run time; 64-bit
    // offsets otherwise).  Fewer address instructions per copy, but the two
    // copies of the step enlarge the code; shapes that gain use it.
    static constexpr bool W32 = W32_;
    // DYN: warps take their items from the partition's counter (P.next, zeroed
    // before each launch) in list order, instead of the fixed share w, w + S,
    // ...: the descending-degree list is then consumed largest first by
    // whichever warp is free, so no warp is left with the last long items.
    // DYN_ > 1 takes the items in batches of consecutive ones, the plan's
    // batch (Partition::batch) capped at DYN_: one atomic per batch, as short
    // rows would otherwise queue on the counter.
    static constexpr bool DYN = DYN_ > 0;
    static constexpr int BATCH = DYN_ > 1 ? DYN_ : 1;
    // walk the plan's item list (else: chunks, then all rows by id)
    static constexpr bool LIST = LIST_;
    static_assert(NSC_ <= 3, "at most three gathered scalar arrays");
    static constexpr int NC = NC_, G = G_, U = U_, NROW = NROW_, NSC = NSC_, NOWN = NOWN_,
                         NOSC = NOSC_, DEPTH = DEPTH_, QD = QD_;
    // bit s set: gathered scalar array s is indexed by the edge's CSR position
    // ([E, H]) rather than by its node ([N, H]); fixed at compile time so that
    // shapes without such arrays pay nothing for them
    static constexpr uint32_t ESC = ESC_;
    static constexpr int NG = 32 / G, STEP = NG * U;
    static_assert(DEPTH >= 2 && DEPTH <= 8, "ring depth");
    static_assert(QD >= 2, "queue depth");
    static_assert(32 % STEP == 0, "a step must not straddle a batch of 32 ids");
    // per-warp shared memory layout (bytes)
    static constexpr int ROW_SLOT = U * NROW * NC * 32 * 16;
    static constexpr int SC_SLOT = U * NSC * 32 * 4;     // [U][NSC][group g * G + head]
    static constexpr int OWN_SLOT = NOWN * NC * 32 * 16;
    static constexpr int OSC_SLOT = NOSC * 32 * 4;       // [NOSC][head]
    static constexpr int OFF_ROW = 0;
    static constexpr int OFF_OWN = OFF_ROW + DEPTH * ROW_SLOT;
    static constexpr int OFF_SC = OFF_OWN + QD * OWN_SLOT;
    static constexpr int OFF_OSC = OFF_SC + DEPTH * SC_SLOT;
    static_assert(U <= 4, "a step's validity masks fill one 16-byte record");
    static constexpr int OFF_MASK = (OFF_OSC + QD * OSC_SLOT + 15) / 16 * 16;   // [DEPTH] uint4: masks of u = 0..3
    static constexpr int OFF_GRP = OFF_MASK + DEPTH * 16;          // [DEPTH] int32
    static constexpr int OFF_Q = (OFF_GRP + DEPTH * 4 + 15) / 16 * 16;   // [QD] int4
    static constexpr int BYTES = OFF_Q + QD * 16;
    // 16-byte regions (cp.async 16, uint4 / int4 accesses) start on 16 bytes,
    // 4-byte regions on 4 bytes; BYTES keeps every warp's base 16-aligned
    static_assert(OFF_ROW % 16 == 0 && OFF_OWN % 16 == 0 && ROW_SLOT % 16 == 0 && OWN_SLOT % 16 == 0,
                  "row slots must be 16-byte aligned");
    static_assert(OFF_SC % 4 == 0 && OFF_OSC % 4 == 0 && OFF_MASK % 16 == 0 && OFF_GRP % 4 == 0,
                  "scalar slots must be 4-byte aligned");
    static_assert(OFF_Q % 16 == 0 && BYTES % 16 == 0, "queue entries and warp bases must be 16-byte aligned");
};

// One queued item, as the consumer sees it.
struct StreamItem {
    int32_t row;      // destination (or source) node
    int32_t nsteps;   // steps of STEP edges; 0 for an empty row
    int32_t item;     // work item index (chunk index when partial)
    int32_t partial;  // 1: a chunk of a split row
};

struct StreamArrays {
    const uint4 *rows[4];   // gathered node rows, [N][R] sixteen-byte chunks
    const float *sc[3];     // gathered per-head scalars, [N][H] (or [E][H], see StreamCfg::ESC)
    const uint4 *own[2];    // the item's own rows
    const float *osc[2];    // the item's own scalars
};

template <typename C> struct EdgeStream {
    // fixed
    unsigned char *sm;       // this warp's shared memory
    uint32_t sa;             // its shared-space address
    StreamArrays arr;
    Partition P;
    const int32_t *ptr, *ids;
    int64_t N;
    int H, R, LH, threshold;
    int32_t *err;
    int64_t stride, n_items;
    int lane, g, gl;
    uint32_t c_in;           // bit k: this lane's chunk gl + G k of a row exists (< R)
    bool off32;              // W32 and every gathered row array below 4 GB: 32-bit byte offsets
    // producer
    // next item to consider, and (DYN) the one after it (else nx_item + stride);
    // 32-bit under DYN, whose items come from a 32-bit counter
    std::conditional_t<C::DYN, uint32_t, int64_t> nx_item, nx2;
    uint32_t b_next, b_left;  // DYN batches: next item of the warp's batch, items left in it
    ItemMeta m1, m2;         // descriptors of nx_item and the item after it
    int32_t ids1;            // first id batch of nx_item (when valid)
    bool v1;                 // nx_item is a valid item (its ids1 were issued)
    ItemRange r1;
    int32_t p_beg, p_deg, p_step, p_nsteps, p_ids, p_ids_nx;
    int32_t p_issued, gc, q_tail, p_slot, q_tslot;
    bool p_done;
    // consumer
    int32_t c_step, q_head, c_slot, q_hslot;
    uint4 c_mask;            // validity masks of the current step (lane bit per neighbour u)

    __device__ __forceinline__ void init(unsigned char *warp_smem, const StreamArrays &a, const Partition &part,
                                         const int32_t *ptr_, const int32_t *ids_, int64_t N_, int H_, int R_,
                                         int LH_, int threshold_, int32_t *err_) {
        sm = warp_smem;
        sa = (uint32_t)__cvta_generic_to_shared(warp_smem);
        arr = a;
        P = part;
        ptr = ptr_;
        ids = ids_;
        N = N_;
        H = H_;
        R = R_;
        LH = LH_;
        threshold = threshold_;
        err = err_;
        lane = threadIdx.x & 31;
        g = lane / C::G;
        gl = lane % C::G;
        c_in = 0;
#pragma unroll
        for (int k = 0; k < C::NC; ++k) c_in |= (gl + C::G * k < R ? 1u : 0u) << k;
        off32 = C::W32 && (uint64_t)N * (uint64_t)R * 16u <= 0xffffffffull;
        stride = (int64_t)gridDim.x * (blockDim.x >> 5);
        n_items = C::LIST ? P.n_items : (int64_t)P.n_chunks + N;
        if constexpr (C::DYN) {
            b_next = b_left = 0;
            nx_item = fetch_item();
            nx2 = fetch_item();
            meta_issue<C::LIST>(nx_item, P, ptr, N, m1);
            meta_issue<C::LIST>(nx2, P, ptr, N, m2);
        } else {   // (nx2 is not kept: nx_item + stride)
            nx_item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
            meta_issue<C::LIST>(nx_item, P, ptr, N, m1);
            meta_issue<C::LIST>(nx_item + stride, P, ptr, N, m2);
        }
        v1 = meta_eval<C::LIST>(nx_item, m1, P, threshold, r1);
        ids1 = first_ids(ids, r1, v1);
        p_beg = p_deg = p_step = p_nsteps = 0;
        p_ids = p_ids_nx = -1;
        p_issued = gc = q_tail = p_slot = q_tslot = 0;
        p_done = false;
        c_step = q_head = c_slot = q_hslot = 0;
        for (int i = 0; i < C::DEPTH - 1; ++i) produce();
    }

    // ---- producer ----------------------------------------------------------

    // The next item of the launch's list (DYN): one atomic of lane 0 per item
    // or per batch of items.
    __device__ __forceinline__ uint32_t fetch_item() {
        if constexpr (C::BATCH == 1) {
            uint32_t v = 0;
            if (lane == 0) v = atomicAdd(reinterpret_cast<unsigned int *>(P.next), 1u);
            return __shfl_sync(SGA_FULL_MASK, v, 0);
        } else {
            if (b_left == 0) {
                const uint32_t n = min((uint32_t)P.batch, (uint32_t)C::BATCH);
                uint32_t v = 0;
                if (lane == 0) v = atomicAdd(reinterpret_cast<unsigned int *>(P.next), n);
                b_next = __shfl_sync(SGA_FULL_MASK, v, 0);
                b_left = n;
            }
            --b_left;
            return b_next++;
        }
    }

    // Queue the next item to be processed here; false when there is none.
    __device__ __forceinline__ bool advance_item() {
        for (;;) {
            if ((int64_t)nx_item >= n_items || m1.row < 0) {
                p_done = true;
                return false;
            }
            const bool valid = v1;
            const ItemRange r = r1;
            const int64_t cur = nx_item;
            int32_t first = ids1;
            // rotate the descriptor pipeline
            m1 = m2;
            if constexpr (C::DYN) {
                nx_item = nx2;
                nx2 = fetch_item();
                meta_issue<C::LIST>(nx2, P, ptr, N, m2);
            } else {
                nx_item += stride;
                meta_issue<C::LIST>(nx_item + stride, P, ptr, N, m2);
            }
            v1 = meta_eval<C::LIST>(nx_item, m1, P, threshold, r1);
            ids1 = first_ids(ids, r1, v1);
            if (!valid) continue;   // a row above the split threshold: its chunks cover it
            const int32_t deg = r.end - r.beg;
            if (lane < deg && lane < 32) {
                if ((uint32_t)first >= (uint32_t)N) {
                    atomicOr(err, kErrIndexRange);
                    first = -1;
                }
            } else {
                first = -1;
            }
            p_beg = r.beg;
            p_deg = deg;
            p_step = 0;
            p_nsteps = (deg + C::STEP - 1) / C::STEP;
            p_ids = first;
            p_ids_nx = deg > 32 ? load_ids(ids, r.beg + 32, min(32, deg - 32), N, err) : -1;
            const int qs = q_tslot;
            if (lane == 0) {
                int4 e;
                e.x = r.row;
                e.y = p_nsteps;
                e.z = (int32_t)cur;
                e.w = r.partial ? 1 : 0;
                *reinterpret_cast<int4 *>(sm + C::OFF_Q + qs * 16) = e;
            }
            // the item's own rows and scalars
            if (p_nsteps > 0) {
#pragma unroll
                for (int o = 0; o < C::NOWN; ++o)
#pragma unroll
                    for (int k = 0; k < C::NC; ++k) {
                        const int c = gl + C::G * k;
                        const bool ok = c < R;
                        cp16_async(sa + C::OFF_OWN + qs * C::OWN_SLOT + ((o * C::NC + k) * 32 + lane) * 16,
                                   ok ? arr.own[o] + (size_t)r.row * R + c : arr.own[o], ok);
                    }
                if (lane < H)
#pragma unroll
                    for (int o = 0; o < C::NOSC; ++o)
                        cp4_async(sa + C::OFF_OSC + qs * C::OSC_SLOT + (o * 32 + lane) * 4,
                                  arr.osc[o] + (size_t)r.row * H + lane, true);
            }
            ++q_tail;
            q_tslot = q_tslot + 1 == C::QD ? 0 : q_tslot + 1;
            return true;
        }
    }

    // (two copies of the step, one per address width, chosen once per step)
    __device__ __forceinline__ void issue_step() {
        if constexpr (C::W32) {
            if (off32) {
                issue_step_w<true>();
                return;
            }
        }
        issue_step_w<false>();
    }
    template <bool O32> __device__ __forceinline__ void issue_step_w() {
        const int slot = p_slot;
        const int32_t e0 = p_step * C::STEP;   // item-local first edge of the step
        uint32_t masks[4] = {0u, 0u, 0u, 0u};
        if (p_step > 0 && (e0 & 31) == 0) {    // next batch of 32 ids
            p_ids = p_ids_nx;
            p_ids_nx = e0 + 32 < p_deg ? load_ids(ids, p_beg + e0 + 32, min(32, p_deg - e0 - 32), N, err) : -1;
        }
        const uint32_t dst0 = sa + C::OFF_ROW + slot * C::ROW_SLOT + lane * 16;
#pragma unroll
        for (int u = 0; u < C::U; ++u) {
            const int32_t e = e0 + g + C::NG * u;
            const int32_t j = __shfl_sync(SGA_FULL_MASK, p_ids, e & 31);
            // (ids past the item's last edge, like out-of-range ids, are -1: a
            // step never straddles a batch of 32, and a batch's lanes past
            // the item hold -1)
            const bool ok = j >= 0;
            // a copy that is skipped (src-size 0) still names an address inside the
            // array: row 0 for a missing neighbour, chunk 0 for a lane past the row
            if constexpr (O32) {   // byte offsets from the array bases fit 32 bits
                const uint32_t boff = (uint32_t)(ok ? j : 0) * (uint32_t)(R * 16);
#pragma unroll
                for (int k = 0; k < C::NC; ++k) {
                    const bool cin = (c_in >> k) & 1u;
                    const uint32_t koff = boff + (cin ? (uint32_t)(gl + C::G * k) * 16u : 0u);
                    const uint32_t sz = (ok && cin) ? 16u : 0u;
#pragma unroll
                    for (int r = 0; r < C::NROW; ++r)
                        cp16_async_sz(dst0 + ((u * C::NROW + r) * C::NC + k) * 32 * 16,
                                      reinterpret_cast<const unsigned char *>(arr.rows[r]) + koff, sz);
                }
            } else {
                const size_t roff = (size_t)(uint32_t)(ok ? j : 0) * R;
#pragma unroll
                for (int k = 0; k < C::NC; ++k) {
                    const bool cin = (c_in >> k) & 1u;
                    const size_t off = roff + (cin ? gl + C::G * k : 0);
                    const uint32_t sz = (ok && cin) ? 16u : 0u;
#pragma unroll
                    for (int r = 0; r < C::NROW; ++r)
                        cp16_async_sz(dst0 + ((u * C::NROW + r) * C::NC + k) * 32 * 16, arr.rows[r] + off, sz);
                }
            }
            if (gl < H)
#pragma unroll
                for (int s = 0; s < C::NSC; ++s) {
                    const size_t at = !ok ? 0 : ((C::ESC >> s) & 1u) ? (size_t)(p_beg + e) : (size_t)j;
                    cp4_async(sa + C::OFF_SC + slot * C::SC_SLOT + ((u * C::NSC + s) * 32 + lane) * 4,
                              arr.sc[s] + at * H + gl, ok);
                }
            masks[u] = __ballot_sync(SGA_FULL_MASK, ok);
        }
        if (lane == 0) {
            *reinterpret_cast<uint4 *>(sm + C::OFF_MASK + slot * 16) = make_uint4(masks[0], masks[1], masks[2], masks[3]);
            reinterpret_cast<int32_t *>(sm + C::OFF_GRP)[slot] = gc;
        }
        ++p_step;
        ++p_issued;
        p_slot = p_slot + 1 == C::DEPTH ? 0 : p_slot + 1;
    }

    // Issue at most one step (queueing items as needed), then commit a group.
    __device__ __forceinline__ void produce() {
        if (!p_done) {
            bool ready = p_step < p_nsteps;
            while (!ready && q_tail - q_head < C::QD && advance_item()) ready = p_step < p_nsteps;
            if (ready && p_issued - c_step < C::DEPTH) issue_step();
        }
        cp_commit_group();
        ++gc;
    }

    // ---- consumer ----------------------------------------------------------

    // The next item in order; false when the warp has no more.  (The producer
    // runs DEPTH - 1 >= 1 steps ahead, so every item up to and including the
    // one holding the next step is already queued.)
    __device__ __forceinline__ bool next_item(StreamItem &it) {
        __syncwarp();
        while (q_head == q_tail && !p_done) produce();
        __syncwarp();
        if (q_head == q_tail) return false;
        const int4 e = *reinterpret_cast<const int4 *>(sm + C::OFF_Q + q_hslot * 16);
        it.row = e.x;
        it.nsteps = e.y;
        it.item = e.z;
        it.partial = e.w;
        return true;
    }
    __device__ __forceinline__ void finish_item() {
        ++q_head;
        q_hslot = q_hslot + 1 == C::QD ? 0 : q_hslot + 1;
    }

    // Make the data of the next step (and the current item's own rows) visible.
    __device__ __forceinline__ void wait_step() {
        __syncwarp();
        produce();
        const int newer = gc - 1 - reinterpret_cast<const int32_t *>(sm + C::OFF_GRP)[c_slot];
        if (newer >= C::DEPTH - 1) cp_wait_group<C::DEPTH - 1>();   // the steady state
        else cp_wait_newer(newer);
        __syncwarp();
        c_mask = *reinterpret_cast<const uint4 *>(sm + C::OFF_MASK + c_slot * 16);
    }
    __device__ __forceinline__ void release_step() {
        ++c_step;
        c_slot = c_slot + 1 == C::DEPTH ? 0 : c_slot + 1;
    }

    __device__ __forceinline__ bool valid(int u) const {
        const uint32_t m = u == 0 ? c_mask.x : (u == 1 ? c_mask.y : (u == 2 ? c_mask.z : c_mask.w));
        return (m >> lane) & 1u;
    }
    __device__ __forceinline__ uint4 row(int u, int r, int k) const {
        return *reinterpret_cast<const uint4 *>(
            sm + C::OFF_ROW + c_slot * C::ROW_SLOT + (((u * C::NROW + r) * C::NC + k) * 32 + lane) * 16);
    }
    // scalar s of this lane's neighbour u, head h
    __device__ __forceinline__ float scalar(int u, int s, int h) const {
        // (lanes past the row's last head read a slot entry they never use)
        return *reinterpret_cast<const float *>(sm + C::OFF_SC + c_slot * C::SC_SLOT +
                                                ((u * C::NSC + s) * 32 + ((g * C::G + h) & 31)) * 4);
    }
    __device__ __forceinline__ uint4 own_row(int o, int k) const {
        return *reinterpret_cast<const uint4 *>(
            sm + C::OFF_OWN + q_hslot * C::OWN_SLOT + ((o * C::NC + k) * 32 + lane) * 16);
    }
    // own scalar o of the current item, head h
    __device__ __forceinline__ float own_scalar(int o, int h) const {
        return *reinterpret_cast<const float *>(sm + C::OFF_OSC + q_hslot * C::OSC_SLOT + (o * 32 + (h & 31)) * 4);
    }

    __device__ __forceinline__ void drain() { cp_wait_group<0>(); }
};

}  // namespace sga
