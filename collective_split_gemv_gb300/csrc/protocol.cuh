// Device-side pieces shared by the fused GEMV kernels: streaming loads,
// bf16 unpacking, and the publish / last-arriver reduction protocol.
//
// Protocol (one row tile t, C = R * splits contributing CTAs: one per rank
// and K-split):
//  0. the launch's epoch e is one more than the epoch word of slot 0's pad,
//     which holds the epoch of the last finished fused launch on the handle
//     (read on the device, so a launch replayed from a CUDA graph gets a new
//     epoch each time);
//  1. every thread stores its share of the contributor's fp32 partial into
//     the rank's scratch slot, one thread also the contributor's flag (= e),
//     then every thread fences (gpu scope);
//  2. after a CTA barrier, one thread takes an arrival ticket with an acq_rel
//     atomic add on counter[t].  Tickets run 0..C-1 in every launch: the
//     holder of C-1 is the tile's reducer and puts the counter back to zero
//     (every contributor of this launch has arrived).  A ticket >= C latches
//     a protocol error;
//  3. the reducer (its acq_rel ticket orders its loads after every
//     contributor's fenced stores) loads the C flags together with the first
//     partials -- each flag must equal e, else nothing is stored -- sums the
//     C partials in fixed order (rank 0..R-1, split 0..splits-1) in fp32,
//     rounds to bf16 (RNE) and stores the value into every rank's output
//     slot;
//  4. the reducer counts the tile on tiles_done (when it takes the ticket).
//     The reducer of the last tile knows that every CTA of the launch has
//     read e (each read it before publishing), so it stores e into the epoch
//     word and clears tiles_done and the work counter the next launch will
//     use.
// No CTA ever waits for another: a tile whose contributors have not all
// arrived is finished by whichever contributor arrives last.  Between
// launches every counter is zero and the flags hold older epochs, so a
// launch depends on no host-side state and the geometry may change from one
// launch to the next.
//
// This is the publish-as-soon-as-done / reduce-locally scheme of the fused
// GEMV + AllReduce ("Overlapping Collective Communication with Dependent
// Computation ...", Abstract) and the one-shot all-reduce ("PyTorch Symmetric
// Memory" talk, one-shot segment), with the start/end signal-pad barriers of
// the symmetric-memory kernels replaced by per-tile release flags; keeping
// the synchronisation state in the signal pad is what makes the calls
// replayable from a CUDA graph (the symmetric-memory pages' CUDA-graph
// compatible synchronisation primitives).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include <type_traits>

#include "internal.h"
#include "timeline.cuh"

namespace symm {

__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_v4(void *p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_u32(uint32_t *p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ float ld_relaxed_gpu_f32(const float *p) {
    float v;
    asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}

// Two bf16 values packed in one 32-bit word (element 2i in the low half):
// a bf16 is the top half of an fp32 word, so widening is a shift / mask.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void latch_status(uint32_t *status, int code, int rank, int tile,
                                             uint32_t epoch) {
    if (atomicCAS(status + kStatusCode, 0u, (uint32_t)code) == 0u) {
        status[kStatusRank] = (uint32_t)rank;
        status[kStatusTile] = (uint32_t)tile;
        status[kStatusEpoch] = epoch;
    }
}

// Step 0: this launch's epoch.  A thread that publishes must have read it
// before its flag store (the release orders the read before the flag); the
// last tile's reducer then knows the read happened before its update.
__device__ __forceinline__ uint32_t read_launch_epoch(const GemvArgs &a) {
    return ld_relaxed_gpu_u32(a.epoch_word) + 1u;
}

// Step 2's ticket for contributor (r, ...) of tile t among C.  Returns the
// ticket; its holder is the reducer when it equals C - 1, and the reducer
// has then also counted the tile on tiles_done (*done: the count before it,
// used later so that the atomic's latency hides behind the flag check) and
// put the tile's counter back to zero.  The count may come before the flag
// check: the acq_rel ticket already orders every contributor's epoch read
// before it, whatever the flags hold.
__device__ __forceinline__ uint32_t take_ticket(const GemvArgs &a, int t, uint32_t C, int r, uint32_t epoch,
                                                uint32_t *done) {
    const uint32_t pos = atom_add_acq_rel_gpu(a.counters + t, 1u);
    if (pos >= C) {
        latch_status(a.status, kProtoBadTicket, r, t, epoch);
    } else if (pos == C - 1u) {
        if (a.tiles_done) *done = atom_add_release_gpu(a.tiles_done, 1u);
        st_relaxed_gpu_u32(a.counters + t, 0u);
    }
    return pos;
}

// Step 4: the reducer of the last tile (every CTA of the launch has read the
// epoch by then) publishes the epoch and clears the counters for the next
// launch.  Run by the thread that took the ticket, before the reduction, so
// that these stores are long done when the grid ends.
__device__ __forceinline__ void finish_launch_if_last(const GemvArgs &a, uint32_t done, uint32_t epoch, int t) {
    if (!a.tiles_done) return;   // a launch counted in units (count_unit)
    const uint32_t T = (uint32_t)a.num_tiles;
    if (done >= T) latch_status(a.status, kProtoBadTicket, -1, t, epoch);
    if (done != T - 1u) return;
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    st_relaxed_gpu_u32(a.tiles_done, 0u);
    st_relaxed_gpu_u32(a.work + ((epoch + 1u) & 1u), 0u);
    st_relaxed_gpu_u32(a.epoch_word, epoch);
}

// Step 4 for a launch that is counted in units instead of reduced tiles (the
// unfused form's GEMV, whose partials no tile reducer sums; and one rank's
// launch on a multi-process handle, whose tiles the other ranks' launches may
// finish): the thread that counts the last of the launch's U units on
// `counter` stores the epoch and clears the counter and the work counter the
// next launch uses.  Every unit is counted after its CTA read the epoch, and
// the acq_rel count orders those reads before the epoch store.
__device__ __forceinline__ void count_unit(const GemvArgs &a, uint32_t *counter, uint32_t epoch, uint32_t U) {
    const uint32_t done = atom_add_acq_rel_gpu(counter, 1u);
    if (done >= U) latch_status(a.status, kProtoBadTicket, -1, -1, epoch);
    if (done != U - 1u) return;
    asm volatile("fence.acq_rel.gpu;" ::: "memory");
    st_relaxed_gpu_u32(counter, 0u);
    st_relaxed_gpu_u32(a.work + ((epoch + 1u) & 1u), 0u);
    st_relaxed_gpu_u32(a.epoch_word, epoch);
}

// Where the tile reducer puts the fp32 sum of output (b, n) (see
// GemvArgs::out_mode): bf16 into every rank's y (all-reduce), bf16 into the
// rank that owns batch row b (reduce-scatter along the batch rows, the
// sequence-parallel ending of the row-parallel layer), or fp32 sum + bias
// into z for the RMS-normalisation stage.
// `e` is the element index b * N + n of the output in a [B][N] array.
__device__ __forceinline__ void store_output(const GemvArgs &a, size_t e, float acc) {
    if (a.out_mode == kOutAllReduce) {
        const __nv_bfloat16 h = __float2bfloat16_rn(acc);
        for (int q = 0; q < a.R; ++q)
            *reinterpret_cast<__nv_bfloat16 *>(a.y + (long long)q * a.stride + e * 2) = h;
        return;
    }
    const int b = (int)(e / (size_t)a.N);
    const int n = (int)(e - (size_t)b * a.N);
    if (a.out_mode == kOutReduceScatter) {
        const int q = b / a.rs_rows;
        const size_t yoff = ((size_t)(b - q * a.rs_rows) * a.N + n) * 2;
        *reinterpret_cast<__nv_bfloat16 *>(a.y + (long long)q * a.stride + yoff) = __float2bfloat16_rn(acc);
    } else {
        float v = acc;
        if (a.bias) v += __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(a.bias)[n]);
        __stcg(a.z + e, v);
    }
}

// The same for the four outputs e .. e + 3 (e % 4 == 0, all in one row b,
// which holds when N % 4 == 0): one 8-byte bf16 store per slot, or one
// 16-byte fp32 store of z.  Each value is rounded or biased exactly as
// store_output does it.
__device__ __forceinline__ void store_output4(const GemvArgs &a, size_t e, float4 acc) {
    if (a.out_mode == kOutBiasZ) {
        if (a.bias) {
            const int n = (int)(e % (size_t)a.N);
            const uint2 bb = *reinterpret_cast<const uint2 *>(a.bias + (size_t)n * 2);
            acc.x += bf16lo(bb.x);
            acc.y += bf16hi(bb.x);
            acc.z += bf16lo(bb.y);
            acc.w += bf16hi(bb.y);
        }
        __stcg(reinterpret_cast<float4 *>(a.z + e), acc);
        return;
    }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    uint2 o;
    o.x = *reinterpret_cast<const uint32_t *>(&lo);
    o.y = *reinterpret_cast<const uint32_t *>(&hi);
    if (a.out_mode == kOutAllReduce) {
        for (int q = 0; q < a.R; ++q) *reinterpret_cast<uint2 *>(a.y + (long long)q * a.stride + e * 2) = o;
        return;
    }
    const int b = (int)(e / (size_t)a.N);
    const int n = (int)(e - (size_t)b * a.N);
    const int q = b / a.rs_rows;
    *reinterpret_cast<uint2 *>(a.y + (long long)q * a.stride + ((size_t)(b - q * a.rs_rows) * a.N + n) * 2) = o;
}

// Waits until the grid this one was launched as a programmatic dependent of
// has completed and its memory is visible; returns at once otherwise.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Entry of the collective kernels and the per-tile fused kernels for chained
// calls (launched as programmatic dependents of the previous kernel on the
// stream): a CTA may be scheduled while that kernel drains, and waits for it,
// and for its memory, before reading anything; it lets its own successor (the
// next chained call, or the RMS-normalisation stage of a bias + RMSNorm call)
// be scheduled likewise.  Both are no-ops in plain stream order.
__device__ __forceinline__ void chain_entry() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    griddep_wait();
}

// Contributor (r, s)'s flag for tile t (S splits per rank) in rank r's pad.
__device__ __forceinline__ uint32_t *flag_of(const GemvArgs &a, int r, int t, int S, int s) {
    return reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(a.flags) + (long long)r * a.stride) +
           (size_t)t * S + s;
}

// The reduction of one tile by its last contributor: for each output (b, n)
// of rows [n0, n0 + rows), sum the C contributors' fp32 partials in
// contributor order j = 0..C-1 (contributor j = (rank j / S, split j % S),
// its [B][N] array at contributor_base(j)) and hand the sum to store_output.
// The caller holds the tile's last ticket (an acq_rel atomic that every
// contributor took after fencing its partial and its flag), and the group
// has passed a barrier since, so plain L2 loads (.cg) see every partial and
// every flag.
// Each thread takes kPer items -- vectors of four consecutive outputs (for
// N % 4 == 0, when then n0 and rows are multiples of 4, and C <= 8), else
// single outputs -- and loads up to kBatch contributors of all of them before
// adding anything, so one L2 round trip serves up to kPer * kBatch loads; the
// additions stay in contributor order, element by element, so vector and
// scalar items give the same bits.
// The flags are checked in the same round trip as the first partials: thread
// i loads the flags of contributors i, i + nthreads, ... and the group agrees
// (all_ok, called exactly once by every thread of the group) before anything
// is stored.  A flag that does not hold `epoch` latches kProtoStaleFlag and
// the tile is left unwritten (returns false).  `issued` runs in every thread
// once its first round of loads is out (the caller's launch bookkeeping,
// whose atomic result it waits for, then overlaps those loads).
template <int kW, class BaseFn, class AllFn, class IssuedFn>
__device__ __forceinline__ bool reduce_items(const GemvArgs &a, int t, uint32_t epoch, int n0, int rows, int C,
                                             BaseFn contributor_base, AllFn all_ok, IssuedFn issued, int tid,
                                             int nthreads) {
    // kW: outputs per item (4: float4 vectors, 1: scalars)
    constexpr int kPer = kW == 4 ? 2 : 4;
    constexpr int kBatch = 8;
    using V = typename std::conditional<kW == 4, float4, float>::type;
    const int S = a.splits;
    const int per_row = rows / kW;           // items per batch row
    const int count = per_row * a.B;         // items of the tile
    bool checked = false;
    for (int i0 = tid; i0 < count || !checked; i0 += nthreads * kPer) {
        const bool active = i0 < count;
        size_t off[kPer];                    // element offset b * N + n of the item's first output
        V acc[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = min(i0 + k * nthreads, max(count - 1, 0));
            const int b = per_row > 0 ? i / per_row : 0;
            const int n = n0 + (i - b * per_row) * kW;
            off[k] = (size_t)b * a.N + n;
        }
        for (int j0 = 0; j0 < C; j0 += kBatch) {
            // First round: this thread's flag (the common case, C <= nthreads:
            // one load) goes out with the partial loads.
            uint32_t f0 = epoch;
            const bool first = !checked;
            if (first && tid < C) f0 = ld_relaxed_gpu_u32(flag_of(a, tid / S, t, S, tid % S));
            V v[kBatch][kPer];
            if (active) {
#pragma unroll
                for (int c = 0; c < kBatch; ++c) {
                    if (j0 + c < C) {
                        const float *base = reinterpret_cast<const float *>(contributor_base(j0 + c));
#pragma unroll
                        for (int k = 0; k < kPer; ++k) v[c][k] = __ldcg(reinterpret_cast<const V *>(base + off[k]));
                    }
                }
            }
            if (first) {
                issued();
                checked = true;
                bool ok = true;
                for (int j = tid; j < C; j += nthreads) {
                    const int q = j / S;
                    const uint32_t f = j == tid ? f0 : ld_relaxed_gpu_u32(flag_of(a, q, t, S, j - q * S));
                    if (f != epoch) {
                        latch_status(a.status, kProtoStaleFlag, q, t, epoch);
                        ok = false;
                    }
                }
                if (!all_ok(ok)) return false;
            }
            if (active) {
#pragma unroll
                for (int c = 0; c < kBatch; ++c) {
                    if (j0 + c < C) {
#pragma unroll
                        for (int k = 0; k < kPer; ++k) {
                            if (j0 + c == 0) {
                                acc[k] = v[c][k];
                            } else if constexpr (kW == 4) {
                                acc[k].x += v[c][k].x;
                                acc[k].y += v[c][k].y;
                                acc[k].z += v[c][k].z;
                                acc[k].w += v[c][k].w;
                            } else {
                                acc[k] += v[c][k];
                            }
                        }
                    }
                }
            }
        }
        if (active) {
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                if (i0 + k * nthreads < count) {
                    if constexpr (kW == 4) {
                        store_output4(a, off[k], acc[k]);
                    } else {
                        store_output(a, off[k], acc[k]);
                    }
                }
            }
        }
    }
    return true;
}

template <class BaseFn, class AllFn, class IssuedFn>
__device__ __forceinline__ bool reduce_tile(const GemvArgs &a, int t, uint32_t epoch, int n0, int rows, int C,
                                            BaseFn contributor_base, AllFn all_ok, IssuedFn issued, int tid,
                                            int nthreads) {
    if ((a.N & 3) == 0 && C <= 8)
        return reduce_items<4>(a, t, epoch, n0, rows, C, contributor_base, all_ok, issued, tid, nthreads);
    return reduce_items<1>(a, t, epoch, n0, rows, C, contributor_base, all_ok, issued, tid, nthreads);
}

// Contributor order: rank 0..R-1, and within a rank split 0..S-1.
__device__ __forceinline__ const uint8_t *contributor_partials(const GemvArgs &a, int j) {
    const int q = j / a.splits;
    return a.scratch + (long long)q * a.stride + (long long)(j - q * a.splits) * a.partial_stride;
}

// Steps 2-4 of the protocol.  Called by ALL threads of the CTA after each
// thread has stored its part of contributor (r, s)'s partial for tile t;
// `epoch` (step 0) is needed in thread 0 only, which publishes.
// Thread 0 stores the contributor's flag next to the partial stores, so one
// fence orders both before the ticket: the flag is a record of which launch
// the partial belongs to, checked by the reducer, while the ticket (an
// acq_rel atomic) is what orders the reducer's loads after every
// contributor's stores.
// Timeline slots of the per-tile kernel (timeline build only): 3 partial
// fenced, 4 ticket taken, 5 reducer: first loads out and launch bookkeeping
// done, 6 reduction stored (reducer), 7 exit, 8 1 if this CTA reduced its
// tile.
__device__ __forceinline__ void publish_and_reduce(const GemvArgs &a, uint32_t epoch, int t, int r, int s) {
    __shared__ int s_last;
    __shared__ uint32_t s_epoch;
    const int S = a.splits;
    const uint32_t C = (uint32_t)a.R * (uint32_t)S;   // contributors per tile
    uint32_t done = 0;                                 // thread 0, reducer: tiles counted before this one
    if (threadIdx.x == 0) st_relaxed_gpu_u32(flag_of(a, r, t, S, s), epoch);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 3);
        s_last = take_ticket(a, t, C, r, epoch, &done) == C - 1u;
        s_epoch = epoch;
        if (a.my_rank >= 0) count_unit(a, a.units_done, epoch, (uint32_t)a.num_tiles);
        tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 4);
        tl_value(a.tl, a.tl_ctas, blockIdx.x, 8, s_last ? 1ull : 0ull);
        if (!s_last) tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 7);
    }
    __syncthreads();
    if (!s_last) return;
    const uint32_t e = s_epoch;
    const int n0 = t * a.rows_per_tile;
    const int rows = min(a.rows_per_tile, a.N - n0);
    reduce_tile(a, t, e, n0, rows, (int)C, [&](int j) { return contributor_partials(a, j); },
                [](bool ok) { return __syncthreads_and(ok) != 0; },
                [&]() {
                    if (threadIdx.x == 0) {
                        finish_launch_if_last(a, done, e, t);
                        tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 5);
                    }
                },
                (int)threadIdx.x, (int)blockDim.x);
    if (threadIdx.x == 0) {
        tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 6);
        tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 7);
    }
}

}  // namespace symm
