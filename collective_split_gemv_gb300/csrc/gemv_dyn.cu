// Persistent, dynamically scheduled fused GEMV + one-shot all-reduce: one or
// more CTAs per SM draw whole (row tile, rank) units from an atomic work
// counter and stream them through a TMA ring into the tcgen05 tensor cores,
// at every batch width.
//
// Why this shape: W is read exactly once, so the kernel is bound by HBM, and
// what costs time besides bytes is (a) a CTA's start-up and wind-down, which
// do not stream, and (b) SMs that finish their share early.  Persistent CTAs
// pay (a) once per launch instead of once per unit, and drawing units from a
// shared counter removes (b) -- a static partition cannot adapt to SMs whose
// bandwidth differs.  A unit's epilogue (partial store, publish, and the
// tile reduction when it is the last contributor) overlaps the streaming of
// the CTA's next unit: the accumulator is double-buffered in TMEM.
//
// Units: a unit is one K split of one (row tile, rank) pair, numbered
// tile-major, u = (t * R + r) * S + s, so that a tile's contributors are
// drawn close together.  S > 1 only serves to make units small enough that
// drawing them balances the SMs.
//
// Work counter: slot 0's signal pad holds two; launch e draws from
// work[e & 1], which starts at zero (the previous launch's last tile reducer
// cleared it).  CTA c starts with unit c (G <= U) and then draws: ticket k
// names unit G + k; U - G tickets name units and each of the G CTAs draws
// exactly one ticket past the end, which tells it to stop.
//
// Roles (192 threads):
//   warp 0, lane 0  draws units, issues the TMA loads of each unit's K blocks
//                   (W 128 rows x 64*kSlabs, x 16 rows x 64*kSlabs, 128-byte
//                   swizzle; W of a packed weight as kSlabs contiguous 16 KB
//                   blocks already in that byte order) and tags every stage
//                   with (unit, block);
//   warp 1          TMEM owner; lane 0 issues the MMAs of each stage and, at a
//                   unit's last block, hands the accumulator and the unit id
//                   to the epilogue;
//   warps 2-5       tcgen05.ld of the accumulator, then the partial store and
//                   the publish / last-arriver protocol of the tile (R * S
//                   contributors).
// Unit ids travel with the stages (producer -> MMA) and through a two-entry
// mailbox (MMA -> epilogue) guarded by its own mbarrier.
// A stage tagged -1 ends the stream.
//
// Follows the fused GEMV + AllReduce of "Overlapping Collective Communication
// with Dependent Computation ... GPU-Initiated Intra-Kernel Networking"
// (Abstract): partials are published as soon as a unit is computed, the
// reduction of a tile overlaps the streaming of other units, and the
// workgroup scheduling is communication-aware (units are drawn tile-major, so
// a tile's R contributors run close together and its partials stay in L2).
//
// Cluster epilogue (kCl): when every unit has a CTA slot of its own (one
// wave), or units are long, the launch is a grid of thread-block clusters of
// C = R * splits CTAs (at most 8), cluster t holding the C units of row tile
// t (CTA rank j = contributor j: rank j / splits, K split j % splits).
// Nothing is drawn; each CTA streams its one unit, and its epilogue puts the
// fp32 partial into the CTA's own shared memory (the drained ring) instead of
// the scratch region.  One cluster barrier (release / acquire) then
// publishes the C partials, and every CTA sums its share of the tile over
// them -- read from the peers' shared memory, in contributor order, in fp32,
// the same additions as the global-memory reducer -- and stores the result; a second barrier keeps
// each CTA's shared memory alive until its peers have read it.  This replaces
// the global-memory protocol's round trips at the end of the launch (partial
// store, fence, ticket, then flag and partial loads by the last arriver),
// which in a one-wave launch are not hidden behind other units.
//
// Safety: all mbarrier waits are bounded (%globaltimer); decisions that
// steer the group's named barrier are made uniform with bar.red.and; a CTA
// that gave up latches a status code, waits (bounded) for its copies and MMAs
// in flight, frees TMEM and exits without publishing.
//
// Timeline slots (timeline build only, timeline.cuh), one row per CTA:
//   0 entry                      1 set-up done (barriers, TMEM)
//   2 first W load issued        3 dependency wait passed (producer)
//   4 first stage full (MMA)     5 first accumulator ready (epilogue)
//   6 last accumulator ready     7 last unit published
//   8 last tile reduction done   9 exit
//  10 units computed (count)    11 tile reductions (count)
//  12 last stage issued         13 producer saw the end of the work
//  14 cluster epilogue: partials published (first cluster barrier passed)
//  15 cluster epilogue: share of the tile stored
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "protocol.cuh"
#include "sm100.cuh"
#include "timeline.cuh"

namespace symm {

namespace {

constexpr int kM = kDynRows;
constexpr int kNmma = 16;
constexpr int kSlabA = kM * 64 * 2;
constexpr int kSlabX = kNmma * 64 * 2;
constexpr int kThreads = 192;
constexpr int kGroupThreads = 128;
constexpr int kGroupBarrier = 1;
constexpr uint32_t kTmemCols = 32;
constexpr uint32_t kIdesc = mma_idesc_bf16_f32(kM, kNmma);

template <int kSlabs, int kCps>
struct Ring {
    static constexpr int kStageBytes = kSlabs * (kSlabA + kSlabX);
    static constexpr int kStages = ((216 * 1024) / kCps) / kStageBytes;
    static constexpr int kSmem = kStages * kStageBytes + 1024;
};

__device__ __forceinline__ bool group_all(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n.reg .pred p, q;\n"
        "setp.ne.u32 q, %1, 0;\n"
        "bar.red.and.pred p, %2, %3, q;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(kGroupBarrier), "r"(kGroupThreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t atom_add_relaxed_gpu(uint32_t *p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Steps 2-4 of the protocol for contributor (r, s) of tile t (C = R * S
// contributors: every rank's K range in S splits), run by the 128 threads of
// warps 2-5 (gt = 0..127).  The caller has stored its partial; the flag goes
// out with it, before the fence, and the reducer checks the flags in the
// same round of loads as its first partials (protocol.cuh).  Returns whether
// this group reduced the tile.
__device__ __forceinline__ bool publish_reduce_unit(const GemvArgs &a, uint32_t epoch, int S, int t, int r, int s,
                                                    int gt, int *s_last) {
    const uint32_t C = (uint32_t)a.R * (uint32_t)S;
    uint32_t done = 0;   // gt == 0, reducer: tiles counted before this one
    if (gt == 0) st_relaxed_gpu_u32(flag_of(a, r, t, S, s), epoch);
    __threadfence();
    named_barrier(kGroupBarrier, kGroupThreads);
    if (gt == 0) *s_last = take_ticket(a, t, C, r, epoch, &done) == C - 1u;
    named_barrier(kGroupBarrier, kGroupThreads);
    if (!*s_last) return false;
    reduce_tile(a, t, epoch, t * kM, min(kM, a.N - t * kM), (int)C,
                [&](int j) { return contributor_partials(a, j); }, [](bool ok) { return group_all(ok); },
                [&]() {
                    if (gt == 0) finish_launch_if_last(a, done, epoch, t);
                },
                gt, kGroupThreads);
    return true;
}

// Unit u of this launch: (tile t, rank r, K split s).  Units are numbered
// tile-major, u = (t * R + r) * S + s; a multi-process handle's launch
// covers its own rank only, u = t * S + s.
__device__ __forceinline__ void unit_of(const GemvArgs &a, int u, int S, int *t, int *r, int *s) {
    const int tr = u / S;
    *s = u - tr * S;
    if (a.my_rank >= 0) {
        *t = tr;
        *r = a.my_rank;
    } else {
        *t = tr / a.R;
        *r = tr - *t * a.R;
    }
}

static_assert(kM == kPackRows && kSlabA == (int)kPackBlockBytes, "a stage slab is one block of the packed layout");

// W slab j (64 columns) of row tile t, rank r, into one stage slab: a TMA box
// of the row-major W_r, or the same bytes as one contiguous block of the
// packed layout (past the last slab: the slot's zero block, as the tensor
// map's fill would give).
// W is read once per call: its lines are marked evict-first in L2, so that
// the stream does not push out what is read again soon (x, the partials).
__device__ __forceinline__ void load_w_slab(uint8_t *dst, const CUtensorMap *tmW, const GemvArgs &a, uint64_t *bar,
                                            int j, int t, int r, uint64_t policy) {
    if (a.w_packed) {
        const int J = (a.Kr + kPackCols - 1) / kPackCols;
        const size_t blk = j < J ? (size_t)t * J + j : (size_t)a.num_tiles * J;
        bulk_load_hint(dst, a.W + (long long)r * a.stride + blk * kPackBlockBytes, (uint32_t)kPackBlockBytes, bar,
                       policy);
    } else {
        tma_load_3d_hint(dst, tmW, bar, j * 64, t * kM, r, policy);
    }
}

// The cluster epilogue's sum (kCl): CTA `me` of the C-CTA cluster of row
// tile t (C = R * splits contributors, CTA rank j = contributor j: rank
// j / splits, K split j % splits) sums its share of the tile's [b][row]
// outputs over the C partials (each CTA's `part`, [b][kM] fp32 in its own
// shared memory), in contributor order, element by element as reduce_items
// does, and stores them; kW = 4: four consecutive rows per item (N % 4 ==
// 0), else single outputs.  All kThreads threads of the CTA take part;
// between the two cluster barriers only the loads from the peers happen, the
// stores follow the second arrive.
template <int kW>
__device__ __forceinline__ void cluster_sum_tile(const GemvArgs &a, const float *part, const int *abort_word, int t,
                                                 int me, int C, int tid) {
    using V = typename std::conditional<kW == 4, float4, float>::type;
    constexpr int kPerRow = kM / kW;                         // items per batch row
    constexpr int kMax = (kNmma * kPerRow + kThreads - 1) / kThreads;   // items per thread at R = 1, B = 16
    const int n0 = t * kM;
    const int rows = min(kM, a.N - n0);
    const int items = a.B * kPerRow;
    const int share = (items + C - 1) / C;
    // A tile is stored only if all C units were computed (a CTA that gave up
    // has latched the status): the C abort words are read in the same round
    // of loads as the partials.
    int bad = 0;
#pragma unroll
    for (int q = 0; q < kMaxClusterRanks; ++q)
        if (q < C) bad |= ld_cluster_s32(cluster_addr(abort_word, (uint32_t)q));
    V acc[kMax];
    size_t off[kMax];
    bool mine[kMax];
#pragma unroll
    for (int k = 0; k < kMax; ++k) {
        const int l = tid + k * kThreads;                    // this thread's k-th item of the share
        const int i = me * share + l;
        const int b = i / kPerRow;
        const int row = (i - b * kPerRow) * kW;
        mine[k] = l < share && i < items && row < rows;
        off[k] = (size_t)b * a.N + n0 + row;
        if (mine[k]) {
            const int e = b * kM + row;
            V v[kMaxClusterRanks];
#pragma unroll
            for (int q = 0; q < kMaxClusterRanks; ++q) {
                if (q < C) {
                    if constexpr (kW == 4) {
                        v[q] = ld_cluster_v4f32(cluster_addr(part + e, (uint32_t)q));
                    } else {
                        v[q] = ld_cluster_f32(cluster_addr(part + e, (uint32_t)q));
                    }
                }
            }
            acc[k] = v[0];
#pragma unroll
            for (int q = 1; q < kMaxClusterRanks; ++q) {
                if (q < C) {
                    if constexpr (kW == 4) {
                        acc[k].x += v[q].x;
                        acc[k].y += v[q].y;
                        acc[k].z += v[q].z;
                        acc[k].w += v[q].w;
                    } else {
                        acc[k] += v[q];
                    }
                }
            }
        }
    }
    // The peers' shared memory has been read (arrive orders the loads before
    // it); every peer waits for this before it leaves.
    cluster_arrive_release();
#pragma unroll
    for (int k = 0; k < kMax; ++k) {
        if (mine[k] && bad == 0) {
            if constexpr (kW == 4) {
                store_output4(a, off[k], acc[k]);
            } else {
                store_output(a, off[k], acc[k]);
            }
        }
    }
}

// At two CTAs per SM the register file must hold both (at most 168
// registers a thread); the three-CTA rings do not fit it and run in two waves.
template <int kSlabs, int kCps, bool kCl>
__global__ void __launch_bounds__(kThreads, kCps == 2 ? 2 : 1)
    gemv_ar_dyn_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                       const GemvArgs a, const DynGeom geo) {
    // Dependents of this launch (the RMSNorm stage, or the next fused call
    // when calls are chained) may be scheduled as CTAs of this one retire;
    // they wait for this grid before touching anything it writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        tl_begin();
        tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 0);
    }
    using RingT = Ring<kSlabs, kCps>;
    static_assert(RingT::kStages >= 2, "the ring needs at least two stages");
    static_assert(!kCl || RingT::kStageBytes >= kNmma * kM * 4, "cluster epilogue: the partial fits in a stage");
    constexpr int kStages = RingT::kStages;
    constexpr int kStageBytes = RingT::kStageBytes;
    constexpr int kBK = 64 * kSlabs;

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t acc_full[2];
    __shared__ __align__(8) uint64_t acc_empty[2];
    __shared__ __align__(8) uint64_t unit_full[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ int stage_unit[kStages];
    __shared__ int stage_flags[kStages];   // bit 0: first block of the unit, bit 1: last
    __shared__ int acc_unit[2];
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    __shared__ int s_last;
    __shared__ uint32_t epoch_sh;

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int U = geo.units;            // (tile, rank, split) triples, tile-major
    const int S = geo.splits;
    const int KBs = geo.KBs;            // K blocks per split (the last split may have fewer)
    const int KB = geo.KB;

    if (threadIdx.x == 0) {
        // The descriptors' fetch overlaps the set-up below (the first TMA
        // load would otherwise wait for it).
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&acc_full[j], 1);
            // Drained by the 4 epilogue warps; the unit id comes from the MMA
            // thread.
            mbar_init(&acc_empty[j], 4);
            mbar_init(&unit_full[j], 1);
        }
        mbar_init(&drain_bar, 1);
        abort_sh = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(&tmem_base_sh, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 1);
    const uint32_t tmem = tmem_base_sh;
    // Launched as a programmatic dependent of the previous kernel (calls
    // chained on one stream), this grid may start while that one drains.
    // Everything below except, for a packed weight, the producer's first W
    // loads can depend on it (x, scratch, the pad, y, a row-major W), so every
    // other thread waits for it here; the wait returns at once when the
    // launch was not a programmatic dependent.
    int pre = 0;   // producer: stages of the first unit issued here
    // Producer's L2 policies: W streamed once (evict first); x_r re-read by
    // every unit of rank r (evict last).
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_x = l2_policy_evict_last();
    if (warp == 0 && lane == 0) {
        // A packed weight is written once, by symm_pack_w (which the host
        // never chains into a call that reads it), so the W loads of the first
        // unit's first stages go out before the dependency wait and x's after
        // it.  A row-major W may be the output of the kernel just before (any
        // kernel, not only this library's): it is loaded after the wait.
        // The first unit is the CTA's own index (G <= U); in a cluster launch
        // the only one, CTA rank r of cluster t holding unit t * R + r.
        const int u = (a.reverse_order && !kCl) ? U - 1 - (int)blockIdx.x : (int)blockIdx.x;
        int t, r, sp;
        unit_of(a, u, S, &t, &r, &sp);
        const int kb0 = sp * KBs;
        const int kb1 = min(kb0 + KBs, KB);
        pre = min(kStages, kb1 - kb0);
        if (!a.w_early) griddep_wait();
        tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 2);
        for (int i = 0; i < pre; ++i) {   // the ring is empty: no wait
            const int kb = kb0 + i;
            stage_unit[i] = u;
            stage_flags[i] = (kb == kb0 ? 1 : 0) | (kb == kb1 - 1 ? 2 : 0);
            mbar_arrive_expect_tx(&full_bar[i], (uint32_t)kStageBytes);
            uint8_t *dst = smem + (size_t)i * kStageBytes;
#pragma unroll
            for (int s = 0; s < kSlabs; ++s)
                load_w_slab(dst + s * kSlabA, &tmW, a, &full_bar[i], kb * kSlabs + s, t, r, pol_w);
        }
        if (a.w_early) griddep_wait();
        tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 3);
        for (int i = 0; i < pre; ++i) {
            const int kb = kb0 + i;
            uint8_t *dst = smem + (size_t)i * kStageBytes;
#pragma unroll
            for (int s = 0; s < kSlabs; ++s)
                tma_load_3d_hint(dst + kSlabs * kSlabA + s * kSlabX, &tmX, &full_bar[i], kb * kBK + s * 64, 0, r,
                                 pol_x);
        }
        // Step 0 of the protocol: the launch epoch, read once per CTA and
        // shared through the barrier below (which orders the read before
        // every publish of this CTA).  Its latency overlaps the loads above.
        epoch_sh = read_launch_epoch(a);
    } else {
        griddep_wait();
    }
    __syncthreads();
    const uint32_t epoch = epoch_sh;
    uint32_t *const work = a.work + (epoch & 1u);

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            int issued = pre;
            // Later units are drawn: ticket k names unit G + k.
            uint32_t tk = blockIdx.x;
            bool ok = true;
            bool first = true;
            while (ok) {
                const int st0 = issued % kStages;
                const uint32_t ph0 = (uint32_t)(issued / kStages) & 1u;
                if (tk >= (uint32_t)U) {
                    tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 13);
                    // End of the stream: an empty stage tagged -1.
                    if (!mbar_wait(&empty_bar[st0], ph0 ^ 1u, &abort_sh)) {
                        ok = false;
                        break;
                    }
                    stage_unit[st0] = -1;
                    stage_flags[st0] = 0;
                    mbar_arrive(&full_bar[st0]);
                    ++issued;
                    break;
                }
                const int u = (a.reverse_order && !kCl) ? U - 1 - (int)tk : (int)tk;
                int t, r, sp;
                unit_of(a, u, S, &t, &r, &sp);
                const int kb0 = sp * KBs;
                const int kb1 = min(kb0 + KBs, KB);
                // The next unit is drawn right after the loads of this unit's
                // last K block are issued: late enough that a CTA on a slow SM
                // does not take a unit a faster one would finish first (the
                // draw decides who gets the remaining units), early enough that
                // the atomic's latency hides behind the stages still in the
                // ring.  The ticket -> unit arithmetic sits in an asm statement
                // after the loop, so no instruction waits on the atomic early.
                const int kb_from = first ? kb0 + pre : kb0;   // the first unit's first stages are out
                first = false;
                uint32_t next_raw = 0u;
                if (!kCl && kb_from >= kb1) next_raw = atom_add_relaxed_gpu(work, 1u);
                for (int kb = kb_from; kb < kb1; ++kb) {
                    const int st = issued % kStages;
                    const uint32_t ph = (uint32_t)(issued / kStages) & 1u;
                    if (!mbar_wait(&empty_bar[st], ph ^ 1u, &abort_sh)) {
                        ok = false;
                        break;
                    }
                    stage_unit[st] = u;
                    stage_flags[st] = (kb == kb0 ? 1 : 0) | (kb == kb1 - 1 ? 2 : 0);
                    mbar_arrive_expect_tx(&full_bar[st], (uint32_t)kStageBytes);
                    uint8_t *dst = smem + (size_t)st * kStageBytes;
#pragma unroll
                    for (int s = 0; s < kSlabs; ++s)
                        load_w_slab(dst + s * kSlabA, &tmW, a, &full_bar[st], kb * kSlabs + s, t, r, pol_w);
#pragma unroll
                    for (int s = 0; s < kSlabs; ++s)
                        tma_load_3d_hint(dst + kSlabs * kSlabA + s * kSlabX, &tmX, &full_bar[st], kb * kBK + s * 64,
                                         0, r, pol_x);
                    if (!kCl && kb == kb1 - 1) next_raw = atom_add_relaxed_gpu(work, 1u);
                    ++issued;
                    tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 12);
                }
                if constexpr (kCl) {
                    tk = (uint32_t)U;   // one unit per CTA, nothing drawn
                } else {
                    asm volatile("add.u32 %0, %1, %2;" : "=r"(tk) : "r"(next_raw), "r"((uint32_t)geo.G));
                }
            }
            if (!ok) {
                latch_status(a.status, kProtoTimeout, -1, -1, epoch);
                abort_sh = 1;
                volatile int never = 0;
                for (int j = max(0, issued - kStages); j < issued; ++j)
                    mbar_wait(&full_bar[j % kStages], (uint32_t)(j / kStages) & 1u, &never);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int i = 0, seg = 0;
            bool ok = true;
            while (true) {
                const int st = i % kStages;
                const uint32_t ph = (uint32_t)(i / kStages) & 1u;
                if (!mbar_wait(&full_bar[st], ph, &abort_sh)) {
                    ok = false;
                    break;
                }
                if (i == 0) tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 4);
                const int u = stage_unit[st];
                const int fl = stage_flags[st];
                const int j = seg & 1;
                const uint32_t use = (uint32_t)(seg >> 1);
                if (u < 0 || (fl & 1)) {
                    // Buffer j must have been drained (its previous unit read out).
                    if (!mbar_wait(&acc_empty[j], (use & 1u) ^ 1u, &abort_sh)) {
                        ok = false;
                        break;
                    }
                }
                if (u < 0) {
                    acc_unit[j] = -1;
                    mbar_arrive(&unit_full[j]);
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(j * kNmma);
                const uint32_t a_addr = smem_u32(smem + (size_t)st * kStageBytes);
                const uint32_t x_addr = a_addr + kSlabs * kSlabA;
#pragma unroll
                for (int s = 0; s < kSlabs; ++s)
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma(d, smem_desc_sw128(a_addr + s * kSlabA + kk * 32),
                               smem_desc_sw128(x_addr + s * kSlabX + kk * 32), kIdesc,
                               ((fl & 1) && s == 0 && kk == 0) ? 0u : 1u);
                tc_commit(&empty_bar[st]);
                ++i;
                if (fl & 2) {
                    acc_unit[j] = u;
                    mbar_arrive(&unit_full[j]);
                    tc_commit(&acc_full[j]);
                    ++seg;
                }
            }
            if (!ok) {
                latch_status(a.status, kProtoTimeout, -1, -1, epoch);
                abort_sh = 1;
            }
            tc_commit(&drain_bar);
            volatile int never = 0;
            mbar_wait(&drain_bar, 0, &never);
        }
    } else {
        // ---------------------------------------------- epilogue (warps 2-5)
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const int gt = threadIdx.x - 64;
        bool ok = true;
        int seg = 0;
        int n_reduced = 0;   // timeline only
        (void)n_reduced;
        while (true) {
            const int j = seg & 1;
            const uint32_t use = (uint32_t)(seg >> 1);
            ok = group_all(mbar_wait_sleepy(&unit_full[j], use & 1u, &abort_sh));
            if (!ok) break;
            const int u = acc_unit[j];
            if (u < 0) break;
            ok = group_all(mbar_wait_sleepy(&acc_full[j], use & 1u, &abort_sh));
            if (!ok) break;
            if (gt == 0) {
                if (seg == 0) tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 5);
                tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 6);
            }
            tc_fence_after();
            float v[16];
            tmem_ld_16(tmem + (uint32_t)(j * kNmma) + ((uint32_t)(q4 * 32) << 16), v);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[j]);
            if constexpr (kCl) {
                // The partial goes to the drained ring (every MMA of the
                // CTA's one unit has completed, no copy is in flight);
                // the proxy fence orders those asynchronous accesses of
                // the ring before these plain stores.
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                float *part = reinterpret_cast<float *>(smem);
#pragma unroll
                for (int b = 0; b < kNmma; ++b)
                    if (b < a.B) part[b * kM + row] = v[b];
                ++seg;
                continue;
            }
            int t, r, sp;
            unit_of(a, u, S, &t, &r, &sp);
            const int n = t * kM + row;
            if (n < a.N) {
                float *P = reinterpret_cast<float *>(a.scratch + (long long)r * a.stride +
                                                     (long long)sp * a.partial_stride);
#pragma unroll
                for (int b = 0; b < kNmma; ++b)
                    if (b < a.B) P[(size_t)b * a.N + n] = v[b];
            }
            bool reduced = false;
            if (a.out_mode == kOutPartials) {
                if (gt == 0) count_unit(a, a.tiles_done, epoch, (uint32_t)U);
            } else {
                reduced = publish_reduce_unit(a, epoch, S, t, r, sp, gt, &s_last);
                if (a.my_rank >= 0 && gt == 0) count_unit(a, a.units_done, epoch, (uint32_t)U);
            }
            ++seg;
            if (gt == 0) {
                tl_stamp(a.tl, a.tl_ctas, blockIdx.x, reduced ? 8 : 7);
                if (reduced) tl_value(a.tl, a.tl_ctas, blockIdx.x, 11, (unsigned long long)++n_reduced);
                tl_value(a.tl, a.tl_ctas, blockIdx.x, 10, (unsigned long long)seg);
            }
        }
        if (!ok) {
            latch_status(a.status, kProtoTimeout, -1, -1, epoch);
            abort_sh = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if constexpr (kCl) {
        // Every CTA of the cluster reaches this point (all waits above are
        // bounded), also one that gave up: the barriers need all of them.
        cluster_arrive_release();
        cluster_wait_acquire();
        if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 14);
        // Unit u = blockIdx.x = t * C + j, j = r * S + s: the cluster of row
        // tile t, CTA rank j.
        const int C = a.R * S;
        const int me = (int)(blockIdx.x % (unsigned)C);
        const int t = (int)(blockIdx.x / (unsigned)C);
        const float *part = reinterpret_cast<const float *>(smem);
        const int *abort_word = const_cast<const int *>(&abort_sh);
        if ((a.N & 3) == 0)
            cluster_sum_tile<4>(a, part, abort_word, t, me, C, (int)threadIdx.x);
        else
            cluster_sum_tile<1>(a, part, abort_word, t, me, C, (int)threadIdx.x);
        if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 15);
        cluster_wait_acquire();
    }
    if (threadIdx.x == 0) {
        // (every other thread's stamps came before the barrier above)
        tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 9);
        tl_end(a.tl, a.tl_ctas, blockIdx.x);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int kSlabs, int kCps, bool kCl>
cudaError_t launch_cfg(const GemvArgs &a, const DynGeom &geo, const CUtensorMap *m, bool chained, cudaStream_t s) {
    auto kern = gemv_ar_dyn_kernel<kSlabs, kCps, kCl>;
    constexpr int smem = Ring<kSlabs, kCps>::kSmem;
    static std::atomic<unsigned long long> attr_devices{0};
    cudaError_t e = set_smem_once(kern, smem, attr_devices);
    if (e != cudaSuccess) return e;
    if (!kCl) return launch_kernel(kern, dim3((unsigned)geo.G), dim3(kThreads), (size_t)smem, s, chained, m[0], m[1], a, geo);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)geo.G, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)geo.cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int nattr = 1;
    if (chained) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        nattr = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    return cudaLaunchKernelEx(&cfg, kern, m[0], m[1], a, geo);
}

cudaError_t launch_pipeline(const GemvArgs &a, const DynGeom &geo, const CUtensorMap *m, int slabs, int cps,
                            bool chained, cudaStream_t s) {
    if (geo.cluster) {
        // Cluster epilogue: rings sized for two CTAs per SM.
        switch (cps * 10 + slabs) {
            case 21: return launch_cfg<1, 2, true>(a, geo, m, chained, s);
            case 22: return launch_cfg<2, 2, true>(a, geo, m, chained, s);
            case 23: return launch_cfg<3, 2, true>(a, geo, m, chained, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (cps * 10 + slabs) {
        case 11: return launch_cfg<1, 1, false>(a, geo, m, chained, s);
        case 12: return launch_cfg<2, 1, false>(a, geo, m, chained, s);
        case 14: return launch_cfg<4, 1, false>(a, geo, m, chained, s);
        case 21: return launch_cfg<1, 2, false>(a, geo, m, chained, s);
        case 22: return launch_cfg<2, 2, false>(a, geo, m, chained, s);
        case 23: return launch_cfg<3, 2, false>(a, geo, m, chained, s);
        case 31: return launch_cfg<1, 3, false>(a, geo, m, chained, s);
        default: return cudaErrorInvalidValue;
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library); looked up once, thread-safe.
EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return nullptr;
    }();
    return fn;
}

// A 3-D view [R][rows][Kr] of bf16 with the slot stride as the rank stride;
// boxes of 64 columns x box_rows rows, 128-byte swizzle, zero fill outside.
int encode_3d(CUtensorMap *m, const void *base, int Kr, int rows, int R, long long stride, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return -1;
    const cuuint64_t dims[3] = {(cuuint64_t)Kr, (cuuint64_t)rows, (cuuint64_t)R};
    const cuuint64_t strides[2] = {(cuuint64_t)Kr * 2, (cuuint64_t)stride};
    const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult rc = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS ? 0 : (int)rc;
}

}  // namespace

int dyn_encode_maps(const GemvArgs &a, void *maps) {
    CUtensorMap *m = static_cast<CUtensorMap *>(maps);
    int rc = encode_3d(&m[0], a.W, a.Kr, a.N, a.R, a.stride, kM);
    if (rc != 0) return rc;
    return encode_3d(&m[1], a.x, a.Kr, a.B, a.R, a.stride, kNmma);
}

int dyn_block_k(int slabs) { return 64 * slabs; }

// Pipeline shapes that are instantiated: (slabs, CTAs per SM) with a ring of
// at least two stages.
bool dyn_config_supported(int slabs, int cps) {
    return (cps == 1 && (slabs == 1 || slabs == 2 || slabs == 4)) ||
           (cps == 2 && (slabs == 1 || slabs == 2 || slabs == 3)) || (cps == 3 && slabs == 1);
}

bool dyn_cluster_supported(int slabs, int cps) {
    return cps == 2 && (slabs == 1 || slabs == 2 || slabs == 3);
}

namespace {

template <int kSlabs>
int max_active_clusters(int R) {
    auto kern = gemv_ar_dyn_kernel<kSlabs, 2, true>;
    constexpr int smem = Ring<kSlabs, 2>::kSmem;
    static std::atomic<unsigned long long> attr_devices{0};
    if (set_smem_once(kern, smem, attr_devices) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)R, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)R;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace

bool dyn_cluster_fits(int slabs, int R) {
    // Per device, slab count and R: 0 unknown, 1 fits, 2 does not.
    static std::atomic<unsigned char> known[64][4][kMaxClusterRanks + 1];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || slabs < 1 || slabs > 3 || R < 1 ||
        R > kMaxClusterRanks)
        return false;
    std::atomic<unsigned char> &k = known[dev][slabs][R];
    unsigned char v = k.load(std::memory_order_acquire);
    if (v == 0) {
        const int n = slabs == 1 ? max_active_clusters<1>(R) : slabs == 2 ? max_active_clusters<2>(R)
                                                                           : max_active_clusters<3>(R);
        v = n > 0 ? 1 : 2;
        k.store(v, std::memory_order_release);
    }
    return v == 1;
}

cudaError_t launch_gemv_dyn(const GemvArgs &a, const DynGeom &geo, const void *maps, int slabs, int cps,
                            bool chained, cudaStream_t s) {
    return launch_pipeline(a, geo, static_cast<const CUtensorMap *>(maps), slabs, cps, chained, s);
}

}  // namespace symm
