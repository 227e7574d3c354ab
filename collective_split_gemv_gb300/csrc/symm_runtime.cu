// Host runtime of the symmetric-slot library: the C ABI of include/symm_gemv.h.
//
// Slot layout (every slot identical; stride rounded up to 2 MiB):
//
//   [user region  slot_bytes][guard 4 KiB][scratch][guard][signal pad][guard]
//
// The user region holds the caller's tensors at symmetric offsets (W_r, x_r,
// y, all-reduce in/out), like the per-peer buffers of a symmetric-memory
// handle ("PyTorch Symmetric Memory" docs, "Write your own kernel":
// buffer_ptrs / signal_pad_ptrs).  The scratch region receives the fused
// kernel's fp32 partials, one slot per rank (the peer-visible buffer the
// fused GEMV + AllReduce writes its partials into).  The signal pad holds the
// per-tile flags, the tile arrival counters and the status words.  Guard bands
// are filled with 0xA5 and checked by symm_check_guards.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include <unistd.h>

#include "../../include/symm_gemv.h"
#include "internal.h"
#include "timeline.cuh"

using namespace symm;

struct symm_handle {
    int R = 0;
    int device = 0;
    size_t slot_bytes = 0, scratch_bytes = 0, pad_bytes = 0;
    size_t stride = 0, total = 0;
    size_t guard0 = 0, scratch_off = 0, guard1 = 0, pad_off = 0, guard2 = 0;
    size_t flags_off = 0, counters_off = 0;   // within the pad
    int max_tiles = 0;
    uint8_t *base = nullptr;
    bool owned = false;
    int opt_gemv_path = 0;
    int opt_tile_order = 0;
    int opt_sk_slabs = 0;
    int opt_sk_cps = 0;
    int opt_sk_grid = 0;
    int opt_dyn_splits = 0;
    int opt_norm_pdl = 1;       // launch the RMSNorm stage as a programmatic dependent
    int opt_chain = 1;          // launch the persistent kernel as a programmatic dependent
    int opt_ar_cps = 0;         // all-reduce / reduce-scatter grid cap per SM (0 = the kernels' default)
    int opt_ar_kernel = 0;      // one-shot all-reduce kernel (kArKernel*)
    int opt_copy_engine = 0;    // symm_copy_*: 1 = always the copy engine, 0 = SMs where possible
    int opt_unfused = 0;        // gemv_all_reduce as two kernels (GEMV partials, then their all-reduce)
    int opt_dyn_cluster = -1;   // persistent kernel's cluster epilogue: -1 auto, 0 off, 1 on
    // y of the last persistent-kernel launch on the handle: a chained launch
    // reads W before its predecessor has finished, so W must not overlap it.
    // Slot-0 range written by the last kernel this handle launched (the same
    // offsets in every slot): a chained persistent-kernel launch, which loads
    // W before its predecessor has finished, must not read it.
    const void *last_write = nullptr;
    size_t last_write_bytes = 0;
    // Timeline rows registered by symm_set_timeline (timeline build only).
    unsigned long long *tl = nullptr;
    int tl_ctas = 0;
    // TMA descriptors of recent tensor-core launches (two CUtensorMap each).
    struct MapEntry {
        const void *W = nullptr, *x = nullptr;
        int N = 0, Kr = 0, B = 0;
        alignas(64) unsigned char maps[2][128];
    };
    MapEntry map_cache[8];
    int map_next = 0;
    // Packed weights made by symm_pack_w: slot-0 address, shape, bytes per slot.
    struct PackedW {
        const void *p = nullptr;
        int N = 0, Kr = 0;
        size_t bytes = 0;
    };
    std::vector<PackedW> packed;
    // Multi-process handle (symm_mp_alloc): this process holds rank mp_rank;
    // every rank's slot is a CUDA VMM allocation of its own process, mapped
    // into one reserved range at base + r * stride in every process.
    int mp_rank = -1;
    unsigned long long va = 0;                       // reserved range (CUdeviceptr)
    unsigned long long mem[kMaxRanks] = {};          // mapped allocation of slot r (0: not mapped)
};

namespace {

constexpr size_t kGuard = 4096;
constexpr size_t kAlign = 256;
constexpr size_t kStrideAlign = 2u << 20;
constexpr unsigned char kGuardByte = 0xA5;

thread_local char g_err[512];

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(SYMM_ECUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool mul_overflows(size_t a, size_t b) { return a != 0 && b > SIZE_MAX / a; }

// Fills a handle's offsets from the sizes; returns false on overflow.
bool compute_layout(symm_handle &h) {
    if (h.slot_bytes > SIZE_MAX / 4 || h.scratch_bytes > SIZE_MAX / 4 || h.pad_bytes > SIZE_MAX / 4)
        return false;
    h.guard0 = round_up(h.slot_bytes, kAlign);
    h.scratch_off = h.guard0 + kGuard;
    h.guard1 = h.scratch_off + round_up(h.scratch_bytes, kAlign);
    h.pad_off = h.guard1 + kGuard;
    h.guard2 = h.pad_off + round_up(h.pad_bytes, kAlign);
    h.stride = round_up(h.guard2 + kGuard, kStrideAlign);
    if (mul_overflows(h.stride, (size_t)h.R)) return false;
    h.total = h.stride * (size_t)h.R;
    // Pad: status, then flags[T] and counters[T], each 128-byte aligned.
    size_t room = round_up(h.pad_bytes, kAlign) - kPadStatusBytes;
    size_t T = room / 8;
    T = T / 32 * 32;
    while (T > 0 && kPadStatusBytes + round_up(4 * T, 128) * 2 > round_up(h.pad_bytes, kAlign)) T -= 32;
    h.max_tiles = (int)std::min<size_t>(T, 1u << 30);
    h.flags_off = kPadStatusBytes;
    h.counters_off = kPadStatusBytes + round_up(4 * (size_t)h.max_tiles, 128);
    return true;
}

uint8_t *slot(const symm_handle *h, int r) { return h->base + (size_t)r * h->stride; }
uint32_t *pad_word(const symm_handle *h, int r, size_t off) {
    return reinterpret_cast<uint32_t *>(slot(h, r) + h->pad_off + off);
}

// Every slot of a multi-process handle is mapped (all peers imported).
bool mp_ready(const symm_handle *h) {
    if (h->mp_rank < 0) return true;
    for (int r = 0; r < h->R; ++r)
        if (!h->mem[r]) return false;
    return true;
}

// The handle's device is the current one.
int check_current_device(const symm_handle *h) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != h->device)
        return fail(SYMM_EINVAL, "current device %d differs from the handle's device %d", dev, h->device);
    return SYMM_OK;
}

// The checks before any launch: the handle's device is current and, for a
// multi-process handle, every rank's slot is mapped.
int check_device(const symm_handle *h) {
    if (!mp_ready(h)) return fail(SYMM_EINVAL, "not every rank's slot is mapped yet (symm_mp_import)");
    return check_current_device(h);
}

// [p, p + bytes) inside slot 0's user region?
bool in_user_region(const symm_handle *h, const void *p, size_t bytes) {
    const uint8_t *q = static_cast<const uint8_t *>(p);
    if (q < h->base) return false;
    size_t off = (size_t)(q - h->base);
    return off <= h->slot_bytes && bytes <= h->slot_bytes - off;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uint8_t *x = static_cast<const uint8_t *>(a), *y = static_cast<const uint8_t *>(b);
    if (na == 0 || nb == 0) return false;
    return x < y + nb && y < x + na;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

void note_write(symm_handle *h, const void *p, size_t bytes) {
    h->last_write = p;
    h->last_write_bytes = bytes;
}

const symm_handle::PackedW *find_packed(const symm_handle *h, const void *p) {
    for (const auto &e : h->packed)
        if (e.p == p) return &e;
    return nullptr;
}

// Zero flags, counters, the work counters and the launch epoch
// (stream-ordered): the pad as symm_alloc leaves it.
// A multi-process handle resets its own slot's pad only (rank 0's holds the
// tile counters every rank shares).
int reset_protocol(symm_handle *h, cudaStream_t s) {
    const int own = h->mp_rank >= 0 ? h->mp_rank : 0;
    uint8_t *pad = slot(h, own) + h->pad_off;
    cudaError_t e0;
    if (h->mp_rank >= 0) {
        // A process keeps its launch count (the epoch word): the other ranks
        // compare theirs with it, and each process resets on its own.
        e0 = cudaMemsetAsync(pad + kPadWorkOffset, 0, kPadEpochOffset - kPadWorkOffset, s);
        if (e0 == cudaSuccess)
            e0 = cudaMemsetAsync(pad + kPadEpochOffset + 4, 0, kPadStatusBytes - kPadEpochOffset - 4, s);
    } else {
        e0 = cudaMemsetAsync(pad + kPadWorkOffset, 0, kPadStatusBytes - kPadWorkOffset, s);
    }
    if (e0 != cudaSuccess) return cuda_fail(e0, "cudaMemsetAsync(work counter)");
    for (int r = 0; r < h->R; ++r) {
        if (h->mp_rank >= 0 && r != h->mp_rank) continue;
        cudaError_t e = cudaMemsetAsync(slot(h, r) + h->pad_off + h->flags_off, 0,
                                        h->pad_bytes - h->flags_off, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(signal pad)");
    }
    return SYMM_OK;
}

// SM count of a device, cached per device ordinal (atomics: host threads may
// plan launches concurrently).
int num_sms(int device) {
    static std::atomic<int> cached[64];
    if (device >= 0 && device < 64) {
        const int c = cached[device].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, device) != cudaSuccess || v <= 0) {
        cudaGetLastError();
        return 148;
    }
    if (device >= 0 && device < 64) cached[device].store(v, std::memory_order_relaxed);
    return v;
}

// Kernels: 1 CUDA-core, one CTA per (tile, rank), 128-bit loads; 4
// persistent CTAs drawing (tile, rank) units from a work counter, or one CTA
// per unit in clusters (TMA ring into tcgen05, double-buffered accumulator in
// TMEM).  The automatic choice is 4 whenever K > 0 (1 for K = 0, and for
// small W, below), with two CTAs per SM and two 64-column slabs per stage: the
// fastest configuration measured on the decode (B = 1), attention-projection
// (B = 8) and large (B = 16) shapes.  Paths 2 (one tensor-core CTA per tile)
// and 3 (static stream-K partition) were retired, and so was the persistent
// kernel's CUDA-core engine: none of them won on any shape measured.  5 is the cluster kernel for
// small layers: one thread-block cluster of R CTAs per row tile, the partials
// exchanged through distributed shared memory instead of the global-memory
// protocol (R <= 8, B <= 4).
constexpr int kPathFfma = 1, kPathDyn = 4, kPathCluster = 5;
// K/R from which the persistent kernel's units (128 rows x K/R bf16, 768 KB
// here) take the cluster epilogue even when they do not fit in one wave.
constexpr int kClusterEpilogueMinKr = 3072;

// Below this many bytes of W a call is latency-bound: the persistent
// kernel's start-up costs more than it saves, and for narrow batches a
// per-tile kernel returns first (measured on 0.3-17 MB): the cluster kernel
// where R and B allow it, else the CUDA-core one.
constexpr size_t kSmallWBytes = 24u << 20;
constexpr int kSmallMaxBatch = 4;
// The cluster kernel does every product on the CUDA cores, one cluster of R
// CTAs per 16 rows: it returns first while its CTAs times the batch width
// stay at most this, beyond that the persistent kernel's tensor cores do.
// Measured per launch, L2 flushed, cluster kernel / persistent kernel, us
// (R, N, K, B; CTAs x B): 2, 256, 512, 1 (32): 7.0 / 12.4; 2, 2048, 4096,
// 1 (256): 10.4 / 13.5; 2, 1024, 4096, 4 (512): 11.0 / 12.4; 4, 2048, 4096,
// 1 (512): 12.3 / 13.5; 8, 1024, 4096, 1 (512): 11.3 / 16.8; 2, 4096, 2048,
// 2 (1024): 13.1 / 13.1; 4, 1024, 4096, 4 (1024): 13.8 / 12.4; 8, 2048,
// 4096, 1 (1024): 14.5 / 13.7; 4, 4096, 2048, 2 (2048): 17.5 / 13.2; 8,
// 1024, 2048, 4 (2048): 20.5 / 15.9; 8, 4096, 2048, 4 (8192): 56.3 / 13.4.
constexpr long long kClusterMaxWork = 512;

// (Not on a multi-process handle: a cluster's CTAs belong to one process.)
bool cluster_ok(const symm_handle *h, int N, int B) {
    return h->mp_rank < 0 && h->R <= kMaxClusterRanks && B <= kClusterMaxBatch && (N + kClusterRows - 1) / kClusterRows <= 65535;
}

int gemv_path(const symm_handle *h, int N, int B, int Kr) {
    if (h->opt_gemv_path != 0) return h->opt_gemv_path;
    if (Kr == 0) return kPathFfma;
    const size_t wbytes = (size_t)N * (size_t)Kr * 2 * (size_t)h->R;
    if (wbytes <= kSmallWBytes && B <= kSmallMaxBatch) {
        // The per-tile kernels do every product on the CUDA cores: the
        // cluster kernel where it can run, else the per-tile one (R > 8, a
        // multi-process handle), each under the same bound.  Per-tile kernel
        // / persistent kernel, per launch, L2 flushed, us (R, N, K, B; CTAs x
        // B): 16, 256, 4096, 1 (256): 12.9 / 16.9; 16, 1024, 8192, 1 (1024):
        // 22.7 / 18.4; 32, 512, 8192, 1 (1024): 24.4 / 19.0; 16, 2048, 4096,
        // 2 (4096): 32.5 / 18.8; 64, 1024, 8192, 1 (4096): 58.4 / 41.1.
        const bool clu = cluster_ok(h, N, B);
        const int rows = clu ? kClusterRows : ffma_rows_per_tile(B);
        const long long ctas = (long long)h->R * ((N + rows - 1) / rows);
        if (ctas * B > kClusterMaxWork) return kPathDyn;
        return clu ? kPathCluster : kPathFfma;
    }
    return kPathDyn;
}

int rows_per_tile_for_path(int path, int B) {
    if (B < 1 || B > SYMM_MAX_BATCH) return 0;
    switch (path) {
        case kPathFfma: return ffma_rows_per_tile(B);
        case kPathDyn: return kDynRows;
        case kPathCluster: return kClusterRows;
        default: return 0;
    }
}

int dyn_slabs(const symm_handle *h) { return h->opt_sk_slabs > 0 ? h->opt_sk_slabs : 2; }
int dyn_cps(const symm_handle *h) { return h->opt_sk_cps > 0 ? h->opt_sk_cps : 2; }

const void *tc_maps_for(symm_handle *h, const GemvArgs &a, int *err) {
    for (auto &e : h->map_cache)
        if (e.W == a.W && e.x == a.x && e.N == a.N && e.Kr == a.Kr && e.B == a.B) return e.maps;
    auto &e = h->map_cache[h->map_next];
    h->map_next = (h->map_next + 1) % 8;
    e.W = nullptr;
    *err = dyn_encode_maps(a, e.maps);
    if (*err != 0) return nullptr;
    e.W = a.W;
    e.x = a.x;
    e.N = a.N;
    e.Kr = a.Kr;
    e.B = a.B;
    return e.maps;
}

// The kernel and launch geometry gemv_all_reduce would use.
struct Plan {
    int path = 0, engine = 0, slabs = 0, cps = 0, rows = 0, tiles = 0, splits = 1, grid = 0, cluster = 0;
    DynGeom dyn = {0, 1, 0, 0, 0, 0};
};

// `cap`: scratch bytes per slot the partials may use (the whole region, or
// less when part of it is reserved for the bias + RMSNorm stage's z).
// `packed`: W is a packed weight, which only the persistent kernel reads
// (a call with K = 0 reads no W and keeps its path).
int make_plan(const symm_handle *h, int N, int Kr, int B, Plan *pl, size_t cap, bool packed = false) {
    if ((size_t)B * (size_t)N * 4 > cap)
        return fail(SYMM_ERANGE, "partials need %zu scratch bytes per slot, %zu available",
                    (size_t)B * (size_t)N * 4, cap);
    pl->path = gemv_path(h, N, B, Kr);
    if (packed && Kr > 0) {
        if (h->opt_gemv_path != 0 && h->opt_gemv_path != kPathDyn)
            return fail(SYMM_EINVAL, "a packed weight is read by the persistent kernel (path 4) only");
        pl->path = kPathDyn;
    }
    if (h->opt_unfused) {
        if (Kr == 0 || (h->opt_gemv_path != 0 && h->opt_gemv_path != kPathDyn))
            return fail(SYMM_EINVAL, "the unfused form runs on the persistent kernel (path 4, K > 0) only");
        pl->path = kPathDyn;
    }
    if (pl->path == kPathCluster && !cluster_ok(h, N, B))
        return fail(SYMM_EINVAL,
                    "the cluster kernel (path 5) needs R <= %d, B <= %d, at most 65535 row tiles and a "
                    "single-process handle", kMaxClusterRanks, kClusterMaxBatch);
    pl->rows = rows_per_tile_for_path(pl->path, B);
    if (pl->rows <= 0) return fail(SYMM_EINVAL, "no GEMV kernel for B=%d", B);
    pl->tiles = (N + pl->rows - 1) / pl->rows;
    if (pl->tiles > h->max_tiles)
        return fail(SYMM_ERANGE, "%d row tiles exceed the signal pad's %d", pl->tiles, h->max_tiles);
    pl->splits = 1;
    pl->grid = pl->tiles * (h->mp_rank >= 0 ? 1 : h->R);
    pl->cluster = pl->path == kPathCluster ? h->R : 0;
    if (pl->path == kPathDyn) {
        if (Kr == 0) return fail(SYMM_EINVAL, "the persistent kernel needs K > 0");
        pl->engine = 0;   // tcgen05 (the CUDA-core engine was retired)
        pl->slabs = dyn_slabs(h);
        pl->cps = dyn_cps(h);
        if (!dyn_config_supported(pl->slabs, pl->cps))
            return fail(SYMM_EINVAL, "no pipeline for %d slabs at %d CTAs per SM", pl->slabs, pl->cps);
        // (tile, rank) pairs this launch computes: every rank's, or on a
        // multi-process handle the own rank's only.
        const long long pairs = (long long)pl->tiles * (h->mp_rank >= 0 ? 1 : h->R);
        const long long KB = (Kr + dyn_block_k(pl->slabs) - 1) / dyn_block_k(pl->slabs);
        if (pairs > (1LL << 26)) return fail(SYMM_ERANGE, "too many row tiles");
        long long G = h->opt_sk_grid > 0 ? h->opt_sk_grid : (long long)num_sms(h->device) * pl->cps;
        // K splits: the requested count (option), else none; limited by the K
        // blocks, the scratch region (one partial per split) and the pad.
        // Automatic: split only when the (tile, rank) pairs fill at most a
        // quarter of the grid, and then to about half of it -- splits cost a
        // partial and a reduction input each, and measured slower whenever
        // the pairs alone already kept most SMs streaming.
        long long S = h->opt_dyn_splits > 0
                          ? h->opt_dyn_splits
                          : (4 * pairs > G ? 1 : std::min<long long>(8, (G + 2 * pairs - 1) / (2 * pairs)));
        // Cluster epilogue: one unit per CTA, the R * S units of a tile one
        // cluster (at most 8 CTAs), partials summed through distributed shared
        // memory; beyond one wave the hardware starts each cluster as slots
        // free up.  Automatic (no K splits) when the units fit the grid in one
        // wave (nothing would be drawn anyway, and the end of such a launch is
        // the global-memory protocol's round trips), or when they are long
        // enough that a CTA's start-up is small against its stream: measured
        // on 268-537 MB layers, chained calls with units of 64-128 KB ran 3-18 %
        // slower than drawn ones, 256-512 KB units about even, 0.9-2 MB units
        // 1-6 % faster.  Forced on, it takes the requested K splits (none by
        // default).
        // (cl_ok: the cluster epilogue could run this shape; the unfused form
        // takes the splits it would have, without the clusters, so that its
        // partials are summed in the fused call's order)
        const bool cl_ok = dyn_cluster_supported(pl->slabs, pl->cps) && h->mp_rank < 0;
        const bool cl_base = cl_ok && !h->opt_unfused;
        bool cl = false;
        if (h->opt_dyn_cluster == 1) {
            cl = true;
            if (h->opt_dyn_splits <= 0) S = 1;
        } else if (h->opt_dyn_cluster < 0) {
            if (cl_ok && 2 * h->R <= kMaxClusterRanks && h->opt_dyn_splits <= 0 && 2 * pairs <= G) {
                // Units that fill at most half of the CTA slots leave SMs
                // idle: split K inside the clusters (R x S CTAs each, at most
                // 8) as far as the launch stays one wave.  Measured (chained
                // us per call, two runs each), against the plan without it
                // (clusters of R, or drawn K-split units for the smallest):
                // R = 2, N = 8192, K/R = 14336: 2 splits, 72.5 -> 66.5-66.9;
                // R = 4, N = 4096, K/R = 2048, B = 8: 14.6 -> 13.2-13.4;
                // R = 3, N = 4096, K/R = 4096: 22.0 -> 17.6; R = 2, N = 4096,
                // K/R = 4096, B = 4: 16.7 -> 13.1; R = 4, N = 2048, K/R = 4096:
                // 20.6-21.0 -> 14.2-14.4; R = 2, N = 2048, K/R = 8192: 19.0-19.7
                // -> 14.3-14.4; one rank (the K splits are then the cluster),
                // N = 8192, K = 28672: 73.9-75.4 -> 65.8 (4 splits); N = 4096,
                // K = 16384, B = 4: 29.6-30.0 -> 23.9.  3 splits on the first
                // (two uneven waves) lost; at R = 8 no split fits a cluster, and
                // clusters of 8 without splits measured 2 % behind drawn K-split
                // units there.
                cl = cl_base;
                S = 1;
                while (h->R * (S + 1) <= kMaxClusterRanks && pairs * (S + 1) <= G) ++S;
            } else {
                cl = cl_base && h->R >= 2 && S == 1 && (pairs <= G || Kr >= kClusterEpilogueMinKr);
            }
        }
        S = std::min<long long>(S, KB);
        while (S > 1 && ((size_t)S * B * N * 4 > cap || (long long)pl->tiles * S > h->max_tiles)) --S;
        const long long KBs = (KB + S - 1) / S;
        S = (KB + KBs - 1) / KBs;   // no empty split
        if (cl && h->opt_dyn_cluster < 0 && h->R * S < 2) cl = false;   // automatic: a cluster of one CTA gains nothing
        if (cl) {
            const long long C = (long long)h->R * S;
            const bool fits = cl_base && C <= kMaxClusterRanks && dyn_cluster_fits(pl->slabs, (int)C);
            if (!fits && h->opt_dyn_cluster == 1)
                return fail(SYMM_EINVAL,
                            "the cluster epilogue needs 2 CTAs per SM (1-3 slabs), R x splits "
                            "<= %d, the fused form, a single-process handle and a device that can hold a cluster "
                            "of that many such CTAs", kMaxClusterRanks);
            cl = fits;
        }
        const long long units = pairs * S;
        G = cl ? units : std::max<long long>(1, std::min<long long>(G, units));
        pl->dyn.cluster = cl ? (int)(h->R * S) : 0;
        pl->cluster = pl->dyn.cluster;
        pl->dyn.units = (int)units;
        pl->dyn.splits = (int)S;
        pl->dyn.KB = (int)KB;
        pl->dyn.KBs = (int)KBs;
        pl->dyn.G = (int)G;
        pl->splits = (int)S;
        pl->grid = (int)G;
    }
    return SYMM_OK;
}

}  // namespace

namespace symm {
// Lets other translation units of the library report through symm_last_error.
int report_error(int code, const char *msg) { return fail(code, "%s", msg); }
}  // namespace symm

namespace {

// CUDA VMM through the runtime's driver entry points (the library links the
// runtime only).
struct Vmm {
    CUresult (*granularity)(size_t *, const CUmemAllocationProp *, CUmemAllocationGranularity_flags) = nullptr;
    CUresult (*reserve)(CUdeviceptr *, size_t, size_t, CUdeviceptr, unsigned long long) = nullptr;
    CUresult (*addr_free)(CUdeviceptr, size_t) = nullptr;
    CUresult (*create)(CUmemGenericAllocationHandle *, size_t, const CUmemAllocationProp *,
                       unsigned long long) = nullptr;
    CUresult (*release)(CUmemGenericAllocationHandle) = nullptr;
    CUresult (*map)(CUdeviceptr, size_t, size_t, CUmemGenericAllocationHandle, unsigned long long) = nullptr;
    CUresult (*unmap)(CUdeviceptr, size_t) = nullptr;
    CUresult (*set_access)(CUdeviceptr, size_t, const CUmemAccessDesc *, size_t) = nullptr;
    CUresult (*export_handle)(void *, CUmemGenericAllocationHandle, CUmemAllocationHandleType,
                              unsigned long long) = nullptr;
    CUresult (*import_handle)(CUmemGenericAllocationHandle *, void *, CUmemAllocationHandleType) = nullptr;
    bool ok = false;
};

template <class F>
bool entry(const char *name, F *fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
        return false;
    *fn = reinterpret_cast<F>(p);
    return true;
}

const Vmm &vmm() {
    static const Vmm v = []() {
        Vmm t;
        t.ok = entry("cuMemGetAllocationGranularity", &t.granularity) && entry("cuMemAddressReserve", &t.reserve) &&
               entry("cuMemAddressFree", &t.addr_free) && entry("cuMemCreate", &t.create) &&
               entry("cuMemRelease", &t.release) && entry("cuMemMap", &t.map) && entry("cuMemUnmap", &t.unmap) &&
               entry("cuMemSetAccess", &t.set_access) &&
               entry("cuMemExportToShareableHandle", &t.export_handle) &&
               entry("cuMemImportFromShareableHandle", &t.import_handle);
        return t;
    }();
    return v;
}

int cu_fail(CUresult r, const char *what) { return fail(SYMM_ECUDA, "%s failed (CUresult %d)", what, (int)r); }

CUmemAllocationProp slot_prop(int device) {
    CUmemAllocationProp prop = {};
    prop.type = CU_MEM_ALLOCATION_TYPE_PINNED;
    prop.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    prop.location.id = device;
    prop.requestedHandleTypes = CU_MEM_HANDLE_TYPE_POSIX_FILE_DESCRIPTOR;
    return prop;
}

// Maps allocation `mem` as slot r of h's reserved range, read-write for the
// handle's device.
int map_slot(symm_handle *h, int r, CUmemGenericAllocationHandle mem) {
    const Vmm &v = vmm();
    const CUdeviceptr at = (CUdeviceptr)(h->va + (unsigned long long)r * h->stride);
    CUresult c = v.map(at, h->stride, 0, mem, 0);
    if (c != CUDA_SUCCESS) return cu_fail(c, "cuMemMap");
    CUmemAccessDesc acc = {};
    acc.location.type = CU_MEM_LOCATION_TYPE_DEVICE;
    acc.location.id = h->device;
    acc.flags = CU_MEM_ACCESS_FLAGS_PROT_READWRITE;
    c = v.set_access(at, h->stride, &acc, 1);
    if (c != CUDA_SUCCESS) {
        v.unmap(at, h->stride);
        return cu_fail(c, "cuMemSetAccess");
    }
    h->mem[r] = (unsigned long long)mem;
    return SYMM_OK;
}

// Unmaps and releases every slot of a multi-process handle, frees its range.
void mp_release(symm_handle *h) {
    const Vmm &v = vmm();
    for (int r = 0; r < h->R; ++r) {
        if (!h->mem[r]) continue;
        v.unmap((CUdeviceptr)(h->va + (unsigned long long)r * h->stride), h->stride);
        v.release((CUmemGenericAllocationHandle)h->mem[r]);
        h->mem[r] = 0;
    }
    if (h->va) v.addr_free((CUdeviceptr)h->va, h->total);
    h->va = 0;
}

// What the fused call does after the tile sums (GemvArgs::out_mode) and the
// extra arguments of each form.
struct Epilogue {
    int mode = kOutAllReduce;
    const void *bias = nullptr;    // kOutBiasZ
    const void *gamma = nullptr;   // kOutBiasZ
    float eps = 0.f;               // kOutBiasZ
};

// The three public forms of the fused row-parallel layer share everything up
// to the tile reducer's store: all-reduce (y [B][N] in every slot),
// reduce-scatter along the batch rows (y [B/R][N] per slot), and all-reduce +
// bias + RMSNorm (fp32 z stage, then the cluster normalisation kernel).
int gemv_common(symm_handle *h, const void *W_r, const void *x_r, void *y, int R, int N, int K, int B,
                symm_stream_t stream, const Epilogue &ep) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (R != h->R) return fail(SYMM_EINVAL, "R=%d but the handle has %d ranks", R, h->R);
    if (N < 0 || K < 0) return fail(SYMM_EINVAL, "N=%d K=%d must be >= 0", N, K);
    if (B < 0 || B > SYMM_MAX_BATCH) return fail(SYMM_EINVAL, "B=%d outside 0..%d", B, SYMM_MAX_BATCH);
    if (K % R) return fail(SYMM_EINVAL, "K=%d is not a multiple of R=%d", K, R);
    const int Kr = K / R;
    if (Kr % 8) return fail(SYMM_EINVAL, "K/R=%d is not a multiple of 8", Kr);
    if (ep.mode == kOutReduceScatter && B % R)
        return fail(SYMM_EINVAL, "reduce-scatter along the batch rows needs B=%d to be a multiple of R=%d", B, R);
    if (ep.mode == kOutBiasZ) {
        if (N % 8) return fail(SYMM_EINVAL, "bias + RMSNorm needs N=%d to be a multiple of 8", N);
        if (N > rmsnorm_max_h()) return fail(SYMM_EINVAL, "bias + RMSNorm supports N <= %d", rmsnorm_max_h());
        if (!(ep.eps >= 0.f) || ep.eps > 3.0e38f) return fail(SYMM_EINVAL, "eps must be finite and >= 0");
    }
    const symm_handle::PackedW *pw = find_packed(h, W_r);
    if (pw && (pw->N != N || pw->Kr != Kr))
        return fail(SYMM_EINVAL, "W_r is a packed weight of N=%d K/R=%d, called with N=%d K/R=%d", pw->N, pw->Kr, N,
                    Kr);
    if (N == 0 || B == 0) return SYMM_OK;
    const size_t wbytes = pw ? pw->bytes : (size_t)N * (size_t)Kr * 2;
    const size_t xbytes = (size_t)B * (size_t)Kr * 2;
    const size_t ybytes = (size_t)(ep.mode == kOutReduceScatter ? B / R : B) * (size_t)N * 2;
    const size_t vbytes = (size_t)N * 2;
    if (!in_user_region(h, W_r, wbytes))
        return fail(SYMM_EINVAL, "W_r (N x K/R bf16, or its packed layout) is not inside slot 0's user region");
    if (!in_user_region(h, x_r, xbytes)) return fail(SYMM_EINVAL, "x_r (B x K/R bf16) is not inside slot 0's user region");
    if (!in_user_region(h, y, ybytes)) return fail(SYMM_EINVAL, "y is not inside slot 0's user region");
    if (!aligned16(W_r) || !aligned16(x_r) || !aligned16(y)) return fail(SYMM_EINVAL, "W_r, x_r and y must be 16-byte aligned");
    if (overlaps(y, ybytes, W_r, wbytes) || overlaps(y, ybytes, x_r, xbytes))
        return fail(SYMM_EINVAL, "y overlaps W_r or x_r");
    for (const void *v : {ep.bias, ep.gamma}) {
        if (!v) continue;
        if (!in_user_region(h, v, vbytes) || !aligned16(v))
            return fail(SYMM_EINVAL, "bias / gamma (N bf16) must be 16-byte aligned inside slot 0's user region");
        if (overlaps(v, vbytes, y, ybytes)) return fail(SYMM_EINVAL, "bias / gamma overlaps y");
    }
    // The bias + RMSNorm form keeps z (fp32 [B][N]) at the top of slot 0's
    // scratch region; the partials get the rest.
    size_t cap = h->scratch_bytes;
    size_t z_off = 0;
    if (ep.mode == kOutBiasZ) {
        const size_t zbytes = (size_t)B * N * 4;
        if (zbytes > h->scratch_bytes) return fail(SYMM_ERANGE, "z needs %zu scratch bytes", zbytes);
        z_off = (h->scratch_bytes - zbytes) / 256 * 256;
        cap = z_off;
    }
    if (h->opt_unfused && ep.mode != kOutAllReduce)
        return fail(SYMM_EINVAL, "the unfused form (SYMM_OPT_UNFUSED) is a form of gemv_all_reduce only");
    if (h->mp_rank >= 0 && (h->opt_unfused || ep.mode == kOutBiasZ))
        return fail(SYMM_EINVAL, "a multi-process handle runs the all-reduce and reduce-scatter forms, fused");
    // (the plan asks the handle's device whether a cluster launch fits)
    int rc = check_device(h);
    if (rc != SYMM_OK) return rc;
    Plan pl;
    rc = make_plan(h, N, Kr, B, &pl, cap, pw != nullptr);
    if (rc != SYMM_OK) return rc;
    const int path = pl.path, rows = pl.rows, tiles = pl.tiles, splits = pl.splits,
              slabs = pl.slabs, cps = pl.cps;
    const DynGeom dyn = pl.dyn;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // The launch epoch, the tickets and the work counter live in the signal
    // pad and are advanced by the kernels themselves (every counter is back
    // at zero when a launch ends), so nothing here depends on earlier calls:
    // a captured call replays correctly and the geometry may change freely.
    GemvArgs a;
    a.W = static_cast<const uint8_t *>(W_r);
    a.x = static_cast<const uint8_t *>(x_r);
    a.y = static_cast<uint8_t *>(y);
    // Multi-process handle: this process launches its own rank's units only;
    // its launch epoch, work counters, unit count and status words are in
    // its own slot's pad, while the tile counters (rank 0's pad) and the
    // flags (each rank's pad) are shared by every rank's launch.
    const int own = h->mp_rank >= 0 ? h->mp_rank : 0;
    a.scratch = h->base + h->scratch_off;
    a.flags = pad_word(h, 0, h->flags_off);
    a.counters = pad_word(h, 0, h->counters_off);
    a.status = pad_word(h, own, 0);
    a.stride = (long long)h->stride;
    a.R = h->R;
    a.N = N;
    a.Kr = Kr;
    a.B = B;
    a.rows_per_tile = rows;
    a.num_tiles = tiles;
    a.epoch_word = pad_word(h, own, kPadEpochOffset);
    a.tiles_done = h->mp_rank >= 0 ? nullptr : pad_word(h, 0, kPadTilesDoneOffset);
    a.units_done = h->mp_rank >= 0 ? pad_word(h, own, kPadTilesDoneOffset) : nullptr;
    a.my_rank = h->mp_rank;
    a.work = pad_word(h, own, kPadWorkOffset);
    a.reverse_order = h->opt_tile_order;
    a.splits = splits;
    a.partial_stride = (long long)B * N * 4;
    a.kc_cap = 0;
    a.out_mode = ep.mode;
    a.chained = h->opt_chain;   // path 1 (path 4 decides below)
    a.rs_rows = ep.mode == kOutReduceScatter ? B / R : B;
    a.z = ep.mode == kOutBiasZ ? reinterpret_cast<float *>(h->base + h->scratch_off + z_off) : nullptr;
    a.bias = ep.mode == kOutBiasZ ? static_cast<const uint8_t *>(ep.bias) : nullptr;
    a.w_packed = pw != nullptr && path == kPathDyn;
    // Early W loads (before the wait for the previous kernel) only for a
    // packed weight: it is written by symm_pack_w alone, and a call whose
    // packed weight the handle's last kernel wrote is not chained (below).
    a.w_early = a.w_packed;
    if (h->opt_unfused) a.out_mode = kOutPartials;
    a.tl = h->tl;
    a.tl_ctas = h->tl_ctas;
    cudaError_t e = cudaSuccess;
    switch (path) {
        case kPathFfma:
            a.kc_cap = ffma_kc_cap(B, Kr);
            e = launch_gemv_ffma(a, s);
            break;
        case kPathCluster:
            e = launch_gemv_cluster(a, s);
            break;
        case kPathDyn: {
            int err = 0;
            const void *maps = tc_maps_for(h, a, &err);
            if (!maps) return fail(SYMM_ECUDA, "cuTensorMapEncodeTiled failed (%d)", err);
            const bool chained = h->opt_chain != 0 && !overlaps(W_r, wbytes, h->last_write, h->last_write_bytes);
            e = launch_gemv_dyn(a, dyn, maps, slabs, cps, chained, s);
            break;
        }
        default:
            return fail(SYMM_EINVAL, "no GEMV kernel for B=%d", B);
    }
    if (e != cudaSuccess) return cuda_fail(e, "gemv_all_reduce launch");
    note_write(h, y, ybytes);   // by the GEMV, or by the norm stage launched next
    if (h->opt_unfused) {
        // The unfused form's all-reduce of the partials, a programmatic
        // dependent of the GEMV (it waits for the GEMV before reading).
        PartialsArArgs pa;
        pa.scratch = a.scratch;
        pa.y = a.y;
        pa.stride = a.stride;
        pa.partial_stride = a.partial_stride;
        pa.R = h->R;
        pa.splits = splits;
        pa.B = B;
        pa.N = N;
        pa.vec = ((size_t)B * (size_t)N) % 4 == 0;
        pa.chained = 1;
        e = launch_partials_ar(pa, s);
        if (e != cudaSuccess) return cuda_fail(e, "unfused all-reduce launch");
        return SYMM_OK;
    }
    if (ep.mode == kOutBiasZ) {
        RmsNormArgs n = {};
        n.z = a.z;
        n.gamma = static_cast<const uint8_t *>(ep.gamma);
        n.out = a.y;
        n.stride = a.stride;
        n.R = h->R;
        n.rows = B;
        n.H = N;
        n.eps = ep.eps;
        n.wait_prior = h->opt_norm_pdl;
        e = launch_rmsnorm_rows(n, s);
        if (e != cudaSuccess) return cuda_fail(e, "RMSNorm stage launch");
    }
    return SYMM_OK;
}


}  // namespace

extern "C" {

const char *symm_last_error(void) { return g_err; }

int symm_layout(int R, size_t slot_bytes, size_t scratch_bytes, size_t signal_pad_bytes,
                size_t *stride_out, size_t *total_bytes_out) {
    if (R < 1 || R > SYMM_MAX_RANKS) return fail(SYMM_EINVAL, "R=%d outside 1..%d", R, SYMM_MAX_RANKS);
    if (slot_bytes == 0) return fail(SYMM_EINVAL, "slot_bytes must be > 0");
    if (signal_pad_bytes < 4096) return fail(SYMM_EINVAL, "signal_pad_bytes must be >= 4096");
    symm_handle h;
    h.R = R;
    h.slot_bytes = slot_bytes;
    h.scratch_bytes = scratch_bytes;
    h.pad_bytes = signal_pad_bytes;
    if (!compute_layout(h)) return fail(SYMM_EINVAL, "sizes overflow");
    if (stride_out) *stride_out = h.stride;
    if (total_bytes_out) *total_bytes_out = h.total;
    g_err[0] = 0;
    return SYMM_OK;
}

int symm_alloc(int R, size_t slot_bytes, size_t scratch_bytes, size_t signal_pad_bytes,
               void *backing, size_t backing_bytes, symm_handle_t **out) {
    if (!out) return fail(SYMM_EINVAL, "out is NULL");
    *out = nullptr;
    int rc = symm_layout(R, slot_bytes, scratch_bytes, signal_pad_bytes, nullptr, nullptr);
    if (rc != SYMM_OK) return rc;
    symm_handle *h = new (std::nothrow) symm_handle;
    if (!h) return fail(SYMM_ENOMEM, "host allocation of the handle failed");
    h->R = R;
    h->slot_bytes = slot_bytes;
    h->scratch_bytes = scratch_bytes;
    h->pad_bytes = signal_pad_bytes;
    compute_layout(*h);
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e, "cudaGetDevice");
    }
    if (backing) {
        if ((reinterpret_cast<uintptr_t>(backing) % kAlign) != 0) {
            delete h;
            return fail(SYMM_EINVAL, "backing pointer is not %zu-byte aligned", kAlign);
        }
        if (backing_bytes < h->total) {
            delete h;
            return fail(SYMM_ENOMEM, "backing holds %zu bytes, layout needs %zu", backing_bytes, h->total);
        }
        h->base = static_cast<uint8_t *>(backing);
        h->owned = false;
    } else {
        e = cudaMalloc(reinterpret_cast<void **>(&h->base), h->total);
        if (e != cudaSuccess) {
            delete h;
            cudaGetLastError();
            return fail(SYMM_ENOMEM, "cudaMalloc(%zu) failed: %s", h->total, cudaGetErrorString(e));
        }
        h->owned = true;
    }
    for (int r = 0; r < R && e == cudaSuccess; ++r) {
        uint8_t *s = slot(h, r);
        e = cudaMemset(s + h->guard0, kGuardByte, kGuard);
        if (e == cudaSuccess) e = cudaMemset(s + h->scratch_off, 0, h->guard1 - h->scratch_off);
        if (e == cudaSuccess) e = cudaMemset(s + h->guard1, kGuardByte, kGuard);
        if (e == cudaSuccess) e = cudaMemset(s + h->pad_off, 0, h->guard2 - h->pad_off);
        if (e == cudaSuccess) e = cudaMemset(s + h->guard2, kGuardByte, kGuard);
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        if (h->owned) cudaFree(h->base);
        delete h;
        return cuda_fail(e, "initialising slots");
    }
    *out = h;
    g_err[0] = 0;
    return SYMM_OK;
}

int symm_mp_alloc(int R, int rank, size_t slot_bytes, size_t scratch_bytes, size_t signal_pad_bytes,
                  symm_handle_t **out, int *fd_out) {
    if (!out || !fd_out) return fail(SYMM_EINVAL, "out or fd_out is NULL");
    *out = nullptr;
    *fd_out = -1;
    int rc = symm_layout(R, slot_bytes, scratch_bytes, signal_pad_bytes, nullptr, nullptr);
    if (rc != SYMM_OK) return rc;
    if (rank < 0 || rank >= R) return fail(SYMM_EINVAL, "rank=%d outside 0..%d", rank, R - 1);
    const Vmm &v = vmm();
    if (!v.ok) return fail(SYMM_ECUDA, "the CUDA virtual memory entry points are not available");
    symm_handle *h = new (std::nothrow) symm_handle;
    if (!h) return fail(SYMM_ENOMEM, "host allocation of the handle failed");
    h->R = R;
    h->slot_bytes = slot_bytes;
    h->scratch_bytes = scratch_bytes;
    h->pad_bytes = signal_pad_bytes;
    compute_layout(*h);
    h->mp_rank = rank;
    h->owned = true;
    cudaError_t e = cudaGetDevice(&h->device);
    if (e != cudaSuccess) {
        delete h;
        return cuda_fail(e, "cudaGetDevice");
    }
    const CUmemAllocationProp prop = slot_prop(h->device);
    size_t gran = 0;
    CUresult c = v.granularity(&gran, &prop, CU_MEM_ALLOC_GRANULARITY_MINIMUM);
    if (c != CUDA_SUCCESS || gran == 0) {
        delete h;
        return cu_fail(c, "cuMemGetAllocationGranularity");
    }
    // Every rank's slot is one allocation of `stride` bytes.
    h->stride = round_up(h->stride, gran);
    h->total = h->stride * (size_t)R;
    CUdeviceptr va = 0;
    c = v.reserve(&va, h->total, gran, 0, 0);
    if (c != CUDA_SUCCESS) {
        delete h;
        return cu_fail(c, "cuMemAddressReserve");
    }
    h->va = (unsigned long long)va;
    h->base = reinterpret_cast<uint8_t *>(va);
    CUmemGenericAllocationHandle mem = 0;
    c = v.create(&mem, h->stride, &prop, 0);
    if (c != CUDA_SUCCESS) {
        const size_t bytes = h->stride;
        mp_release(h);
        delete h;
        return c == CUDA_ERROR_OUT_OF_MEMORY ? fail(SYMM_ENOMEM, "cuMemCreate(%zu) failed", bytes)
                                             : cu_fail(c, "cuMemCreate");
    }
    rc = map_slot(h, rank, mem);
    if (rc != SYMM_OK) {
        v.release(mem);
        mp_release(h);
        delete h;
        return rc;
    }
    int fd = -1;
    c = v.export_handle(&fd, mem, CU_MEM_HANDLE_TYPE_POSIX_FILE_DESCRIPTOR, 0);
    if (c != CUDA_SUCCESS) {
        mp_release(h);
        delete h;
        return cu_fail(c, "cuMemExportToShareableHandle");
    }
    // The own slot as symm_alloc leaves every slot: guard bands, zero scratch
    // and pad.
    uint8_t *sl = slot(h, rank);
    e = cudaMemset(sl + h->guard0, kGuardByte, kGuard);
    if (e == cudaSuccess) e = cudaMemset(sl + h->scratch_off, 0, h->guard1 - h->scratch_off);
    if (e == cudaSuccess) e = cudaMemset(sl + h->guard1, kGuardByte, kGuard);
    if (e == cudaSuccess) e = cudaMemset(sl + h->pad_off, 0, h->guard2 - h->pad_off);
    if (e == cudaSuccess) e = cudaMemset(sl + h->guard2, kGuardByte, kGuard);
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        close(fd);   // never handed out
        mp_release(h);
        delete h;
        return cuda_fail(e, "initialising the slot");
    }
    *fd_out = fd;
    *out = h;
    g_err[0] = 0;
    return SYMM_OK;
}

int symm_mp_import(symm_handle_t *h, int peer, int fd) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (h->mp_rank < 0) return fail(SYMM_EINVAL, "not a multi-process handle (symm_mp_alloc)");
    if (peer < 0 || peer >= h->R || peer == h->mp_rank)
        return fail(SYMM_EINVAL, "peer=%d must be another rank in 0..%d", peer, h->R - 1);
    if (h->mem[peer]) return fail(SYMM_EINVAL, "rank %d's slot is already mapped", peer);
    if (fd < 0) return fail(SYMM_EINVAL, "fd=%d is not a descriptor", fd);
    int rc = check_current_device(h);
    if (rc != SYMM_OK) return rc;
    const Vmm &v = vmm();
    CUmemGenericAllocationHandle mem = 0;
    CUresult c = v.import_handle(&mem, reinterpret_cast<void *>((uintptr_t)fd), CU_MEM_HANDLE_TYPE_POSIX_FILE_DESCRIPTOR);
    if (c != CUDA_SUCCESS) return cu_fail(c, "cuMemImportFromShareableHandle");
    rc = map_slot(h, peer, mem);
    if (rc != SYMM_OK) {
        v.release(mem);
        return rc;
    }
    g_err[0] = 0;
    return SYMM_OK;
}

int symm_rendezvous(symm_handle_t *h, void **slot_ptrs, void **signal_pad_ptrs, size_t *stride_out) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (h->mp_rank >= 0)
        for (int r = 0; r < h->R; ++r)
            if (!h->mem[r]) return fail(SYMM_EINVAL, "rank %d's slot is not mapped yet (symm_mp_import)", r);
    for (int r = 0; r < h->R; ++r) {
        if (slot_ptrs) slot_ptrs[r] = slot(h, r);
        if (signal_pad_ptrs) signal_pad_ptrs[r] = slot(h, r) + h->pad_off;
    }
    if (stride_out) *stride_out = h->stride;
    return SYMM_OK;
}

int symm_info(symm_handle_t *h, symm_info_t *info) {
    if (!h || !info) return fail(SYMM_EINVAL, "NULL argument");
    info->R = h->R;
    info->device = h->device;
    info->stride = h->stride;
    info->slot_bytes = h->slot_bytes;
    info->scratch_bytes = h->scratch_bytes;
    info->signal_pad_bytes = h->pad_bytes;
    info->max_tiles = h->max_tiles;
    return SYMM_OK;
}

int symm_set_option(symm_handle_t *h, int option, int value) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    switch (option) {
        case SYMM_OPT_GEMV_PATH:
            if (value == 2 || value == 3)
                return fail(SYMM_EINVAL, "GEMV path %d was retired (0 auto, 1 CUDA-core, 4 persistent, 5 cluster)",
                            value);
            if (value < 0 || value > 5)
                return fail(SYMM_EINVAL, "GEMV path %d unknown (0 auto, 1 CUDA-core, 4 persistent, 5 cluster)", value);
            h->opt_gemv_path = value;
            return SYMM_OK;
        case SYMM_OPT_TILE_ORDER:
            if (value < 0 || value > 1) return fail(SYMM_EINVAL, "tile order %d unknown", value);
            h->opt_tile_order = value;
            return SYMM_OK;
        case SYMM_OPT_SK_SLABS:
            if (value < 0 || value > 4)
                return fail(SYMM_EINVAL, "persistent-kernel slabs %d not in {0 auto, 1, 2, 3, 4}", value);
            h->opt_sk_slabs = value;
            return SYMM_OK;
        case SYMM_OPT_SK_ENGINE:
            if (value == 1)
                return fail(SYMM_EINVAL, "the persistent kernel's CUDA-core engine (1) was retired; -1 auto or 0 tcgen05");
            if (value < -1 || value > 0) return fail(SYMM_EINVAL, "persistent-kernel engine %d not in {-1 auto, 0}", value);
            return SYMM_OK;   // tcgen05, the only engine
        case SYMM_OPT_SK_GRID:
            if (value < 0) return fail(SYMM_EINVAL, "persistent grid %d: 0 auto or a CTA count > 0", value);
            h->opt_sk_grid = value;
            return SYMM_OK;
        case SYMM_OPT_DYN_SPLITS:
            if (value < 0 || value > 16) return fail(SYMM_EINVAL, "persistent-kernel splits %d not in 0..16", value);
            h->opt_dyn_splits = value;
            return SYMM_OK;
        case SYMM_OPT_AR_CTAS_PER_SM:
            if (value < 0 || value > 64) return fail(SYMM_EINVAL, "all-reduce CTAs per SM %d not in 0..64", value);
            h->opt_ar_cps = value;
            return SYMM_OK;
        case SYMM_OPT_COPY_ENGINE:
            if (value < 0 || value > 1) return fail(SYMM_EINVAL, "copy engine %d not in {0, 1}", value);
            h->opt_copy_engine = value;
            return SYMM_OK;
        case SYMM_OPT_AR_KERNEL:
            if (value < 0 || value > 2) return fail(SYMM_EINVAL, "all-reduce kernel %d not in {0 auto, 1, 2}", value);
            h->opt_ar_kernel = value;
            return SYMM_OK;
        case SYMM_OPT_CHAIN:
            if (value < 0 || value > 1) return fail(SYMM_EINVAL, "chain %d not in {0, 1}", value);
            h->opt_chain = value;
            return SYMM_OK;
        case SYMM_OPT_NORM_PDL:
            if (value < 0 || value > 1) return fail(SYMM_EINVAL, "RMSNorm-stage PDL %d not in {0, 1}", value);
            h->opt_norm_pdl = value;
            return SYMM_OK;
        case SYMM_OPT_UNFUSED:
            if (value < 0 || value > 1) return fail(SYMM_EINVAL, "unfused %d not in {0, 1}", value);
            h->opt_unfused = value;
            return SYMM_OK;
        case SYMM_OPT_SK_CTAS_PER_SM:
            if (value < 0 || value > 3) return fail(SYMM_EINVAL, "persistent-kernel CTAs per SM %d not in 0..3", value);
            h->opt_sk_cps = value;
            return SYMM_OK;
        case SYMM_OPT_DYN_CLUSTER:
            if (value < -1 || value > 1) return fail(SYMM_EINVAL, "cluster epilogue %d not in {-1 auto, 0, 1}", value);
            h->opt_dyn_cluster = value;
            return SYMM_OK;
        default:
            return fail(SYMM_EINVAL, "unknown option %d", option);
    }
}

int symm_gemv_plan(symm_handle_t *h, int N, int K, int B, symm_gemv_plan_t *out) {
    if (!h || !out) return fail(SYMM_EINVAL, "NULL argument");
    if (N < 1 || K < 0 || B < 1 || B > SYMM_MAX_BATCH || K % h->R || (K / h->R) % 8)
        return fail(SYMM_EINVAL, "no plan for N=%d K=%d B=%d on %d ranks", N, K, B, h->R);
    int rc = check_current_device(h);   // the plan depends on the device's occupancy
    if (rc != SYMM_OK) return rc;
    Plan pl;
    rc = make_plan(h, N, K / h->R, B, &pl, h->scratch_bytes);
    if (rc != SYMM_OK) return rc;
    out->path = pl.path;
    out->engine = pl.engine;
    out->slabs = pl.slabs;
    out->rows_per_tile = pl.rows;
    out->tiles = pl.tiles;
    out->splits = pl.splits;
    out->grid = pl.grid;
    out->parts_max = 1;
    out->kblocks = pl.dyn.KB;
    out->ctas_per_sm = pl.cps;
    out->cluster = pl.cluster;
    return SYMM_OK;
}

int one_shot_all_reduce(symm_handle_t *h, const void *in, void *out, int R, size_t n, symm_stream_t stream) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (R != h->R) return fail(SYMM_EINVAL, "R=%d but the handle has %d ranks", R, h->R);
    if (n == 0) return SYMM_OK;
    if (n > SIZE_MAX / 2) return fail(SYMM_EINVAL, "n too large");
    const size_t bytes = n * 2;
    if (!in_user_region(h, in, bytes)) return fail(SYMM_EINVAL, "in + n elements is not inside slot 0's user region");
    if (!in_user_region(h, out, bytes)) return fail(SYMM_EINVAL, "out + n elements is not inside slot 0's user region");
    if (!aligned16(in) || !aligned16(out)) return fail(SYMM_EINVAL, "in/out must be 16-byte aligned");
    if (in != out && overlaps(in, bytes, out, bytes)) return fail(SYMM_EINVAL, "in and out partially overlap");
    int rc = check_device(h);
    if (rc != SYMM_OK) return rc;
    AllReduceArgs a;
    a.in = static_cast<const uint8_t *>(in);
    a.out = static_cast<uint8_t *>(out);
    a.stride = (long long)h->stride;
    a.R = h->R;
    a.n = n;
    a.ctas_per_sm = h->opt_ar_cps;
    // A multi-process handle: the real one-shot -- this process reads every
    // rank's input and writes its own rank's output (the per-thread kernel).
    a.kernel = h->mp_rank >= 0 ? kArKernelPerThread : h->opt_ar_kernel;
    a.chained = h->opt_chain;
    a.my_rank = h->mp_rank;
    cudaError_t e = launch_one_shot_all_reduce(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "one_shot_all_reduce launch");
    note_write(h, out, bytes);
    return SYMM_OK;
}

int gemv_all_reduce(symm_handle_t *h, const void *W_r, const void *x_r, void *y, int R, int N, int K, int B,
                    symm_stream_t stream) {
    return gemv_common(h, W_r, x_r, y, R, N, K, B, stream, Epilogue());
}

int symm_packed_w_bytes(int R, int N, int K, size_t *bytes_out) {
    if (!bytes_out) return fail(SYMM_EINVAL, "bytes_out is NULL");
    if (R < 1 || R > SYMM_MAX_RANKS) return fail(SYMM_EINVAL, "R=%d outside 1..%d", R, SYMM_MAX_RANKS);
    if (N < 0 || K < 0) return fail(SYMM_EINVAL, "N=%d K=%d must be >= 0", N, K);
    if (K % R) return fail(SYMM_EINVAL, "K=%d is not a multiple of R=%d", K, R);
    if ((K / R) % 8) return fail(SYMM_EINVAL, "K/R=%d is not a multiple of 8", K / R);
    *bytes_out = packed_w_blocks(N, K / R) * kPackBlockBytes;
    return SYMM_OK;
}

int symm_pack_w(symm_handle_t *h, const void *W_r, void *Wp, int R, int N, int K, symm_stream_t stream) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (R != h->R) return fail(SYMM_EINVAL, "R=%d but the handle has %d ranks", R, h->R);
    size_t pbytes = 0;
    int rc = symm_packed_w_bytes(R, N, K, &pbytes);
    if (rc != SYMM_OK) return rc;
    const int Kr = K / R;
    const size_t wbytes = (size_t)N * (size_t)Kr * 2;
    if (!in_user_region(h, W_r, wbytes)) return fail(SYMM_EINVAL, "W_r (N x K/R bf16) is not inside slot 0's user region");
    if (!in_user_region(h, Wp, pbytes))
        return fail(SYMM_EINVAL, "Wp (%zu packed bytes per slot) is not inside slot 0's user region", pbytes);
    if (!aligned16(W_r) || !aligned16(Wp)) return fail(SYMM_EINVAL, "W_r and Wp must be 16-byte aligned");
    if (overlaps(W_r, wbytes, Wp, pbytes)) return fail(SYMM_EINVAL, "W_r and Wp overlap");
    if (find_packed(h, W_r) && wbytes > 0) return fail(SYMM_EINVAL, "W_r is itself a packed weight");
    rc = check_device(h);
    if (rc != SYMM_OK) return rc;
    PackWArgs a;
    a.W = static_cast<const uint8_t *>(W_r);
    a.Wp = static_cast<uint8_t *>(Wp);
    a.stride = (long long)h->stride;
    a.R = h->mp_rank >= 0 ? 1 : h->R;   // a multi-process handle packs its own rank's weight
    a.r0 = h->mp_rank >= 0 ? h->mp_rank : 0;
    a.N = N;
    a.Kr = Kr;
    cudaError_t e = launch_pack_w(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "symm_pack_w launch");
    note_write(h, Wp, pbytes);
    // Wp's bytes now belong to this weight alone: earlier packed weights it
    // overlaps are gone.
    auto &v = h->packed;
    v.erase(std::remove_if(v.begin(), v.end(),
                           [&](const symm_handle::PackedW &q) { return overlaps(q.p, q.bytes, Wp, pbytes); }),
            v.end());
    symm_handle::PackedW q;
    q.p = Wp;
    q.N = N;
    q.Kr = Kr;
    q.bytes = pbytes;
    v.push_back(q);
    return SYMM_OK;
}

int symm_release_w(symm_handle_t *h, const void *Wp) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    auto &v = h->packed;
    for (auto it = v.begin(); it != v.end(); ++it) {
        if (it->p == Wp) {
            v.erase(it);
            return SYMM_OK;
        }
    }
    return fail(SYMM_EINVAL, "%p is not a packed weight of this handle", Wp);
}

int gemv_reduce_scatter(symm_handle_t *h, const void *W_r, const void *x_r, void *y, int R, int N, int K, int B,
                        symm_stream_t stream) {
    Epilogue ep;
    ep.mode = kOutReduceScatter;
    return gemv_common(h, W_r, x_r, y, R, N, K, B, stream, ep);
}

int gemv_all_reduce_bias_rmsnorm(symm_handle_t *h, const void *W_r, const void *x_r, const void *bias,
                                 const void *gamma, void *y, int R, int N, int K, int B, float eps,
                                 symm_stream_t stream) {
    Epilogue ep;
    ep.mode = kOutBiasZ;
    ep.bias = bias;
    ep.gamma = gamma;
    ep.eps = eps;
    return gemv_common(h, W_r, x_r, y, R, N, K, B, stream, ep);
}

int reduce_scatter(symm_handle_t *h, const void *in, void *out, int R, size_t n, symm_stream_t stream) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (h->mp_rank >= 0) return fail(SYMM_EINVAL, "not available on a multi-process handle");
    if (R != h->R) return fail(SYMM_EINVAL, "R=%d but the handle has %d ranks", R, h->R);
    if (n % (size_t)R) return fail(SYMM_EINVAL, "n=%zu is not a multiple of R=%d", n, R);
    if (n == 0) return SYMM_OK;
    if (n > SIZE_MAX / 2) return fail(SYMM_EINVAL, "n too large");
    const size_t ib = n * 2, ob = n / (size_t)R * 2;
    if (!in_user_region(h, in, ib)) return fail(SYMM_EINVAL, "in + n elements is not inside slot 0's user region");
    if (!in_user_region(h, out, ob)) return fail(SYMM_EINVAL, "out + n/R elements is not inside slot 0's user region");
    if (!aligned16(in) || !aligned16(out)) return fail(SYMM_EINVAL, "in/out must be 16-byte aligned");
    if (overlaps(in, ib, out, ob)) return fail(SYMM_EINVAL, "in and out overlap");
    int rc = check_device(h);
    if (rc != SYMM_OK) return rc;
    ReduceScatterArgs a;
    a.in = static_cast<const uint8_t *>(in);
    a.out = static_cast<uint8_t *>(out);
    a.stride = (long long)h->stride;
    a.R = h->R;
    a.n = n;
    a.chunk = n / (size_t)R;
    a.shift = 0;
    a.ctas_per_sm = h->opt_ar_cps;
    a.chained = h->opt_chain;
    cudaError_t e = launch_reduce_scatter(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "reduce_scatter launch");
    note_write(h, out, ob);
    return SYMM_OK;
}

int two_shot_all_reduce(symm_handle_t *h, const void *in, void *out, int R, size_t n, symm_stream_t stream) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (h->mp_rank >= 0) return fail(SYMM_EINVAL, "not available on a multi-process handle");
    if (R != h->R) return fail(SYMM_EINVAL, "R=%d but the handle has %d ranks", R, h->R);
    if (n == 0) return SYMM_OK;
    if (n > SIZE_MAX / 2) return fail(SYMM_EINVAL, "n too large");
    const size_t bytes = n * 2;
    if (!in_user_region(h, in, bytes)) return fail(SYMM_EINVAL, "in + n elements is not inside slot 0's user region");
    if (!in_user_region(h, out, bytes)) return fail(SYMM_EINVAL, "out + n elements is not inside slot 0's user region");
    if (!aligned16(in) || !aligned16(out)) return fail(SYMM_EINVAL, "in/out must be 16-byte aligned");
    if (in != out && overlaps(in, bytes, out, bytes)) return fail(SYMM_EINVAL, "in and out partially overlap");
    int rc = check_device(h);
    if (rc != SYMM_OK) return rc;
    // Owner s reduces elements [s*chunk, (s+1)*chunk); chunk is a multiple of
    // 8 elements so that every owner's block starts on a 16-byte boundary.
    const size_t per = (n + (size_t)R - 1) / (size_t)R;
    ReduceScatterArgs a;
    a.in = static_cast<const uint8_t *>(in);
    a.out = static_cast<uint8_t *>(out);
    a.stride = (long long)h->stride;
    a.R = h->R;
    a.n = n;
    a.chunk = (per + 7) / 8 * 8;
    a.shift = 1;
    a.ctas_per_sm = h->opt_ar_cps;
    a.chained = h->opt_chain;   // phase 1; phase 2 is always a programmatic dependent of phase 1
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = launch_reduce_scatter(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "two_shot_all_reduce reduce-scatter launch");
    e = launch_all_gather_blocks(a, s);
    if (e != cudaSuccess) return cuda_fail(e, "two_shot_all_reduce all-gather launch");
    note_write(h, out, bytes);
    return SYMM_OK;
}

int all_reduce_bias_rmsnorm(symm_handle_t *h, const void *in, const void *bias, const void *gamma, void *out, int R,
                            int rows, int H, float eps, symm_stream_t stream) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (h->mp_rank >= 0) return fail(SYMM_EINVAL, "not available on a multi-process handle");
    if (R != h->R) return fail(SYMM_EINVAL, "R=%d but the handle has %d ranks", R, h->R);
    if (rows < 0 || rows > 65535) return fail(SYMM_EINVAL, "rows=%d outside 0..65535", rows);
    if (H < 8 || H % 8 || H > rmsnorm_max_h())
        return fail(SYMM_EINVAL, "H=%d must be a multiple of 8 in 8..%d", H, rmsnorm_max_h());
    if (!(eps >= 0.f) || eps > 3.0e38f) return fail(SYMM_EINVAL, "eps must be finite and >= 0");
    if (rows == 0) return SYMM_OK;
    const size_t bytes = (size_t)rows * H * 2, vb = (size_t)H * 2;
    if (!in_user_region(h, in, bytes)) return fail(SYMM_EINVAL, "in (rows x H bf16) is not inside slot 0's user region");
    if (!in_user_region(h, out, bytes)) return fail(SYMM_EINVAL, "out (rows x H bf16) is not inside slot 0's user region");
    if (!aligned16(in) || !aligned16(out)) return fail(SYMM_EINVAL, "in/out must be 16-byte aligned");
    if (in != out && overlaps(in, bytes, out, bytes)) return fail(SYMM_EINVAL, "in and out partially overlap");
    for (const void *v : {bias, gamma}) {
        if (!v) continue;
        if (!in_user_region(h, v, vb) || !aligned16(v))
            return fail(SYMM_EINVAL, "bias / gamma (H bf16) must be 16-byte aligned inside slot 0's user region");
        if (overlaps(v, vb, out, bytes)) return fail(SYMM_EINVAL, "bias / gamma overlaps out");
    }
    int rc = check_device(h);
    if (rc != SYMM_OK) return rc;
    RmsNormArgs a = {};
    a.in = static_cast<const uint8_t *>(in);
    a.bias = static_cast<const uint8_t *>(bias);
    a.gamma = static_cast<const uint8_t *>(gamma);
    a.out = static_cast<uint8_t *>(out);
    a.stride = (long long)h->stride;
    a.R = h->R;
    a.rows = rows;
    a.H = H;
    a.eps = eps;
    // Chained: gamma and bias are loaded before the wait for the previous
    // kernel, so not when that kernel (the handle's last) wrote them.
    const bool chained = h->opt_chain != 0 && !overlaps(bias, bias ? vb : 0, h->last_write, h->last_write_bytes) &&
                         !overlaps(gamma, gamma ? vb : 0, h->last_write, h->last_write_bytes);
    a.wait_prior = chained;
    a.release_next = chained;
    a.tl = h->tl;
    a.tl_ctas = h->tl_ctas;
    cudaError_t e = launch_rmsnorm_rows(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "all_reduce_bias_rmsnorm launch");
    note_write(h, out, bytes);

    return SYMM_OK;
}

int multi_root_tile_reduce(symm_handle_t *h, const void *const *in_tiles, void *out_tile, const int *roots,
                           int ntiles, int rows, int cols, long long ld_in, long long ld_out, symm_stream_t stream) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (h->mp_rank >= 0) return fail(SYMM_EINVAL, "not available on a multi-process handle");
    if (!in_tiles || !roots || !out_tile) return fail(SYMM_EINVAL, "NULL argument");
    if (ntiles < 1 || ntiles > h->R || ntiles > kMaxTiles)
        return fail(SYMM_EINVAL, "ntiles=%d outside 1..%d (one root per rank at most)", ntiles, std::min(h->R, kMaxTiles));
    if (rows < 0 || cols < 0) return fail(SYMM_EINVAL, "rows=%d cols=%d must be >= 0", rows, cols);
    if (rows > 0 && cols > 0 && (ld_in < cols || ld_out < cols))
        return fail(SYMM_EINVAL, "leading dimensions (%lld, %lld) must be >= cols=%d", ld_in, ld_out, cols);
    bool used[SYMM_MAX_RANKS] = {};
    for (int i = 0; i < ntiles; ++i) {
        if (roots[i] < 0 || roots[i] >= h->R) return fail(SYMM_EINVAL, "root %d outside 0..%d", roots[i], h->R - 1);
        if (used[roots[i]]) return fail(SYMM_EINVAL, "rank %d is the root of more than one tile", roots[i]);
        used[roots[i]] = true;
    }
    if (rows == 0 || cols == 0) return SYMM_OK;
    const size_t in_ext = ((size_t)(rows - 1) * (size_t)ld_in + (size_t)cols) * 2;
    const size_t out_ext = ((size_t)(rows - 1) * (size_t)ld_out + (size_t)cols) * 2;
    if (!in_user_region(h, out_tile, out_ext) || (reinterpret_cast<uintptr_t>(out_tile) & 1))
        return fail(SYMM_EINVAL, "the output tile is not inside slot 0's user region (or not 2-byte aligned)");
    for (int i = 0; i < ntiles; ++i) {
        if (!in_tiles[i] || !in_user_region(h, in_tiles[i], in_ext) || (reinterpret_cast<uintptr_t>(in_tiles[i]) & 1))
            return fail(SYMM_EINVAL, "input tile %d is not inside slot 0's user region (or not 2-byte aligned)", i);
        // the output tile is written while other threads still read inputs
        if (overlaps(in_tiles[i], in_ext, out_tile, out_ext))
            return fail(SYMM_EINVAL, "input tile %d overlaps the output tile", i);
    }
    int rc = check_device(h);
    if (rc != SYMM_OK) return rc;
    TileReduceArgs a;
    for (int i = 0; i < ntiles; ++i) {
        a.in[i] = static_cast<const uint8_t *>(in_tiles[i]);
        a.root[i] = roots[i];
    }
    a.out = static_cast<uint8_t *>(out_tile);
    a.stride = (long long)h->stride;
    a.R = h->R;
    a.ntiles = ntiles;
    a.rows = rows;
    a.cols = cols;
    a.ld_in = ld_in;
    a.ld_out = ld_out;
    a.chained = h->opt_chain;
    cudaError_t e = launch_tile_reduce(a, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "tile reduce launch");
    note_write(h, out_tile, out_ext);
    return SYMM_OK;
}

int tile_reduce(symm_handle_t *h, const void *in_tile, void *out_tile, int root, int rows, int cols, long long ld_in,
                long long ld_out, symm_stream_t stream) {
    const void *tiles[1] = {in_tile};
    const int roots[1] = {root};
    return multi_root_tile_reduce(h, tiles, out_tile, roots, 1, rows, cols, ld_in, ld_out, stream);
}

int symm_set_timeline(symm_handle_t *h, void *buf, size_t bytes) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (!buf || bytes == 0) {
        h->tl = nullptr;
        h->tl_ctas = 0;
        return SYMM_OK;
    }
    if (!kTimeline) return fail(SYMM_EINVAL, "this library was built without timeline stamps (-DSYMM_TIMELINE)");
    if (reinterpret_cast<uintptr_t>(buf) % 8) return fail(SYMM_EINVAL, "the timeline buffer must be 8-byte aligned");
    h->tl = static_cast<unsigned long long *>(buf);
    h->tl_ctas = (int)std::min<size_t>(bytes / (sizeof(unsigned long long) * kTlSlots), 1u << 30);
    return SYMM_OK;
}

int symm_status(symm_handle_t *h, symm_stream_t stream, int *code, int *rank, int *tile) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t st[4] = {0, 0, 0, 0};
    const int own = h->mp_rank >= 0 ? h->mp_rank : 0;   // a process latches into its own slot's words
    e = cudaMemcpy(st, pad_word(h, own, 0), sizeof st, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
    // A multi-process handle also compares the ranks' launch counts (each
    // rank's epoch word, advanced by its own launches): read after a
    // barrier that every live rank passed with its calls finished, a count
    // that differs names a rank that skipped a call (or left).
    int lag = -1;
    uint32_t own_epoch = 0, lag_epoch = 0;
    if (h->mp_rank >= 0 && !st[kStatusCode]) {
        e = cudaMemcpy(&own_epoch, pad_word(h, own, kPadEpochOffset), 4, cudaMemcpyDeviceToHost);
        for (int r = 0; r < h->R && e == cudaSuccess && lag < 0; ++r) {
            if (r == own) continue;
            uint32_t ep = 0;
            e = cudaMemcpy(&ep, pad_word(h, r, kPadEpochOffset), 4, cudaMemcpyDeviceToHost);
            if (e == cudaSuccess && ep != own_epoch) {
                lag = r;
                lag_epoch = ep;
            }
        }
        if (e != cudaSuccess) return cuda_fail(e, "reading the ranks' launch counts");
    }
    const bool err = st[kStatusCode] != 0 || lag >= 0;
    if (code) *code = err ? SYMM_EPROTO : SYMM_OK;
    if (rank) *rank = st[kStatusCode] ? (int)st[kStatusRank] : lag;
    if (tile) *tile = st[kStatusCode] ? (int)st[kStatusTile] : -1;
    if (err) {
        if (st[kStatusCode])
            snprintf(g_err, sizeof g_err, "protocol error %u at rank %u tile %u epoch %u", st[kStatusCode],
                     st[kStatusRank], st[kStatusTile], st[kStatusEpoch]);
        else
            snprintf(g_err, sizeof g_err, "rank %d has made %u fused calls, this rank (%d) %u", lag, lag_epoch, own,
                     own_epoch);
        // the four status words only: reset_protocol clears the counters and
        // keeps a multi-process rank's launch count, which the others compare
        e = cudaMemsetAsync(pad_word(h, own, 0), 0, 4 * sizeof(uint32_t), s);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
        int rc = reset_protocol(h, s);
        if (rc != SYMM_OK) return rc;
        e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    }
    return SYMM_OK;
}

// The handle's device can copy to or from [p, p + bytes) with its SMs: its
// own device memory, or pinned host memory mapped into the device's address
// space at the same address (both ends checked).
bool sm_addressable(const symm_handle *h, const void *p, size_t bytes) {
    for (const uint8_t *q : {static_cast<const uint8_t *>(p), static_cast<const uint8_t *>(p) + bytes - 1}) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
            cudaGetLastError();   // an unregistered host pointer is not an error here
            return false;
        }
        if (at.type == cudaMemoryTypeDevice && at.device == h->device) continue;
        if (at.type == cudaMemoryTypeHost && at.devicePointer == q) continue;
        return false;
    }
    return true;
}

int symm_copy_to_slots(symm_handle_t *h, void *dst, const void *src, size_t bytes_per_rank, int nranks,
                       symm_stream_t stream) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (!mp_ready(h)) return fail(SYMM_EINVAL, "not every rank's slot is mapped yet (symm_mp_import)");
    if (nranks < 0 || nranks > h->R) return fail(SYMM_EINVAL, "nranks=%d outside 0..%d", nranks, h->R);
    if (bytes_per_rank == 0 || nranks == 0) return SYMM_OK;
    if (!src) return fail(SYMM_EINVAL, "src is NULL");
    if (!in_user_region(h, dst, bytes_per_rank)) return fail(SYMM_EINVAL, "dst is not inside slot 0's user region");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (h->opt_copy_engine == 0 && sm_addressable(h, src, bytes_per_rank * (size_t)nranks)) {
        int rc = check_device(h);
        if (rc != SYMM_OK) return rc;
        CopySlotsArgs a;
        a.src = static_cast<const uint8_t *>(src);
        a.dst = static_cast<uint8_t *>(dst);
        a.src_stride = (long long)bytes_per_rank;
        a.dst_stride = (long long)h->stride;
        a.bytes = bytes_per_rank;
        a.nranks = nranks;
        a.chained = h->opt_chain;
        cudaError_t e = launch_copy_slots(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "copy to slots launch");
        note_write(h, dst, bytes_per_rank);
        return SYMM_OK;
    }
    // One strided copy: rank r's bytes land at dst + r * stride.
    cudaError_t e = cudaMemcpy2DAsync(dst, h->stride, src, bytes_per_rank, bytes_per_rank, (size_t)nranks,
                                      cudaMemcpyDefault, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync (to slots)");
    return SYMM_OK;
}

int symm_copy_from_slots(symm_handle_t *h, void *dst, const void *src, size_t bytes_per_rank, int nranks,
                         symm_stream_t stream) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (!mp_ready(h)) return fail(SYMM_EINVAL, "not every rank's slot is mapped yet (symm_mp_import)");
    if (nranks < 0 || nranks > h->R) return fail(SYMM_EINVAL, "nranks=%d outside 0..%d", nranks, h->R);
    if (bytes_per_rank == 0 || nranks == 0) return SYMM_OK;
    if (!dst) return fail(SYMM_EINVAL, "dst is NULL");
    if (!in_user_region(h, src, bytes_per_rank)) return fail(SYMM_EINVAL, "src is not inside slot 0's user region");
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (h->opt_copy_engine == 0 && sm_addressable(h, dst, bytes_per_rank * (size_t)nranks)) {
        int rc = check_device(h);
        if (rc != SYMM_OK) return rc;
        CopySlotsArgs a;
        a.src = static_cast<const uint8_t *>(src);
        a.dst = static_cast<uint8_t *>(dst);
        a.src_stride = (long long)h->stride;
        a.dst_stride = (long long)bytes_per_rank;
        a.bytes = bytes_per_rank;
        a.nranks = nranks;
        a.chained = h->opt_chain;
        cudaError_t e = launch_copy_slots(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "copy from slots launch");
        return SYMM_OK;
    }
    cudaError_t e = cudaMemcpy2DAsync(dst, bytes_per_rank, src, h->stride, bytes_per_rank, (size_t)nranks,
                                      cudaMemcpyDefault, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy2DAsync (from slots)");
    return SYMM_OK;
}

int symm_check_guards(symm_handle_t *h, int *bad_rank, int *bad_band) {
    if (!h) return fail(SYMM_EINVAL, "handle is NULL");
    if (bad_rank) *bad_rank = -1;
    if (bad_band) *bad_band = -1;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    static thread_local unsigned char buf[kGuard];
    const size_t offs[3] = {h->guard0, h->guard1, h->guard2};
    for (int r = 0; r < h->R; ++r)
        for (int band = 0; band < 3; ++band) {
            if (h->mp_rank >= 0 && r != h->mp_rank) continue;   // each process checks its own slot
            e = cudaMemcpy(buf, slot(h, r) + offs[band], kGuard, cudaMemcpyDeviceToHost);
            if (e != cudaSuccess) return cuda_fail(e, "reading a guard band");
            for (size_t i = 0; i < kGuard; ++i)
                if (buf[i] != kGuardByte) {
                    if (bad_rank) *bad_rank = r;
                    if (bad_band) *bad_band = band;
                    return fail(SYMM_ECORRUPT, "guard band %d of rank %d overwritten at byte %zu", band, r, i);
                }
        }
    return SYMM_OK;
}

int symm_free(symm_handle_t *h) {
    if (!h) return SYMM_OK;
    int rc = SYMM_OK;
    if (h->mp_rank >= 0) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e != cudaSuccess) rc = cuda_fail(e, "cudaDeviceSynchronize");
        mp_release(h);
    } else if (h->owned && h->base) {
        cudaError_t e = cudaDeviceSynchronize();
        if (e == cudaSuccess) e = cudaFree(h->base);
        if (e != cudaSuccess) rc = cuda_fail(e, "cudaFree");
    }
    delete h;
    return rc;
}

}  // extern "C"
