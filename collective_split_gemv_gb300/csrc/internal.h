// Internal interface between the host runtime (symm_runtime.cu) and the
// kernels.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace symm {

// Sets kern's dynamic shared-memory limit to `bytes` once per device (the
// attribute is per device).  Host threads may launch concurrently: the
// devices already set form an atomic bit mask, and setting the attribute
// twice is harmless.  Devices past 63 set it on every call.
template <class... KArgs>
cudaError_t set_smem_once(void (*kern)(KArgs...), int bytes, std::atomic<unsigned long long> &done) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 64;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

// Launches kern<<<grid, block, smem, s>>>(args...); when `chained`, as a
// programmatic dependent of the previous kernel on the stream (its CTAs may
// be scheduled while that kernel drains; the kernel itself waits for it with
// griddepcontrol.wait before touching what it wrote).
template <class... KArgs, class... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          bool chained, Args &&...args) {
    if (!chained) {
        kern<<<grid, block, smem, s>>>(std::forward<Args>(args)...);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Signal-pad layout of every slot (byte offsets from the pad start):
//   [0, 16)                 status words {code, rank, tile, epoch} (slot 0 only)
//   [64, 72)                work[2]      work counters of the persistent kernel,
//                                        launch e uses work[e & 1] (slot 0 only)
//   [96, 100)               epoch        epoch of the last finished fused launch
//                                        (slot 0 only)
//   [112, 116)              tiles_done   tiles of the running launch that have
//                                        been reduced (slot 0 only)
//   [128, 128 + 4*T)        flags[T]     tile t of rank r published (epoch)
//   [cnt_off, cnt_off+4*T)  counters[T]  arrivals at tile t (slot 0 only)
// Between launches every counter is zero; only the epoch and the flags carry
// over.  So a launch needs no host-side state: the same launch replayed from
// a CUDA graph, or launches of different geometries interleaved, see a
// consistent pad.
constexpr size_t kPadStatusBytes = 128;
constexpr size_t kPadWorkOffset = 64;
constexpr size_t kPadEpochOffset = 96;
constexpr size_t kPadTilesDoneOffset = 112;
constexpr int kStatusCode = 0, kStatusRank = 1, kStatusTile = 2, kStatusEpoch = 3;
constexpr int kProtoStaleFlag = 1;    // device codes; host maps them to SYMM_EPROTO
constexpr int kProtoBadTicket = 2;

constexpr int kProtoTimeout = 3;      // a bounded wait inside a kernel gave up
constexpr int kMaxRanks = 64;

// Arguments of one fused GEMV + all-reduce launch.  Every pointer is the
// slot-0 instance; rank r's instance is ptr + r * stride bytes.
//
// A tile's contributors are the (rank r, K-split s) pairs, r < R, s < splits:
// contributor (r, s) sums k in its split of rank r's K/R columns, writes the
// fp32 partial to scratch + r * stride + s * partial_stride ([B][N]) and
// publishes flags_r[t * splits + s].
struct GemvArgs {
    const uint8_t *W;        // bf16 [N][Kr]
    const uint8_t *x;        // bf16 [B][Kr]
    uint8_t *y;              // bf16 [B][N]
    uint8_t *scratch;        // fp32 [splits][B][N] partials of the slot's rank
    uint32_t *flags;         // [max_tiles]
    uint32_t *counters;      // [max_tiles], slot 0
    uint32_t *status;        // [4], slot 0
    long long stride;        // bytes between slots
    long long partial_stride;  // bytes between the splits' partial arrays (4 * B * N)
    int R, N, Kr, B;
    int splits;              // K-splits per rank (1 for the per-tile kernel)
    int rows_per_tile;
    int num_tiles;
    int kc_cap;              // 16-byte chunks of x staged in shared memory per pass
    uint32_t *epoch_word;    // slot 0: epoch of the last finished fused launch
    uint32_t *tiles_done;    // slot 0: tiles reduced so far in this launch
    uint32_t *work;          // slot 0: the persistent kernel's two work counters
    int reverse_order;       // 1: CTAs take work in reverse (arrival-order tests)
    // What the tile reducer does with the fp32 sum of output (b, n):
    //   kOutAllReduce      bf16 into y of every rank (y: [B][N] per slot);
    //   kOutReduceScatter  bf16 into y of rank b / rs_rows only, at row
    //                      b % rs_rows (y: [rs_rows][N] per slot);
    //   kOutBiasZ          fp32 sum + bias[n] into z[b][n] (slot 0), for the
    //                      RMS-normalisation stage that follows;
    //   kOutPartials       no tile reduction (persistent kernel only): the
    //                      partials stay in scratch for the separate
    //                      all-reduce kernel of the unfused form.
    int out_mode;
    int chained;             // per-tile and cluster kernels (paths 1, 5): launch as a programmatic dependent
    int rs_rows;             // kOutReduceScatter: B / R
    float *z;                // kOutBiasZ: fp32 [B][N]
    const uint8_t *bias;     // kOutBiasZ: bf16 [N] (slot 0) or nullptr
    int w_packed;            // persistent kernel: W is in the packed layout (below), not [N][Kr]
    // Persistent kernel, chained launch: the first stages' W loads may go out
    // before the wait for the previous kernel (packed weights only: they are
    // written once, by symm_pack_w, never by the kernel a call follows).
    int w_early;
    unsigned long long *tl;  // timeline rows (timeline build only; nullptr: none), see timeline.cuh
    int tl_ctas;             // CTAs the timeline buffer has rows for
    // Multi-process handle: this launch computes rank my_rank's units only
    // (-1: every rank's).  tiles_done is then nullptr and the launch is
    // finished by the CTA that counts the last of its units on units_done
    // (the own slot's pad).
    int my_rank;
    uint32_t *units_done;
};
constexpr int kOutAllReduce = 0, kOutReduceScatter = 1, kOutBiasZ = 2, kOutPartials = 3;

// The unfused form's second kernel: y_s = bf16(sum of the R * splits fp32
// partials in contributor order) for every slot s (partials_ar.cu).
struct PartialsArArgs {
    const uint8_t *scratch;  // fp32 [splits][B][N] partials of rank q at + q * stride
    uint8_t *y;              // bf16 [B][N], slot 0
    long long stride;
    long long partial_stride;  // bytes between a rank's split partials (4 * B * N)
    int R, splits, B, N;
    int vec;                 // 1: B * N % 4 == 0 (16-byte loads, 8-byte stores)
    int chained;             // launch as a programmatic dependent of the GEMV
};
cudaError_t launch_partials_ar(const PartialsArArgs &a, cudaStream_t s);

// Sets the calling thread's last-error message (see symm_last_error) and
// returns `code`.
int report_error(int code, const char *msg);

struct AllReduceArgs {
    const uint8_t *in;       // bf16 [n], slot 0
    uint8_t *out;            // bf16 [n], slot 0
    long long stride;
    int R;
    size_t n;
    int ctas_per_sm;         // grid cap per SM (grid-stride beyond it); 0 = the default
    int kernel;              // one-shot kernel: kArKernelAuto / PerThread / Staged
    int chained;             // one-shot: launch as a programmatic dependent of the previous kernel
    int my_rank;             // multi-process handle: store the result into this rank's slot only (-1: all)
};
// The one-shot all-reduce has two kernels: per-thread 16-byte loads and
// stores, and one staged through shared memory by bulk (TMA) copies.  Auto
// takes the per-thread one: it measured faster at every size (R = 8, 32 KB
// to 33.5 MB per rank).
constexpr int kArKernelAuto = 0, kArKernelPerThread = 1, kArKernelStaged = 2;

// Kernel launchers; return the launch's cudaError_t.
cudaError_t launch_one_shot_all_reduce(const AllReduceArgs &a, cudaStream_t s);
bool one_shot_uses_staged(const AllReduceArgs &a);

// Reduce-scatter over the slots: element i (i < n) belongs to owner
// i / chunk; its sum over the R slots goes to slot owner's out at element
// (i - owner * chunk) + shift * owner * chunk.  shift = 0: the compact
// reduce-scatter output (chunk elements per slot); shift = 1: the owner's
// block of a full-length output (phase 1 of the two-shot all-reduce).
struct ReduceScatterArgs {
    const uint8_t *in;       // bf16 [n], slot 0
    uint8_t *out;            // bf16, slot 0
    long long stride;
    int R;
    size_t n;
    size_t chunk;            // elements per owner
    int shift;
    int ctas_per_sm;         // grid cap per SM; 0 = the default
    int chained;             // launch as a programmatic dependent of the previous kernel
};
cudaError_t launch_reduce_scatter(const ReduceScatterArgs &a, cudaStream_t s);
// Phase 2 of the two-shot all-reduce: out_q[i] = out_owner(i)[i] for q != owner.
cudaError_t launch_all_gather_blocks(const ReduceScatterArgs &a, cudaStream_t s);

// Sum of a 2-D tile over the R slots into one root slot's output tile.
constexpr int kMaxTiles = 64;
struct TileReduceArgs {
    const uint8_t *in[kMaxTiles];  // tile i's first element, slot 0
    int root[kMaxTiles];
    uint8_t *out;                  // output tile's first element, slot 0
    long long stride;
    int R, ntiles, rows, cols;
    long long ld_in, ld_out;       // elements
    int chained;                   // launch as a programmatic dependent of the previous kernel
};
cudaError_t launch_tile_reduce(const TileReduceArgs &a, cudaStream_t s);

// RMS normalisation of `rows` rows of H elements, one thread-block cluster
// per row.  Source: either R bf16 slots plus an optional bf16 bias (the
// all-reduce + bias + RMSNorm kernel), or one fp32 array that already holds
// sum + bias (the fused layer's epilogue stage).  The result is stored as
// bf16 into every slot's out.
struct RmsNormArgs {
    const uint8_t *in;       // bf16 [rows][H], slot 0 (source kind 0)
    const float *z;          // fp32 [rows][H] (source kind 1)
    const uint8_t *bias;     // bf16 [H], slot 0, or nullptr (kind 0 only)
    const uint8_t *gamma;    // bf16 [H], slot 0, or nullptr
    uint8_t *out;            // bf16 [rows][H], slot 0
    long long stride;
    int R, rows, H;
    float eps;
    int wait_prior;          // 1: launched as a dependent of the previous kernel (PDL)
    int release_next;        // 1: let the next kernel on the stream be scheduled early
    unsigned long long *tl;  // timeline rows (timeline build only; nullptr: none), see timeline.cuh
    int tl_ctas;
};
int rmsnorm_max_h();
cudaError_t launch_rmsnorm_rows(const RmsNormArgs &a, cudaStream_t s);

// Strided copy by the SMs: block r (bytes) from src + r * src_stride to
// dst + r * dst_stride, r < nranks (copy_slots.cu).
struct CopySlotsArgs {
    const uint8_t *src;
    uint8_t *dst;
    long long src_stride, dst_stride;
    size_t bytes;
    int nranks;
    int chained;             // launch as a programmatic dependent of the previous kernel
};
cudaError_t launch_copy_slots(const CopySlotsArgs &a, cudaStream_t s);

// Packed weight layout (symm_pack_w): W_r cut into 128-row x 64-column
// blocks, block (t, j) = rows 128t.., columns 64j.. stored as 16 KB at
// ((t * J + j) * 16 KB), J = ceil(Kr / 64), in the byte order a TMA load with
// 128-byte swizzle leaves the same box in shared memory: row i at i * 128,
// its 16-byte chunk c at chunk position c ^ (i % 8).  Rows past N and
// columns past Kr are zero, and one more all-zero block follows the last
// (the persistent kernel reads it for the stage slabs past Kr).
constexpr int kPackRows = 128, kPackCols = 64;
constexpr size_t kPackBlockBytes = (size_t)kPackRows * kPackCols * 2;
inline size_t packed_w_blocks(int N, int Kr) {
    return (size_t)((N + kPackRows - 1) / kPackRows) * (size_t)((Kr + kPackCols - 1) / kPackCols) + 1;
}
struct PackWArgs {
    const uint8_t *W;        // bf16 [N][Kr], slot 0
    uint8_t *Wp;             // packed, slot 0
    long long stride;
    int R, N, Kr;
    int r0;                  // first rank packed (R ranks from it; a multi-process handle packs its own)
};
cudaError_t launch_pack_w(const PackWArgs &a, cudaStream_t s);

// Cluster fused kernel for small layers (gemv_cluster.cu): one thread-block
// cluster of R CTAs per 16-row tile, partials exchanged through distributed
// shared memory; R <= kMaxClusterRanks, B <= 4.
constexpr int kClusterRows = 16;
constexpr int kMaxClusterRanks = 8;
constexpr int kClusterMaxBatch = 4;
cudaError_t launch_gemv_cluster(const GemvArgs &a, cudaStream_t s);

// FFMA (CUDA-core) fused kernel: any B in 1..16.
int ffma_rows_per_tile(int B);
size_t ffma_smem_bytes(int B, int kc_cap);
int ffma_kc_cap(int B, int Kr);
cudaError_t launch_gemv_ffma(const GemvArgs &a, cudaStream_t s);

// Persistent dynamically scheduled kernel (TMA ring into tcgen05): 128-row
// tiles, batch padded to 16.  G CTAs draw the U = T*R*splits units (KB
// K-blocks each) from the work counter work[epoch & 1] (slot 0's pad), or,
// with the cluster epilogue, one unit per CTA in clusters of R*splits.
constexpr int kDynRows = 128;
struct DynGeom {
    int units;      // T * R * splits
    int splits;     // K splits per (tile, rank)
    int KB;         // K blocks per (tile, rank)
    int KBs;        // K blocks per split
    int G;
    int cluster;    // 0: units drawn, global-memory protocol; R: cluster epilogue
                    // (G = units, one per CTA, splits 1, clusters of R CTAs)
};
// Encodes the TMA descriptors of a launch (cached by the caller): `maps`
// points at two CUtensorMap objects (W, x), 64-byte aligned.
int dyn_encode_maps(const GemvArgs &a, void *maps);
// K elements per ring stage, and the (slabs, CTAs per SM) pipelines built.
int dyn_block_k(int slabs);
bool dyn_config_supported(int slabs, int ctas_per_sm);
// Pipelines the cluster epilogue is built for (two CTAs per SM).
bool dyn_cluster_supported(int slabs, int ctas_per_sm);
// Whether a cluster of R CTAs of that kernel can be resident on the current
// device at all (the occupancy query, cached per device; false on a device
// or partition whose GPCs cannot hold one).
bool dyn_cluster_fits(int slabs, int R);
// chained: launch as a programmatic dependent of the previous kernel on the
// stream (its CTAs may start while that one drains; see the kernel).
cudaError_t launch_gemv_dyn(const GemvArgs &a, const DynGeom &geo, const void *maps, int slabs, int ctas_per_sm,
                            bool chained, cudaStream_t s);

}  // namespace symm
