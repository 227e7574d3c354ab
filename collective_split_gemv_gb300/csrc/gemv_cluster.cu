// Fused row-parallel GEMV + one-shot all-reduce for small layers: one
// thread-block cluster per row tile, one CTA of the cluster per rank.
//
// On small layers a call is bound by latency, not bandwidth: the per-tile
// publish protocol through global memory (fence, arrival ticket, flag and
// partial loads by the last arriver) costs three to four L2 round trips after
// the dot products.  Here the R contributors of a tile are the R CTAs of one
// cluster, which the hardware schedules together, so the exchange goes
// through distributed shared memory instead: CTA r computes rank r's fp32
// partial of the tile into its own shared memory, one cluster barrier
// (release / acquire) publishes all R partials, and every CTA then sums its
// share of the tile's outputs over the R partials -- read from the peers'
// shared memory, in rank order 0..R-1, in fp32 -- rounds to bf16 and stores
// the value into every rank's output slot.  A second cluster barrier keeps
// each CTA's shared memory alive until its peers have read it.  No scratch,
// no signal pad, no atomics: the kernel reads W and x and writes y.
//
// This is the fused GEMV + AllReduce of "Overlapping Collective Communication
// with Dependent Computation ..." (Abstract: partials are pushed as soon as
// each share is done and reduced where they land) with the R emulated ranks
// co-scheduled as a cluster; distributed shared memory plays the part of the
// peers' memory the pages' kernel writes into.  The sum order is the fixed
// rank order of the global-memory protocol, so the results do not depend on
// timing.
//
// Per CTA (256 threads = 8 warps; warp w owns G consecutive rows of the
// tile): each lane streams 16-byte chunks c = lane, lane + 32, ... of its
// rows of W_r and the same chunks of x_r straight into registers (U chunks in
// flight), multiplies in fp32 in ascending k within a chunk, chunks in the
// lane's order, and ends with a fixed xor-shuffle tree across the warp.
//
// Timeline slots (timeline build only, timeline.cuh; row = tile * R + rank):
// 0 entry, 1 dot products done, 2 partials published (first cluster barrier
// passed), 3 share of the tile summed and stored, 4 exit.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "protocol.cuh"
#include "sm100.cuh"
#include "timeline.cuh"

namespace symm {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kG = 2;                       // rows per warp
constexpr int kRows = kWarps * kG;          // rows per tile
constexpr int kU = 4;                       // 16-byte chunks per row in flight per lane

static_assert(kRows == kClusterRows, "tile height");

__device__ __forceinline__ uint4 ld_nc_v4(const void *p) {
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float dot8(const uint4 &w, const uint4 &x, float acc) {
    acc = fmaf(bf16lo(w.x), bf16lo(x.x), acc);
    acc = fmaf(bf16hi(w.x), bf16hi(x.x), acc);
    acc = fmaf(bf16lo(w.y), bf16lo(x.y), acc);
    acc = fmaf(bf16hi(w.y), bf16hi(x.y), acc);
    acc = fmaf(bf16lo(w.z), bf16lo(x.z), acc);
    acc = fmaf(bf16hi(w.z), bf16hi(x.z), acc);
    acc = fmaf(bf16lo(w.w), bf16lo(x.w), acc);
    acc = fmaf(bf16hi(w.w), bf16hi(x.w), acc);
    return acc;
}

template <int B>
__global__ void __launch_bounds__(kThreads, 1) gemv_ar_cluster_kernel(const GemvArgs a) {
    __shared__ float part[B * kRows];       // this rank's partial of the tile, [b][row]

    const int r = blockIdx.x;               // the CTA's rank = its rank in the cluster
    const int t = blockIdx.y;
    const int R = a.R;
    const int tl_cta = t * R + r;
    if (threadIdx.x == 0) {
        tl_begin();
        tl_stamp(a.tl, a.tl_ctas, tl_cta, 0);
    }
    // Chained calls: let the next kernel be scheduled early; wait for the one
    // before (which may have written W, x or y) before touching memory.
    chain_entry();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nchunk = a.Kr >> 3;
    const int n_base = t * kRows;
    const uint8_t *Wr = a.W + (long long)r * a.stride;
    const uint8_t *xr = a.x + (long long)r * a.stride;

    const uint4 *wrow[kG];
    bool rowok[kG];
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        const int n = n_base + warp * kG + g;
        rowok[g] = n < a.N;
        wrow[g] = reinterpret_cast<const uint4 *>(Wr + (size_t)(rowok[g] ? n : 0) * a.Kr * 2);
    }
    float acc[kG][B];
#pragma unroll
    for (int g = 0; g < kG; ++g)
#pragma unroll
        for (int b = 0; b < B; ++b) acc[g][b] = 0.f;

    for (int c = lane; c < nchunk; c += 32 * kU) {
        uint4 w[kU][kG], xv[kU][B];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int cc = c + 32 * u;
#pragma unroll
            for (int g = 0; g < kG; ++g)
                w[u][g] = (cc < nchunk && rowok[g]) ? ld_stream_v4(wrow[g] + cc) : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int b = 0; b < B; ++b)
                xv[u][b] = cc < nchunk ? ld_nc_v4(xr + ((size_t)b * a.Kr + (size_t)cc * 8) * 2) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            if (c + 32 * u < nchunk) {
#pragma unroll
                for (int b = 0; b < B; ++b)
#pragma unroll
                    for (int g = 0; g < kG; ++g) acc[g][b] = dot8(w[u][g], xv[u][b], acc[g][b]);
            }
        }
    }
    // Fixed butterfly across the warp; every lane ends with every sum.
#pragma unroll
    for (int g = 0; g < kG; ++g)
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float v = acc[g][b];
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
            acc[g][b] = v;
        }
#pragma unroll
    for (int g = 0; g < kG; ++g)
#pragma unroll
        for (int b = 0; b < B; ++b)
            if (lane == ((g * B + b) & 31)) part[b * kRows + warp * kG + g] = acc[g][b];
    if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, tl_cta, 1);

    // Publish: every rank's partial is in its CTA's shared memory once all
    // CTAs of the cluster have passed this barrier (release / acquire).
    cluster_arrive_release();
    cluster_wait_acquire();
    if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, tl_cta, 2);

    // This CTA's share of the tile's outputs: a contiguous range of the
    // [b][row] items, so that the stores of neighbouring threads are
    // neighbouring elements of y.
    const int rows = min(kRows, a.N - n_base);
    const int items = B * kRows;
    const int share = (items + R - 1) / R;
    const int i = r * share + (int)threadIdx.x;
    const bool mine = (int)threadIdx.x < share && i < items && (i % kRows) < rows;
    float sum = 0.f;
    if (mine) {
        // The R partials in rank order, their loads issued back to back.
        float v[kMaxClusterRanks];
#pragma unroll
        for (int q = 0; q < kMaxClusterRanks; ++q)
            if (q < R) v[q] = ld_cluster_f32(cluster_addr(&part[i], (uint32_t)q));
        sum = v[0];
#pragma unroll
        for (int q = 1; q < kMaxClusterRanks; ++q)
            if (q < R) sum += v[q];
    }
    // Done reading the peers' shared memory; the stores need none of it.
    cluster_arrive_release();
    if (mine) {
        const int b = i / kRows;
        store_output(a, (size_t)b * a.N + n_base + (i - b * kRows), sum);
    }
    if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, tl_cta, 3);
    // No CTA leaves while a peer may still read its shared memory.
    cluster_wait_acquire();
    if (threadIdx.x == 0) {
        tl_stamp(a.tl, a.tl_ctas, tl_cta, 4);
        tl_end(a.tl, a.tl_ctas, tl_cta);
    }
}

template <int B>
cudaError_t launch_b(const GemvArgs &a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.R, (unsigned)a.num_tiles, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.R;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int nattr = 1;
    if (a.chained) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        nattr = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    return cudaLaunchKernelEx(&cfg, gemv_ar_cluster_kernel<B>, a);
}

}  // namespace

cudaError_t launch_gemv_cluster(const GemvArgs &a, cudaStream_t s) {
    if (a.R < 1 || a.R > kMaxClusterRanks || a.num_tiles < 1 || a.num_tiles > 65535) return cudaErrorInvalidValue;
    switch (a.B) {
        case 1: return launch_b<1>(a, s);
        case 2: return launch_b<2>(a, s);
        case 3: return launch_b<3>(a, s);
        case 4: return launch_b<4>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace symm
