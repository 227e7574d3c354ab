// Fused row-parallel GEMV + one-shot all-reduce on the CUDA cores (FFMA).
//
// Grid: one CTA per (row tile t, rank r), blockIdx = t * R + r, so the R
// contributors of a tile are adjacent in launch order and run close together:
// their partials are still in L2 when the last one reduces them (the
// communication-aware workgroup ordering of the fused GEMV + AllReduce in
// "Overlapping Collective Communication with Dependent Computation ...",
// Abstract).
//
// Per CTA (256 threads = 8 warps; warp w owns G consecutive rows):
//  - x_r is widened to fp32 once into shared memory, laid out as
//    [b][half][chunk] float4 so that lane-consecutive chunks are
//    bank-conflict free;
//  - each lane streams 16-byte chunks of its rows of W_r
//    (ld.global.nc.L1::no_allocate.v4), U chunks per row in flight, lane l
//    taking chunks l, l+32, l+64, ...; the first batch is issued before x is
//    staged so that HBM latency overlaps the staging;
//  - fp32 FMA in ascending order within a chunk, chunks in the lane's order,
//    then a fixed xor-shuffle tree across the warp;
//  - the fp32 partial goes to the rank's scratch slot and the CTA enters the
//    publish / last-arriver protocol (protocol.cuh).
//
// Timeline slots (timeline build only, timeline.cuh): 0 entry, 1 x staged
// (first pass), 2 dot products done; 3-8 are the protocol's.
#include <cuda_bf16.h>

#include "internal.h"
#include "protocol.cuh"

namespace symm {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <int B>
struct FfmaShape;
// G rows per warp, U chunks (16 B) per row in flight per lane.
template <> struct FfmaShape<1> { static constexpr int G = 2, U = 8; };
template <> struct FfmaShape<2> { static constexpr int G = 2, U = 4; };
template <> struct FfmaShape<3> { static constexpr int G = 2, U = 4; };
template <> struct FfmaShape<4> { static constexpr int G = 2, U = 4; };
template <int B> struct FfmaShape { static constexpr int G = (B <= 8) ? 2 : 1, U = 2; };

__device__ __forceinline__ float dot8(const uint4 &w, const float4 &lo, const float4 &hi, float acc) {
    acc = fmaf(bf16lo(w.x), lo.x, acc);
    acc = fmaf(bf16hi(w.x), lo.y, acc);
    acc = fmaf(bf16lo(w.y), lo.z, acc);
    acc = fmaf(bf16hi(w.y), lo.w, acc);
    acc = fmaf(bf16lo(w.z), hi.x, acc);
    acc = fmaf(bf16hi(w.z), hi.y, acc);
    acc = fmaf(bf16lo(w.w), hi.z, acc);
    acc = fmaf(bf16hi(w.w), hi.w, acc);
    return acc;
}

template <int B>
__global__ void __launch_bounds__(kThreads, 1) gemv_ar_ffma_kernel(const GemvArgs a) {
    if (threadIdx.x == 0) {
        tl_begin();
        tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 0);
    }
    chain_entry();
    // Thread 0 publishes; its read of the launch epoch overlaps the streaming.
    const uint32_t epoch = threadIdx.x == 0 ? read_launch_epoch(a) : 0u;
    constexpr int G = FfmaShape<B>::G;
    constexpr int U = FfmaShape<B>::U;
    extern __shared__ float4 xs4[];   // [B][2][kc_cap]

    const int bid = a.reverse_order ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    // CTA (tile, rank); a multi-process handle's launch covers its own rank.
    const int t = a.my_rank >= 0 ? bid : bid / a.R;
    const int r = a.my_rank >= 0 ? a.my_rank : bid - t * a.R;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nchunk = a.Kr >> 3;
    const int kc_cap = a.kc_cap;

    const int row_in_tile = warp * G;
    const int row0 = t * a.rows_per_tile + row_in_tile;
    const uint8_t *Wr = a.W + (long long)r * a.stride;
    const uint8_t *xr = a.x + (long long)r * a.stride;

    const uint4 *wrow[G];
    bool rowok[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const int n = row0 + g;
        rowok[g] = (row_in_tile + g < a.rows_per_tile) && (n < a.N);
        wrow[g] = reinterpret_cast<const uint4 *>(Wr + (size_t)(rowok[g] ? n : 0) * a.Kr * 2);
    }

    float acc[G][B];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int b = 0; b < B; ++b) acc[g][b] = 0.f;

    uint4 w[U][G];
    // First batch of W for pass 0, issued before x is staged.
    {
        const int kc = min(kc_cap, nchunk);
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int cc = lane + 32 * u;
                w[u][g] = (cc < kc && rowok[g]) ? ld_stream_v4(wrow[g] + cc) : make_uint4(0, 0, 0, 0);
            }
    }

    for (int c0 = 0; c0 < nchunk; c0 += kc_cap) {
        const int kc = min(kc_cap, nchunk - c0);
        if (c0 > 0) __syncthreads();   // previous pass finished reading xs4
        for (int i = threadIdx.x; i < B * kc; i += kThreads) {
            const int b = i / kc;
            const int c = i - b * kc;
            const uint4 v = ld_stream_v4(xr + ((size_t)b * a.Kr + (size_t)(c0 + c) * 8) * 2);
            xs4[(b * 2 + 0) * kc_cap + c] = make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
            xs4[(b * 2 + 1) * kc_cap + c] = make_float4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w));
        }
        __syncthreads();
        if (c0 == 0 && threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 1);

        for (int c = lane; c < kc; c += 32 * U) {
            if (c != lane || c0 > 0) {
#pragma unroll
                for (int u = 0; u < U; ++u)
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const int cc = c + 32 * u;
                        w[u][g] = (cc < kc && rowok[g]) ? ld_stream_v4(wrow[g] + c0 + cc)
                                                        : make_uint4(0, 0, 0, 0);
                    }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cc = c + 32 * u;
                if (cc < kc) {
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        const float4 lo = xs4[(b * 2 + 0) * kc_cap + cc];
                        const float4 hi = xs4[(b * 2 + 1) * kc_cap + cc];
#pragma unroll
                        for (int g = 0; g < G; ++g) acc[g][b] = dot8(w[u][g], lo, hi, acc[g][b]);
                    }
                }
            }
        }
    }

    // Fixed butterfly across the warp; every lane ends with every sum.
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float v = acc[g][b];
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
            acc[g][b] = v;
        }
    if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, blockIdx.x, 2);

    float *P = reinterpret_cast<float *>(a.scratch + (long long)r * a.stride);
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int b = 0; b < B; ++b)
            if (rowok[g] && lane == ((g * B + b) & 31)) P[(size_t)b * a.N + row0 + g] = acc[g][b];

    publish_and_reduce(a, epoch, t, r, 0);
    if (threadIdx.x == 0) tl_end(a.tl, a.tl_ctas, blockIdx.x);
}

template <int B>
cudaError_t launch_b(const GemvArgs &a, cudaStream_t s) {
    const size_t smem = ffma_smem_bytes(B, a.kc_cap);
    auto kern = gemv_ar_ffma_kernel<B>;
    if (smem > 46 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const unsigned grid = (unsigned)a.num_tiles * (a.my_rank >= 0 ? 1u : (unsigned)a.R);
    return launch_kernel(kern, dim3(grid), dim3(kThreads), smem, s, a.chained != 0, a);
}

template <int B>
int rows_b() { return kWarps * FfmaShape<B>::G; }

}  // namespace

int ffma_rows_per_tile(int B) {
    switch (B) {
        case 1: return rows_b<1>();   case 2: return rows_b<2>();   case 3: return rows_b<3>();
        case 4: return rows_b<4>();   case 5: return rows_b<5>();   case 6: return rows_b<6>();
        case 7: return rows_b<7>();   case 8: return rows_b<8>();   case 9: return rows_b<9>();
        case 10: return rows_b<10>(); case 11: return rows_b<11>(); case 12: return rows_b<12>();
        case 13: return rows_b<13>(); case 14: return rows_b<14>(); case 15: return rows_b<15>();
        case 16: return rows_b<16>();
        default: return 0;
    }
}

size_t ffma_smem_bytes(int B, int kc_cap) { return (size_t)B * 2 * (size_t)kc_cap * sizeof(float4); }

// Chunks of x staged per pass: all of K/R when B * K/R * 4 bytes fit in
// 46 KB (the default 48 KB limit also covers the kernel's static shared
// memory), otherwise passes of that size.
int ffma_kc_cap(int B, int Kr) {
    const int nchunk = Kr / 8;
    const int cap = (46 * 1024) / (B * 2 * (int)sizeof(float4));
    return nchunk < 1 ? 1 : (nchunk < cap ? nchunk : cap);
}

cudaError_t launch_gemv_ffma(const GemvArgs &a, cudaStream_t s) {
    switch (a.B) {
        case 1: return launch_b<1>(a, s);   case 2: return launch_b<2>(a, s);
        case 3: return launch_b<3>(a, s);   case 4: return launch_b<4>(a, s);
        case 5: return launch_b<5>(a, s);   case 6: return launch_b<6>(a, s);
        case 7: return launch_b<7>(a, s);   case 8: return launch_b<8>(a, s);
        case 9: return launch_b<9>(a, s);   case 10: return launch_b<10>(a, s);
        case 11: return launch_b<11>(a, s); case 12: return launch_b<12>(a, s);
        case 13: return launch_b<13>(a, s); case 14: return launch_b<14>(a, s);
        case 15: return launch_b<15>(a, s); case 16: return launch_b<16>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace symm
