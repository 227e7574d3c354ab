// One-shot all-reduce over R symmetric slots.
//
// out_s[i] = bf16_rne( in_0[i] + in_1[i] + ... + in_{R-1}[i] ) (fp32, rank
// order) for every slot s.  This is the one-shot algorithm of the "PyTorch
// Symmetric Memory" talk (outer loop over data blocks, inner loop over ranks,
// local or remote loads alike, reduce locally) with the accumulation the
// symmetric-memory docs give for bf16 ("higher-precision reduction": fp32).
// Because the R ranks are slots of one GPU, one thread computes the sum once
// and stores it into all R output slots instead of R GPUs each computing it.
//
// The start/end signal-pad barriers of the symmetric-memory kernel exist to
// order a rank's reads after its peers' writes and to protect buffer reuse
// across ranks.  On one GPU with one stream per handle, stream order gives
// both: the inputs were produced by earlier work on the stream, and the next
// launch starts after this one ends.
//
// Each thread owns one 16-byte vector (8 elements) at a time and reads it in
// every slot before writing it anywhere, so in == out is safe.  The loads of
// the R slots are issued back to back (R x 16 B in flight per thread).
#include <cuda_bf16.h>

#include "internal.h"
#include "protocol.cuh"

namespace symm {

namespace {

constexpr int kThreads = 256;
// Grid cap per SM.  Twice the 8 CTAs an SM holds at once: the hardware then
// starts a fresh CTA wherever one retires, which measured faster (R=8, 8 MiB
// per rank: one-shot 26.7 -> 25.6 us, two-shot 29.0 -> 27.3 us) than eight
// resident CTAs walking a grid-stride loop of uneven length.
constexpr int kDefaultCtasPerSm = 16;

__device__ __forceinline__ void add8(float (&acc)[8], const uint4 &v) {
    acc[0] += bf16lo(v.x); acc[1] += bf16hi(v.x);
    acc[2] += bf16lo(v.y); acc[3] += bf16hi(v.y);
    acc[4] += bf16lo(v.z); acc[5] += bf16hi(v.z);
    acc[6] += bf16lo(v.w); acc[7] += bf16hi(v.w);
}

__device__ __forceinline__ void set8(float (&acc)[8], const uint4 &v) {
    acc[0] = bf16lo(v.x); acc[1] = bf16hi(v.x);
    acc[2] = bf16lo(v.y); acc[3] = bf16hi(v.y);
    acc[4] = bf16lo(v.z); acc[5] = bf16hi(v.z);
    acc[6] = bf16lo(v.w); acc[7] = bf16hi(v.w);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);   // .x = lo (low half)
    return *reinterpret_cast<const uint32_t *>(&p);
}

// RT > 0: rank count known at compile time; RT == 0: runtime a.R.
template <int RT>
__global__ void __launch_bounds__(kThreads) one_shot_ar_kernel(const AllReduceArgs a) {
    const int R = RT > 0 ? RT : a.R;
    const size_t nvec = a.n / 8;
    const size_t step = (size_t)gridDim.x * kThreads;
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < nvec; i += step) {
        const uint8_t *src = a.in + i * 16;
        float acc[8];
        if (RT > 0) {
            uint4 v[RT > 0 ? RT : 1];
#pragma unroll
            for (int q = 0; q < (RT > 0 ? RT : 1); ++q) v[q] = ld_v4(src + (long long)q * a.stride);
            acc[0] = bf16lo(v[0].x); acc[1] = bf16hi(v[0].x);
            acc[2] = bf16lo(v[0].y); acc[3] = bf16hi(v[0].y);
            acc[4] = bf16lo(v[0].z); acc[5] = bf16hi(v[0].z);
            acc[6] = bf16lo(v[0].w); acc[7] = bf16hi(v[0].w);
#pragma unroll
            for (int q = 1; q < (RT > 0 ? RT : 1); ++q) add8(acc, v[q]);
        } else {
            const uint4 v0 = ld_v4(src);
            acc[0] = bf16lo(v0.x); acc[1] = bf16hi(v0.x);
            acc[2] = bf16lo(v0.y); acc[3] = bf16hi(v0.y);
            acc[4] = bf16lo(v0.z); acc[5] = bf16hi(v0.z);
            acc[6] = bf16lo(v0.w); acc[7] = bf16hi(v0.w);
            int q = 1;
            for (; q + 4 <= R; q += 4) {
                uint4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = ld_v4(src + (long long)(q + j) * a.stride);
#pragma unroll
                for (int j = 0; j < 4; ++j) add8(acc, v[j]);
            }
            for (; q < R; ++q) add8(acc, ld_v4(src + (long long)q * a.stride));
        }
        uint4 o;
        o.x = pack2(acc[0], acc[1]);
        o.y = pack2(acc[2], acc[3]);
        o.z = pack2(acc[4], acc[5]);
        o.w = pack2(acc[6], acc[7]);
        uint8_t *dst = a.out + i * 16;
#pragma unroll 8
        for (int s = 0; s < R; ++s) st_v4(dst + (long long)s * a.stride, o);
    }
    // Ragged tail (n % 8 elements): scalar, handled by the first threads of CTA 0.
    const size_t tail0 = nvec * 8;
    if (blockIdx.x == 0 && tail0 + threadIdx.x < a.n) {
        const size_t e = tail0 + threadIdx.x;
        const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(a.in) + e;
        float acc = __bfloat162float(*src);
        for (int q = 1; q < R; ++q)
            acc += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(
                reinterpret_cast<const uint8_t *>(src) + (long long)q * a.stride));
        const __nv_bfloat16 v = __float2bfloat16_rn(acc);
        for (int s = 0; s < R; ++s)
            *reinterpret_cast<__nv_bfloat16 *>(a.out + e * 2 + (long long)s * a.stride) = v;
    }
}

// Reduce-scatter (and phase 1 of the two-shot all-reduce): element i belongs
// to owner s = i / chunk, whose slot alone receives the sum of the R inputs
// (fp32, rank order 0..R-1, RNE to bf16).  kVec: chunk % 8 == 0, so a
// 16-byte vector never straddles two owners; otherwise one element per
// thread.  A thread reads its element(s) in every slot before its one store,
// so in == out is safe for the two-shot layout (shift = 1).
template <int RT, bool kVec>
__global__ void __launch_bounds__(kThreads) reduce_scatter_kernel(const ReduceScatterArgs a) {
    // As phase 1 of the two-shot all-reduce, let phase 2 (launched as a
    // programmatic dependent; it waits for this grid before touching memory)
    // be scheduled as this grid's CTAs retire.
    if (a.shift) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int R = RT > 0 ? RT : a.R;
    const size_t step = (size_t)gridDim.x * kThreads;
    const size_t first = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (kVec) {
        const size_t nvec = a.n / 8;
        for (size_t v = first; v < nvec; v += step) {
            const size_t i = v * 8;
            const size_t s = i / a.chunk;
            const uint8_t *src = a.in + i * 2;
            float acc[8];
            if (RT > 0) {
                uint4 x[RT > 0 ? RT : 1];
#pragma unroll
                for (int q = 0; q < (RT > 0 ? RT : 1); ++q) x[q] = ld_v4(src + (long long)q * a.stride);
                set8(acc, x[0]);
#pragma unroll
                for (int q = 1; q < (RT > 0 ? RT : 1); ++q) add8(acc, x[q]);
            } else {
                set8(acc, ld_v4(src));
                for (int q = 1; q < R; ++q) add8(acc, ld_v4(src + (long long)q * a.stride));
            }
            uint4 o;
            o.x = pack2(acc[0], acc[1]);
            o.y = pack2(acc[2], acc[3]);
            o.z = pack2(acc[4], acc[5]);
            o.w = pack2(acc[6], acc[7]);
            const size_t j = i - s * a.chunk + (a.shift ? s * a.chunk : 0);
            st_v4(a.out + (long long)s * a.stride + j * 2, o);
        }
    }
    // Elements not covered by vectors: all of them (scalar layout) or the
    // ragged tail n % 8.
    const size_t e0 = kVec ? (a.n / 8) * 8 : 0;
    for (size_t i = e0 + first; i < a.n; i += step) {
        const size_t s = i / a.chunk;
        float acc = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(a.in + i * 2));
        for (int q = 1; q < R; ++q)
            acc += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(a.in + i * 2 + (long long)q * a.stride));
        const size_t j = i - s * a.chunk + (a.shift ? s * a.chunk : 0);
        *reinterpret_cast<__nv_bfloat16 *>(a.out + (long long)s * a.stride + j * 2) = __float2bfloat16_rn(acc);
    }
}

// Phase 2 of the two-shot all-reduce: every slot q copies each owner's block
// from the owner's slot (out_q[i] = out_s[i], s = i / chunk, q != s).  The
// owner's values were stored by phase 1, an earlier launch on the stream.
template <bool kVec>
__global__ void __launch_bounds__(kThreads) all_gather_blocks_kernel(const ReduceScatterArgs a) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // phase 1 has completed and is visible
    const size_t step = (size_t)gridDim.x * kThreads;
    const size_t first = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (kVec) {
        const size_t nvec = a.n / 8;
        for (size_t v = first; v < nvec; v += step) {
            const size_t i = v * 8;
            const int s = (int)(i / a.chunk);
            const uint4 val = ld_v4(a.out + (long long)s * a.stride + i * 2);
            for (int q = 0; q < a.R; ++q)
                if (q != s) st_v4(a.out + (long long)q * a.stride + i * 2, val);
        }
    }
    const size_t e0 = kVec ? (a.n / 8) * 8 : 0;
    for (size_t i = e0 + first; i < a.n; i += step) {
        const int s = (int)(i / a.chunk);
        const uint16_t val = *reinterpret_cast<const uint16_t *>(a.out + (long long)s * a.stride + i * 2);
        for (int q = 0; q < a.R; ++q)
            if (q != s) *reinterpret_cast<uint16_t *>(a.out + (long long)q * a.stride + i * 2) = val;
    }
}

unsigned grid_for(size_t work_items, int ctas_per_sm) {
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    size_t blocks = (work_items + kThreads - 1) / kThreads;
    const size_t cap = (size_t)sms * (size_t)(ctas_per_sm > 0 ? ctas_per_sm : kDefaultCtasPerSm);
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    return (unsigned)blocks;
}

}  // namespace

cudaError_t launch_reduce_scatter(const ReduceScatterArgs &a, cudaStream_t s) {
    const bool vec = a.chunk % 8 == 0;
    const unsigned g = grid_for(vec ? a.n / 8 + (a.n % 8) : a.n, a.ctas_per_sm);
    if (vec) {
        switch (a.R) {
            case 2: reduce_scatter_kernel<2, true><<<g, kThreads, 0, s>>>(a); break;
            case 4: reduce_scatter_kernel<4, true><<<g, kThreads, 0, s>>>(a); break;
            case 8: reduce_scatter_kernel<8, true><<<g, kThreads, 0, s>>>(a); break;
            default: reduce_scatter_kernel<0, true><<<g, kThreads, 0, s>>>(a); break;
        }
    } else {
        reduce_scatter_kernel<0, false><<<g, kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

cudaError_t launch_all_gather_blocks(const ReduceScatterArgs &a, cudaStream_t s) {
    const bool vec = a.chunk % 8 == 0;
    const unsigned g = grid_for(vec ? a.n / 8 + (a.n % 8) : a.n, a.ctas_per_sm);
    // A programmatic dependent of phase 1: its launch overlaps phase 1's end.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return vec ? cudaLaunchKernelEx(&cfg, all_gather_blocks_kernel<true>, a)
               : cudaLaunchKernelEx(&cfg, all_gather_blocks_kernel<false>, a);
}

cudaError_t launch_one_shot_all_reduce(const AllReduceArgs &a, cudaStream_t s) {
    const size_t nvec = a.n / 8;
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    // Enough CTAs for one vector per thread, capped at ctas_per_sm per SM
    // (grid-stride beyond that); at least one CTA for the ragged tail.
    size_t blocks = (nvec + kThreads - 1) / kThreads;
    const size_t cap = (size_t)sms * (size_t)(a.ctas_per_sm > 0 ? a.ctas_per_sm : kDefaultCtasPerSm);
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    switch (a.R) {
        case 1: one_shot_ar_kernel<1><<<(unsigned)blocks, kThreads, 0, s>>>(a); break;
        case 2: one_shot_ar_kernel<2><<<(unsigned)blocks, kThreads, 0, s>>>(a); break;
        case 4: one_shot_ar_kernel<4><<<(unsigned)blocks, kThreads, 0, s>>>(a); break;
        case 8: one_shot_ar_kernel<8><<<(unsigned)blocks, kThreads, 0, s>>>(a); break;
        default: one_shot_ar_kernel<0><<<(unsigned)blocks, kThreads, 0, s>>>(a); break;
    }
    return cudaGetLastError();
}

}  // namespace symm
