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
//
// The staged variant (one_shot_ar_staged_kernel, selected by option) moves
// the same bytes with the bulk-copy (TMA) engine instead of per-thread loads
// and stores: each CTA owns one contiguous range of the vectors, brings a
// chunk of it from all R slots into shared memory with R bulk loads on one
// mbarrier (three chunks in flight), sums the chunk there, and writes the
// bf16 result back to the R slots with R bulk stores from shared memory.
// It measured 4-14 % slower than the per-thread kernel from 0.5 MB per rank
// up (R = 8; equal below), so the per-thread kernel is the default.
#include <cuda_bf16.h>

#include "internal.h"
#include "protocol.cuh"
#include "sm100.cuh"

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
    chain_entry();
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
        if (a.my_rank >= 0) {   // multi-process handle: this rank's output only
            st_v4(dst + (long long)a.my_rank * a.stride, o);
            continue;
        }
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
            if (a.my_rank < 0 || s == a.my_rank)
                *reinterpret_cast<__nv_bfloat16 *>(a.out + e * 2 + (long long)s * a.stride) = v;
    }
}

// ---------------------------------------------------------------- staged
constexpr int kStagedThreads = 128;
constexpr int kStagedStages = 3;
// Shared memory of one CTA (two fit on an SM): kStagedStages input stages of
// R chunks plus two output chunks.
constexpr int kStagedSmemBudget = 110 * 1024;

__device__ __forceinline__ void bulk_store(void *dst, const void *src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src_smem)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Waits until at most one committed group of bulk stores still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// Waits until every committed group of bulk stores has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Vectors (16 bytes) per chunk and slot for R slots: the largest multiple of 8
// with (kStagedStages * R + 2) chunks inside the budget.
__host__ __device__ __forceinline__ int staged_chunk_vectors(int R) {
    int v = kStagedSmemBudget / (16 * (kStagedStages * R + 2));
    v &= ~7;
    return v < 8 ? 8 : (v > 1024 ? 1024 : v);
}

// CTA c reduces vectors [V c / G, V (c + 1) / G) of the n / 8 whole vectors,
// chunk by chunk; CTA 0 then adds the ragged tail (n % 8 elements) with
// scalar code.
template <int RT>
__global__ void __launch_bounds__(kStagedThreads, 2) one_shot_ar_staged_kernel(const AllReduceArgs a) {
    chain_entry();
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full_bar[kStagedStages];
    __shared__ int abort_sh;
    const int R = RT > 0 ? RT : a.R;
    const int chv = staged_chunk_vectors(R);
    const uint32_t chunk_bytes = (uint32_t)chv * 16u;
    const size_t V = a.n / 8;
    const size_t v0 = V * blockIdx.x / gridDim.x;
    const size_t v1 = V * (blockIdx.x + 1) / gridDim.x;
    const int nch = (int)((v1 - v0 + chv - 1) / chv);
    uint8_t *in_buf = smem;                                              // [stage][R][chunk]
    uint8_t *out_buf = smem + (size_t)kStagedStages * R * chunk_bytes;   // [2][chunk]

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStagedStages; ++i) mbar_init(&full_bar[i], 1);
        abort_sh = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    // Thread 0 issues the R bulk loads of chunk c into stage c % kStagedStages.
    auto issue = [&](int c) {
        const size_t cv0 = v0 + (size_t)c * chv;
        const uint32_t bytes = (uint32_t)min((size_t)chv, v1 - cv0) * 16u;
        uint64_t *bar = &full_bar[c % kStagedStages];
        uint8_t *dst = in_buf + (size_t)(c % kStagedStages) * R * chunk_bytes;
        mbar_arrive_expect_tx(bar, bytes * (uint32_t)R);
        for (int q = 0; q < R; ++q) bulk_load(dst + (size_t)q * chunk_bytes, a.in + (long long)q * a.stride + cv0 * 16, bytes, bar);
    };
    int issued = 0;
    if (threadIdx.x == 0)
        for (; issued < min(kStagedStages, nch); ++issued) issue(issued);

    int c = 0;
    for (; c < nch; ++c) {
        const size_t cv0 = v0 + (size_t)c * chv;
        const int nv = (int)min((size_t)chv, v1 - cv0);
        uint8_t *ob = out_buf + (size_t)(c & 1) * chunk_bytes;
        // The stores of chunk c - 2 have finished reading ob.
        if (threadIdx.x == 0 && c >= 2) bulk_wait_read_1();
        __syncthreads();
        const bool ok = mbar_wait(&full_bar[c % kStagedStages], (uint32_t)(c / kStagedStages) & 1u, &abort_sh);
        if (!ok) abort_sh = 1;
        if (ok) {
            const uint8_t *ib = in_buf + (size_t)(c % kStagedStages) * R * chunk_bytes;
            for (int v = threadIdx.x; v < nv; v += kStagedThreads) {
                float acc[8];
                set8(acc, *reinterpret_cast<const uint4 *>(ib + (size_t)v * 16));
                if (RT > 0) {
#pragma unroll
                    for (int q = 1; q < (RT > 0 ? RT : 1); ++q)
                        add8(acc, *reinterpret_cast<const uint4 *>(ib + (size_t)q * chunk_bytes + (size_t)v * 16));
                } else {
                    for (int q = 1; q < R; ++q)
                        add8(acc, *reinterpret_cast<const uint4 *>(ib + (size_t)q * chunk_bytes + (size_t)v * 16));
                }
                uint4 o;
                o.x = pack2(acc[0], acc[1]);
                o.y = pack2(acc[2], acc[3]);
                o.z = pack2(acc[4], acc[5]);
                o.w = pack2(acc[6], acc[7]);
                *reinterpret_cast<uint4 *>(ob + (size_t)v * 16) = o;
            }
        }
        // The results in ob are read by the bulk stores (the async proxy).
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncthreads();
        if (abort_sh) break;
        if (threadIdx.x == 0) {
            for (int q = 0; q < R; ++q) bulk_store(a.out + (long long)q * a.stride + cv0 * 16, ob, (uint32_t)nv * 16u);
            bulk_commit();
            if (issued < nch) issue(issued++);
        }
    }
    if (threadIdx.x == 0) {
        // Loads still in flight after a give-up land before shared memory is released.
        volatile int never = 0;
        for (int j = c; j < issued; ++j)
            mbar_wait(&full_bar[j % kStagedStages], (uint32_t)(j / kStagedStages) & 1u, &never);
        bulk_wait_all();
    }
    const size_t tail0 = V * 8;
    if (blockIdx.x == 0 && tail0 + threadIdx.x < a.n) {
        const size_t e = tail0 + threadIdx.x;
        float acc = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(a.in + e * 2));
        for (int q = 1; q < R; ++q)
            acc += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(a.in + e * 2 + (long long)q * a.stride));
        const __nv_bfloat16 v = __float2bfloat16_rn(acc);
        for (int q = 0; q < R; ++q) *reinterpret_cast<__nv_bfloat16 *>(a.out + e * 2 + (long long)q * a.stride) = v;
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
    // Chained: wait for the previous kernel before reading; let the next one
    // (phase 2 of the two-shot all-reduce, or the next chained call) be
    // scheduled as this grid's CTAs retire.
    chain_entry();
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

// Plain launch, or (a.chained) a launch as a programmatic dependent of the
// previous kernel on the stream.
template <class Kern, class Args>
cudaError_t launch_maybe_chained(Kern kern, const Args &a, unsigned grid, int threads, size_t smem,
                                 cudaStream_t s) {
    return launch_kernel(kern, dim3(grid), dim3((unsigned)threads), smem, s, a.chained != 0, a);
}

}  // namespace

cudaError_t launch_reduce_scatter(const ReduceScatterArgs &a, cudaStream_t s) {
    const bool vec = a.chunk % 8 == 0;
    const unsigned g = grid_for(vec ? a.n / 8 + (a.n % 8) : a.n, a.ctas_per_sm);
    if (vec) {
        switch (a.R) {
            case 2: return launch_maybe_chained(reduce_scatter_kernel<2, true>, a, g, kThreads, 0, s);
            case 4: return launch_maybe_chained(reduce_scatter_kernel<4, true>, a, g, kThreads, 0, s);
            case 8: return launch_maybe_chained(reduce_scatter_kernel<8, true>, a, g, kThreads, 0, s);
            default: return launch_maybe_chained(reduce_scatter_kernel<0, true>, a, g, kThreads, 0, s);
        }
    }
    return launch_maybe_chained(reduce_scatter_kernel<0, false>, a, g, kThreads, 0, s);
}

cudaError_t launch_all_gather_blocks(const ReduceScatterArgs &a, cudaStream_t s) {
    const bool vec = a.chunk % 8 == 0;
    const unsigned g = grid_for(vec ? a.n / 8 + (a.n % 8) : a.n, a.ctas_per_sm);
    // A programmatic dependent of phase 1: its launch overlaps phase 1's end.
    return vec ? launch_kernel(all_gather_blocks_kernel<true>, dim3(g), dim3(kThreads), 0, s, true, a)
               : launch_kernel(all_gather_blocks_kernel<false>, dim3(g), dim3(kThreads), 0, s, true, a);
}

namespace {

template <int RT>
cudaError_t launch_staged(const AllReduceArgs &a, unsigned grid, cudaStream_t s) {
    auto kern = one_shot_ar_staged_kernel<RT>;
    static std::atomic<unsigned long long> attr_devices{0};
    cudaError_t e = set_smem_once(kern, kStagedSmemBudget, attr_devices);
    if (e != cudaSuccess) return e;
    const int chv = staged_chunk_vectors(a.R);
    const size_t smem = (size_t)(kStagedStages * a.R + 2) * (size_t)chv * 16;
    return launch_maybe_chained(kern, a, grid, kStagedThreads, smem, s);
}

}  // namespace

bool one_shot_uses_staged(const AllReduceArgs &a) { return a.kernel == kArKernelStaged; }

cudaError_t launch_one_shot_all_reduce(const AllReduceArgs &a, cudaStream_t s) {
    const size_t nvec = a.n / 8;
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (one_shot_uses_staged(a)) {
        // Two CTAs per SM (the shared-memory budget), each with a contiguous
        // range of at least 64 vectors.
        size_t g = nvec / 64;
        if (g > (size_t)sms * 2) g = (size_t)sms * 2;
        if (g == 0) g = 1;
        switch (a.R) {
            case 2: return launch_staged<2>(a, (unsigned)g, s);
            case 4: return launch_staged<4>(a, (unsigned)g, s);
            case 8: return launch_staged<8>(a, (unsigned)g, s);
            default: return launch_staged<0>(a, (unsigned)g, s);
        }
    }
    // Enough CTAs for one vector per thread, capped at ctas_per_sm per SM
    // (grid-stride beyond that); at least one CTA for the ragged tail.
    size_t blocks = (nvec + kThreads - 1) / kThreads;
    const size_t cap = (size_t)sms * (size_t)(a.ctas_per_sm > 0 ? a.ctas_per_sm : kDefaultCtasPerSm);
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    switch (a.R) {
        case 1: return launch_maybe_chained(one_shot_ar_kernel<1>, a, (unsigned)blocks, kThreads, 0, s);
        case 2: return launch_maybe_chained(one_shot_ar_kernel<2>, a, (unsigned)blocks, kThreads, 0, s);
        case 4: return launch_maybe_chained(one_shot_ar_kernel<4>, a, (unsigned)blocks, kThreads, 0, s);
        case 8: return launch_maybe_chained(one_shot_ar_kernel<8>, a, (unsigned)blocks, kThreads, 0, s);
        default: return launch_maybe_chained(one_shot_ar_kernel<0>, a, (unsigned)blocks, kThreads, 0, s);
    }
}

}  // namespace symm
