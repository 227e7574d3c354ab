// gemv_all_reduce_noalloc: the fused GEMV + one-shot all-reduce for callers
// that cannot allocate device memory.
//
// Who needs it: code that runs under a memory manager owning every device
// allocation (a framework's caching allocator, an inference server with a
// fixed memory budget), or on a serving hot path where cudaMalloc's implicit
// device synchronisation is not acceptable.  Such callers own their inputs and
// outputs but cannot create a handle (symm_alloc allocates the slots, the
// scratch region and the signal pad).
//
// What it uses instead: one fixed array of this library, g_noalloc_scratch
// (kNoAllocBytes = 16 MiB of device memory on every GPU that loads the
// library, held until the process exits).  It holds the fp32 partial of every
// rank ([R][B][N]) followed by one arrival counter per row tile.  Nothing in
// this file calls cudaMalloc, cudaFree or any allocating library routine.
//
// The kernel is a variant of the CUDA-core fused kernel: each CTA computes one
// (row tile, rank) partial with 128-bit streaming loads and FFMA, publishes it
// with an acq_rel ticket on the tile's counter, and the last of the R
// contributors sums the partials in rank order 0..R-1 (fp32), rounds to bf16
// and stores the result into every rank's y.  The counters are cleared with a
// stream-ordered memset at the start of every call.
//
// Sharing rules: every call on a device uses the same array and it keeps the
// previous call's contents; calls that overlap on the GPU (different streams,
// or different host threads without ordering) race on it and give wrong
// results.  Issue the calls on one stream.
//
// Set-up: the first call on each device, with that device current, looks up
// the array's device address with cudaGetSymbolAddress (host code cannot use
// the array's name as a device pointer).  Make that first call before any
// stream capture.  The address is cached per device together with the
// identity of the CUDA context it was looked up in: after the context is torn
// down and created again (cudaDeviceReset, or the primary context released
// and retained anew) the array may have moved, and the next call on that
// device looks the address up again.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "../../include/symm_gemv.h"
#include "internal.h"
#include "protocol.cuh"

namespace symm {

namespace {

constexpr size_t kNoAllocBytes = 16u << 20;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

struct NoAllocArgs {
    const uint8_t *W;       // bf16 [N][Kr], rank r at + r * stride
    const uint8_t *x;       // bf16 [B][Kr], rank r at + r * stride
    uint8_t *y;             // bf16 [B][N],  rank r at + r * stride
    float *partials;        // fp32 [R][B][N] inside the fixed array
    uint32_t *counters;     // [num_tiles] inside the fixed array
    long long stride;
    int R, N, Kr, B;
    int rows_per_tile, num_tiles, kc_cap;
};

template <int B>
struct Shape {
    static constexpr int G = B <= 8 ? 2 : 1;   // rows per warp
    static constexpr int U = B <= 4 ? 4 : 2;   // 16-byte chunks per row in flight per lane
};

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
__global__ void __launch_bounds__(kThreads) gemv_ar_noalloc_kernel(const NoAllocArgs a) {
    constexpr int G = Shape<B>::G;
    constexpr int U = Shape<B>::U;
    extern __shared__ float4 xs4[];   // [B][2][kc_cap]
    __shared__ int s_last;

    const int t = blockIdx.x / a.R;
    const int r = blockIdx.x - t * a.R;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nchunk = a.Kr >> 3;
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

    for (int c0 = 0; c0 < nchunk; c0 += a.kc_cap) {
        const int kc = min(a.kc_cap, nchunk - c0);
        __syncthreads();
        for (int i = threadIdx.x; i < B * kc; i += kThreads) {
            const int b = i / kc;
            const int c = i - b * kc;
            const uint4 v = ld_stream_v4(xr + ((size_t)b * a.Kr + (size_t)(c0 + c) * 8) * 2);
            xs4[(b * 2 + 0) * a.kc_cap + c] = make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
            xs4[(b * 2 + 1) * a.kc_cap + c] = make_float4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w));
        }
        __syncthreads();
        for (int c = lane; c < kc; c += 32 * U) {
            uint4 w[U][G];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int cc = c + 32 * u;
                    w[u][g] = (cc < kc && rowok[g]) ? ld_stream_v4(wrow[g] + c0 + cc) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int cc = c + 32 * u;
                if (cc < kc) {
#pragma unroll
                    for (int b = 0; b < B; ++b) {
                        const float4 lo = xs4[(b * 2 + 0) * a.kc_cap + cc];
                        const float4 hi = xs4[(b * 2 + 1) * a.kc_cap + cc];
#pragma unroll
                        for (int g = 0; g < G; ++g) acc[g][b] = dot8(w[u][g], lo, hi, acc[g][b]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int b = 0; b < B; ++b) {
            float v = acc[g][b];
#pragma unroll
            for (int m = 16; m >= 1; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
            acc[g][b] = v;
        }
    float *P = a.partials + (size_t)r * B * a.N;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int b = 0; b < B; ++b)
            if (rowok[g] && lane == ((g * B + b) & 31)) P[(size_t)b * a.N + row0 + g] = acc[g][b];

    // Publish: partial stores -> fence -> barrier -> acq_rel ticket.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atom_add_acq_rel_gpu(a.counters + t, 1u) == (uint32_t)a.R - 1u;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int n0 = t * a.rows_per_tile;
    const int rows = min(a.rows_per_tile, a.N - n0);
    for (int i = threadIdx.x; i < rows * B; i += kThreads) {
        const int b = i / rows;
        const int n = n0 + (i - b * rows);
        float s = ld_relaxed_gpu_f32(a.partials + (size_t)b * a.N + n);
        for (int q = 1; q < a.R; ++q) s += ld_relaxed_gpu_f32(a.partials + ((size_t)q * B + b) * a.N + n);
        const __nv_bfloat16 v = __float2bfloat16_rn(s);
        for (int q = 0; q < a.R; ++q)
            *reinterpret_cast<__nv_bfloat16 *>(a.y + (long long)q * a.stride + ((size_t)b * a.N + n) * 2) = v;
    }
}

template <int B>
cudaError_t launch_b(const NoAllocArgs &a, cudaStream_t s) {
    const size_t smem = (size_t)B * 2 * (size_t)a.kc_cap * sizeof(float4);
    gemv_ar_noalloc_kernel<B><<<(unsigned)a.num_tiles * (unsigned)a.R, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int B>
int rows_b() { return kWarps * Shape<B>::G; }

int rows_per_tile(int B) {
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

cudaError_t launch(const NoAllocArgs &a, cudaStream_t s) {
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

std::mutex g_setup_mu;
void *g_scratch_ptr[kMaxDevices];
unsigned long long g_scratch_ctx[kMaxDevices];   // context ID the address was looked up in

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// Unique ID of the calling thread's current CUDA context (the driver's
// cuCtxGetId, reached through the runtime's entry-point query); 0 if it
// cannot be had.  Called with a device current, after the runtime has
// initialised it.
unsigned long long current_context_id() {
    static const CtxGetCurrentFn get_current = []() -> CtxGetCurrentFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrentFn>(p);
        return nullptr;
    }();
    static const CtxGetIdFn get_id = []() -> CtxGetIdFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetIdFn>(p);
        return nullptr;
    }();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the fixed array on the current device: looked up once
// per device and context (a context created anew may hold the array
// elsewhere).
int scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    char msg[256];
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "cudaGetDevice: %s", cudaGetErrorString(e));
        return report_error(SYMM_ECUDA, msg);
    }
    if (dev < 0 || dev >= kMaxDevices) return report_error(SYMM_EINVAL, "device ordinal out of range");
    unsigned long long ctx = current_context_id();
    if (ctx == 0) {
        // No context is current on this thread yet: cudaSetDevice on the
        // current device makes the runtime create or bind that device's
        // primary context (it allocates nothing), the one the launch will run
        // in.
        e = cudaSetDevice(dev);
        if (e != cudaSuccess) {
            snprintf(msg, sizeof msg, "initialising the device's context: %s", cudaGetErrorString(e));
            return report_error(SYMM_ECUDA, msg);
        }
        ctx = current_context_id();
    }
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            snprintf(msg, sizeof msg, "cudaGetSymbolAddress of the no-alloc scratch: %s", cudaGetErrorString(e));
            return report_error(SYMM_ECUDA, msg);
        }
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return SYMM_OK;
}

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uint8_t *x = static_cast<const uint8_t *>(a), *y = static_cast<const uint8_t *>(b);
    return na && nb && x < y + nb && y < x + na;
}

}  // namespace

}  // namespace symm

extern "C" int gemv_all_reduce_noalloc(const void *W_r, const void *x_r, void *y, size_t stride, int R, int N, int K,
                                       int B, symm_stream_t stream) {
    using namespace symm;
    char msg[256];
    if (R < 1 || R > SYMM_MAX_RANKS) return report_error(SYMM_EINVAL, "R outside 1..64");
    if (N < 0 || K < 0 || B < 0 || B > SYMM_MAX_BATCH)
        return report_error(SYMM_EINVAL, "need N >= 0, K >= 0 and B in 0..16");
    if (K % R) return report_error(SYMM_EINVAL, "K is not a multiple of R");
    const int Kr = K / R;
    if (Kr % 8) return report_error(SYMM_EINVAL, "K/R is not a multiple of 8");
    if (N == 0 || B == 0) return SYMM_OK;
    const int rows = rows_per_tile(B);
    const int tiles = (N + rows - 1) / rows;
    const size_t part_bytes = up256((size_t)R * B * N * 4);
    const size_t need = part_bytes + (size_t)tiles * 4;
    if (need > kNoAllocBytes) {
        snprintf(msg, sizeof msg,
                 "R*B*N=%lld partials need %zu bytes of working memory; the fixed no-alloc array holds %zu",
                 (long long)R * B * N, need, kNoAllocBytes);
        return report_error(SYMM_ERANGE, msg);
    }
    if (!W_r || !x_r || !y) return report_error(SYMM_EINVAL, "NULL tensor pointer");
    if (!aligned16(W_r) || !aligned16(x_r) || !aligned16(y) || stride % 16)
        return report_error(SYMM_EINVAL, "W_r, x_r, y and stride must be 16-byte aligned");
    const size_t wbytes = (size_t)N * Kr * 2, xbytes = (size_t)B * Kr * 2, ybytes = (size_t)B * N * 2;
    const size_t extent = std::max(wbytes, std::max(xbytes, ybytes));
    if (R > 1 && stride < extent) return report_error(SYMM_EINVAL, "stride is smaller than a rank's tensor");
    // No rank's y may overlap any rank's W_r or x_r.
    for (int d = -(R - 1); d <= R - 1; ++d) {
        const uint8_t *yd = static_cast<const uint8_t *>(y) + (long long)d * (long long)stride;
        if (overlaps(yd, ybytes, W_r, wbytes) || overlaps(yd, ybytes, x_r, xbytes))
            return report_error(SYMM_EINVAL, "an instance of y overlaps an instance of W_r or x_r");
    }
    void *base = nullptr;
    int rc = scratch_address(&base);
    if (rc != SYMM_OK) return rc;

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    NoAllocArgs a;
    a.W = static_cast<const uint8_t *>(W_r);
    a.x = static_cast<const uint8_t *>(x_r);
    a.y = static_cast<uint8_t *>(y);
    a.partials = static_cast<float *>(base);
    a.counters = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(base) + part_bytes);
    a.stride = (long long)stride;
    a.R = R;
    a.N = N;
    a.Kr = Kr;
    a.B = B;
    a.rows_per_tile = rows;
    a.num_tiles = tiles;
    // x staged in passes that keep dynamic shared memory under 46 KB.
    const int nchunk = Kr / 8;
    const int cap = (46 * 1024) / (B * 2 * (int)sizeof(float4));
    a.kc_cap = nchunk < 1 ? 1 : std::min(nchunk, cap);
    cudaError_t e = cudaMemsetAsync(a.counters, 0, (size_t)tiles * 4, s);
    if (e == cudaSuccess) e = launch(a, s);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof msg, "gemv_all_reduce_noalloc: %s", cudaGetErrorString(e));
        return report_error(SYMM_ECUDA, msg);
    }
    return SYMM_OK;
}
