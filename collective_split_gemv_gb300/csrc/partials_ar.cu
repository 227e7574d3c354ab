// The second kernel of the unfused form of the row-parallel layer
// (SYMM_OPT_UNFUSED): an all-reduce of the fp32 partials the GEMV kernel
// left in every rank's scratch slot.
//
// y_s[e] = bf16_rne( P_(0,0)[e] + P_(0,1)[e] + ... + P_(R-1,S-1)[e] ) for
// every slot s, where P_(q,k) is rank q's partial of K split k ([B][N] fp32,
// e = b * N + n).  The contributors are summed one after another in that
// order in fp32 -- the order the fused kernel's tile reducer uses -- so both
// forms give the same bits.  The fused GEMV + AllReduce of "Overlapping
// Collective Communication with Dependent Computation ..." (Abstract) is
// measured against this form: the same GEMV, then a separate all-reduce of
// its partials.
//
// Each thread takes four consecutive outputs (16-byte loads of every
// contributor, issued back to back) and stores them as one 8-byte bf16
// vector into each slot; a ragged tail is done element by element.  The
// kernel is launched as a programmatic dependent of the GEMV: its CTAs may be
// scheduled while the GEMV drains, and wait for it (griddepcontrol.wait)
// before reading a partial.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "protocol.cuh"

namespace symm {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxContrib = 16;   // contributors loaded before the first add

__global__ void __launch_bounds__(kThreads) partials_ar_kernel(const PartialsArArgs a) {
    chain_entry();
    const int C = a.R * a.splits;
    const size_t total = (size_t)a.B * (size_t)a.N;
    const size_t nvec = a.vec ? total / 4 : 0;
    const size_t step = (size_t)gridDim.x * kThreads;
    for (size_t i = (size_t)blockIdx.x * kThreads + threadIdx.x; i < nvec; i += step) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < C; j0 += kMaxContrib) {
            const int m = min(kMaxContrib, C - j0);
            float4 v[kMaxContrib];
#pragma unroll
            for (int u = 0; u < kMaxContrib; ++u) {
                if (u < m) {
                    const int j = j0 + u;
                    const int q = j / a.splits;
                    const uint8_t *base = a.scratch + (long long)q * a.stride +
                                          (long long)(j - q * a.splits) * a.partial_stride;
                    v[u] = __ldcg(reinterpret_cast<const float4 *>(base) + i);
                }
            }
#pragma unroll
            for (int u = 0; u < kMaxContrib; ++u) {
                if (u < m) {
                    if (j0 + u == 0) {
                        acc = v[u];
                    } else {
                        acc.x += v[u].x;
                        acc.y += v[u].y;
                        acc.z += v[u].z;
                        acc.w += v[u].w;
                    }
                }
            }
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t *>(&lo);
        o.y = *reinterpret_cast<const uint32_t *>(&hi);
        for (int q = 0; q < a.R; ++q)
            *reinterpret_cast<uint2 *>(a.y + (long long)q * a.stride + i * 8) = o;
    }
    // Elements past the last whole vector (all of them when not vectorised).
    for (size_t e = nvec * 4 + (size_t)blockIdx.x * kThreads + threadIdx.x; e < total; e += step) {
        float acc = 0.f;
        for (int j = 0; j < C; ++j) {
            const int q = j / a.splits;
            const float *base = reinterpret_cast<const float *>(a.scratch + (long long)q * a.stride +
                                                                (long long)(j - q * a.splits) * a.partial_stride);
            const float v = __ldcg(base + e);
            acc = j == 0 ? v : acc + v;
        }
        const __nv_bfloat16 h = __float2bfloat16_rn(acc);
        for (int q = 0; q < a.R; ++q)
            *reinterpret_cast<__nv_bfloat16 *>(a.y + (long long)q * a.stride + e * 2) = h;
    }
}

}  // namespace

cudaError_t launch_partials_ar(const PartialsArArgs &a, cudaStream_t s) {
    const size_t total = (size_t)a.B * (size_t)a.N;
    const size_t work = a.vec ? total / 4 + total % 4 : total;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t cap = (size_t)sms * 8;
    const unsigned grid = (unsigned)std::max<size_t>(1, std::min(cap, (work + kThreads - 1) / kThreads));
    return launch_kernel(partials_ar_kernel, dim3(grid), dim3(kThreads), 0, s, a.chained != 0, a);
}

}  // namespace symm
