// RMS normalisation of rows over the symmetric slots, one thread-block
// cluster per row.
//
// Two sources of the pre-normalisation row z:
//   kind 0  the all-reduce + bias kernel of the "PyTorch Symmetric Memory"
//           talk (fused-kernel segment: reduce, add the bias in the same
//           element-wise loop, then RMS-normalise, all in one launch):
//           z[h] = (sum_r in_r[h]) + bias[h], fp32, ranks in order 0..R-1;
//   kind 1  the fused GEMV's tile reducers, which already stored
//           z = sum + bias in fp32 (the second stage of the fused layer's
//           bias + RMSNorm epilogue; launched as a programmatic dependent of
//           the GEMV so that its launch overlaps the GEMV's tail).
// Then y[h] = z[h] / sqrt(mean_h z^2 + eps) * gamma[h], rounded to bf16 and
// stored into every slot's out.
//
// A row of H elements is split over the C CTAs of a cluster (C <= 8, grid
// (C, rows)); every thread keeps its z values in registers.  The sum of
// squares is reduced in a fixed tree (thread -> warp shuffle -> CTA in warp
// order -> cluster in CTA-rank order: each CTA pushes its sum into every
// CTA's shared memory, then a cluster barrier), so every CTA derives the
// same scale and the result does not depend on timing.  The cluster barriers
// (one split into an arrive at entry and a wait before the first remote
// store, so that no CTA writes into a CTA that has not started; one after the
// stores) are hardware barriers among CTAs that are co-scheduled by
// construction: no CTA spins on memory, and none touches another's shared
// memory after the last barrier, so any may exit.
//
// Timeline slots (timeline build only, timeline.cuh; row = blockIdx.y * C +
// cluster rank): 0 entry, 1 gamma / bias loads issued, 2 dependency wait
// passed, 3 row loaded and squared, 4 first cluster barrier passed, 5 second
// cluster barrier passed, 6 stores issued.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "internal.h"
#include "protocol.cuh"
#include "timeline.cuh"

namespace symm {

namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 8;
constexpr int kMaxVecPerThread = 8;

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Store v at the same shared-memory variable of CTA `cta` of the cluster.
__device__ __forceinline__ void st_cluster_f32(float *local, uint32_t cta, float v) {
    const uint32_t addr = (uint32_t)__cvta_generic_to_shared(local);
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(addr), "r"(cta));
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    f[0] = bf16lo(v.x); f[1] = bf16hi(v.x);
    f[2] = bf16lo(v.y); f[3] = bf16hi(v.y);
    f[4] = bf16lo(v.z); f[5] = bf16hi(v.z);
    f[6] = bf16lo(v.w); f[7] = bf16hi(v.w);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    const __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&p);
}

// kV: 16-byte vectors (8 elements) per thread; chunk: vectors per CTA.
template <int kSrc, int kV>
__global__ void __launch_bounds__(kThreads) rmsnorm_rows_kernel(const RmsNormArgs a, int chunk) {
    __shared__ float s_warp[kWarps];
    __shared__ float s_part[kMaxCluster];   // s_part[c]: CTA c's sum of squares

    uint32_t crank;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(crank));
    uint32_t csize;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(csize));
    const int row = blockIdx.y;
    const int tl_cta = (int)(blockIdx.y * gridDim.x + blockIdx.x);
    if (threadIdx.x == 0) {
        tl_begin();
        tl_stamp(a.tl, a.tl_ctas, tl_cta, 0);
    }
    const int H8 = a.H / 8;
    const int v0 = (int)crank * chunk;
    const int v1 = min(H8, v0 + chunk);

    // A standalone chained call lets the next kernel on the stream be
    // scheduled as this one's clusters retire.
    if (a.release_next) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Distributed shared memory may be written only once every CTA of the
    // cluster runs: arrive now, wait just before the first remote store (the
    // row loads in between hide the wait).
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    // gamma and bias do not depend on the kernel this one may follow: load
    // them first, so their latency hides under the wait and the row loads.
    uint4 gv[kV], bv[kV];
#pragma unroll
    for (int j = 0; j < kV; ++j) {
        const int v = v0 + (int)threadIdx.x + j * kThreads;
        gv[j] = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);   // bf16 1.0 pairs
        bv[j] = make_uint4(0u, 0u, 0u, 0u);
        if (v < v1) {
            if (a.gamma) gv[j] = ld_v4(a.gamma + (size_t)v * 16);
            if (kSrc == 0 && a.bias) bv[j] = ld_v4(a.bias + (size_t)v * 16);
        }
    }
    if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, tl_cta, 1);
    if (a.wait_prior) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, tl_cta, 2);

    float z[kV][8];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kV; ++j) {
        const int v = v0 + (int)threadIdx.x + j * kThreads;
        if (v < v1) {
            const size_t e = (size_t)row * a.H + (size_t)v * 8;
            if (kSrc == 0) {
                const uint8_t *src = a.in + e * 2;
                for (int q0 = 0; q0 < a.R; q0 += 8) {   // up to eight ranks' loads in flight, then add in order
                    const int m = min(8, a.R - q0);
                    uint4 x[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (u < m) x[u] = ld_v4(src + (long long)(q0 + u) * a.stride);
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        if (u < m) {
                            float f[8];
                            unpack8(x[u], f);
#pragma unroll
                            for (int k = 0; k < 8; ++k) z[j][k] = (q0 + u == 0) ? f[k] : z[j][k] + f[k];
                        }
                    }
                }
                if (a.bias) {
                    float f[8];
                    unpack8(bv[j], f);
#pragma unroll
                    for (int k = 0; k < 8; ++k) z[j][k] += f[k];
                }
            } else {
                const float4 lo = __ldcg(reinterpret_cast<const float4 *>(a.z + e));
                const float4 hi = __ldcg(reinterpret_cast<const float4 *>(a.z + e) + 1);
                z[j][0] = lo.x; z[j][1] = lo.y; z[j][2] = lo.z; z[j][3] = lo.w;
                z[j][4] = hi.x; z[j][5] = hi.y; z[j][6] = hi.z; z[j][7] = hi.w;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) ss = fmaf(z[j][k], z[j][k], ss);
        }
    }
    // Fixed-shape reduction of the sum of squares.
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, tl_cta, 3);
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
    if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, tl_cta, 4);
    // Thread c < C of warp 0 pushes this CTA's sum (warps in order) into
    // s_part[crank] of CTA c; one cluster barrier (release / acquire) makes
    // all pushes visible, and no CTA touches another's memory after it.
    if (threadIdx.x < csize) {
        float t = s_warp[0];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) t += s_warp[w];
        st_cluster_f32(&s_part[crank], threadIdx.x, t);
    }
    cluster_sync_all();
    if (threadIdx.x == 0) tl_stamp(a.tl, a.tl_ctas, tl_cta, 5);
    float tot = s_part[0];
    for (uint32_t c = 1; c < csize; ++c) tot += s_part[c];   // CTA-rank order: the same in every CTA
    const float scale = 1.0f / sqrtf(tot / (float)a.H + a.eps);

#pragma unroll
    for (int j = 0; j < kV; ++j) {
        const int v = v0 + (int)threadIdx.x + j * kThreads;
        if (v < v1) {
            float g[8];
            unpack8(gv[j], g);
            float y[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) y[k] = z[j][k] * scale * g[k];
            uint4 o;
            o.x = pack2(y[0], y[1]);
            o.y = pack2(y[2], y[3]);
            o.z = pack2(y[4], y[5]);
            o.w = pack2(y[6], y[7]);
            uint8_t *dst = a.out + ((size_t)row * a.H + (size_t)v * 8) * 2;
            for (int q = 0; q < a.R; ++q) st_v4(dst + (long long)q * a.stride, o);
        }
    }
    if (threadIdx.x == 0) {
        tl_stamp(a.tl, a.tl_ctas, tl_cta, 6);
        tl_end(a.tl, a.tl_ctas, tl_cta);
    }
}

template <int kSrc, int kV>
cudaError_t launch_kv(const RmsNormArgs &a, int C, int chunk, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C, (unsigned)a.rows, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int nattr = 1;
    if (a.wait_prior) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        nattr = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = nattr;
    return cudaLaunchKernelEx(&cfg, rmsnorm_rows_kernel<kSrc, kV>, a, chunk);
}

template <int kSrc>
cudaError_t launch_src(const RmsNormArgs &a, cudaStream_t s) {
    const int H8 = a.H / 8;
    const int C = std::max(1, std::min(kMaxCluster, (H8 + kThreads - 1) / kThreads));
    const int chunk = (H8 + C - 1) / C;
    const int need = (chunk + kThreads - 1) / kThreads;
    if (need <= 1) return launch_kv<kSrc, 1>(a, C, chunk, s);
    if (need <= 2) return launch_kv<kSrc, 2>(a, C, chunk, s);
    if (need <= 4) return launch_kv<kSrc, 4>(a, C, chunk, s);
    return launch_kv<kSrc, kMaxVecPerThread>(a, C, chunk, s);
}

}  // namespace

int rmsnorm_max_h() { return kMaxCluster * kThreads * kMaxVecPerThread * 8; }

cudaError_t launch_rmsnorm_rows(const RmsNormArgs &a, cudaStream_t s) {
    if (a.rows <= 0) return cudaSuccess;
    return a.z ? launch_src<1>(a, s) : launch_src<0>(a, s);
}

}  // namespace symm
