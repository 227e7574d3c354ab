// Persistent stream-K fused GEMV + one-shot all-reduce: a TMA ring feeding
// either the tcgen05 tensor cores or (an option for B <= 2) CUDA-core FFMA,
// one CTA per SM.
//
// Work decomposition.  A unit is one (row tile t of 128 rows, rank r) pair,
// u = t * R + r (tile-major, so a tile's R contributors are neighbours); each
// unit is KB K-blocks of 64 * kSlabs columns of W_r.  The U * KB blocks form
// one sequence that is cut into G equal contiguous ranges, one per CTA:
// every CTA streams the same number of bytes, whatever N, R and K are, so no
// wave quantisation or tail imbalance remains.  A CTA's range crosses unit
// boundaries, and a unit may be shared by two or more CTAs: each maximal
// piece of a unit inside one CTA's range is a "part" with its own fp32
// partial, published like a contributor of the tile.  For unit u the parts
// are numbered by CTA, p = c - first_cta(u).
//
// Pipeline inside a CTA (192 threads):
//   warp 0      one lane walks the range and issues TMA loads of the W block
//               (128 rows x 64 * kSlabs, 128-byte swizzle) and of the x
//               block into a kStages ring;
//   warp 1      MMA engine: owns a 32-column TMEM allocation (two 16-column
//               accumulators, so the next part accumulates while the
//               previous one is drained) and one lane issues
//               tcgen05.mma.kind::f16 (M=128, N=16, K=16) per 16 columns;
//   warps 2-5   MMA engine: drain the accumulator with tcgen05.ld;
//               FFMA engine: each thread owns one row of the tile and
//               multiplies it with the x block straight from the swizzled
//               shared-memory stage.
//   Warps 2-5 then store the part's partial into rank r's scratch slot and
//   run the publish / last-arriver protocol of the tile (release flag,
//   acq_rel ticket; the last contributor sums all parts in rank order, then
//   part order, and stores bf16 into every rank's y), while warps 0-1 keep
//   streaming the next blocks.
//
// This follows the fused GEMV + AllReduce of "Overlapping Collective
// Communication with Dependent Computation ... GPU-Initiated Intra-Kernel
// Networking" (Abstract): partials are pushed as soon as a share of the
// computation is complete and the collective's reduction is overlapped with
// the streaming of the rest of W.
//
// Safety: every mbarrier wait is bounded (%globaltimer); timeouts latch a
// status code.  Decisions that steer named barriers are made uniform across
// warps 2-5 with bar.red.and, so a timeout can never leave a barrier short of
// threads; a CTA that gave up skips publishing, waits (bounded) for its
// copies and MMAs in flight, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "protocol.cuh"
#include "sm100.cuh"

namespace symm {

namespace {

constexpr int kM = 128;
constexpr int kNmma = 16;
constexpr int kSlabA = kM * 64 * 2;       // one 128-byte-swizzled slab of W: 16 KiB
constexpr int kSlabX = kNmma * 64 * 2;    // one slab of x: 2 KiB
constexpr int kThreads = 192;
constexpr int kGroupThreads = 128;        // warps 2-5
constexpr int kGroupBarrier = 1;
constexpr uint32_t kTmemCols = 32;
constexpr uint32_t kIdesc = mma_idesc_bf16_f32(kM, kNmma);

// Ring of one CTA when kCps CTAs share an SM's 228 KB of shared memory.
template <int kSlabs, int kCps>
struct Ring {
    static constexpr int kStageBytes = kSlabs * (kSlabA + kSlabX);
    static constexpr int kStages = ((216 * 1024) / kCps) / kStageBytes;
    static constexpr int kSmem = kStages * kStageBytes + 1024;
    static_assert(kStageBytes % 1024 == 0, "stages keep 1024-byte alignment");
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

// CTA whose range contains block g: the largest c with floor(total * c / G) <= g.
__device__ __forceinline__ int cta_of_block(long long g, long long total, int G) {
    return (int)(((g + 1) * (long long)G + total - 1) / total) - 1;
}

__device__ __forceinline__ int parts_of_unit(long long u, const SkGeom &geo) {
    return cta_of_block((u + 1) * geo.KB - 1, geo.total, geo.G) - cta_of_block(u * geo.KB, geo.total, geo.G) + 1;
}

// The reduction of tile t by its last contributor (flags acquired): the
// tile's parts in fixed order, run by the 128 threads of warps 2-5.
__device__ __forceinline__ void sk_reduce_tile(const GemvArgs &a, int t, int gt, const int *s_parts) {
    // Partials of the tile in fixed order (rank, then part): plain L2 loads
    // after the reducer's acquire of the flags.  Each thread owns up to kPer outputs and loads
    // all of them for one contributor before adding, so one L2 round trip
    // serves kPer outputs; contributions are added strictly in order.
    const int n0 = t * kM;
    const int rows = min(kM, a.N - n0);
    const int count = rows * a.B;
    constexpr int kPer = 16;
    for (int i0 = gt; i0 < count; i0 += kGroupThreads * kPer) {
        size_t off[kPer];
        float acc[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i = min(i0 + k * kGroupThreads, count - 1);
            const int b = i / rows;
            const int n = n0 + (i - b * rows);
            off[k] = ((size_t)b * a.N + n) * sizeof(float);
        }
        bool first = true;
        for (int q = 0; q < a.R; ++q)
            for (int qp = 0; qp < s_parts[q]; ++qp) {
                const uint8_t *base = a.scratch + (long long)q * a.stride + (long long)qp * a.partial_stride;
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const float v = __ldcg(reinterpret_cast<const float *>(base + off[k]));
                    acc[k] = first ? v : acc[k] + v;
                }
                first = false;
            }
#pragma unroll
        for (int k = 0; k < kPer; ++k)
            if (i0 + k * kGroupThreads < count) store_output(a, off[k] / sizeof(float), acc[k]);
    }
}

// Steps 2-4 of the protocol for one part (r, p) of tile t, run by the 128
// threads of warps 2-5 (gt = 0..127).  The caller has stored its partial;
// `epoch` (step 0) is needed in gt == 0 only, which publishes.
__device__ __forceinline__ void sk_publish_reduce(const GemvArgs &a, const SkGeom &geo, uint32_t epoch, int t,
                                                  int r, int p, int gt, int *s_last, int *s_bad, int *s_parts,
                                                  uint32_t *s_epoch) {
    uint32_t done = 0;   // gt == 0, reducer: tiles counted before this one
    __threadfence();
    named_barrier(kGroupBarrier, kGroupThreads);
    if (gt == 0) {
        int C = 0;
        for (int q = 0; q < a.R; ++q) {
            const int P = parts_of_unit((long long)t * a.R + q, geo);
            s_parts[q] = P;
            C += P;
        }
        uint32_t *flag = reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(a.flags) +
                                                      (long long)r * a.stride) + (size_t)t * geo.Pmax + p;
        st_release_gpu(flag, epoch);
        *s_last = take_ticket(a, t, (uint32_t)C, r, epoch, &done) == (uint32_t)C - 1u;
        *s_bad = 0;
        *s_epoch = epoch;
    }
    named_barrier(kGroupBarrier, kGroupThreads);
    if (!*s_last) return;
    const uint32_t e = *s_epoch;
    // The acquire loads of the flags (and the barrier after them) order the
    // partial loads of the reduction after every contributor's stores.
    for (int i = gt; i < a.R * geo.Pmax; i += kGroupThreads) {
        const int q = i / geo.Pmax;
        const int qp = i - q * geo.Pmax;
        if (qp < s_parts[q]) {
            const uint32_t *f = reinterpret_cast<const uint32_t *>(
                                    reinterpret_cast<const uint8_t *>(a.flags) + (long long)q * a.stride) +
                                (size_t)t * geo.Pmax + qp;
            if (ld_acquire_gpu(f) != e) {
                latch_status(a.status, kProtoStaleFlag, q, t, e);
                *s_bad = 1;
            }
        }
    }
    named_barrier(kGroupBarrier, kGroupThreads);
    if (gt == 0) finish_launch_if_last(a, done, e, t);
    if (!*s_bad) sk_reduce_tile(a, t, gt, s_parts);
}

// 8 bf16 of W (one 16-byte chunk) times 8 bf16 of x, fp32, ascending order.
__device__ __forceinline__ float dot8_bf16(const uint4 &w, const uint4 &x, float acc) {
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

// kEngine 0: tcgen05 MMA (any B <= 16); kEngine 1: CUDA-core FFMA with kB batch columns.
template <int kEngine, int kSlabs, int kB, int kCps>
__global__ void __launch_bounds__(kThreads, 1)
    gemv_ar_sk_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const GemvArgs a, const SkGeom geo) {
    chain_entry();
    using RingT = Ring<kSlabs, kCps>;
    static_assert(RingT::kStages >= 2, "the ring needs at least two stages");
    constexpr int kStages = RingT::kStages;
    constexpr int kStageBytes = RingT::kStageBytes;
    constexpr int kBK = 64 * kSlabs;

    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t acc_full[2];
    __shared__ __align__(8) uint64_t acc_empty[2];
    __shared__ __align__(8) uint64_t drain_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;
    __shared__ int s_last, s_bad;
    __shared__ uint32_t s_epoch;
    __shared__ int s_parts[kMaxRanks];

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c = a.reverse_order ? geo.G - 1 - (int)blockIdx.x : (int)blockIdx.x;
    const long long beg = geo.total * c / geo.G;
    const long long end = geo.total * (c + 1) / geo.G;
    const long long KB = geo.KB;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], kEngine == 0 ? 1 : 4);
        }
        for (int j = 0; j < 2; ++j) {
            mbar_init(&acc_full[j], 1);
            mbar_init(&acc_empty[j], 4);
        }
        mbar_init(&drain_bar, 1);
        abort_sh = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (kEngine == 0 && warp == 1) tmem_alloc(&tmem_base_sh, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = kEngine == 0 ? tmem_base_sh : 0u;

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
            int issued = 0;
            // (unit, K-block) of block g, advanced without divisions.
            const long long u0 = beg / KB;
            int kb = (int)(beg - u0 * KB);
            int t = (int)(u0 / a.R);
            int r = (int)(u0 - (long long)t * a.R);
            for (long long g = beg; g < end; ++g) {
                const int st = issued % kStages;
                const uint32_t ph = (uint32_t)(issued / kStages) & 1u;
                if (!mbar_wait(&empty_bar[st], ph ^ 1u, &abort_sh)) {
                    latch_status(a.status, kProtoTimeout, r, t, read_launch_epoch(a));
                    abort_sh = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full_bar[st], (uint32_t)kStageBytes);
                uint8_t *dst = smem + (size_t)st * kStageBytes;
#pragma unroll
                for (int s = 0; s < kSlabs; ++s)
                    tma_load_3d(dst + s * kSlabA, &tmW, &full_bar[st], kb * kBK + s * 64, t * kM, r);
#pragma unroll
                for (int s = 0; s < kSlabs; ++s)
                    tma_load_3d(dst + kSlabs * kSlabA + s * kSlabX, &tmX, &full_bar[st], kb * kBK + s * 64, 0, r);
                ++issued;
                if (++kb == geo.KB) {
                    kb = 0;
                    if (++r == a.R) {
                        r = 0;
                        ++t;
                    }
                }
            }
            if (abort_sh) {
                volatile int never = 0;
                for (int j = max(0, issued - kStages); j < issued; ++j)
                    mbar_wait(&full_bar[j % kStages], (uint32_t)(j / kStages) & 1u, &never);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issuer
        if constexpr (kEngine == 0) {
          if (lane == 0) {
            int i = 0, seg = 0;
            long long g = beg;
            bool ok = true;
            while (g < end && ok) {
                const long long u = g / KB;
                const long long seg_end = min(end, (u + 1) * KB);
                const int j = seg & 1;
                const uint32_t use = (uint32_t)(seg >> 1);
                ok = mbar_wait(&acc_empty[j], (use & 1u) ^ 1u, &abort_sh);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(j * kNmma);
                bool first = true;
                for (; g < seg_end; ++g, ++i) {
                    const int st = i % kStages;
                    const uint32_t ph = (uint32_t)(i / kStages) & 1u;
                    if (!mbar_wait(&full_bar[st], ph, &abort_sh)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_u32(smem + (size_t)st * kStageBytes);
                    const uint32_t x_addr = a_addr + kSlabs * kSlabA;
#pragma unroll
                    for (int s = 0; s < kSlabs; ++s)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma(d, smem_desc_sw128(a_addr + s * kSlabA + kk * 32),
                                   smem_desc_sw128(x_addr + s * kSlabX + kk * 32), kIdesc,
                                   (first && s == 0 && kk == 0) ? 0u : 1u);
                    first = false;
                    tc_commit(&empty_bar[st]);
                }
                if (!ok) break;
                tc_commit(&acc_full[j]);
                ++seg;
            }
            if (!ok) {
                latch_status(a.status, kProtoTimeout, -1, -1, read_launch_epoch(a));
                abort_sh = 1;
            }
            // Every MMA issued by this thread has finished once this commit arrives.
            tc_commit(&drain_bar);
            volatile int never = 0;
            mbar_wait(&drain_bar, 0, &never);
          }
        }
    } else {
        // ------------------------------------- drain / FFMA (warps 2-5)
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const int gt = threadIdx.x - 64;
        // gt == 0 publishes; its read of the launch epoch overlaps the streaming.
        const uint32_t epoch = gt == 0 ? read_launch_epoch(a) : 0u;
        int i = 0, seg = 0;
        long long g = beg;
        while (g < end) {
            const long long u = g / KB;
            const long long seg_end = min(end, (u + 1) * KB);
            const int t = (int)(u / a.R);
            const int r = (int)(u - (long long)t * a.R);
            float v[kEngine == 0 ? kNmma : kB];
            bool ok = true;
            if constexpr (kEngine == 0) {
                const int j = seg & 1;
                const uint32_t use = (uint32_t)(seg >> 1);
                ok = mbar_wait_sleepy(&acc_full[j], use & 1u, &abort_sh);
                ok = group_all(ok);
                if (!ok) break;
                tc_fence_after();
                tmem_ld_16(tmem + (uint32_t)(j * kNmma) + ((uint32_t)(q4 * 32) << 16), v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[j]);
                g = seg_end;
            } else {
                float acc0[kB], acc1[kB];
#pragma unroll
                for (int b = 0; b < kB; ++b) acc0[b] = acc1[b] = 0.f;
                for (; g < seg_end; ++g, ++i) {
                    const int st = i % kStages;
                    const uint32_t ph = (uint32_t)(i / kStages) & 1u;
                    if (ok) ok = mbar_wait(&full_bar[st], ph, &abort_sh);
                    const uint8_t *A = smem + (size_t)st * kStageBytes;
                    const uint8_t *X = A + kSlabs * kSlabA;
#pragma unroll
                    for (int s = 0; s < kSlabs; ++s)
#pragma unroll
                        for (int jj = 0; jj < 8; jj += 2) {
                            const uint4 w0 = *reinterpret_cast<const uint4 *>(A + s * kSlabA + row * 128 +
                                                                              ((jj ^ (row & 7)) << 4));
                            const uint4 w1 = *reinterpret_cast<const uint4 *>(A + s * kSlabA + row * 128 +
                                                                              (((jj + 1) ^ (row & 7)) << 4));
#pragma unroll
                            for (int b = 0; b < kB; ++b) {
                                const uint4 x0 = *reinterpret_cast<const uint4 *>(X + s * kSlabX + b * 128 +
                                                                                  ((jj ^ (b & 7)) << 4));
                                const uint4 x1 = *reinterpret_cast<const uint4 *>(X + s * kSlabX + b * 128 +
                                                                                  (((jj + 1) ^ (b & 7)) << 4));
                                acc0[b] = dot8_bf16(w0, x0, acc0[b]);
                                acc1[b] = dot8_bf16(w1, x1, acc1[b]);
                            }
                        }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty_bar[st]);
                }
                ok = group_all(ok);
                if (!ok) break;
#pragma unroll
                for (int b = 0; b < kB; ++b) v[b] = acc0[b] + acc1[b];
            }
            const int p = c - cta_of_block(u * KB, geo.total, geo.G);
            const int n = t * kM + row;
            if (n < a.N) {
                float *P = reinterpret_cast<float *>(a.scratch + (long long)r * a.stride +
                                                     (long long)p * a.partial_stride);
#pragma unroll
                for (int b = 0; b < (kEngine == 0 ? kNmma : kB); ++b)
                    if (b < a.B) P[(size_t)b * a.N + n] = v[b];
            }
            sk_publish_reduce(a, geo, epoch, t, r, p, gt, &s_last, &s_bad, s_parts, &s_epoch);
            ++seg;
        }
        if (g < end) {
            latch_status(a.status, kProtoTimeout, -1, -1, read_launch_epoch(a));
            abort_sh = 1;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (kEngine == 0 && warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int kEngine, int kSlabs, int kB, int kCps>
cudaError_t launch_cfg(const GemvArgs &a, const SkGeom &geo, const CUtensorMap *m, cudaStream_t s) {
    auto kern = gemv_ar_sk_kernel<kEngine, kSlabs, kB, kCps>;
    constexpr int smem = Ring<kSlabs, kCps>::kSmem;
    // The shared-memory attribute is per device: set it once for each device
    // a launch happens on (devices past 63 set it every time).
    static unsigned long long attr_devices = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 64;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit == 0 || !(attr_devices & bit)) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        attr_devices |= bit;
    }
    return launch_kernel(kern, dim3((unsigned)geo.G), dim3(kThreads), (size_t)smem, s, a.chained != 0, m[0], m[1], a,
                         geo);
}

}  // namespace

int sk_block_k(int slabs) { return 64 * slabs; }

// Pipeline shapes that are instantiated: (slabs, CTAs per SM) with a ring of
// at least two stages.
bool sk_config_supported(int slabs, int cps) {
    return (cps == 1 && (slabs == 1 || slabs == 2 || slabs == 4)) ||
           (cps == 2 && (slabs == 1 || slabs == 2 || slabs == 3)) || (cps == 3 && slabs == 1);
}

template <int kEngine, int kB>
cudaError_t launch_engine(const GemvArgs &a, const SkGeom &geo, const CUtensorMap *m, int slabs, int cps,
                          cudaStream_t s) {
    switch (cps * 10 + slabs) {
        case 11: return launch_cfg<kEngine, 1, kB, 1>(a, geo, m, s);
        case 12: return launch_cfg<kEngine, 2, kB, 1>(a, geo, m, s);
        case 14: return launch_cfg<kEngine, 4, kB, 1>(a, geo, m, s);
        case 21: return launch_cfg<kEngine, 1, kB, 2>(a, geo, m, s);
        case 22: return launch_cfg<kEngine, 2, kB, 2>(a, geo, m, s);
        case 23: return launch_cfg<kEngine, 3, kB, 2>(a, geo, m, s);
        case 31: return launch_cfg<kEngine, 1, kB, 3>(a, geo, m, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv_sk(const GemvArgs &a, const SkGeom &geo, const void *maps, int engine, int slabs, int cps,
                           cudaStream_t s) {
    const CUtensorMap *m = static_cast<const CUtensorMap *>(maps);
    if (engine == 0) return launch_engine<0, 0>(a, geo, m, slabs, cps, s);
    if (a.B == 1) return launch_engine<1, 1>(a, geo, m, slabs, cps, s);
    if (a.B == 2) return launch_engine<1, 2>(a, geo, m, slabs, cps, s);
    return cudaErrorInvalidValue;
}

}  // namespace symm
